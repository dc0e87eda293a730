"""Decode benchmark: the 32-layer Qwen3.5-4B-shape stack at batch 1.

Workload (default): layer i is full attention when i % 4 == 3, else Gated
DeltaNet; int8 group-64 synthetic weights (3.79 GB, larger than L2, so every
step streams them from HBM); bf16 KV caches prefilled to 8192 tokens; GDN
states N(0, 0.1); conv states zero. One step = one token through all 32 layers,
replayed as one CUDA graph (qwen35_graph_*); the graph advances the device
position, so the context grows by one token per step.

Prints one JSON line. --impl reference times the CPU oracle on the same
workload instead (bounded sample per step; see cpu_sample).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s (32-layer 4B-shape stack, batch 1); achieved HBM GB/s vs peak"
PREFILL = 8192
SEED = 0


KERNEL_SOURCES = ["full_attention_decode_gb300/csrc/decode_kernel.cuh", "full_attention_decode_gb300/csrc/decode.cu",
                  "full_attention_decode_gb300/csrc/decode_d64.cu", "full_attention_decode_gb300/csrc/decode_d128.cu",
                  "full_attention_decode_gb300/csrc/decode_d256.cu", "full_attention_decode_gb300/csrc/decode.h",
                  "full_attention_decode_gb300/csrc/common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_kernel_stack_dram_traffic.txt")


def kernel_sha() -> str:
    """sha256 over the decode kernel's sources without comments and blank lines
    (ties a profile to the code it measured, not to its commentary)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f)) as fh:
            for line in fh:
                if '"' not in line:
                    line = re.sub(r"//.*$", "", line)
                line = line.strip()
                if line:
                    h.update(line.encode() + b"\n")
    return h.hexdigest()


def profiled_traffic(step_bytes: int):
    """DRAM bytes (read + write) per launch of the decode kernel from the committed
    ncu capture, scaled from the captured stack to this launch by algorithmic bytes
    (traffic grows with the layers streamed); None when the kernel's sources have
    changed since the capture or no capture is committed."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if "=" in line and not line.lstrip().startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sources_sha256") != kernel_sha():
            return None, "stale: the kernel changed since the capture"
        dram = float(kv["dram_bytes_per_launch"])
        alg = float(kv["algorithmic_bytes_per_launch"])
        return int(round(dram * step_bytes / alg)), f"scaled from the {kv.get('captured')} capture ({dram / alg:.4f} x algorithmic)"
    except Exception:
        return None, "no capture committed"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def algorithmic_bytes(cfg: dict, seq_len: int, kinds: list | None = None, kv_dtype: str = "bf16") -> dict:
    """Bytes a decode step must move: every weight, scale and bias once, K/V rows
    [0, seq_len) once per full-attention layer plus the appended row, GDN and conv
    state read and written once, norm vectors and the small per-head vectors."""
    from full_attention_decode_gb300 import synth
    E, I, H, Hkv, D = cfg["hidden"], cfg["intermediate"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    Hk, Hv, Dk, Dv, Kc = (cfg["num_k_heads_lin"], cfg["num_v_heads_lin"], cfg["k_head_dim_lin"],
                          cfg["v_head_dim_lin"], cfg["conv_kernel_size"])
    C = 2 * Hk * Dk + Hv * Dv

    def q(n, k):
        return n * k + 2 * n * (k // 64) * 2  # codes + bf16 scale + bf16 bias per group

    mlp = q(I, E) * 2 + q(E, I)
    fa_w = q(2 * H * D, E) + 2 * q(Hkv * D, E) + q(E, H * D) + mlp + 2 * (2 * E + 2 * D)
    gdn_w = q(Hv, E) * 2 + q(C, E) + q(Hv * Dv, E) + q(E, Hv * Dv) + mlp + 2 * (2 * E + Dv) + \
        Hv * (4 + 2) + C * Kc * 2
    gdn_state = 2 * (Hv * Dk * Dv * 4 + C * Kc * 4)
    # per token and kv-head: bf16 rows, or Turbo8 codes plus one bf16 scale per 16
    row = D * 2 if kv_dtype == "bf16" else D + D // 8
    kv = lambda S: 2 * S * Hkv * row + 2 * Hkv * row  # noqa: E731
    kinds = kinds if kinds is not None else synth.layer_kinds(cfg)
    n_fa = kinds.count("fa")
    n_gdn = kinds.count("gdn")
    weights = n_fa * fa_w + n_gdn * gdn_w
    return {"weights": weights, "gemv_weights": n_fa * (q(2 * H * D, E) + 2 * q(Hkv * D, E) + q(E, H * D) + mlp)
            + n_gdn * (q(Hv, E) * 2 + q(C, E) + q(Hv * Dv, E) + q(E, Hv * Dv) + mlp),
            "step": weights + n_gdn * gdn_state + n_fa * kv(seq_len), "fa_layer_w": fa_w, "gdn_layer_w": gdn_w,
            "gdn_state": gdn_state, "gdn_state_all": n_gdn * gdn_state}


# ---------------------------------------------------------------------- clocks


class Clocks:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.rows.append(f)

    def summary(self) -> dict:
        if not getattr(self, "rows", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(sm)}


# ---------------------------------------------------------------------- the job across ranks


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest of the ranks' values: the job takes as long as its slowest rank.
    `dist` is torch.distributed (or None for one process); `device` the device a
    rank's collectives use (cuda under NCCL, cpu under gloo)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tok_s(ms_per_step: float, world: int, batch: int) -> float:
    """Whole-job decode throughput: every rank decodes `batch` sequences of its own
    (independent replicas), one token each per step."""
    return 1000.0 / ms_per_step * world * batch


def replica_seed(rank: int) -> int:
    """Each replica decodes its own synthetic sequences."""
    return SEED + rank


# ---------------------------------------------------------------------- GPU arm


def run_gpu(args) -> dict | None:
    import numpy as np
    import torch

    from full_attention_decode_gb300 import binding as B
    from full_attention_decode_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    B.qwen35_init()

    cfg = synth.config("4b")
    kinds = synth.layer_kinds(cfg)[:args.layers]
    cfg = dict(cfg, num_layers=len(kinds))
    c = B.make_config(cfg)
    nb = args.batch
    seed = replica_seed(rank)
    if nb > 1:  # each sequence at its own position, U{1024..65536}, seeded
        positions = [int(p) for p in np.random.default_rng([seed, 4242]).integers(1024, 65537, size=nb)]
    else:
        positions = [args.prefill]
    grow = args.warmup + args.steps + 2 * (args.steps + 4) + 8
    cap = max(positions) + grow
    t0 = time.time()
    dev_layers, caches, entries = [], [], []
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    device_fill = nb > 1 or args.prefill != PREFILL  # large caches: filled on the device (seeded)
    t8 = args.kv == "turbo8"
    for i, kind in enumerate(kinds):
        if kind == "fa":
            dl = B.DeviceFaLayer(synth.fa_layer(seed, i, cfg))
            if t8:  # Turbo8 caches filled on the device: finite E4M3 codes, scales of N(0, 1) groups
                Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
                cc = B.DeviceKvBatch.__new__(B.DeviceKvBatch)
                codes = []
                for _ in range(2):
                    c8 = torch.randint(0, 254, (nb, cap, Hkv, D), generator=gen, device="cuda", dtype=torch.int16)
                    codes.append(torch.where(c8 >= 0x7F, c8 + 1, c8).to(torch.uint8))
                ss = B.turbo8_sstride(cfg)
                scl = [(torch.rand((nb, cap, ss), generator=gen, device="cuda") + 0.5) * (2.0 / 448.0) for _ in range(2)]
                cc.k, cc.v = codes
                cc.ks, cc.vs = [x.to(torch.bfloat16).view(torch.int16) for x in scl]
                cc.struct = B.qwen35_kv_cache(cc.k.data_ptr(), cc.v.data_ptr(), cap, B.QWEN35_KV_TURBO8,
                                              cc.ks.data_ptr(), cc.vs.data_ptr())
            elif args.paged:  # one pool of 16-token blocks placed by a shuffled table, filled on the device
                bt = 16
                nbl = nb * ((cap + bt - 1) // bt)
                shape = (nbl, bt, cfg["num_kv_heads"], cfg["head_dim"])
                cc = B.DeviceKvBatch.__new__(B.DeviceKvBatch)
                cc.k = torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16).view(torch.int16)
                cc.v = torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16).view(torch.int16)
                cc.table = torch.randperm(nbl, generator=gen, device="cuda").to(torch.int32)
                cc.struct = B.qwen35_kv_cache(cc.k.data_ptr(), cc.v.data_ptr(), nbl // nb * bt, B.QWEN35_KV_BF16,
                                              None, None, cc.table.data_ptr(), bt, 0)
            elif device_fill:
                shape = (nb, cap, cfg["num_kv_heads"], cfg["head_dim"])
                cc = B.DeviceKvBatch.__new__(B.DeviceKvBatch)
                cc.k = torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16).view(torch.int16)
                cc.v = torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16).view(torch.int16)
                cc.struct = B.qwen35_kv_cache(cc.k.data_ptr(), cc.v.data_ptr(), cap)
            else:
                kb, vb = synth.kv_cache(seed, i, cfg, cap, PREFILL)
                cc = B.DeviceKv(kb, vb)
        else:
            dl = B.DeviceGdnLayer(synth.gdn_layer(seed, i, cfg))
            if nb > 1:
                conv, ssm = synth.gdn_state(seed, i, cfg, std=0.1)
                cc = B.DeviceStateBatch([conv] * nb, [ssm] * nb)
            else:
                conv, ssm = synth.gdn_state(seed, i, cfg, std=0.1)
                cc = B.DeviceState(conv, ssm)
        dev_layers.append(dl)
        caches.append(cc)
        entries.append(B.stack_layer(kind, dl, cc))
    setup_s = time.time() - t0

    stream = torch.cuda.Stream()
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb), stream=stream)
    x_in = torch.empty(nb * cfg["hidden"], dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    d_pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        x_in.copy_(B.to_device(np.concatenate([synth.x_in(seed + 97 * b, 0, cfg) for b in range(nb)])))
    stream.synchronize()
    with torch.cuda.stream(stream):
        graph = B.Graph(c, entries, scratch, x_in, x_out, d_pos, cap, batch=nb)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timing: K graph replays
    for _ in range(args.warmup):
        graph.launch(stream)
    barrier()
    pos0 = positions[0] + args.warmup
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            graph.launch(stream)
        ev1.record(stream)
        stream.synchronize()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, dist, "cuda")
    status = B.qwen35_read_device_status(scratch, stream)
    if args.stack_only:  # profiling runs: the graph replays alone
        graph.close()
        return {"ms_per_step": ms, "status": status, "layers": len(kinds)} if rank == 0 else None

    # ---- end to end through the C ABI with host buffers: H2D of the step's
    # input vector, the graph, D2H of its output, every step
    h_in = torch.empty_like(x_in, device="cpu").pin_memory()
    h_out = torch.empty_like(x_out, device="cpu").pin_memory()
    h_in.copy_(torch.from_numpy(np.concatenate([synth.x_in(seed + 97 * b, 1, cfg) for b in range(nb)]).view(np.int16)))
    barrier()
    t_e0 = time.perf_counter()
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            x_in.copy_(h_in, non_blocking=True)
            graph.launch(stream)
            h_out.copy_(x_out, non_blocking=True)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t_e0) * 1e3 / args.steps
    barrier()
    e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")

    # ---- the quantised GEMV phase alone (the same kernel on a one-GEMV program):
    # every layer's gate_proj (9216 x 2560, 25.1 MB) back to back, 32 distinct
    # matrices, so nothing is served from L2
    mats = [dl.m["gate_proj"] for dl in dev_layers]
    xv = torch.zeros(cfg["hidden"], dtype=torch.int16, device="cuda")
    yv = torch.empty(cfg["intermediate"], dtype=torch.int16, device="cuda")
    gs = B.new_scratch(4096, stream=stream)
    cw = [m.c() for m in mats]
    reps = 4
    with torch.cuda.stream(stream):
        for w in cw:
            B.qwen35_gemv(w, xv, yv, gs, stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            for w in cw:
                assert B.qwen35_gemv(w, xv, yv, gs, stream) == 0
        e1.record(stream)
    stream.synchronize()
    gemv_ms = e0.elapsed_time(e1) / (reps * len(cw))
    m0 = mats[0]
    gemv_bytes = m0.n * m0.k + 2 * m0.n * (m0.k // 64) * 2

    # ---- the output head after the stack: final norm + lm_head GEMV over the full
    # vocabulary + greedy token (qwen35_lm_head_greedy), back to back
    head = synth.head(seed, cfg)
    vocab, E = cfg["vocab"], cfg["hidden"]
    h_nw = B.to_device(head["final_norm"])
    h_w = B.DeviceQWeight(head["lm_head"])
    h_logits = torch.empty(vocab, dtype=torch.int16, device="cuda")
    h_tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    h_scr = B.new_scratch(4096, stream=stream)
    h_x = x_out[:E]
    with torch.cuda.stream(stream):
        for _ in range(3):
            assert B.qwen35_lm_head_greedy(c, h_nw, h_w.c(), h_x, h_logits, h_tok, h_scr, stream) == 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            assert B.qwen35_lm_head_greedy(c, h_nw, h_w.c(), h_x, h_logits, h_tok, h_scr, stream) == 0
        e1.record(stream)
    stream.synchronize()
    head_ms = e0.elapsed_time(e1) / 10
    head_bytes = vocab * E + 2 * vocab * (E // 64) * 2 + E * 2
    head_status = B.qwen35_read_device_status(h_scr, stream)
    del h_w
    graph.close()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    peak, peak_kind = _peaks()
    mid = args.warmup + args.steps // 2 + 1  # tokens each sequence gained by mid-run
    per_seq = [algorithmic_bytes(cfg, p + mid, kinds, args.kv) for p in positions]
    kv_seq = [a["step"] - a["weights"] - a["gdn_state_all"] for a in per_seq]
    ab = dict(per_seq[0])
    ab["step"] = per_seq[0]["weights"] + sum(kv_seq) + nb * per_seq[0]["gdn_state_all"]
    seq_mid = positions[0] + mid
    traffic, traffic_note = profiled_traffic(ab["step"]) if nb == 1 and args.prefill == PREFILL and not t8 \
        and not args.paged \
        else (None, "not captured")
    tok_s = job_tok_s(ms, world, nb)
    step_gbs = ab["step"] / (ms * 1e-3) / 1e9
    gemv_gbs = gemv_bytes / (gemv_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(tok_s, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8-weight/bf16-act/fp32-acc", "data": "synthetic",
        "config": {"workload": ("qwen3.5-4b-shape 32-layer decode stack, batch 1, KV prefilled to 8192" if nb == 1
                                and args.prefill == PREFILL and not t8 and not args.paged else
                                f"qwen3.5-4b-shape 32-layer decode stack, batch {nb}, KV prefilled to {positions}"
                                + (", Turbo8 KV cache" if t8 else "") + (", paged KV (16-token blocks)"
                                                                          if args.paged else "")),
                   "kv_dtype": args.kv, "paged": bool(args.paged),
                   "batch": nb, "positions": positions,
                   "layers": "24 gated-deltanet + 8 full-attention (i % 4 == 3)",
                   "context": [pos0 + 1, pos0 + args.steps], "global_batch": world, "seq_len": seq_mid,
                   "parallelism": f"replicas x{world}" if world > 1 else "single gpu",
                   "l2": "inputs larger than L2: 3.79 GB of weights streamed per step",
                   "graph": "one CUDA graph per step (a memset of the scratch's tagged words + one decode_kernel launch)",
                   "seed": SEED, "bytes_per_step": ab["step"], "peak_gbs": peak,
                   "frac_step_of_8000": round(step_gbs / 8000.0, 4),
                   "gemv_phase_alone": {"matrix": "9216x2560", "bytes": gemv_bytes,
                                        "us": round(gemv_ms * 1e3, 2), "gbs": round(gemv_gbs, 1)},
                   "lm_head_greedy": {"vocab": vocab, "bytes": head_bytes, "us": round(head_ms * 1e3, 2),
                                      "gbs": round(head_bytes / (head_ms * 1e-3) / 1e9, 1),
                                      "frac_of_peak": round(head_bytes / (head_ms * 1e-3) / 1e9 / peak, 4),
                                      "tok_s_stack_plus_head": round(1000.0 / (ms + head_ms) * world * nb, 2)
                                      if nb == 1 else None,
                                      "device_status": head_status},
                   "device_status": status, "setup_s": round(setup_s, 1)},
        "roofline": {"bound": "hbm", "achieved": round(step_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(step_gbs / peak, 4), "traffic": traffic, "traffic_source": traffic_note,
                     "kernel": "decode_kernel (one launch = the whole 32-layer step)",
                     "bytes_per_launch": ab["step"], "us_per_launch": round(ms * 1e3, 2),
                     "peak_kind": peak_kind},
        "e2e": {"value": round(job_tok_s(e2e_ms, world, nb), 2), "unit": "tok/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": nb * cfg["hidden"] * 2, "d2h_bytes_per_step": nb * cfg["hidden"] * 2},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    if dist is not None:
        dist.destroy_process_group()
    return res


# ---------------------------------------------------------------------- prompt prefill


def prefill_flops(cfg: dict, T: int, kinds: list) -> dict:
    """Tensor-core FLOPs of one prefill of T tokens from position 0: 2 T N K per
    projection, plus the causal attention's 4 D per (token, head, key) (keys 0..t)."""
    E, I, H, Hkv, D = cfg["hidden"], cfg["intermediate"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    Hk, Hv, Dk, Dv = cfg["num_k_heads_lin"], cfg["num_v_heads_lin"], cfg["k_head_dim_lin"], cfg["v_head_dim_lin"]
    C = 2 * Hk * Dk + Hv * Dv
    mlp = 3 * E * I
    fa = 2 * H * D * E + 2 * Hkv * D * E + H * D * E + mlp
    gdn = 2 * Hv * E + C * E + Hv * Dv * E + Hv * Dv * E + mlp
    gemm = 2 * T * (kinds.count("fa") * fa + kinds.count("gdn") * gdn)
    attn = kinds.count("fa") * 4 * D * H * T * (T + 1) // 2
    return {"gemm": gemm, "attention": attn, "gate_proj_one": 2 * T * I * E}


def prefill_launches(cfg: dict, T: int, kinds: list) -> int:
    """Kernel launches of one prefill step: 12 per full-attention and 16 per
    linear-attention layer, plus the split-K sum after each projection whose
    128-row x 256-token tiles would leave more than half of the 152 SMs idle (the
    rule of the library's prefill GEMM)."""
    E, I, H, Hkv, D = cfg["hidden"], cfg["intermediate"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    Hk, Hv, Dk, Dv = cfg["num_k_heads_lin"], cfg["num_v_heads_lin"], cfg["k_head_dim_lin"], cfg["v_head_dim_lin"]
    C = 2 * Hk * Dk + Hv * Dv

    def split(n, k):
        tiles = -(-n // 128) * -(-T // 256)
        return 1 if tiles * 2 <= 152 and min(152 // tiles, 8, k // 64) >= 2 else 0

    mlp = 2 * split(I, E) + split(E, I)
    fa = 12 + split(2 * H * D, E) + 2 * split(Hkv * D, E) + split(E, H * D) + mlp
    gdn = 16 + 2 * split(Hv, E) + split(C, E) + split(Hv * Dv, E) + split(E, Hv * Dv) + mlp
    return kinds.count("fa") * fa + kinds.count("gdn") * gdn


def run_prompt(args) -> dict | None:
    """The multi-token prefill of a T-token prompt through the 32-layer stack from
    position 0 (qwen35_prefill_step): one step = the whole prompt through every
    layer; K steps timed after W warm-up steps (each rewrites the same cache rows;
    the linear-attention states keep advancing)."""
    import numpy as np
    import torch

    from full_attention_decode_gb300 import binding as B
    from full_attention_decode_gb300 import synth

    rank = int(os.environ.get("RANK", "0"))
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    B.qwen35_init()
    cfg = synth.config("4b")
    kinds = synth.layer_kinds(cfg)[:args.layers]
    cfg = dict(cfg, num_layers=len(kinds))
    c = B.make_config(cfg)
    T, E = args.prompt, cfg["hidden"]
    seed = replica_seed(rank)
    t0 = time.time()
    dev_layers, caches, entries = [], [], []
    for i, kind in enumerate(kinds):
        if kind == "fa":
            dl = B.DeviceFaLayer(synth.fa_layer(seed, i, cfg))
            kb, vb = synth.kv_cache(seed, i, cfg, T, 0)
            cc = B.DeviceKv(kb, vb)
        else:
            dl = B.DeviceGdnLayer(synth.gdn_layer(seed, i, cfg))
            conv, ssm = synth.gdn_state(seed, i, cfg, std=0.1)
            cc = B.DeviceState(conv, ssm)
        dev_layers.append(dl)
        caches.append(cc)
        entries.append(B.stack_layer(kind, dl, cc))
    setup_s = time.time() - t0
    stream = torch.cuda.Stream()
    scratch = B.new_scratch(B.qwen35_prefill_scratch_bytes(c, T), stream=stream)
    X = np.stack([synth.x_in(seed, 5000 + t, cfg) for t in range(T)])
    x_in = B.to_device(X)
    x_out = torch.empty_like(x_in)
    torch.cuda.synchronize()

    def step():
        assert B.qwen35_prefill_step(c, entries, scratch, x_in, x_out, 0, T, stream) == 0

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    # the same step enqueued call by call (eager), then as one CUDA graph (the timed value)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
    stream.synchronize()
    eager_ms = ev0.elapsed_time(ev1) / args.steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        step()
    with torch.cuda.stream(stream):
        for _ in range(2):
            graph.replay()
    stream.synchronize()
    with Clocks(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            ev1.record(stream)
        stream.synchronize()
    ms = ev0.elapsed_time(ev1) / args.steps
    status = B.qwen35_read_device_status(scratch, stream)

    # end to end: the prompt from pinned host memory, the outputs back, every step
    h_in = torch.from_numpy(X.view(np.int16)).pin_memory()
    h_out = torch.empty_like(x_out, device="cpu").pin_memory()
    torch.cuda.synchronize()
    t_e0 = time.perf_counter()
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            x_in.copy_(h_in, non_blocking=True)
            graph.replay()
            h_out.copy_(x_out, non_blocking=True)
        stream.synchronize()
    e2e_ms = (time.perf_counter() - t_e0) * 1e3 / args.steps
    del graph

    # the projection alone: every layer's gate_proj (9216 x 2560) over the T tokens
    gs = B.new_scratch(4096, stream=stream)
    xs = torch.zeros((T, E), dtype=torch.int16, device="cuda")
    ys = torch.empty((T, cfg["intermediate"]), dtype=torch.int16, device="cuda")
    cw = [dl.m["gate_proj"].c() for dl in dev_layers]
    gemm_ms = {}
    for exact in (False, True):
        with torch.cuda.stream(stream):
            for w in cw:
                assert B.qwen35_prefill_gemm(w, xs, ys, T, gs, stream, exact) == 0
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            reps = 4
            for _ in range(reps):
                for w in cw:
                    assert B.qwen35_prefill_gemm(w, xs, ys, T, gs, stream, exact) == 0
            e1.record(stream)
        stream.synchronize()
        gemm_ms[exact] = e0.elapsed_time(e1) / (reps * len(cw))
    if rank != 0:
        return None
    fl = prefill_flops(cfg, T, kinds)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        peak_burst, peak_sus, peak_kind = float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), "measured"
    except Exception:
        peak_burst, peak_sus, peak_kind = 1900.0, 1700.0, "fallback"
    step_tf = fl["gemm"] / (ms * 1e-3) / 1e12
    gemm_tf = fl["gate_proj_one"] / (gemm_ms[False] * 1e-3) / 1e12
    gemm_tf_x = fl["gate_proj_one"] / (gemm_ms[True] * 1e-3) / 1e12
    return {
        "metric": "prefill tok/s (32-layer 4B-shape stack, one prompt from position 0); tensor TFLOP/s vs peak",
        "value": round(T / (ms * 1e-3), 1), "unit": "tok/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16-dequantised-weight/bf16-act/fp32-acc", "data": "synthetic",
        "config": {"workload": f"qwen3.5-4b-shape 32-layer prefill of a {T}-token prompt from position 0",
                   "prompt_tokens": T, "layers": "24 gated-deltanet + 8 full-attention (i % 4 == 3)",
                   "graph": "one CUDA graph per prompt (the qwen35_prefill_step launches captured once)",
                   "eager_ms_per_step": round(eager_ms, 4),
                   "l2": "inputs larger than L2: 3.79 GB of weights per step",
                   "flops_per_step": fl, "device_status": status, "setup_s": round(setup_s, 1),
                   "gemm_alone": {"matrix": "9216x2560", "tokens": T, "us": round(gemm_ms[False] * 1e3, 2),
                                  "tflops": round(gemm_tf, 1), "frac_of_burst_peak": round(gemm_tf / peak_burst, 4),
                                  "exact_us": round(gemm_ms[True] * 1e3, 2),
                                  "exact_tflops": round(gemm_tf_x, 1),
                                  "exact_note": "hi + lo bf16 weights: two MMAs per weight; the tensor work is "
                                                "twice the useful FLOPs counted here"}},
        "roofline": {"bound": "tensor", "achieved": round(gemm_tf, 1), "peak": peak_burst, "unit": "TFLOP/s",
                     "frac": round(gemm_tf / peak_burst, 4), "traffic": None,
                     "kernel": f"gemm_kernel alone: the 9216x2560 gate_proj over the {T}-token prompt (bf16 "
                               "weights), 2 T N K FLOPs per launch over its CUDA-event time",
                     "peak_kind": peak_kind + " (burst bf16)",
                     "step_tflops": round(step_tf, 1), "step_frac_of_sustained": round(step_tf / peak_sus, 4)},
        "e2e": {"value": round(T / (e2e_ms * 1e-3), 1), "unit": "tok/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": T * E * 2, "d2h_bytes_per_step": T * E * 2},
        "gpu_launches": args.steps * prefill_launches(cfg, T, kinds),
        "clocks": clk.summary(),
    }


# ---------------------------------------------------------------------- CPU oracle


def cpu_sample(n_steps: int, threads: int) -> dict:
    """Time the oracle as it stands on a bounded sample of the workload.

    The sample is the first four layers of the stack (three Gated DeltaNet layers
    and the first full-attention layer at 8192 tokens of context), cycled one
    layer per sample step; tok/s = 1 / (32 x mean layer time). Each layer's
    matrices are dequantised once before the timed region (the oracle caches them
    per layer; that one-time cost is reported apart as dequant_ms). `threads`:
    the BLAS threads the caller pinned before numpy loaded (the oracle's matrix
    products are its only multi-threaded part).
    """
    import numpy as np

    from full_attention_decode_gb300 import synth
    from oracle import qwen35_oracle as O
    cfg = synth.config("4b")
    kinds = synth.layer_kinds(cfg)[:4]
    layers, caches = [], []
    for i, kind in enumerate(kinds):
        if kind == "fa":
            layers.append(synth.fa_layer(SEED, i, cfg))
            kb, vb = synth.kv_cache(SEED, i, cfg, PREFILL + n_steps + 8, PREFILL)
            caches.append(O.kv_from_bits(kb, vb))
        else:
            layers.append(synth.gdn_layer(SEED, i, cfg))
            conv, ssm = synth.gdn_state(SEED, i, cfg, std=0.1)
            caches.append(O.state_from_arrays(conv, ssm))
    t0 = time.perf_counter()
    for lay in layers:  # the oracle's per-layer dequantisation, once, untimed
        for name, v in list(lay.items()):
            if isinstance(v, dict) and "codes" in v:
                O._W(lay, name)
    dequant_s = time.perf_counter() - t0
    x = O.bf16_to_f64(synth.x_in(SEED, 0, cfg))
    times = []
    pos = PREFILL
    for s in range(n_steps):
        i = s % 4
        t0 = time.perf_counter()
        if kinds[i] == "fa":
            x = O.forward_full_attention(cfg, layers[i], caches[i], x, pos, pos + 1)
            pos += 1
        else:
            x = O.forward_linear_attention(cfg, layers[i], caches[i], x)
        times.append(time.perf_counter() - t0)
    mean = float(np.mean(times))
    return {"value": 1.0 / (32 * mean), "unit": "tok/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_steps} single-layer forwards cycling the stack's first 4 layers "
                      f"(3 GDN + 1 FA at 8192 context), float64 numpy, {threads} BLAS thread(s); "
                      f"tok/s = 1/(32 x mean layer time); mean {mean * 1e3:.1f} ms/layer; each layer's "
                      f"dequantisation done once before the timed region",
            "layer_ms": round(mean * 1e3, 2), "dequant_ms_per_layer": round(dequant_s * 1e3 / len(layers), 1),
            "host_cores": os.cpu_count()}


def cpu_sample_subprocess(n_steps: int, threads: int = 1) -> dict | None:
    t = str(threads)
    env = dict(os.environ, OPENBLAS_NUM_THREADS=t, OMP_NUM_THREADS=t, MKL_NUM_THREADS=t,
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample", str(n_steps),
                            "--cpu-threads", t], env=env, capture_output=True, text=True, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not fatal
        return {"value": None, "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": f"failed: {e}"}


def cpu_baseline(n_steps: int) -> dict:
    """The oracle on all host cores, with the single-threaded figure beside it."""
    cores = os.cpu_count() or 1
    allc = cpu_sample_subprocess(n_steps, cores)
    one = cpu_sample_subprocess(n_steps, 1)
    res = dict(allc) if allc and allc.get("value") else dict(one or {})
    res["single_thread"] = one
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-threads", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-steps", type=int, default=24)
    ap.add_argument("--layers", type=int, default=32, help="first N layers of the stack (profiling a small case)")
    ap.add_argument("--stack-only", action="store_true", help="graph replays only (for ncu captures)")
    ap.add_argument("--batch", type=int, default=1, help="sequences per step (multi-sequence workload)")
    ap.add_argument("--prefill", type=int, default=PREFILL, help="KV tokens before the first step (batch 1)")
    ap.add_argument("--kv", choices=["bf16", "turbo8"], default="bf16", help="KV cache format")
    ap.add_argument("--paged", action="store_true", help="paged bf16 KV (16-token blocks, shuffled table)")
    ap.add_argument("--prompt", type=int, default=0,
                    help="time the multi-token prefill of a prompt of this many tokens instead of decode")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.cpu_sample:
        print(json.dumps(cpu_sample(args.cpu_sample, args.cpu_threads)))
        return

    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        n = max(4, min(args.steps, 96))
        s = cpu_baseline(n + args.warmup)
        res = {"metric": METRIC, "value": s["value"], "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps,
               "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "f64", "data": "synthetic", "impl": "reference",
               "config": {"workload": "qwen3.5-4b-shape 32-layer decode stack, batch 1, KV prefilled to 8192"},
               "cpu_baseline": s,
               "e2e": {"value": s["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(res))
        return

    if args.prompt > 0:
        res = run_prompt(args)
        if res is None:
            return
        if args.cpu_steps > 0:  # the oracle's prefill is its single-token forward per token
            cb = cpu_baseline(args.cpu_steps)
            cb["sample"] = "the oracle's prefill runs its single-token forward token after token: " + cb["sample"]
            res["cpu_baseline"] = cb
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res))
        return
    res = run_gpu(args)
    if res is None:
        return
    if args.stack_only:
        print(json.dumps(res))
        return
    res["cpu_baseline"] = cpu_baseline(args.cpu_steps) if args.cpu_steps > 0 else None
    print(json.dumps(res))


if __name__ == "__main__":
    main()
