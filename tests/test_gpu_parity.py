"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Tolerances: bit-exact for dequantised weights, KV-append positions and the
[Q_h | gate_h] split; relative L2 <= 1e-2 on every layer output (bf16
activations) and <= 2e-3 on the fp32 Gated DeltaNet state after 64 steps.
"""

import numpy as np
import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O

from harness import FaRunner, GdnRunner, bf16_ulps, bits, f32, f64, init, rel_l2

pytestmark = pytest.mark.gpu

TOL_X = 1e-2
TOL_STATE = 2e-3


# ------------------------------------------------------------------ GEMV


@pytest.mark.parametrize("n,k", [(300, 2560), (77, 4096), (50, 9216), (8, 256), (3, 128), (37, 192),
                                 (1, 12288), (1031, 320)])
def test_dequant_bit_exact(n, k):
    init()
    qw = synth.qweight(11, ("dq", n, k), n, k)
    if k == 192:  # a general affine bias, not tied to the scale
        qw["biases"][:, :3] = synth.to_bf16_bits(np.random.default_rng(1).standard_normal((n, 3)) * 1e-2)
    d = B.DeviceQWeight(qw)
    out = torch.empty((n, k), dtype=torch.float32, device="cuda")
    assert B.qwen35_dequant(d.c(), out) == 0
    ref = O.dequant(qw).astype(np.float32)  # exact values, rounded once to fp32
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


def bf16_ulp(x):
    """The spacing of bf16 values at |x| (2^(e-7) for 2^e <= |x| < 2^(e+1))."""
    x = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(x)).astype(int) - 7)


def gemv_bound(W, x, K):
    """Elementwise bound on |GPU - oracle| for y = bf16(W x) with bf16 x.

    The kernel's sum before its bf16 rounding, y', differs from the exact W x by at
    most delta = (K/16 + W_parts + 3) * 2^-24 * sum_k |W_rk x_k|: a bf16 input is
    exact in the 16-bit fixed point it is quantised to (8 significant bits within
    2^8 of its chunk's largest element, 2^-15 of it below), the chunk dot products
    are exact integers, and each of the K/16 chunk terms and each step of the fp32
    running sum rounds once (relative 2^-24, against at most sum |W_rk x_k|).
    Both sides then round to bf16, each by at most half a unit in the last place of
    its own value: |got - ref| <= ulp(max(|got|, |ref|)) + delta. In practice the
    error is one bf16 step on the rows whose exact value falls near a rounding
    boundary, and zero elsewhere.
    """
    ax = np.abs(W) @ np.abs(x)
    return (K / 16 + 6 + 3) * 2.0 ** -24 * ax


@pytest.mark.parametrize("n,k", [(300, 2560), (77, 4096), (50, 9216), (8, 256), (3, 128), (37, 192),
                                 (5, 12288), (1031, 320), (18432, 2560)])
def test_gemv_matches_oracle(n, k):
    init()
    qw = synth.qweight(5, ("gv", n, k), n, k)
    x = synth.to_bf16_bits(np.random.default_rng(n + k).standard_normal(k))
    d = B.DeviceQWeight(qw)
    y = torch.empty(n, dtype=torch.int16, device="cuda")
    scratch = B.new_scratch(4096)
    assert B.qwen35_gemv(d.c(), B.to_device(x), y, scratch) == 0
    got = f64(y)
    W = O.dequant(qw)
    xf = O.bf16_to_f64(x)
    ref = O.bf16_round(W @ xf)
    assert rel_l2(got, ref) <= 2e-3
    bound = bf16_ulp(np.maximum(np.abs(got), np.abs(ref))) + gemv_bound(W, xf, k)
    assert np.all(np.abs(got - ref) <= bound), np.max(np.abs(got - ref) / bound)
    # in bf16 steps: exact on almost every row, one step on the rows whose exact value
    # sits near a rounding boundary; more only where the absolute term of the bound
    # dominates (outputs near zero after cancellation)
    ulps = bf16_ulps(got, ref)
    big = gemv_bound(W, xf, k) < 0.5 * bf16_ulp(ref)
    assert not big.any() or ulps[big].max() <= 1, ulps[big].max()
    assert np.mean(ulps == 0) >= 0.9
    assert B.qwen35_read_device_status(scratch) == 0


@pytest.mark.parametrize("n,k", [(300, 2560), (77, 4096), (50, 9216), (37, 192), (1031, 320), (5, 12288)])
def test_gemv_one_hot_input_returns_dequantised_column(n, k):
    """The hot path's own dequantisation, bit for bit: with x = e_j the GEMV's output
    is bf16(W[:, j]), and W[r][j] = scale * code + bias is exact in fp32 (an 8-bit
    scale times a code, the bias -128 * scale), so every row must equal the
    oracle's dequantised weight rounded once to bf16. Columns j cover the first and
    last column of groups, of the K-parts a row is split into across warps (9216:
    six parts of 1536), of the per-lane chunks, and the matrix's last column."""
    init()
    qw = synth.qweight(9, ("onehot", n, k), n, k)
    d = B.DeviceQWeight(qw)
    W = O.dequant(qw)
    scratch = B.new_scratch(4096)
    y = torch.empty(n, dtype=torch.int16, device="cuda")
    cols = sorted(c for c in {0, 1, 15, 16, 63, 64, 65, 511, 512, k // 2 - 1, k // 2, k - 64, k - 1,
                              1535, 1536, 3071, 4607, 6144, 9215} if c < k)
    for j in cols:
        x = np.zeros(k, dtype=np.uint16)
        x[j] = 0x3F80  # bf16 1.0
        assert B.qwen35_gemv(d.c(), B.to_device(x), y, scratch) == 0
        got = bits(y)
        np.testing.assert_array_equal(got, O.bf16_bits(O.bf16_round(W[:, j])), err_msg=f"column {j}")
    assert B.qwen35_read_device_status(scratch) == 0


# ------------------------------------------------------------------ layers, tiny


def test_gdn_layer_tiny_16_steps():
    r = GdnRunner("tiny")
    for t in range(16):
        tr = {}
        got, ref = r.step(t, tr)
        assert rel_l2(got, ref) <= TOL_X, t
        assert rel_l2(r.view("qkv", len(tr["qkv"])), tr["qkv"]) <= TOL_X
        assert rel_l2(r.view("y", len(tr["y"])), tr["y"]) <= TOL_X
    assert rel_l2(f32(r.state.ssm_matrix()), r.ostate["ssm"]) <= TOL_STATE
    assert rel_l2(f32(r.state.conv), r.ostate["conv"]) <= TOL_STATE
    assert B.qwen35_read_device_status(r.scratch) == 0


def test_fa_layer_tiny_16_steps_and_append_rows():
    cap = 20
    r = FaRunner("tiny", cap, 0)
    sentinel = torch.full_like(r.kv.k, 0x7F7F)  # a bf16 pattern no computed value takes
    r.kv.k.copy_(sentinel)
    r.kv.v.copy_(sentinel)
    r.okv["k"][:] = O.bf16_to_f64(np.full(r.okv["k"].shape, 0x7F7F, np.uint16))
    r.okv["v"][:] = r.okv["k"]
    for t in range(16):
        tr = {}
        got, ref = r.step(t, t, trace=tr)
        assert rel_l2(got, ref) <= TOL_X, t
        # rows above the newest append are untouched, bit for bit
        kb = bits(r.kv.k)
        assert np.all(kb[t + 1:] == 0x7F7F)
        assert not np.any(kb[t] == 0x7F7F)
        assert rel_l2(O.bf16_to_f64(kb[t]), tr["k_rope"]) <= TOL_X
        assert rel_l2(f64(r.kv.v)[t], tr["v"].reshape(kb[t].shape)) <= TOL_X
    assert B.qwen35_read_device_status(r.scratch) == 0


def test_fa_seq1_is_gated_v_and_split_is_exact():
    # zero gate rows of q_proj: gate = 0, sigmoid = 1/2, so at one token the gated
    # attention output is exactly v / 2 of the head's kv-head
    cfg = synth.config("tiny")
    r = FaRunner("tiny", 8, 0)
    H, Hkv, D = cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    codes = r.layer["q_proj"]["codes"]
    for h in range(H):
        codes[h * 2 * D + D:(h + 1) * 2 * D] = 128
    r.dev = B.DeviceFaLayer(r.layer)
    r.layer.pop("_deq_q_proj", None)
    got, ref = r.step(0, 0)
    assert rel_l2(got, ref) <= TOL_X
    v = r.view("v", Hkv * D).reshape(Hkv, D)
    ga = r.view("gated_attn", H * D).reshape(H, D)
    for h in range(H):
        np.testing.assert_array_equal(ga[h], v[h // (H // Hkv)] / 2)
    qf = r.view("q_full", 2 * H * D).reshape(H, 2 * D)
    assert not np.any(qf[:, D:])


def test_fa_prefix_attention_and_last_row():
    # seq_len_attn below cache_pos + 1 (the new row is appended but not attended),
    # and an append at the last row of the cache
    cap = 12
    r = FaRunner("tiny", cap, 11)
    got, ref = r.step(0, 11, seq_len=7)
    assert rel_l2(got, ref) <= TOL_X
    got, ref = r.step(1, cap - 1)
    assert rel_l2(got, ref) <= TOL_X
    assert rel_l2(f64(r.kv.k), r.okv["k"]) <= TOL_X


def test_device_position_out_of_range_sets_status_and_skips():
    r = FaRunner("tiny", 8, 4)
    before = bits(r.kv.k).copy()
    dpos = torch.full((1,), 8, dtype=torch.int32, device="cuda")  # == capacity
    rc = B.qwen35_forward_full_attention_dpos(r.c, r.dev.struct, r.scratch, r.kv.struct, r.x_in, r.x_out, dpos, 8)
    assert rc == 0
    assert B.qwen35_read_device_status(r.scratch) == B.QWEN35_ERR_DEVICE_RANGE
    np.testing.assert_array_equal(bits(r.kv.k), before)
    B.qwen35_scratch_init(r.scratch)
    dpos.fill_(-1)
    rc = B.qwen35_forward_full_attention_dpos(r.c, r.dev.struct, r.scratch, r.kv.struct, r.x_in, r.x_out, dpos, 8)
    assert rc == 0
    assert B.qwen35_read_device_status(r.scratch) == B.QWEN35_ERR_DEVICE_RANGE
    np.testing.assert_array_equal(bits(r.kv.k), before)


def test_fa_device_position_matches_host_position():
    r = FaRunner("tiny", 16, 0)
    dpos = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(6):
        got, ref = r.step(t, t, dpos=dpos)
        assert rel_l2(got, ref) <= TOL_X, t
    assert B.qwen35_read_device_status(r.scratch) == 0


# ------------------------------------------------------------------ tiny stack (config 0)


def _tiny_stack(seed=0):
    cfg = synth.config("tiny")
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(seed, 0, cfg), synth.fa_layer(seed, 1, cfg)]
    conv, ssm = synth.gdn_state(seed, 0, cfg)
    kb, vb = synth.kv_cache(seed, 1, cfg, 16, 0)
    dev = [B.DeviceGdnLayer(layers[0]), B.DeviceFaLayer(layers[1])]
    caches = [B.DeviceState(conv, ssm), B.DeviceKv(kb, vb)]
    ocaches = [O.state_from_arrays(conv, ssm), O.kv_from_bits(kb, vb)]
    return cfg, kinds, layers, dev, caches, ocaches


@pytest.mark.parametrize("use_graph", [False, True])
def test_tiny_stack_16_steps(use_graph):
    init()
    cfg, kinds, layers, dev, caches, ocaches = _tiny_stack()
    c = B.make_config(cfg)
    entries = [B.stack_layer(k, l, cc) for k, l, cc in zip(kinds, dev, caches)]
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes(c))
    x_in = torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    d_pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    g = None
    if use_graph:
        with torch.cuda.stream(stream):
            g = B.Graph(c, entries, scratch, x_in, x_out, d_pos, 16)
    for t in range(16):
        x = synth.x_in(0, t, cfg)
        with torch.cuda.stream(stream):
            x_in.copy_(B.to_device(x))
            if g is not None:
                g.launch()
            else:
                assert B.qwen35_decode_step(c, entries, scratch, x_in, x_out, d_pos, 16) == 0
        ref = O.decode_step(cfg, kinds, layers, ocaches, O.bf16_to_f64(x), t)
        stream.synchronize()
        assert rel_l2(f64(x_out), ref) <= TOL_X, t
    assert int(d_pos.item()) == 16
    assert rel_l2(f32(caches[0].ssm_matrix()), ocaches[0]["ssm"]) <= TOL_STATE
    assert rel_l2(f64(caches[1].k), ocaches[1]["k"]) <= TOL_X
    assert B.qwen35_read_device_status(scratch, stream) == 0
    if g is not None:
        g.close()


def test_resume_from_snapshot_is_bit_exact():
    """Checkpoint and resume: the caller owns the KV cache, the linear-attention
    state and the device position, so copying them mid-run and restoring them later
    reproduces the uninterrupted run bit for bit (every reduction of the decode runs
    in a fixed order)."""
    init()
    cfg, kinds, layers, dev, caches, _ = _tiny_stack()
    c = B.make_config(cfg)
    entries = [B.stack_layer(k, l, cc) for k, l, cc in zip(kinds, dev, caches)]
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes(c))
    x_in = torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    d_pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    persistent = [caches[0].conv, caches[0].ssm, caches[1].k, caches[1].v, d_pos]

    def run(t0, t1):
        outs = []
        for t in range(t0, t1):
            x_in.copy_(B.to_device(synth.x_in(0, t, cfg)))
            assert B.qwen35_decode_step(c, entries, scratch, x_in, x_out, d_pos, 16) == 0
            outs.append(x_out.clone())
        torch.cuda.synchronize()
        return outs

    run(0, 6)
    snapshot = [b.clone() for b in persistent]
    uninterrupted = run(6, 12)
    final = [b.clone() for b in persistent]
    for b, s in zip(persistent, snapshot):
        b.copy_(s)
    resumed = run(6, 12)
    for t, (a, b) in enumerate(zip(uninterrupted, resumed)):
        assert torch.equal(a, b), t
    for a, b in zip(final, persistent):
        assert torch.equal(a, b)
    assert int(d_pos.item()) == 12
    assert B.qwen35_read_device_status(scratch) == 0


# ------------------------------------------------------------------ output head (lm_head, greedy token)


def _run_head(cfg, head, x_bits):
    init()
    c = B.make_config(cfg)
    nw = B.to_device(head["final_norm"])
    w = B.DeviceQWeight(head["lm_head"])
    x = B.to_device(x_bits)
    logits = torch.empty(head["lm_head"]["n"], dtype=torch.int16, device="cuda")
    tok = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    scratch = B.new_scratch(4096)
    assert B.qwen35_lm_head_greedy(c, nw, w.c(), x, logits, tok, scratch) == 0
    torch.cuda.synchronize()
    assert B.qwen35_read_device_status(scratch) == 0
    return f64(logits), int(tok.item())


@pytest.mark.parametrize("name,vocab", [("tiny", 1000), ("4b", None)])
def test_lm_head_greedy_matches_oracle(name, vocab):
    cfg = synth.config(name)
    head = synth.head(7, cfg, vocab)  # 4b: the full 248 320-token vocabulary
    x_bits = synth.x_in(7, 0, cfg)
    got, tok = _run_head(cfg, head, x_bits)
    ref, _ = O.lm_head_greedy(cfg, head, O.bf16_to_f64(x_bits))
    assert rel_l2(got, ref) <= TOL_X
    # the token is decided on the kernel's own bf16 logits: their first maximal index
    assert tok == int(np.argmax(got))


def test_lm_head_ties_and_planted_winner():
    cfg = synth.config("tiny")
    x_bits = synth.x_in(6, 0, cfg)

    def head_with_identical_rows(winner=None, factor=1.0):
        h = synth.head(6, cfg, 1000)
        w = h["lm_head"]
        for key in ("codes", "scales", "biases"):
            w[key][:] = w[key][0]
        if winner is not None:
            for key in ("scales", "biases"):
                w[key][winner] = synth.to_bf16_bits(synth.bf16_bits_to_f32(w[key][winner]) * factor)
        return h

    got, tok = _run_head(cfg, head_with_identical_rows(), x_bits)
    assert np.all(got == got[0]) and tok == 0  # equal logits: the lowest index
    factor = 2.0 if got[0] > 0 else 0.5
    got2, tok2 = _run_head(cfg, head_with_identical_rows(winner=637, factor=factor), x_bits)
    assert tok2 == 637 and got2[637] == got[0] * factor


# ------------------------------------------------------------------ 4B-shape layers (configs 1, 2)


def test_gdn_layer_4b_64_steps():
    r = GdnRunner("4b")
    worst = 0.0
    for t in range(64):
        got, ref = r.step(t)
        worst = max(worst, rel_l2(got, ref))
        assert worst <= TOL_X, (t, worst)
    err = rel_l2(f32(r.state.ssm_matrix()), r.ostate["ssm"])
    assert err <= TOL_STATE, err
    assert rel_l2(f32(r.state.conv), r.ostate["conv"]) <= TOL_STATE
    assert B.qwen35_read_device_status(r.scratch) == 0


def check_append_rows(r, tr, cache_pos):
    """The KV rows appended at cache_pos, elementwise.

    v: the appended row is the kernel's own v projection output, bit for bit.
    k: the kernel's own k projection output taken through the pages' per-head
    RMSNorm (rounded to bf16) and partial RoPE (rounded to bf16) by the oracle's
    functions. The kernel forms the norm in fp32, so a normed element whose exact
    value lies within fp32 error of a bf16 rounding boundary may land one bf16 step
    away; RoPE mixes the pair (x_i, x_{i+R/2}), so on rotated dims that step reaches
    the output scaled by |cos| + |sin| <= 1.5, plus the fp32 rotation's own error
    (below 2^-20 of the pair's norm); both sides' final roundings add one step of
    the output. The projections themselves are held to the oracle's by the GEMV
    bound in test_gemv_matches_oracle and by the layer output.
    """
    cfg = r.cfg
    Hkv, D, R = cfg["num_kv_heads"], cfg["head_dim"], cfg["rotary_dim"]
    k_own = r.view("k", Hkv * D).reshape(Hkv, D)
    v_own = r.view("v", Hkv * D).reshape(Hkv, D)
    np.testing.assert_array_equal(f64(r.kv.v)[cache_pos], v_own)
    kn = O.bf16_round(O.rms_norm(k_own, O.bf16_to_f64(r.layer["k_norm"]), cfg["rms_eps"]))
    want = O.bf16_round(O.rope_apply(kn, cache_pos, O.rope_inv_freq(cfg["rope_theta"], R), R))
    got = f64(r.kv.k)[cache_pos]
    h = R // 2
    pair_max = np.abs(kn).copy()
    pm = np.maximum(np.abs(kn[:, :h]), np.abs(kn[:, h:R]))
    pair_max[:, :h] = pm
    pair_max[:, h:R] = pm
    pair_norm = np.abs(kn).copy()
    pn = np.hypot(kn[:, :h], kn[:, h:R])
    pair_norm[:, :h] = pn
    pair_norm[:, h:R] = pn
    rot = np.zeros((Hkv, D), dtype=bool)
    rot[:, :R] = True
    bound = bf16_ulp(np.maximum(np.abs(got), np.abs(want))) + np.where(rot, 1.5, 1.0) * bf16_ulp(pair_max) + \
        2.0 ** -20 * pair_norm
    assert np.all(np.abs(got - want) <= bound), np.max(np.abs(got - want) / bound)
    # and against the oracle's own k row (its k projection): per layer tolerance
    assert rel_l2(got, tr["k_rope"]) <= TOL_X


@pytest.mark.parametrize("cache_pos", [511, 4095, 16383])
def test_fa_layer_4b(cache_pos):
    r = FaRunner("4b", cache_pos + 8, cache_pos)
    tr = {}
    got, ref = r.step(0, cache_pos, trace=tr)
    assert rel_l2(got, ref) <= TOL_X
    check_append_rows(r, tr, cache_pos)
    assert not np.any(bits(r.kv.k)[cache_pos + 1:])  # rows above the append stay zero
    np.testing.assert_array_equal(bits(r.kv.k)[:cache_pos], O.bf16_bits(r.okv["k"][:cache_pos]))
    assert B.qwen35_read_device_status(r.scratch) == 0


# ------------------------------------------------------------------ long context (config 4a)


def test_fa_layer_4b_long_context():
    # 131072 tokens of context: the appended row is the cache's 131072nd
    cache_pos = 131071
    r = FaRunner("4b", cache_pos + 8, cache_pos)
    tr = {}
    got, ref = r.step(0, cache_pos, trace=tr)
    assert rel_l2(got, ref) <= TOL_X
    check_append_rows(r, tr, cache_pos)
    assert rel_l2(f64(r.kv.v)[cache_pos], tr["v"].reshape(-1, r.cfg["head_dim"])) <= TOL_X
    assert B.qwen35_read_device_status(r.scratch) == 0


# ------------------------------------------------------------------ the 32-layer stack (config 3)


def test_stack_4b_teacher_forced_per_layer():
    """One decode step of the 32-layer 4B-shape stack at 8192 tokens of context,
    checked layer by layer: the GPU runs the stack's prefixes [0, i] from the same
    states; the oracle applies layer i to the GPU's own input of that layer, and its
    output, its new state (GDN) or appended row (FA) must match."""
    init()
    cfg = synth.config("4b")
    kinds = synth.layer_kinds(cfg)
    c = B.make_config(cfg)
    prefill, cap = 8192, 8192 + 8
    dev, caches, entries, layers, ocaches = [], [], [], [], []
    for i, kind in enumerate(kinds):
        if kind == "fa":
            layers.append(synth.fa_layer(0, i, cfg))
            kb, vb = synth.kv_cache(0, i, cfg, cap, prefill)
            dev.append(B.DeviceFaLayer(layers[-1]))
            caches.append(B.DeviceKv(kb, vb))
            ocaches.append(O.kv_from_bits(kb, vb))
        else:
            layers.append(synth.gdn_layer(0, i, cfg))
            conv, ssm = synth.gdn_state(0, i, cfg, std=0.1)
            dev.append(B.DeviceGdnLayer(layers[-1]))
            caches.append(B.DeviceState(conv, ssm))
            ocaches.append(O.state_from_arrays(conv, ssm))
        entries.append(B.stack_layer(kind, dev[-1], caches[-1]))
    saved = [(cc.conv.clone(), cc.ssm.clone()) for cc in caches if isinstance(cc, B.DeviceState)]
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes(c))
    x_in = torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    d_pos = torch.empty(1, dtype=torch.int32, device="cuda")
    x0 = synth.x_in(0, 0, cfg)
    x_layer = O.bf16_to_f64(x0)  # the GPU's input of layer i
    worst = 0.0
    for i, kind in enumerate(kinds):
        j = 0
        for cc in caches:  # every linear-attention state back to its initial value
            if isinstance(cc, B.DeviceState):
                cc.conv.copy_(saved[j][0])
                cc.ssm.copy_(saved[j][1])
                j += 1
        d_pos.fill_(prefill)
        x_in.copy_(B.to_device(x0))
        assert B.qwen35_decode_step(c, entries[:i + 1], scratch, x_in, x_out, d_pos, cap) == 0
        torch.cuda.synchronize()
        got = f64(x_out)
        tr = {}
        if kind == "fa":
            ref = O.forward_full_attention(cfg, layers[i], ocaches[i], x_layer, prefill, prefill + 1, tr)
            assert rel_l2(f64(caches[i].k)[prefill], tr["k_rope"]) <= TOL_X, i
        else:
            ref = O.forward_linear_attention(cfg, layers[i], ocaches[i], x_layer, tr)
            assert rel_l2(f32(caches[i].ssm_matrix()), ocaches[i]["ssm"]) <= TOL_STATE, i
        for key in [k for k in layers[i] if k.startswith("_deq_")]:
            del layers[i][key]  # the oracle's dequantised weights, one layer at a time
        err = rel_l2(got, ref)
        worst = max(worst, err)
        assert err <= TOL_X, (i, kind, err)
        x_layer = got
    assert int(d_pos.item()) == prefill + 1
    assert B.qwen35_read_device_status(scratch) == 0


# ------------------------------------------------------------------ multi-sequence batch (config 4b)


def _batch_case(cfg_name, n_layers, positions, cap, seeds):
    """Layers shared by the batch; per sequence its own caches at its own position."""
    cfg = synth.config(cfg_name)
    kinds = synth.layer_kinds(cfg)[:n_layers]
    cfg = dict(cfg, num_layers=len(kinds))
    layers, dev = [], []
    per_seq = [[] for _ in positions]  # per sequence: its numpy caches per layer
    for i, kind in enumerate(kinds):
        if kind == "fa":
            layers.append(synth.fa_layer(0, i, cfg))
            dev.append(B.DeviceFaLayer(layers[-1]))
            for s, (pos, sd) in enumerate(zip(positions, seeds)):
                per_seq[s].append(synth.kv_cache(sd, i, cfg, cap, pos))
        else:
            layers.append(synth.gdn_layer(0, i, cfg))
            dev.append(B.DeviceGdnLayer(layers[-1]))
            for s, sd in enumerate(seeds):
                per_seq[s].append(synth.gdn_state(sd, i, cfg, std=0.1))
    return cfg, kinds, layers, dev, per_seq


@pytest.mark.parametrize("cfg_name,n_layers,positions,use_graph",
                         [("tiny", 2, [0, 5, 11], False), ("tiny", 2, [3, 0, 7], True),
                          ("tiny", 2, [0, 5, 11, 2, 7, 1, 9, 4], True),
                          ("4b", 4, [1000, 3100, 257, 2048], False)])
def test_batch_matches_single_sequence_decodes(cfg_name, n_layers, positions, use_graph):
    # the batch's projections run on tensor cores with inputs quantised per 64
    # columns (16-bit), the single path per 16: each sequence of the batch is held
    # to the oracle at the per-layer tolerances, and batch and single path, both
    # within those of the oracle, to twice them of each other. Only the first
    # layer's state sees the exact input; a deeper layer's input carries the
    # earlier layers' output error (<= TOL_X), which its decay gate passes on to
    # the state, so deeper states are held to TOL_X here and to TOL_STATE in the
    # teacher-forced test below
    init()
    nb, steps = len(positions), 3
    cap = max(positions) + steps + 8
    seeds = [10 + s for s in range(nb)]
    cfg, kinds, layers, dev, per_seq = _batch_case(cfg_name, n_layers, positions, cap, seeds)
    c = B.make_config(cfg)
    E = cfg["hidden"]
    # the batch: caches stacked per layer
    bcaches = []
    for i, kind in enumerate(kinds):
        if kind == "fa":
            bcaches.append(B.DeviceKvBatch([per_seq[s][i][0] for s in range(nb)], [per_seq[s][i][1] for s in range(nb)]))
        else:
            bcaches.append(B.DeviceStateBatch([per_seq[s][i][0] for s in range(nb)],
                                              [per_seq[s][i][1] for s in range(nb)]))
    bent = [B.stack_layer(k, d, cc) for k, d, cc in zip(kinds, dev, bcaches)]
    bscr = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb))
    bx_in = torch.empty(nb * E, dtype=torch.int16, device="cuda")
    bx_out = torch.empty_like(bx_in)
    bpos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    g = None
    if use_graph:
        with torch.cuda.stream(stream):
            g = B.Graph(c, bent, bscr, bx_in, bx_out, bpos, cap, batch=nb)
    # the same sequences one at a time
    singles = []
    for s in range(nb):
        caches = []
        for i, kind in enumerate(kinds):
            caches.append(B.DeviceKv(*per_seq[s][i]) if kind == "fa" else B.DeviceState(*per_seq[s][i]))
        ent = [B.stack_layer(k, d, cc) for k, d, cc in zip(kinds, dev, caches)]
        singles.append(dict(caches=caches, ent=ent, scr=B.new_scratch(B.qwen35_stack_scratch_bytes(c)),
                            x_in=torch.empty(E, dtype=torch.int16, device="cuda"),
                            x_out=torch.empty(E, dtype=torch.int16, device="cuda"),
                            pos=torch.tensor([positions[s]], dtype=torch.int32, device="cuda")))
    ocaches = [[O.kv_from_bits(*per_seq[s][i]) if kind == "fa" else O.state_from_arrays(*per_seq[s][i])
                for i, kind in enumerate(kinds)] for s in range(nb)]
    for t in range(steps):
        xs = [synth.x_in(seeds[s], t, cfg) for s in range(nb)]
        refs = [O.decode_step(cfg, kinds, layers, ocaches[s], O.bf16_to_f64(xs[s]), positions[s] + t)
                for s in range(nb)]
        with torch.cuda.stream(stream):
            bx_in.copy_(B.to_device(np.concatenate(xs)))
            if g is not None:
                g.launch(stream)
            else:
                assert B.qwen35_decode_step_batched(c, bent, nb, bscr, bx_in, bx_out, bpos, cap, stream) == 0
            for s, sg in enumerate(singles):
                sg["x_in"].copy_(B.to_device(xs[s]))
                assert B.qwen35_decode_step(c, sg["ent"], sg["scr"], sg["x_in"], sg["x_out"], sg["pos"], cap,
                                            stream) == 0
        stream.synchronize()
        bo = O.bf16_to_f64(bits(bx_out).reshape(nb, E))
        for s, sg in enumerate(singles):
            assert rel_l2(bo[s], refs[s]) <= TOL_X, (t, s)
            assert rel_l2(bo[s], f64(sg["x_out"])) <= 2 * TOL_X, (t, s)
    assert bpos.tolist() == [p + steps for p in positions]
    for i, kind in enumerate(kinds):
        for s, sg in enumerate(singles):
            if kind == "fa":
                assert rel_l2(f64(bcaches[i].k)[s], ocaches[s][i]["k"]) <= TOL_X, (i, s)
                assert rel_l2(f64(bcaches[i].v)[s], ocaches[s][i]["v"]) <= TOL_X, (i, s)
                assert rel_l2(f64(bcaches[i].k)[s], f64(sg["caches"][i].k)) <= 2 * TOL_X, (i, s)
            else:
                tol = TOL_STATE if i == 0 else TOL_X
                assert rel_l2(f32(bcaches[i].ssm_matrix(s)), ocaches[s][i]["ssm"]) <= tol, (i, s)
                assert rel_l2(f32(bcaches[i].conv[s]), ocaches[s][i]["conv"]) <= tol, (i, s)
                assert rel_l2(f32(bcaches[i].ssm_matrix(s)), f32(sg["caches"][i].ssm_matrix())) <= 2 * tol, (i, s)
    assert B.qwen35_read_device_status(bscr, stream) == 0
    if g is not None:
        g.close()


@pytest.mark.parametrize("positions", [[1000, 3100, 257, 2048],
                                       # the multi-sequence workload: 8 sequences, positions U{1024..65536}
                                       [int(p) for p in synth.cache_positions(0, 8)]])
def test_batch_4b_teacher_forced_per_layer(positions):
    """One batched step of a 4-layer 4B-shape stack (3 linear-attention layers, then
    full attention), each sequence at its own position, checked layer by layer: the
    GPU runs the prefixes [0, i] from the same caches; the oracle applies layer i to
    each sequence's GPU input of that layer; output, new state or appended row must
    match at the per-layer tolerances. With 8 sequences every n-column of the
    tensor-core products (one per sequence) and every per-sequence cache and
    scratch stride up to b = 7 is checked."""
    init()
    nb, cap = len(positions), max(positions) + 8
    seeds = [30 + s for s in range(nb)]
    cfg, kinds, layers, dev, per_seq = _batch_case("4b", 4, positions, cap, seeds)
    c = B.make_config(cfg)
    E = cfg["hidden"]
    bcaches = []
    for i, kind in enumerate(kinds):
        if kind == "fa":
            bcaches.append(B.DeviceKvBatch([per_seq[s][i][0] for s in range(nb)], [per_seq[s][i][1] for s in range(nb)]))
        else:
            bcaches.append(B.DeviceStateBatch([per_seq[s][i][0] for s in range(nb)],
                                              [per_seq[s][i][1] for s in range(nb)]))
    saved = [(cc.conv.clone(), cc.ssm.clone()) if kind == "gdn" else None for kind, cc in zip(kinds, bcaches)]
    bent = [B.stack_layer(k, d, cc) for k, d, cc in zip(kinds, dev, bcaches)]
    bscr = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb))
    bx_in = torch.empty(nb * E, dtype=torch.int16, device="cuda")
    bx_out = torch.empty_like(bx_in)
    bpos = torch.empty(nb, dtype=torch.int32, device="cuda")
    xs = [synth.x_in(seeds[s], 0, cfg) for s in range(nb)]
    x_layer = [O.bf16_to_f64(x) for x in xs]  # each sequence's GPU input of layer i
    for i, kind in enumerate(kinds):
        for sv, cc in zip(saved, bcaches):
            if sv is not None:
                cc.conv.copy_(sv[0])
                cc.ssm.copy_(sv[1])
        bpos.copy_(torch.tensor(positions, dtype=torch.int32))
        bx_in.copy_(B.to_device(np.concatenate(xs)))
        assert B.qwen35_decode_step_batched(c, bent[:i + 1], nb, bscr, bx_in, bx_out, bpos, cap) == 0
        torch.cuda.synchronize()
        got = O.bf16_to_f64(bits(bx_out).reshape(nb, E))
        for s in range(nb):
            tr = {}
            if kind == "fa":
                okv = O.kv_from_bits(*per_seq[s][i])
                ref = O.forward_full_attention(cfg, layers[i], okv, x_layer[s], positions[s], positions[s] + 1, tr)
                assert rel_l2(f64(bcaches[i].k)[s][positions[s]], tr["k_rope"]) <= TOL_X, (i, s)
                assert rel_l2(f64(bcaches[i].v)[s][positions[s]], tr["v"].reshape(-1, cfg["head_dim"])) <= TOL_X
            else:
                ost = O.state_from_arrays(*per_seq[s][i])
                ref = O.forward_linear_attention(cfg, layers[i], ost, x_layer[s], tr)
                assert rel_l2(f32(bcaches[i].ssm_matrix(s)), ost["ssm"]) <= TOL_STATE, (i, s)
                assert rel_l2(f32(bcaches[i].conv[s]), ost["conv"]) <= TOL_STATE, (i, s)
            assert rel_l2(got[s], ref) <= TOL_X, (i, s)
        x_layer = list(got)
    assert bpos.tolist() == [p + 1 for p in positions]
    assert B.qwen35_read_device_status(bscr) == 0


def test_batch_sequence_matches_oracle():
    # a batched sequence against the oracle stack (tiny dims, 3 sequences, 8 steps)
    init()
    positions, steps = [2, 0, 6], 8
    nb, cap = len(positions), 6 + steps + 4
    seeds = [20, 21, 22]
    cfg, kinds, layers, dev, per_seq = _batch_case("tiny", 2, positions, cap, seeds)
    c = B.make_config(cfg)
    E = cfg["hidden"]
    bcaches = [B.DeviceStateBatch([per_seq[s][0][0] for s in range(nb)], [per_seq[s][0][1] for s in range(nb)]),
               B.DeviceKvBatch([per_seq[s][1][0] for s in range(nb)], [per_seq[s][1][1] for s in range(nb)])]
    bent = [B.stack_layer(k, d, cc) for k, d, cc in zip(kinds, dev, bcaches)]
    bscr = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb))
    bx_in = torch.empty(nb * E, dtype=torch.int16, device="cuda")
    bx_out = torch.empty_like(bx_in)
    bpos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    s = 2  # the sequence checked against the oracle
    oc = [O.state_from_arrays(*per_seq[s][0]), O.kv_from_bits(*per_seq[s][1])]
    for t in range(steps):
        xs = [synth.x_in(seeds[q], t, cfg) for q in range(nb)]
        bx_in.copy_(B.to_device(np.concatenate(xs)))
        assert B.qwen35_decode_step_batched(c, bent, nb, bscr, bx_in, bx_out, bpos, cap) == 0
        ref = O.decode_step(cfg, kinds, layers, oc, O.bf16_to_f64(xs[s]), positions[s] + t)
        torch.cuda.synchronize()
        assert rel_l2(O.bf16_to_f64(bits(bx_out).reshape(nb, E)[s]), ref) <= TOL_X, t
    assert rel_l2(f32(bcaches[0].ssm_matrix(s)), oc[0]["ssm"]) <= TOL_STATE
    assert B.qwen35_read_device_status(bscr) == 0


# ------------------------------------------------------------------ per-layer batched forwards


@pytest.mark.parametrize("cfg_name,nb", [("tiny", 3), ("4b", 8)])
def test_linear_attention_batched_forward(cfg_name, nb):
    """qwen35_forward_linear_attention_batched: each of nb sequences (own state, own
    input) against the oracle's single-sequence forward, output and state."""
    init()
    cfg = synth.config(cfg_name)
    c = B.make_config(cfg)
    E = cfg["hidden"]
    layer = synth.gdn_layer(2, 0, cfg)
    dev = B.DeviceGdnLayer(layer)
    states = [synth.gdn_state(40 + s, 0, cfg, std=0.1) for s in range(nb)]
    bst = B.DeviceStateBatch([cs for cs, _ in states], [ss for _, ss in states])
    ost = [O.state_from_arrays(cs, ss) for cs, ss in states]
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb))
    x_in = torch.empty(nb * E, dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    for t in range(2):
        xs = [synth.x_in(40 + s, t, cfg) for s in range(nb)]
        x_in.copy_(B.to_device(np.concatenate(xs)))
        assert B.qwen35_forward_linear_attention_batched(c, dev.struct, nb, scratch, bst.struct, x_in, x_out) == 0
        torch.cuda.synchronize()
        got = O.bf16_to_f64(bits(x_out).reshape(nb, E))
        for s in range(nb):
            ref = O.forward_linear_attention(cfg, layer, ost[s], O.bf16_to_f64(xs[s]))
            assert rel_l2(got[s], ref) <= TOL_X, (t, s)
    for s in range(nb):
        assert rel_l2(f32(bst.ssm_matrix(s)), ost[s]["ssm"]) <= TOL_STATE, s
        assert rel_l2(f32(bst.conv[s]), ost[s]["conv"]) <= TOL_STATE, s
    assert B.qwen35_read_device_status(scratch) == 0


@pytest.mark.parametrize("cfg_name,positions", [("tiny", [0, 5, 11]), ("4b", [300, 4095, 1024, 2047, 17, 999, 3000, 511])])
def test_full_attention_batched_forward(cfg_name, positions):
    """qwen35_forward_full_attention_batched: each sequence at its own device position
    against the oracle's single-sequence forward (output, appended row), and the
    positions left as they were."""
    init()
    cfg = synth.config(cfg_name)
    c = B.make_config(cfg)
    E, D = cfg["hidden"], cfg["head_dim"]
    nb, cap = len(positions), max(positions) + 4
    layer = synth.fa_layer(3, 1, cfg)
    dev = B.DeviceFaLayer(layer)
    kvs = [synth.kv_cache(50 + s, 1, cfg, cap, p) for s, p in enumerate(positions)]
    bkv = B.DeviceKvBatch([k for k, _ in kvs], [v for _, v in kvs])
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb))
    x_in = torch.empty(nb * E, dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    dpos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    xs = [synth.x_in(50 + s, 0, cfg) for s in range(nb)]
    x_in.copy_(B.to_device(np.concatenate(xs)))
    assert B.qwen35_forward_full_attention_batched(c, dev.struct, nb, scratch, bkv.struct, x_in, x_out, dpos, cap) == 0
    torch.cuda.synchronize()
    got = O.bf16_to_f64(bits(x_out).reshape(nb, E))
    for s, p in enumerate(positions):
        tr = {}
        ref = O.forward_full_attention(cfg, layer, O.kv_from_bits(*kvs[s]), O.bf16_to_f64(xs[s]), p, p + 1, tr)
        assert rel_l2(got[s], ref) <= TOL_X, s
        assert rel_l2(f64(bkv.k)[s][p], tr["k_rope"]) <= TOL_X, s
        assert rel_l2(f64(bkv.v)[s][p], tr["v"].reshape(-1, D)) <= TOL_X, s
        assert not np.any(bits(bkv.k)[s][p + 1:])  # nothing above the append
    assert dpos.tolist() == positions  # a per-layer forward does not advance the positions
    assert B.qwen35_read_device_status(scratch) == 0
