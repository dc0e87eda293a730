"""The debug hooks through the C ABI: the stage dumps of the steps fused inside the
kernel (the page "linear_attention.rs" intra_dump names x_norm, qkv_smooth, y_norm,
and x_norm2) against the oracle, and the device-side wait limit: a wait that runs
out is reported in the status word, the call returns, and the next forward on the
same context is correct.
"""

import numpy as np
import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O

from harness import FaRunner, GdnRunner, bf16_ulps, bits, f64, init, rel_l2

pytestmark = pytest.mark.gpu

TOL_X = 1e-2


def _dump(r, kind, name, n):
    return O.bf16_to_f64(bits(B.scratch_view(r.scratch, r.c, kind, name, n)))


@pytest.fixture
def stage_dump():
    init()
    B.qwen35_debug_stage_dump(True)
    yield
    B.qwen35_debug_stage_dump(False)


def test_stage_dump_linear_attention(stage_dump):
    r = GdnRunner("tiny", state_std=0.1)
    cfg = r.cfg
    E, Hv, Dv = cfg["hidden"], cfg["num_v_heads_lin"], cfg["v_head_dim_lin"]
    C = 2 * cfg["num_k_heads_lin"] * cfg["k_head_dim_lin"] + Hv * Dv
    for t in range(3):
        tr = {}
        got, ref = r.step(t, tr)
        assert rel_l2(got, ref) <= TOL_X
        # x_norm: the same bf16 input on both sides, one rounding each: one step at most
        assert bf16_ulps(_dump(r, 1, "x_norm", E), tr["x_norm"]).max() <= 1
        # the fused steps applied by the oracle's functions to the kernel's own inputs
        # of them: y_norm from the kernel's y, x_norm2 from its x_resid
        y = r.view("y", Hv * Dv).reshape(Hv, Dv)
        yn = O.bf16_round(O.rms_norm(y, O.bf16_to_f64(r.layer["norm_weight"]), cfg["rms_eps"])).reshape(-1)
        assert bf16_ulps(_dump(r, 1, "y_norm", Hv * Dv), yn).max() <= 1
        xr = r.view("x_resid", E)
        xn2 = O.bf16_round(O.rms_norm(xr, O.bf16_to_f64(r.layer["post_ln"]), cfg["rms_eps"]))
        assert bf16_ulps(_dump(r, 1, "x_norm2", E), xn2).max() <= 1
        # qkv_smooth: conv, SiLU and the per-head L2 norm, against the oracle's trace
        qs = _dump(r, 1, "qkv_smooth", C)
        assert rel_l2(qs, tr["qkv_smooth"]) <= TOL_X
        nqk = 2 * cfg["num_k_heads_lin"] * cfg["k_head_dim_lin"]
        heads = qs[:nqk].reshape(-1, cfg["k_head_dim_lin"])
        np.testing.assert_allclose(np.linalg.norm(heads, axis=1), 1.0, atol=1e-2)
    assert B.qwen35_read_device_status(r.scratch) == 0


def test_stage_dump_full_attention(stage_dump):
    r = FaRunner("tiny", 16, 5)
    E = r.cfg["hidden"]
    tr = {}
    got, ref = r.step(0, 5, trace=tr)
    assert rel_l2(got, ref) <= TOL_X
    assert bf16_ulps(_dump(r, 0, "x_norm", E), tr["x_norm"]).max() <= 1
    xr = r.view("x_resid", E)
    xn2 = O.bf16_round(O.rms_norm(xr, O.bf16_to_f64(r.layer["post_ln"]), r.cfg["rms_eps"]))
    assert bf16_ulps(_dump(r, 0, "x_norm2", E), xn2).max() <= 1
    assert B.qwen35_read_device_status(r.scratch) == 0


def test_stage_dump_off_by_default():
    init()
    B.qwen35_debug_stage_dump(False)
    r = GdnRunner("tiny")
    E = r.cfg["hidden"]
    off = B.qwen35_debug_scratch_offset(r.c, 1, "x_norm")
    r.scratch[off:off + 2 * E].fill_(0x5A)
    r.step(0)
    assert torch.all(r.scratch[off:off + 2 * E] == 0x5A)  # nothing written there


# ------------------------------------------------------------------ bounded waits


def _tiny_stack(seed):
    cfg = synth.config("tiny")
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(seed, 0, cfg), synth.fa_layer(seed, 1, cfg)]
    conv, ssm = synth.gdn_state(seed, 0, cfg)
    kb, vb = synth.kv_cache(seed, 1, cfg, 16, 0)
    dev = [B.DeviceGdnLayer(layers[0]), B.DeviceFaLayer(layers[1])]
    caches = [B.DeviceState(conv, ssm), B.DeviceKv(kb, vb)]
    entries = [B.stack_layer(k, l, cc) for k, l, cc in zip(kinds, dev, caches)]
    ocaches = [O.state_from_arrays(conv, ssm), O.kv_from_bits(kb, vb)]
    c = B.make_config(cfg)
    return dict(cfg=cfg, c=c, kinds=kinds, layers=layers, keep=(dev, caches), entries=entries, ocaches=ocaches,
                scratch=B.new_scratch(B.qwen35_stack_scratch_bytes(c)),
                x_in=torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda"),
                x_out=torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda"),
                d_pos=torch.zeros(1, dtype=torch.int32, device="cuda"))


def _run_stack(st, t):
    x = synth.x_in(0, t, st["cfg"])
    st["x_in"].copy_(B.to_device(x))
    assert B.qwen35_decode_step(st["c"], st["entries"], st["scratch"], st["x_in"], st["x_out"], st["d_pos"], 16) == 0
    torch.cuda.synchronize()
    return x


def test_device_wait_that_runs_out_is_reported_and_recoverable():
    """Three launches of the tiny two-layer stack (config 0).

    1. Every CTA, after its work, waits on a flag that nothing sets, with a 2 ms
       limit: the wait runs out, the status word reads QWEN35_ERR_DEVICE_TIMEOUT,
       and the step's output is still the oracle's (the forward's own waits all
       completed well inside the limit).
    2. A 1 ns limit: the forward's own waits (tagged inputs, ring tiles, split
       flags) give up as soon as they are not satisfied at once; the call returns
       and the status reads the timeout (its results are meaningless).
    3. Defaults restored, on fresh buffers: the context is usable and the step
       matches the oracle with a clean status.
    """
    init()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = _tiny_stack(0)
    try:
        assert B.qwen35_debug_set_wait_limit(2_000_000) == 0
        assert B.qwen35_debug_wait_probe(flag) == 0
        x = _run_stack(st, 0)
    finally:
        B.qwen35_debug_wait_probe(None)
        B.qwen35_debug_set_wait_limit(0)
    assert B.qwen35_read_device_status(st["scratch"]) == B.QWEN35_ERR_DEVICE_TIMEOUT
    ref = O.decode_step(st["cfg"], st["kinds"], st["layers"], st["ocaches"], O.bf16_to_f64(x), 0)
    assert rel_l2(f64(st["x_out"]), ref) <= TOL_X
    assert int(st["d_pos"].item()) == 1

    st2 = _tiny_stack(1)
    try:
        assert B.qwen35_debug_set_wait_limit(1) == 0
        assert B.qwen35_debug_wait_probe(flag) == 0
        _run_stack(st2, 0)
    finally:
        B.qwen35_debug_wait_probe(None)
        B.qwen35_debug_set_wait_limit(0)
    assert B.qwen35_read_device_status(st2["scratch"]) == B.QWEN35_ERR_DEVICE_TIMEOUT

    st3 = _tiny_stack(0)
    for t in range(2):
        x = _run_stack(st3, t)
        ref = O.decode_step(st3["cfg"], st3["kinds"], st3["layers"], st3["ocaches"], O.bf16_to_f64(x), t)
        assert rel_l2(f64(st3["x_out"]), ref) <= TOL_X, t
    assert B.qwen35_read_device_status(st3["scratch"]) == 0
