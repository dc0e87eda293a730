"""Multi-token prefill on the GPU against the oracle's prefill (the single-token
forward applied token after token).

Tolerances: those of the decode path (relative L2 <= 1e-2 on every token's layer
output and on the KV rows written, <= 2e-3 on the fp32 Gated DeltaNet state). The
projections whose outputs are kept (KV rows, conv and delta-rule states) multiply
each dequantised weight as the sum of two bf16 values (exact to 2^-16 relative);
the others multiply it rounded to bf16, and the inputs the single-token path keeps
unrounded (SiLU(gate) * up, SiLU(z) * y_norm) are rounded to bf16. The projection
alone is checked against the product of the weights its form defines: within one
bf16 unit, plus the tensor cores' accumulation error (a small part of the rms) on
outputs near zero.
"""

import numpy as np
import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O

from harness import bf16_ulps, bits, f32, f64, init, rel_l2

pytestmark = pytest.mark.gpu

TOL_X = 1e-2
TOL_STATE = 2e-3


def _prompt(seed, T, cfg):
    return np.stack([synth.x_in(seed, 1000 + t, cfg) for t in range(T)])


# ------------------------------------------------------------------ the projection


def _ulp(v):
    """The bf16 spacing at each |v| (v holds bf16 values; 0 for 0)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 0.0)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("exact", [True, False])
@pytest.mark.parametrize("n,k,T", [(300, 320, 200), (128, 64, 1), (37, 256, 129), (9216, 2560, 256),
                                   (32, 2560, 77), (2560, 9216, 300)])
def test_prefill_gemm_matches_weight_product(n, k, T, exact, split):
    """Rows past a 128-row tile and tokens past a 256-token tile (ragged tails), K
    past the 4-slot ring. Against bf16(X W^T) with the weights the form defines (the
    exact dequantised weights, or each rounded to bf16): a misplaced operand or a
    stage read before it is written puts errors of the outputs' own size on whole
    rows or tokens; here every output is within one bf16 unit of the reference plus
    1e-3 of the rms (the tensor cores' fp32 accumulation and, exact, the weights'
    2^-16 split, which move only outputs near a rounding boundary or near zero),
    and 99.9% are within one unit. With the split-K workspace, shapes of few tiles
    sum K in up to eight ranges (the same bounds hold)."""
    init()
    qw = synth.qweight(3, ("pf", n, k), n, k)
    w = B.DeviceQWeight(qw)
    X = synth.to_bf16_bits(np.random.default_rng(n + k + T).standard_normal((T, k)))
    x = B.to_device(X)
    y = torch.empty((T, n), dtype=torch.int16, device="cuda")
    scratch = B.new_scratch(B.QWEN35_PREFILL_GEMM_SPLIT_SCRATCH if split else 256)
    assert B.qwen35_prefill_gemm(w.c(), x, y, T, scratch, exact=exact) == 0
    wt = O.dequant(qw) if exact else O.bf16_round(O.dequant(qw))
    ref = O.bf16_round(O.bf16_to_f64(X) @ wt.T)
    torch.cuda.synchronize()
    got = f64(y)
    rms = np.sqrt(np.mean(ref * ref))
    err = np.abs(got - ref)
    excess = np.maximum(err - _ulp(ref), 0.0)
    ulps = bf16_ulps(got, ref)
    print(f"n={n} k={k} T={T} exact={exact} split={split}: max err / rms {err.max() / rms:.3e}, beyond one unit / rms "
          f"{excess.max() / rms:.3e}, rel-L2 {rel_l2(got, ref):.3e}, within 1 unit {np.mean(ulps <= 1):.6f}")
    assert excess.max() <= 1e-3 * rms
    assert np.mean(ulps <= 1) >= 0.999
    assert B.qwen35_read_device_status(scratch) == 0


# ------------------------------------------------------------------ layers


class PrefillFa:
    def __init__(self, cfg_name, capacity, n_filled, T, seed=0, layer=1):
        init()
        self.cfg = synth.config(cfg_name)
        self.c = B.make_config(self.cfg)
        self.layer = synth.fa_layer(seed, layer, self.cfg)
        self.k0, self.v0 = synth.kv_cache(seed, layer, self.cfg, capacity, n_filled)
        self.dev = B.DeviceFaLayer(self.layer)
        self.kv = B.DeviceKv(self.k0, self.v0)
        self.okv = O.kv_from_bits(self.k0, self.v0)
        self.T = T
        self.X = _prompt(seed, T, self.cfg)
        self.x_in = B.to_device(self.X)
        self.x_out = torch.empty_like(self.x_in)
        self.scratch = B.new_scratch(B.qwen35_prefill_scratch_bytes(self.c, T))

    def run(self, cache_pos, traces=None):
        rc = B.qwen35_prefill_full_attention(self.c, self.dev.struct, self.scratch, self.kv.struct, self.x_in,
                                             self.x_out, cache_pos, self.T)
        assert rc == 0, rc
        ref = O.prefill_full_attention(self.cfg, self.layer, self.okv, O.bf16_to_f64(self.X), cache_pos, traces)
        torch.cuda.synchronize()
        return f64(self.x_out), ref


def _check_fa(r, cache_pos, got, ref, traces):
    for t in range(r.T):
        assert rel_l2(got[t], ref[t]) <= TOL_X, t
    kb, vb = bits(r.kv.k), bits(r.kv.v)
    for t in range(r.T):  # the appended rows
        assert rel_l2(O.bf16_to_f64(kb[cache_pos + t]), traces[t]["k_rope"]) <= TOL_X, t
        assert rel_l2(O.bf16_to_f64(vb[cache_pos + t]).reshape(-1), traces[t]["v"]) <= TOL_X, t
    # rows below the prompt and above it are untouched, bit for bit
    assert np.array_equal(kb[:cache_pos], r.k0[:cache_pos]) and np.array_equal(vb[:cache_pos], r.v0[:cache_pos])
    end = cache_pos + r.T
    assert np.array_equal(kb[end:], r.k0[end:]) and np.array_equal(vb[end:], r.v0[end:])
    assert B.qwen35_read_device_status(r.scratch) == 0


def test_prefill_fa_tiny_after_cached_rows():
    r = PrefillFa("tiny", capacity=64, n_filled=5, T=37)
    traces = []
    got, ref = r.run(5, traces)
    _check_fa(r, 5, got, ref, traces)


def test_prefill_fa_tiny_whole_capacity_from_zero():
    r = PrefillFa("tiny", capacity=48, n_filled=0, T=48)
    traces = []
    got, ref = r.run(0, traces)
    _check_fa(r, 0, got, ref, traces)


def test_prefill_fa_4b():
    """Two token tiles (128 + 22) after 300 cached rows at the 4B dims."""
    r = PrefillFa("4b", capacity=512, n_filled=300, T=150)
    traces = []
    got, ref = r.run(300, traces)
    _check_fa(r, 300, got, ref, traces)


class PrefillGdn:
    def __init__(self, cfg_name, T, seed=0, layer=0, state_std=0.1):
        init()
        self.cfg = synth.config(cfg_name)
        self.c = B.make_config(self.cfg)
        self.layer = synth.gdn_layer(seed, layer, self.cfg)
        conv, ssm = synth.gdn_state(seed, layer, self.cfg, state_std)
        self.dev = B.DeviceGdnLayer(self.layer)
        self.state = B.DeviceState(conv, ssm)
        self.ostate = O.state_from_arrays(conv, ssm)
        self.T = T
        self.X = _prompt(seed, T, self.cfg)
        self.x_in = B.to_device(self.X)
        self.x_out = torch.empty_like(self.x_in)
        self.scratch = B.new_scratch(B.qwen35_prefill_scratch_bytes(self.c, T))

    def run(self):
        rc = B.qwen35_prefill_linear_attention(self.c, self.dev.struct, self.scratch, self.state.struct,
                                               self.x_in, self.x_out, self.T)
        assert rc == 0, rc
        ref = O.prefill_linear_attention(self.cfg, self.layer, self.ostate, O.bf16_to_f64(self.X))
        torch.cuda.synchronize()
        return f64(self.x_out), ref


@pytest.mark.parametrize("cfg_name,T", [("tiny", 37), ("tiny", 1), ("4b", 150)])
def test_prefill_gdn(cfg_name, T):
    r = PrefillGdn(cfg_name, T)
    got, ref = r.run()
    for t in range(T):
        assert rel_l2(got[t], ref[t]) <= TOL_X, t
    assert rel_l2(f32(r.state.ssm_matrix()), r.ostate["ssm"]) <= TOL_STATE
    assert rel_l2(f32(r.state.conv), r.ostate["conv"]) <= TOL_STATE
    assert B.qwen35_read_device_status(r.scratch) == 0


# ------------------------------------------------------------------ stack, then decode


def test_prefill_stack_tiny_then_decode():
    """A 20-token prompt through the tiny stack in one call, then 6 decode steps on
    the caches and states it left: every output against the oracle."""
    init()
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(0, 0, cfg), synth.fa_layer(0, 1, cfg)]
    conv, ssm = synth.gdn_state(0, 0, cfg, 0.1)
    kb, vb = synth.kv_cache(0, 1, cfg, 32, 0)
    dev = [B.DeviceGdnLayer(layers[0]), B.DeviceFaLayer(layers[1])]
    caches = [B.DeviceState(conv, ssm), B.DeviceKv(kb, vb)]
    ocaches = [O.state_from_arrays(conv, ssm), O.kv_from_bits(kb, vb)]
    entries = [B.stack_layer(k, l, cc) for k, l, cc in zip(kinds, dev, caches)]
    T = 20
    X = _prompt(0, T, cfg)
    x_in = B.to_device(X)
    x_out = torch.empty_like(x_in)
    pscr = B.new_scratch(B.qwen35_prefill_scratch_bytes(c, T))
    assert B.qwen35_prefill_step(c, entries, pscr, x_in, x_out, 0, T) == 0
    ref = O.prefill_step(cfg, kinds, layers, ocaches, O.bf16_to_f64(X), 0)
    torch.cuda.synchronize()
    got = f64(x_out)
    for t in range(T):
        assert rel_l2(got[t], ref[t]) <= TOL_X, t
    assert B.qwen35_read_device_status(pscr) == 0
    # decode continues from position T on what the prefill left
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes(c))
    xi = torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda")
    xo = torch.empty_like(xi)
    d_pos = torch.full((1,), T, dtype=torch.int32, device="cuda")
    for s in range(6):
        x = synth.x_in(0, s, cfg)
        xi.copy_(B.to_device(x))
        assert B.qwen35_decode_step(c, entries, scratch, xi, xo, d_pos, 32) == 0
        ref = O.decode_step(cfg, kinds, layers, ocaches, O.bf16_to_f64(x), T + s)
        torch.cuda.synchronize()
        assert rel_l2(f64(xo), ref) <= TOL_X, s
    assert rel_l2(f32(caches[0].ssm_matrix()), ocaches[0]["ssm"]) <= TOL_STATE
    assert rel_l2(f64(caches[1].k)[:T + 6], ocaches[1]["k"][:T + 6]) <= TOL_X
    assert B.qwen35_read_device_status(scratch) == 0


def test_prefill_argument_errors():
    init()
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    layer = synth.fa_layer(0, 1, cfg)
    dev = B.DeviceFaLayer(layer)
    kb, vb = synth.kv_cache(0, 1, cfg, 16, 0)
    kv = B.DeviceKv(kb, vb)
    X = _prompt(0, 8, cfg)
    x = B.to_device(X)
    y = torch.empty_like(x)
    small = B.new_scratch(B.qwen35_prefill_scratch_bytes(c, 4))
    big = B.new_scratch(B.qwen35_prefill_scratch_bytes(c, 8))
    assert B.qwen35_prefill_full_attention(c, dev.struct, small, kv.struct, x, y, 0, 8) == B.QWEN35_ERR_INVALID_ARGUMENT
    assert B.qwen35_prefill_full_attention(c, dev.struct, big, kv.struct, x, y, 9, 8) == B.QWEN35_ERR_OUT_OF_RANGE
    assert B.qwen35_prefill_full_attention(c, dev.struct, big, kv.struct, x, y, 0, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    assert B.qwen35_prefill_full_attention(c, dev.struct, big, kv.struct, x, y, 8, 8) == 0
    torch.cuda.synchronize()


# ------------------------------------------------------------------ paged caches, long context


@pytest.mark.parametrize("cfg_name,capacity,n_filled,T,bt", [("tiny", 64, 5, 37, 8), ("4b", 512, 300, 150, 16)])
def test_prefill_fa_paged_equals_contiguous(cfg_name, capacity, n_filled, T, bt):
    """The prompt over a paged cache (blocks placed by a shuffled table, every block
    the table does not name filled with bf16 NaN) gives the contiguous cache's
    outputs and rows bit for bit, and the oracle's within the layer tolerance."""
    r = PrefillFa(cfg_name, capacity=capacity, n_filled=n_filled, T=T)
    nl = capacity // bt
    table = synth.block_table(11, 1, nl, nl + 3)
    paged = B.DeviceKvPaged([r.k0], [r.v0], bt, table, nl + 3, fill=0x7FC0)
    out_p = torch.empty_like(r.x_out)
    scr_p = B.new_scratch(B.qwen35_prefill_scratch_bytes(r.c, T))
    assert B.qwen35_prefill_full_attention(r.c, r.dev.struct, scr_p, paged.struct, r.x_in, out_p, n_filled, T) == 0
    got, ref = r.run(n_filled)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(out_p), bits(r.x_out))
    for t in range(T):
        assert rel_l2(got[t], ref[t]) <= TOL_X, t
    for w, flat in (("k", r.kv.k), ("v", r.kv.v)):
        np.testing.assert_array_equal(paged.logical(w), bits(flat))
        pool = paged.pool(w)
        unused = sorted(set(range(pool.shape[0])) - set(table.reshape(-1).tolist()))
        assert np.all(pool[unused] == 0x7FC0)
    assert B.qwen35_read_device_status(scr_p) == 0


def test_prefill_fa_4b_after_long_context():
    """A 64-token prompt after 8192 cached rows at the 4B dims: each token attends
    over 8193 .. 8256 rows."""
    r = PrefillFa("4b", capacity=8320, n_filled=8192, T=64)
    traces = []
    got, ref = r.run(8192, traces)
    _check_fa(r, 8192, got, ref, traces)


def test_prefill_fa_one_token_equals_decode():
    """A one-token prompt is the single-token forward: against the oracle and the
    decode path on the same cache."""
    r = PrefillFa("4b", capacity=512, n_filled=200, T=1)
    traces = []
    got, ref = r.run(200, traces)
    _check_fa(r, 200, got, ref, traces)
    # the decode path on a fresh copy of the same cache and input
    kv2 = B.DeviceKv(r.k0, r.v0)
    scr = B.new_scratch(B.qwen35_scratch_bytes(r.c, B.QWEN35_LAYER_FULL_ATTENTION))
    xo = torch.empty(r.cfg["hidden"], dtype=torch.int16, device="cuda")
    assert B.qwen35_forward_full_attention(r.c, r.dev.struct, scr, kv2.struct, r.x_in[0], xo, 200, 201) == 0
    torch.cuda.synchronize()
    assert rel_l2(got[0], f64(xo)) <= TOL_X


# ------------------------------------------------------------------ Turbo8 caches


@pytest.mark.parametrize("cfg_name,capacity,n_filled,T", [("tiny", 64, 5, 37), ("4b", 512, 300, 150)])
def test_prefill_fa_turbo8(cfg_name, capacity, n_filled, T):
    """A prompt appended to a Turbo8 cache (rows WHT-rotated, FP8 E4M3 codes with a
    bf16 scale per 16) and attending over it: every token's output within the layer
    tolerance; the appended rows decode to the oracle's within it (a code can move
    one E4M3 step where the two sides' rotated rows differ in the last bf16 bit), and
    most codes are the oracle's; the rows outside the prompt untouched."""
    init()
    cfg = synth.config(cfg_name)
    c = B.make_config(cfg)
    layer = synth.fa_layer(0, 1, cfg)
    dev = B.DeviceFaLayer(layer)
    kc, ks, vc, vs = synth.kv_cache_turbo8(0, 1, cfg, capacity, n_filled)
    kv = B.DeviceKvTurbo8(kc, ks, vc, vs, cfg)
    okv = O.turbo8_kv(kc, ks, vc, vs)
    X = _prompt(0, T, cfg)
    x_in = B.to_device(X)
    x_out = torch.empty_like(x_in)
    scratch = B.new_scratch(B.qwen35_prefill_scratch_bytes(c, T))
    assert B.qwen35_prefill_full_attention(c, dev.struct, scratch, kv.struct, x_in, x_out, n_filled, T) == 0
    ref = O.prefill_full_attention(cfg, layer, okv, O.bf16_to_f64(X), n_filled)
    torch.cuda.synchronize()
    got = f64(x_out)
    for t in range(T):
        assert rel_l2(got[t], ref[t]) <= TOL_X, t
    end = n_filled + T
    for w, codes0 in (("k", kc), ("v", vc)):
        gc = (kv.k if w == "k" else kv.v).cpu().numpy().view(np.uint8)
        gs = O.bf16_to_f64(kv.scales(w))
        oc, osc = okv[w + "_codes"], okv[w + "_scales"]
        deq_g = O.turbo8_dequantize(gc[n_filled:end], gs[n_filled:end])
        deq_o = O.turbo8_dequantize(oc[n_filled:end], osc[n_filled:end])
        assert rel_l2(deq_g, deq_o) <= TOL_X, w
        assert np.mean(gc[n_filled:end] == oc[n_filled:end]) >= 0.9, w
        np.testing.assert_array_equal(gc[:n_filled], codes0[:n_filled])
        assert not gc[end:].any()
    assert B.qwen35_read_device_status(scratch) == 0


def test_prefill_stack_turbo8_then_decode():
    """A 20-token prompt through the tiny stack with a Turbo8 cache, then 4 decode
    steps on what it left, against the oracle."""
    init()
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(0, 0, cfg), synth.fa_layer(0, 1, cfg)]
    conv, ssm = synth.gdn_state(0, 0, cfg, 0.1)
    kc, ks, vc, vs = synth.kv_cache_turbo8(0, 1, cfg, 32, 0)
    dev = [B.DeviceGdnLayer(layers[0]), B.DeviceFaLayer(layers[1])]
    caches = [B.DeviceState(conv, ssm), B.DeviceKvTurbo8(kc, ks, vc, vs, cfg)]
    ocaches = [O.state_from_arrays(conv, ssm), O.turbo8_kv(kc, ks, vc, vs)]
    entries = [B.stack_layer(k, l, cc) for k, l, cc in zip(kinds, dev, caches)]
    T = 20
    X = _prompt(0, T, cfg)
    x_in = B.to_device(X)
    x_out = torch.empty_like(x_in)
    pscr = B.new_scratch(B.qwen35_prefill_scratch_bytes(c, T))
    assert B.qwen35_prefill_step(c, entries, pscr, x_in, x_out, 0, T) == 0
    ref = O.prefill_step(cfg, kinds, layers, ocaches, O.bf16_to_f64(X), 0)
    torch.cuda.synchronize()
    got = f64(x_out)
    for t in range(T):
        assert rel_l2(got[t], ref[t]) <= TOL_X, t
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes(c))
    xi = torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda")
    xo = torch.empty_like(xi)
    d_pos = torch.full((1,), T, dtype=torch.int32, device="cuda")
    for s in range(4):
        x = synth.x_in(0, s, cfg)
        xi.copy_(B.to_device(x))
        assert B.qwen35_decode_step(c, entries, scratch, xi, xo, d_pos, 32) == 0
        ref = O.decode_step(cfg, kinds, layers, ocaches, O.bf16_to_f64(x), T + s)
        torch.cuda.synchronize()
        assert rel_l2(f64(xo), ref) <= TOL_X, s
    assert B.qwen35_read_device_status(pscr) == 0 and B.qwen35_read_device_status(scratch) == 0


def test_prefill_step_captured_in_a_graph():
    """A stack prefill captured once as a CUDA graph and replayed computes what the
    call computes eagerly, bit for bit (outputs, caches and states)."""
    init()
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(0, 0, cfg), synth.fa_layer(0, 1, cfg)]
    conv, ssm = synth.gdn_state(0, 0, cfg, 0.1)
    kb, vb = synth.kv_cache(0, 1, cfg, 32, 0)
    T = 20
    X = _prompt(3, T, cfg)
    runs = []
    for use_graph in (False, True):
        dev = [B.DeviceGdnLayer(layers[0]), B.DeviceFaLayer(layers[1])]
        caches = [B.DeviceState(conv, ssm), B.DeviceKv(kb, vb)]
        entries = [B.stack_layer(k, l, cc) for k, l, cc in zip(kinds, dev, caches)]
        x_in = B.to_device(X)
        x_out = torch.empty_like(x_in)
        scr = B.new_scratch(B.qwen35_prefill_scratch_bytes(c, T))
        stream = torch.cuda.Stream()
        torch.cuda.synchronize()
        if use_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                assert B.qwen35_prefill_step(c, entries, scr, x_in, x_out, 0, T, stream) == 0
            with torch.cuda.stream(stream):
                g.replay()
        else:
            with torch.cuda.stream(stream):
                assert B.qwen35_prefill_step(c, entries, scr, x_in, x_out, 0, T, stream) == 0
        stream.synchronize()
        runs.append((bits(x_out), f32(caches[0].ssm_matrix()), bits(caches[1].k), bits(caches[1].v)))
        assert B.qwen35_read_device_status(scr) == 0
    for a, b in zip(*runs):
        np.testing.assert_array_equal(a, b)
