"""Parity of the Turbo8 KV-cache path (page "mod.rs", MetalKvDtype::Turbo8; page
"full_attention.rs", the Turbo path) with the oracle, through the C ABI.

Tolerances: the layer output within the layer tolerance (relative L2 1e-2); the
appended codes and scales bit for bit against the oracle's quantiser applied to
the kernel's own rotated rows (both sides decide each E4M3 code on the same fp32
quotient); the rotated rows themselves within one bf16 step of the oracle's
rotation of the kernel's own (normed, RoPE'd) k and v, up to the fp32 vs float64
rotation near a rounding boundary.
"""

import numpy as np
import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O

from harness import bits, f64, init, rel_l2

pytestmark = pytest.mark.gpu

TOL_X = 1e-2


class TurboFa:
    """One full-attention layer with a Turbo8 cache, on the GPU and in the oracle."""

    def __init__(self, cfg_name, capacity, n_prefill, seed=0):
        init()
        self.cfg = synth.config(cfg_name)
        self.c = B.make_config(self.cfg)
        self.seed = seed
        self.layer = synth.fa_layer(seed, 1, self.cfg)
        kc, ks, vc, vs = synth.kv_cache_turbo8(seed, 1, self.cfg, capacity, n_prefill)
        self.dev = B.DeviceFaLayer(self.layer)
        self.kv = B.DeviceKvTurbo8(kc, ks, vc, vs, self.cfg)
        self.okv = O.turbo8_kv(kc, ks, vc, vs)
        self.scratch = B.new_scratch(B.qwen35_scratch_bytes(self.c, B.QWEN35_LAYER_FULL_ATTENTION))
        self.x_in = torch.empty(self.cfg["hidden"], dtype=torch.int16, device="cuda")
        self.x_out = torch.empty_like(self.x_in)

    def step(self, t, cache_pos, trace=None):
        x = synth.x_in(self.seed, t, self.cfg)
        self.x_in.copy_(B.to_device(x))
        rc = B.qwen35_forward_full_attention(self.c, self.dev.struct, self.scratch, self.kv.struct, self.x_in,
                                             self.x_out, cache_pos, cache_pos + 1)
        assert rc == 0, rc
        ref = O.forward_full_attention(self.cfg, self.layer, self.okv, O.bf16_to_f64(x), cache_pos, cache_pos + 1,
                                       trace)
        torch.cuda.synchronize()
        return f64(self.x_out), ref

    def dump(self, name):
        n = self.cfg["num_kv_heads"] * self.cfg["head_dim"]
        return O.bf16_to_f64(bits(B.scratch_view(self.scratch, self.c, 0, name, n))).reshape(
            self.cfg["num_kv_heads"], self.cfg["head_dim"])


def check_append(r, pos, tr):
    """Row pos of the cache: codes and scales equal the oracle's quantiser applied to
    the kernel's own rotated k and v rows (from the stage dump), bit for bit; those
    rows are within one bf16 step of the oracle's rotation of the kernel's own k."""
    k_rot, v_rot = r.dump("k_rot"), r.dump("v_rot")
    ck, sk = O.turbo8_quantize(k_rot)
    cv, sv = O.turbo8_quantize(v_rot)
    got_kc = r.kv.k.cpu().numpy().view(np.uint8)[pos]
    got_vc = r.kv.v.cpu().numpy().view(np.uint8)[pos]
    np.testing.assert_array_equal(got_kc, ck)
    np.testing.assert_array_equal(got_vc, cv)
    np.testing.assert_array_equal(O.bf16_to_f64(r.kv.scales("k")[pos]), sk)
    np.testing.assert_array_equal(O.bf16_to_f64(r.kv.scales("v")[pos]), sv)
    # against the oracle's own rotated rows (its k, v projections): the layer tolerance
    assert rel_l2(k_rot, tr["k_rot"]) <= TOL_X
    assert rel_l2(v_rot, tr["v_rot"]) <= TOL_X


@pytest.fixture
def stage_dump():
    init()
    B.qwen35_debug_stage_dump(True)
    yield
    B.qwen35_debug_stage_dump(False)


def test_turbo8_layer_tiny_16_steps(stage_dump):
    cap = 20
    r = TurboFa("tiny", cap, 0)
    for t in range(16):
        tr = {}
        got, ref = r.step(t, t, trace=tr)
        assert rel_l2(got, ref) <= TOL_X, t
        check_append(r, t, tr)
        # nothing above the append
        assert not r.kv.k.cpu().numpy().view(np.uint8)[t + 1:].any()
    assert B.qwen35_read_device_status(r.scratch) == 0


@pytest.mark.parametrize("cache_pos", [511, 4095, 16383])
def test_turbo8_layer_4b(stage_dump, cache_pos):
    r = TurboFa("4b", cache_pos + 8, cache_pos)
    tr = {}
    got, ref = r.step(0, cache_pos, trace=tr)
    assert rel_l2(got, ref) <= TOL_X
    check_append(r, cache_pos, tr)
    # the prefilled rows are untouched
    kc0, _, _, _ = synth.kv_cache_turbo8(0, 1, r.cfg, cache_pos + 8, cache_pos)
    np.testing.assert_array_equal(r.kv.k.cpu().numpy().view(np.uint8)[:cache_pos], kc0[:cache_pos])
    assert B.qwen35_read_device_status(r.scratch) == 0


def test_turbo8_layer_4b_long_context(stage_dump):
    """131072 tokens of Turbo8 context (config 4a's length): the layer output, the
    appended codes and scales, and the prefilled rows untouched."""
    cache_pos = 131071
    r = TurboFa("4b", cache_pos + 8, cache_pos)
    tr = {}
    got, ref = r.step(0, cache_pos, trace=tr)
    assert rel_l2(got, ref) <= TOL_X
    check_append(r, cache_pos, tr)
    kc0, _, _, _ = synth.kv_cache_turbo8(0, 1, r.cfg, cache_pos + 8, cache_pos)
    np.testing.assert_array_equal(r.kv.k.cpu().numpy().view(np.uint8)[:cache_pos], kc0[:cache_pos])
    assert B.qwen35_read_device_status(r.scratch) == 0


@pytest.mark.parametrize("use_graph", [False, True])
def test_turbo8_tiny_stack(use_graph):
    init()
    cfg = synth.config("tiny")
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(0, 0, cfg), synth.fa_layer(0, 1, cfg)]
    conv, ssm = synth.gdn_state(0, 0, cfg)
    tk = synth.kv_cache_turbo8(0, 1, cfg, 16, 0)
    dev = [B.DeviceGdnLayer(layers[0]), B.DeviceFaLayer(layers[1])]
    caches = [B.DeviceState(conv, ssm), B.DeviceKvTurbo8(*tk, cfg)]
    ocaches = [O.state_from_arrays(conv, ssm), O.turbo8_kv(*tk)]
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
    for t in range(10):
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
    assert int(d_pos.item()) == 10
    assert B.qwen35_read_device_status(scratch, stream) == 0
    if g is not None:
        g.close()


def test_turbo8_batched_forward():
    """qwen35_forward_full_attention_batched on a batch of Turbo8 caches
    ([B][capacity][Hkv][D] codes, [B][capacity][sstride] scales)."""
    init()
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    E = cfg["hidden"]
    positions = [0, 5, 11]
    nb, cap = len(positions), 16
    layer = synth.fa_layer(4, 1, cfg)
    dev = B.DeviceFaLayer(layer)
    caches = [synth.kv_cache_turbo8(60 + s, 1, cfg, cap, p) for s, p in enumerate(positions)]
    bkv = B.DeviceKvTurbo8(*[np.stack([cc[i] for cc in caches]) for i in range(4)], cfg)
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb))
    x_in = torch.empty(nb * E, dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    dpos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    xs = [synth.x_in(60 + s, 0, cfg) for s in range(nb)]
    x_in.copy_(B.to_device(np.concatenate(xs)))
    assert B.qwen35_forward_full_attention_batched(c, dev.struct, nb, scratch, bkv.struct, x_in, x_out, dpos, cap) == 0
    torch.cuda.synchronize()
    got = O.bf16_to_f64(bits(x_out).reshape(nb, E))
    for s, p in enumerate(positions):
        okv = O.turbo8_kv(*caches[s])
        tr = {}
        ref = O.forward_full_attention(cfg, layer, okv, O.bf16_to_f64(xs[s]), p, p + 1, tr)
        assert rel_l2(got[s], ref) <= TOL_X, s
        # the appended row decodes to the oracle's within its quantisation
        kc = bkv.k.cpu().numpy().view(np.uint8)[s][p]
        ks = O.bf16_to_f64(bkv.scales("k")[s][p])
        assert rel_l2(O.turbo8_dequantize(kc, ks), O.turbo8_dequantize(okv["k_codes"][p], okv["k_scales"][p])) <= 0.1
    assert B.qwen35_read_device_status(scratch) == 0
