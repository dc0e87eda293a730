"""The C-ABI entries not covered by the layer-forward tests, without a GPU: every
malformed call is rejected before anything touches the device (the pointers here
are fake, aligned or deliberately misaligned, and never dereferenced), and a
well-formed call with no device present fails with QWEN35_ERR_CUDA.

The whole file is skipped where a CUDA device is present: a check lost in a later
change would otherwise let a fake address reach a kernel on a real GPU. The debug
setters are only ever called with their default values, so the library's global
state is left as it was for whatever runs next in the process.
"""

import ctypes as C

import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth

_BASE = 0x10000000  # fake device addresses, 16-byte aligned
_NO_STREAM = 0
_no_device = pytest.mark.skipif(torch.cuda.is_available(), reason="a CUDA device is present")
pytestmark = _no_device


def _qw(n, k, i):
    base = _BASE + i * 0x4000000
    return B.qwen35_qweight(base, base + 0x1000000, base + 0x2000000, n, k)


def _fake_gdn(cfg):
    E, I = cfg["hidden"], cfg["intermediate"]
    Hk, Hv, Dk, Dv = cfg["num_k_heads_lin"], cfg["num_v_heads_lin"], cfg["k_head_dim_lin"], cfg["v_head_dim_lin"]
    Cq, Z = 2 * Hk * Dk + Hv * Dv, Hv * Dv
    g = B.qwen35_gdn_layer()
    g.input_ln, g.a_log, g.dt_bias, g.conv1d_weight = 0x1000, 0x2000, 0x3000, 0x4000
    g.norm_weight, g.post_ln = 0x5000, 0x6000
    g.in_proj_a, g.in_proj_b = _qw(Hv, E, 1), _qw(Hv, E, 2)
    g.in_proj_qkv, g.in_proj_z = _qw(Cq, E, 3), _qw(Z, E, 4)
    g.out_proj = _qw(E, Z, 5)
    g.gate_proj, g.up_proj, g.down_proj = _qw(I, E, 6), _qw(I, E, 7), _qw(E, I, 8)
    return g


def _fake_fa(cfg):
    E, I, H, Hkv, D = cfg["hidden"], cfg["intermediate"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    shapes = [(2 * H * D, E), (Hkv * D, E), (Hkv * D, E), (E, H * D), (I, E), (I, E), (E, I)]
    return B.qwen35_fa_layer(0x1000, 0x2000, 0x3000, 0x4000, *[_qw(n, k, i + 1) for i, (n, k) in enumerate(shapes)])


class _Scratch:  # a fake buffer: an address and a size
    def __init__(self, n, addr=0x70000000):
        self.n, self.addr = n, addr

    def numel(self):
        return self.n

    def data_ptr(self):
        return self.addr


X, Y = 0x80000000, 0x90000000
_STATIC_BYTES = 256 * 1024  # QWEN35_STATIC_SCRATCH_BYTES


# ------------------------------------------------ the no-alloc linear-attention forward


def test_static_forward_rejects_malformed_calls_before_the_device():
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    g = _fake_gdn(cfg)
    st = B.qwen35_gdn_state(0xA0000000, 0xB0000000)
    f = B.qwen35_forward_linear_attention_static
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    assert f(c, g, st, X + 2, Y, _NO_STREAM) == INV            # misaligned x_in
    assert f(c, g, st, X, Y + 8, _NO_STREAM) == INV            # misaligned x_out
    assert f(c, g, B.qwen35_gdn_state(0xA0000004, 0xB0000000), X, Y, _NO_STREAM) == INV  # conv state
    assert f(c, g, B.qwen35_gdn_state(0xA0000000, None), X, Y, _NO_STREAM) == INV         # no ssm state
    bad = _fake_gdn(cfg)
    bad.out_proj.k += 64                                        # wrong shape
    assert f(c, bad, st, X, Y, _NO_STREAM) == INV
    bad = _fake_gdn(cfg)
    bad.a_log = 0x2002                                          # a_log is fp32: 4-byte aligned
    assert f(c, bad, st, X, Y, _NO_STREAM) == INV
    L = B.lib()
    assert L.qwen35_forward_linear_attention_static(C.byref(c), None, C.byref(st), X, Y, None) == INV
    assert L.qwen35_forward_linear_attention_static(C.byref(c), C.byref(g), None, X, Y, None) == INV
    assert L.qwen35_forward_linear_attention_static(None, C.byref(g), C.byref(st), X, Y, None) == INV
    # the same errors as the scratch form for the config
    cb = synth.config("tiny")
    cb["k_head_dim_lin"] = 48
    assert f(B.make_config(cb), g, st, X, Y, _NO_STREAM) == B.QWEN35_ERR_UNSUPPORTED
    cb = synth.config("tiny")
    cb["num_v_heads_lin"] = 3                                   # not a multiple of the k-heads
    assert f(B.make_config(cb), g, st, X, Y, _NO_STREAM) == INV


def test_static_forward_rejects_configs_larger_than_the_array():
    cfg = synth.config("4b")
    cfg["hidden"], cfg["intermediate"] = 12288, 12288
    c = B.make_config(cfg)
    assert B.qwen35_scratch_bytes(c, B.QWEN35_LAYER_LINEAR_ATTENTION) > _STATIC_BYTES
    st = B.qwen35_gdn_state(0xA0000000, 0xB0000000)
    assert B.qwen35_forward_linear_attention_static(c, _fake_gdn(cfg), st, X, Y, _NO_STREAM) == \
        B.QWEN35_ERR_UNSUPPORTED
    # the size is judged on the config alone, before the pointers: an empty layer
    # and null state are still unsupported, not invalid
    assert B.qwen35_forward_linear_attention_static(c, B.qwen35_gdn_layer(), B.qwen35_gdn_state(0, 0), 0, 0,
                                                    _NO_STREAM) == B.QWEN35_ERR_UNSUPPORTED
    # the 4B shape fits
    c4 = B.make_config(synth.config("4b"))
    assert B.qwen35_scratch_bytes(c4, B.QWEN35_LAYER_LINEAR_ATTENTION) <= _STATIC_BYTES


@_no_device
def test_static_forward_and_status_without_a_device_fail_cleanly():
    cfg = synth.config("tiny")
    st = B.qwen35_gdn_state(0xA0000000, 0xB0000000)
    assert B.qwen35_forward_linear_attention_static(B.make_config(cfg), _fake_gdn(cfg), st, X, Y, _NO_STREAM) == \
        B.QWEN35_ERR_CUDA
    out = C.c_int32(7)
    assert B.lib().qwen35_read_static_status(C.byref(out), None) == B.QWEN35_ERR_CUDA
    assert out.value == 7


def test_static_status_needs_a_host_word():
    assert B.lib().qwen35_read_static_status(None, None) == B.QWEN35_ERR_INVALID_ARGUMENT


# ------------------------------------------------ the device-position and batched stack forms


def test_dpos_forward_argument_errors():
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    kv = B.qwen35_kv_cache(0xA0000000, 0xB0000000, 16)
    S = _Scratch(B.qwen35_scratch_bytes(c, B.QWEN35_LAYER_FULL_ATTENTION))
    f = B.qwen35_forward_full_attention_dpos
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    assert f(c, _fake_fa(cfg), S, kv, X, Y, None, 16, _NO_STREAM) == INV          # no device position
    assert f(c, _fake_fa(cfg), S, kv, X, Y, 0xC0000002, 16, _NO_STREAM) == INV    # misaligned int32
    assert f(c, _fake_fa(cfg), S, kv, X, Y, 0xC0000000, 0, _NO_STREAM) == INV     # no attention length bound
    assert f(c, _fake_fa(cfg), _Scratch(S.n - 16), kv, X, Y, 0xC0000000, 16, _NO_STREAM) == INV


def _stack(cfg):
    fa = _fake_fa(cfg)
    g = _fake_gdn(cfg)
    kv = B.qwen35_kv_cache(0xA0000000, 0xB0000000, 16)
    st = B.qwen35_gdn_state(0xA8000000, 0xB8000000)
    keep = (fa, g, kv, st)
    layers = [B.qwen35_layer(B.QWEN35_LAYER_LINEAR_ATTENTION, None, None, C.pointer(g), C.pointer(st)),
              B.qwen35_layer(B.QWEN35_LAYER_FULL_ATTENTION, C.pointer(fa), C.pointer(kv), None, None)]
    return layers, keep


def test_batched_decode_step_argument_errors():
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    layers, _keep = _stack(cfg)
    S2 = _Scratch(B.qwen35_stack_scratch_bytes_batched(c, 2))
    f = B.qwen35_decode_step_batched
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    pos = 0xC0000000
    assert f(c, layers, 0, S2, X, Y, pos, 16, _NO_STREAM) == INV               # empty batch
    assert f(c, layers, 9, S2, X, Y, pos, 16, _NO_STREAM) == INV               # above 8 sequences
    assert f(c, layers, 3, S2, X, Y, pos, 16, _NO_STREAM) == INV               # scratch sized for 2
    assert f(c, layers, 2, S2, X, Y, None, 16, _NO_STREAM) == INV              # a step advances positions
    assert f(c, layers, 2, S2, X, Y, pos + 2, 16, _NO_STREAM) == INV
    assert f(c, layers, 2, S2, X, Y, pos, 0, _NO_STREAM) == INV
    assert f(c, layers, 2, S2, X + 4, Y, pos, 16, _NO_STREAM) == INV
    assert f(c, [], 2, S2, X, Y, pos, 16, _NO_STREAM) == INV                   # no layers
    odd = [B.qwen35_layer(5, None, None, None, None)]
    assert f(c, odd, 2, S2, X, Y, pos, 16, _NO_STREAM) == INV                  # unknown layer kind
    # the batch scratch: the shared status block plus one block per sequence
    one, two = B.qwen35_stack_scratch_bytes_batched(c, 1), S2.n
    assert B.qwen35_stack_scratch_bytes_batched(c, 8) == one + 7 * (two - one)
    assert B.qwen35_stack_scratch_bytes_batched(c, 0) == 0 and B.qwen35_stack_scratch_bytes_batched(c, 9) == 0


@_no_device
def test_stack_forms_without_a_device_fail_cleanly():
    """The well-formed calls beside the rejected ones above pass every check and
    only then fail, at the first device query."""
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    kv = B.qwen35_kv_cache(0xA0000000, 0xB0000000, 16)
    S = _Scratch(B.qwen35_scratch_bytes(c, B.QWEN35_LAYER_FULL_ATTENTION))
    assert B.qwen35_forward_full_attention_dpos(c, _fake_fa(cfg), S, kv, X, Y, 0xC0000000, 16, _NO_STREAM) == \
        B.QWEN35_ERR_CUDA
    layers, _keep = _stack(cfg)
    S2 = _Scratch(B.qwen35_stack_scratch_bytes_batched(c, 2))
    assert B.qwen35_decode_step_batched(c, layers, 2, S2, X, Y, 0xC0000000, 16, _NO_STREAM) == B.QWEN35_ERR_CUDA


def test_graph_entries_argument_errors():
    """Graph creation checks its handle, its stream and the whole step before it
    begins a capture; launch and destroy reject a null graph."""
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    layers, _keep = _stack(cfg)
    arr = (B.qwen35_layer * len(layers))(*layers)
    S = _Scratch(B.qwen35_stack_scratch_bytes(c))
    L = B.lib()
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    h = C.c_void_p(0x1234)
    assert L.qwen35_graph_create(C.byref(c), arr, 2, S.addr, S.n, X, Y, 0xC0000000, 16, None, C.byref(h)) == INV
    assert h.value is None                                      # cleared on failure
    assert L.qwen35_graph_create(C.byref(c), arr, 2, S.addr, S.n, X, Y, 0xC0000000, 16, 0x5000, None) == INV
    assert L.qwen35_graph_create_batched(C.byref(c), arr, 2, 2, S.addr, S.n, X, Y, 0xC0000000, 16, None,
                                         C.byref(h)) == INV
    # a malformed step is rejected before the capture begins: the stream (a fake
    # handle here) is never used
    fake_stream = 0x5000
    small = _Scratch(S.n - 16)
    assert L.qwen35_graph_create(C.byref(c), arr, 2, small.addr, small.n, X, Y, 0xC0000000, 16, fake_stream,
                                 C.byref(h)) == INV
    assert L.qwen35_graph_create(C.byref(c), arr, 2, S.addr, S.n, X + 2, Y, 0xC0000000, 16, fake_stream,
                                 C.byref(h)) == INV
    assert L.qwen35_graph_create(C.byref(c), arr, 2, S.addr, S.n, X, Y, None, 16, fake_stream, C.byref(h)) == INV
    assert L.qwen35_graph_create_batched(C.byref(c), arr, 2, 9, S.addr, S.n, X, Y, 0xC0000000, 16, fake_stream,
                                         C.byref(h)) == INV
    assert h.value is None
    assert L.qwen35_graph_launch(None, None) == INV
    assert L.qwen35_graph_destroy(None) == INV


# ------------------------------------------------ component entries


def test_gemv_argument_errors():
    f = B.qwen35_gemv
    S = _Scratch(256)
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    w = _qw(1000, 2560, 1)
    assert f(w, X + 2, Y, S, _NO_STREAM) == INV                 # misaligned x
    assert f(w, X, Y + 2, S, _NO_STREAM) == INV                 # misaligned y
    assert f(w, X, Y, _Scratch(255), _NO_STREAM) == INV         # no room for the status block
    assert f(w, X, Y, _Scratch(256, 0x70000008), _NO_STREAM) == INV
    assert f(_qw(1000, 2560 + 32, 1), X, Y, S, _NO_STREAM) == INV   # k not whole groups
    assert f(_qw(0, 2560, 1), X, Y, S, _NO_STREAM) == INV
    w_mis = _qw(1000, 2560, 1)
    w_mis.scales += 2
    assert f(w_mis, X, Y, S, _NO_STREAM) == INV
    assert f(_qw(64, 12288 + 64, 1), X, Y, S, _NO_STREAM) == B.QWEN35_ERR_UNSUPPORTED


def test_dequant_argument_errors():
    L = B.lib()
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    w = _qw(300, 320, 1)
    assert L.qwen35_dequant(C.byref(w), None, None) == INV
    assert L.qwen35_dequant(None, 0xC0000000, None) == INV
    assert L.qwen35_dequant(C.byref(_qw(300, 100, 1)), 0xC0000000, None) == INV
    assert L.qwen35_dequant(C.byref(_qw(0, 320, 1)), 0xC0000000, None) == INV


@_no_device
def test_component_entries_without_a_device_fail_cleanly():
    L = B.lib()
    assert B.qwen35_gemv(_qw(1000, 2560, 1), X, Y, _Scratch(256), _NO_STREAM) == B.QWEN35_ERR_CUDA
    assert L.qwen35_dequant(C.byref(_qw(300, 320, 1)), 0xC0000000, None) == B.QWEN35_ERR_CUDA
    assert L.qwen35_scratch_init(0x70000000, 256, None) == B.QWEN35_ERR_CUDA
    out = C.c_int32(7)
    assert L.qwen35_read_device_status(0x70000000, C.byref(out), None) == B.QWEN35_ERR_CUDA
    assert out.value == 7


def test_status_word_entries_argument_errors():
    L = B.lib()
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    assert L.qwen35_scratch_init(0x70000008, 4096, None) == INV  # misaligned
    assert L.qwen35_scratch_init(0x70000000, 255, None) == INV   # below the status block
    assert L.qwen35_scratch_init(None, 4096, None) == INV
    out = C.c_int32(0)
    assert L.qwen35_read_device_status(0x70000000, None, None) == INV
    assert L.qwen35_read_device_status(0x70000004, C.byref(out), None) == INV


def test_debug_hooks_check_arguments_and_accept_their_defaults():
    L = B.lib()
    INV = B.QWEN35_ERR_INVALID_ARGUMENT
    assert L.qwen35_debug_trace(None, 4) == INV                 # a phase count without a buffer
    assert L.qwen35_debug_trace(0xC0000000, 0) == INV           # a buffer without a phase count
    assert L.qwen35_debug_wait_probe(0xC0000002) == INV          # the flag is a 32-bit word
    # the defaults: no trace, no probe, the default wait limit, no stage dumps
    assert L.qwen35_debug_trace(None, 0) == B.QWEN35_OK
    assert L.qwen35_debug_wait_probe(None) == B.QWEN35_OK
    assert L.qwen35_debug_set_wait_limit(0) == B.QWEN35_OK
    assert L.qwen35_debug_stage_dump(0) == B.QWEN35_OK
    assert L.qwen35_status_string(B.QWEN35_ERR_DEVICE_TIMEOUT) == b"device wait timed out"
    assert L.qwen35_status_string(12345) == b"unknown status"


# ------------------------------------------------ prefill head groups


@pytest.mark.parametrize("H,Hkv", [(3, 1), (16, 1), (12, 4)])
def test_prefill_rejects_head_groups_its_attention_lacks(H, Hkv):
    """The prefill's causal attention takes 1, 2, 4 or 8 q-heads per kv-head; other
    groups, which the single-token forward accepts, are unsupported before anything
    is enqueued (the layer and the stack form)."""
    cfg = synth.config("tiny")
    cfg["num_heads"], cfg["num_kv_heads"] = H, Hkv
    c = B.make_config(cfg)
    assert B.qwen35_scratch_bytes(c, B.QWEN35_LAYER_FULL_ATTENTION) > 0  # a valid decode config
    fa = _fake_fa(cfg)
    kv = B.qwen35_kv_cache(0xA0000000, 0xB0000000, 64)
    S = _Scratch(B.qwen35_prefill_scratch_bytes(c, 16))
    assert B.qwen35_prefill_full_attention(c, fa, S, kv, X, Y, 0, 16, _NO_STREAM) == B.QWEN35_ERR_UNSUPPORTED
    layers = [B.qwen35_layer(B.QWEN35_LAYER_FULL_ATTENTION, C.pointer(fa), C.pointer(kv), None, None)]
    arr = (B.qwen35_layer * 1)(*layers)
    assert B.lib().qwen35_prefill_step(C.byref(c), arr, 1, S.addr, S.n, X, Y, 0, 16, None) == \
        B.QWEN35_ERR_UNSUPPORTED


@_no_device
def test_prefill_accepts_supported_head_groups():
    for H, Hkv in [(4, 1), (8, 4), (8, 1), (4, 4)]:
        cfg = synth.config("tiny")
        cfg["num_heads"], cfg["num_kv_heads"] = H, Hkv
        c = B.make_config(cfg)
        kv = B.qwen35_kv_cache(0xA0000000, 0xB0000000, 64)
        S = _Scratch(B.qwen35_prefill_scratch_bytes(c, 16))
        assert B.qwen35_prefill_full_attention(c, _fake_fa(cfg), S, kv, X, Y, 0, 16, _NO_STREAM) == \
            B.QWEN35_ERR_CUDA, (H, Hkv)
