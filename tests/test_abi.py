"""The C-ABI library without a GPU: it loads, exports every declared symbol, its
structs have the C layout, and argument errors are reported before any launch."""

import ctypes as C
import os
import re
import subprocess

import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qwen35_decode.h")


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"QWEN35_API\s+[\w\s\*]+?\b(qwen35_\w+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    L = B.lib()
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (qwen35_\w+)", out))
    assert set(names) <= exported
    # the binding declares a prototype for each of them
    assert set(names) == set(B.exported_symbols())


def test_struct_layout_matches_c_compiler(tmp_path):
    src = tmp_path / "layout.c"
    fields = {
        "qwen35_config": [f for f, _ in B.qwen35_config._fields_],
        "qwen35_qweight": [f for f, _ in B.qwen35_qweight._fields_],
        "qwen35_fa_layer": [f for f, _ in B.qwen35_fa_layer._fields_],
        "qwen35_gdn_layer": [f for f, _ in B.qwen35_gdn_layer._fields_],
        "qwen35_kv_cache": [f for f, _ in B.qwen35_kv_cache._fields_],
        "qwen35_gdn_state": [f for f, _ in B.qwen35_gdn_state._fields_],
        "qwen35_layer": [f for f, _ in B.qwen35_layer._fields_],
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void) {"]
    for s, fs in fields.items():
        lines.append(f'printf("{s} %zu\\n", sizeof({s}));')
        for f in fs:
            lines.append(f'printf("{s}.{f} %zu\\n", offsetof({s}, {f}));')
    lines.append("return 0; }")
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", str(src), "-o", str(exe)], check=True)
    got = dict(l.split() for l in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    for s, fs in fields.items():
        cls = getattr(B, s)
        assert int(got[s]) == C.sizeof(cls), s
        for f in fs:
            assert int(got[f"{s}.{f}"]) == getattr(cls, f).offset, (s, f)


def test_scratch_sizes():
    c4 = B.make_config(synth.config("4b"))
    fa = B.qwen35_scratch_bytes(c4, B.QWEN35_LAYER_FULL_ATTENTION)
    gdn = B.qwen35_scratch_bytes(c4, B.QWEN35_LAYER_LINEAR_ATTENTION)
    assert fa > 0 and gdn > 0
    # a stack keeps both kinds' intermediates apart: more than either kind alone
    assert max(fa, gdn) < B.qwen35_stack_scratch_bytes(c4) < fa + gdn
    assert B.qwen35_scratch_bytes(c4, 7) == 0
    bad = synth.config("4b")
    bad["group_size"] = 32
    assert B.qwen35_scratch_bytes(B.make_config(bad), 0) == 0
    bad = synth.config("4b")
    bad["head_dim"] = 96
    assert B.qwen35_scratch_bytes(B.make_config(bad), 0) == 0
    assert B.qwen35_scratch_bytes(B.make_config(bad), 1) > 0  # the GDN layer does not use head_dim


def test_debug_offsets():
    c = B.make_config(synth.config("tiny"))
    none = C.c_size_t(-1).value
    for n in ["q_full", "k", "v", "gated_attn", "o", "x_resid", "gate_act", "up_act"]:
        assert B.qwen35_debug_scratch_offset(c, 0, n) != none, n
    for n in ["dt_raw", "b_raw", "qkv", "z", "y", "out", "x_resid", "gate_act", "up_act"]:
        assert B.qwen35_debug_scratch_offset(c, 1, n) != none, n
    assert B.qwen35_debug_scratch_offset(c, 0, "qkv") == none
    assert B.qwen35_debug_scratch_offset(c, 1, "nope") == none
    # the fused steps' stage dumps (the page's intra_dump names)
    for n in ["x_norm", "x_norm2"]:
        assert B.qwen35_debug_scratch_offset(c, 0, n) != none, n
    for n in ["x_norm", "x_norm2", "qkv_smooth", "y_norm"]:
        assert B.qwen35_debug_scratch_offset(c, 1, n) != none, n
    assert B.qwen35_debug_scratch_offset(c, 0, "y_norm") == none
    # a stack's layout holds both kinds' names at distinct offsets, inside its scratch
    names = ["q_full", "k", "v", "gated_attn", "o", "dt_raw", "b_raw", "qkv", "z", "y", "out", "x_resid",
             "gate_act", "up_act", "x_norm", "x_norm2", "qkv_smooth", "y_norm"]
    offs = [B.qwen35_debug_stack_scratch_offset(c, n) for n in names]
    assert none not in offs and len(set(offs)) == len(offs)
    assert max(offs) < B.qwen35_stack_scratch_bytes(c)
    assert B.qwen35_debug_stack_scratch_offset(c, "nope") == none


# ---- argument validation with fake (never dereferenced) aligned pointers; skipped
# where a CUDA device is present, so that a check lost in a later change cannot let
# a fake address reach a kernel on a real GPU

_no_device = pytest.mark.skipif(torch.cuda.is_available(), reason="fake device addresses: run without a GPU")

_FAKE = 0x10000


def _fake_qw(n, k, base):
    return B.qwen35_qweight(base, base + 0x1000000, base + 0x2000000, n, k)


def _fake_fa(cfg):
    E, I, H, Hkv, D = cfg["hidden"], cfg["intermediate"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    shapes = [(2 * H * D, E), (Hkv * D, E), (Hkv * D, E), (E, H * D), (I, E), (I, E), (E, I)]
    qws = [_fake_qw(n, k, _FAKE * (i + 10) * 0x100) for i, (n, k) in enumerate(shapes)]
    return B.qwen35_fa_layer(_FAKE, _FAKE * 2, _FAKE * 3, _FAKE * 4, *qws)


class _FakeScratch:
    def __init__(self, n):
        self.n = n

    def numel(self):
        return self.n

    def data_ptr(self):
        return 0x7000000


@_no_device
def test_full_attention_argument_errors_precede_launch():
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    lay = _fake_fa(cfg)
    kv = B.qwen35_kv_cache(0x5000000, 0x6000000, 16)
    sb = B.qwen35_scratch_bytes(c, 0)
    S = _FakeScratch(sb)
    x, y = 0x8000000, 0x9000000
    f = B.qwen35_forward_full_attention
    assert f(c, lay, S, kv, x, y, 16, 17, 0) == B.QWEN35_ERR_OUT_OF_RANGE  # cache_pos >= capacity
    assert f(c, lay, S, kv, x, y, 3, 0, 0) == B.QWEN35_ERR_OUT_OF_RANGE    # empty attention
    assert f(c, lay, S, kv, x, y, 3, 5, 0) == B.QWEN35_ERR_OUT_OF_RANGE    # beyond cache_pos + 1
    assert f(c, lay, _FakeScratch(sb - 1), kv, x, y, 3, 4, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    assert f(c, lay, S, kv, x + 2, y, 3, 4, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # misaligned
    bad = _fake_fa(cfg)
    bad.down_proj.k = 256
    assert f(c, bad, S, kv, x, y, 3, 4, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # wrong shape
    bad = _fake_fa(cfg)
    bad.q_norm = None
    assert f(c, bad, S, kv, x, y, 3, 4, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    cb = synth.config("tiny")
    cb["rotary_dim"] = 15
    assert f(B.make_config(cb), lay, S, kv, x, y, 3, 4, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    cb = synth.config("tiny")
    cb["num_kv_heads"] = 3
    assert f(B.make_config(cb), lay, S, kv, x, y, 3, 4, 0) == B.QWEN35_ERR_INVALID_ARGUMENT


@_no_device
def test_linear_attention_and_stack_argument_errors():
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    g = B.qwen35_gdn_layer()
    st = B.qwen35_gdn_state(0x5000000, 0x6000000)
    S = _FakeScratch(B.qwen35_scratch_bytes(c, 1))
    assert B.qwen35_forward_linear_attention(c, g, S, st, 0x8000000, 0x9000000, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    cb = synth.config("tiny")
    cb["k_head_dim_lin"] = 48
    assert B.qwen35_forward_linear_attention(B.make_config(cb), g, S, st, 0x8000000, 0x9000000, 0) == \
        B.QWEN35_ERR_UNSUPPORTED
    bad_layer = B.qwen35_layer(9, None, None, None, None)
    assert B.qwen35_decode_step(c, [bad_layer], S, 0x8000000, 0x9000000, 0x100, 16, 0) == \
        B.QWEN35_ERR_INVALID_ARGUMENT
    assert B.lib().qwen35_status_string(2) == b"position out of range"


@_no_device
def test_lm_head_argument_errors_precede_launch():
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    E = cfg["hidden"]
    w = B.qwen35_qweight(0x1000000, 0x2000000, 0x3000000, 1000, E)
    S = _FakeScratch(4096)
    nw, x, logits, tok = 0x4000000, 0x5000000, 0x6000000, 0x7000000
    f = B.qwen35_lm_head_greedy
    assert f(c, nw, w, x + 2, logits, tok, S, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # misaligned x
    assert f(c, nw, w, x, logits, tok + 2, S, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # misaligned token
    assert f(c, None, w, x, logits, tok, S, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # no final norm
    assert f(c, nw, w, x, logits, tok, _FakeScratch(255), 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    bad = B.qwen35_qweight(0x1000000, 0x2000000, 0x3000000, 1000, E + 64)
    assert f(c, nw, bad, x, logits, tok, S, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # k != hidden
    empty = B.qwen35_qweight(0x1000000, 0x2000000, 0x3000000, 0, E)
    assert f(c, nw, empty, x, logits, tok, S, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # no vocabulary
    big = synth.config("tiny")
    big["hidden"] = 12288 + 64
    wbig = B.qwen35_qweight(0x1000000, 0x2000000, 0x3000000, 1000, 12288 + 64)
    assert f(B.make_config(big), nw, wbig, x, logits, tok, S, 0) == B.QWEN35_ERR_UNSUPPORTED


def test_well_formed_calls_without_a_device_fail_cleanly():
    """With no CUDA device the runtime's device queries fail: a call that passes
    every argument check returns QWEN35_ERR_CUDA (no crash, nothing launched)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    assert B.lib().qwen35_init() == B.QWEN35_ERR_CUDA
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    kv = B.qwen35_kv_cache(0x5000000, 0x6000000, 16)
    S = _FakeScratch(B.qwen35_scratch_bytes(c, 0))
    assert B.qwen35_forward_full_attention(c, _fake_fa(cfg), S, kv, 0x8000000, 0x9000000, 3, 4, 0) == \
        B.QWEN35_ERR_CUDA
    w = B.qwen35_qweight(0x1000000, 0x2000000, 0x3000000, 1000, cfg["hidden"])
    assert B.qwen35_lm_head_greedy(c, 0x4000000, w, 0x5000000, 0x6000000, 0x7000000, _FakeScratch(4096), 0) == \
        B.QWEN35_ERR_CUDA


@_no_device
def test_batched_layer_forwards_argument_errors():
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    fa = _fake_fa(cfg)
    kv = B.qwen35_kv_cache(_FAKE * 5, _FAKE * 6, 16)
    scr = _FakeScratch(B.qwen35_stack_scratch_bytes_batched(c, 2))
    L = B.lib()
    import ctypes as C
    # batch outside 1..8, missing positions, a misaligned vector: rejected before any launch
    for batch, dpos, x in [(0, _FAKE * 9, _FAKE * 7), (9, _FAKE * 9, _FAKE * 7), (2, None, _FAKE * 7),
                           (2, _FAKE * 9, _FAKE * 7 + 2)]:
        rc = L.qwen35_forward_full_attention_batched(C.byref(c), C.byref(fa), batch, scr.data_ptr(), scr.numel(),
                                                     C.byref(kv), x, _FAKE * 8, dpos, 16, None)
        assert rc == B.QWEN35_ERR_INVALID_ARGUMENT, (batch, dpos, x)
    # scratch too small for the batch
    small = _FakeScratch(B.qwen35_stack_scratch_bytes_batched(c, 1))
    rc = L.qwen35_forward_full_attention_batched(C.byref(c), C.byref(fa), 2, small.data_ptr(), small.numel(),
                                                 C.byref(kv), _FAKE * 7, _FAKE * 8, _FAKE * 9, 16, None)
    assert rc == B.QWEN35_ERR_INVALID_ARGUMENT
    rc = L.qwen35_forward_linear_attention_batched(C.byref(c), None, 2, scr.data_ptr(), scr.numel(), None,
                                                   _FAKE * 7, _FAKE * 8, None)
    assert rc == B.QWEN35_ERR_INVALID_ARGUMENT


@_no_device
def test_prefill_argument_errors_precede_launch():
    """Prefill entries: scratch sized per token count, range and format checks
    before anything is enqueued; a well-formed call without a device is a CUDA error."""
    import torch
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    s8, s16 = B.qwen35_prefill_scratch_bytes(c, 8), B.qwen35_prefill_scratch_bytes(c, 16)
    assert 0 < s8 < s16
    assert B.qwen35_prefill_scratch_bytes(c, 0) == 0 and B.qwen35_prefill_scratch_bytes(c, 65537) == 0
    fa = _fake_fa(cfg)
    kv = B.qwen35_kv_cache(_FAKE * 5, _FAKE * 6, 16)
    S = _FakeScratch(s8)
    x, y = _FAKE * 7, _FAKE * 8
    f = B.qwen35_prefill_full_attention
    assert f(c, fa, S, kv, x, y, 9, 8, 0) == B.QWEN35_ERR_OUT_OF_RANGE        # rows 9..16 past capacity 16
    assert f(c, fa, S, kv, x, y, 0, 9, 0) == B.QWEN35_ERR_INVALID_ARGUMENT    # scratch for 8 tokens
    assert f(c, fa, S, kv, x, y, 0, 0, 0) == B.QWEN35_ERR_INVALID_ARGUMENT    # no tokens
    assert f(c, fa, S, kv, x + 2, y, 0, 8, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    t8 = B.qwen35_kv_cache(_FAKE * 5, _FAKE * 6, 16, 1, None, _FAKE * 4)
    assert f(c, fa, S, t8, x, y, 0, 8, 0) == B.QWEN35_ERR_INVALID_ARGUMENT    # Turbo8 without k scales
    badpaged = B.qwen35_kv_cache(_FAKE * 5, _FAKE * 6, 16, 0, None, None, _FAKE * 2, 12)
    assert f(c, fa, S, badpaged, x, y, 0, 8, 0) == B.QWEN35_ERR_INVALID_ARGUMENT  # blocks not a power of 2
    g = B.qwen35_gdn_layer()
    st = B.qwen35_gdn_state(_FAKE * 5, _FAKE * 6)
    assert B.qwen35_prefill_linear_attention(c, g, S, st, x, y, 8, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    bad_layer = B.qwen35_layer(9, None, None, None, None)
    assert B.qwen35_prefill_step(c, [bad_layer], S, x, y, 0, 8, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    w = B.qwen35_qweight(_FAKE * 1, _FAKE * 2, _FAKE * 3, 100, 256)
    assert B.qwen35_prefill_gemm(w, x, y, 0, S, 0, True) == B.QWEN35_ERR_INVALID_ARGUMENT
    if not torch.cuda.is_available():
        assert f(c, fa, S, kv, x, y, 0, 8, 0) == B.QWEN35_ERR_CUDA
        assert B.qwen35_prefill_gemm(w, x, y, 4, S, 0, False) == B.QWEN35_ERR_CUDA
