"""Python binding of the C ABI in include/qwen35_decode.h.

Argument marshalling only: the ctypes structs mirror the C structs, the
functions carry the C names and forward torch tensors' device pointers and the
current CUDA stream. Every step of the decode runs in the library's kernels.
Loading fails loudly when the library has not been built (there is no fallback).

Upload helpers turn the numpy weight dicts of `synth` into device tensors (torch
owns the memory) and the matching C structs.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libqwen35_decode.so")

QWEN35_OK = 0
QWEN35_PREFILL_GEMM_SPLIT_SCRATCH = 256 + 152 * 128 * 256 * 4  # include/qwen35_decode.h
QWEN35_ERR_INVALID_ARGUMENT = 1
QWEN35_ERR_OUT_OF_RANGE = 2
QWEN35_ERR_UNSUPPORTED = 3
QWEN35_ERR_CUDA = 4
QWEN35_ERR_DEVICE_TIMEOUT = 5
QWEN35_ERR_DEVICE_RANGE = 6
QWEN35_LAYER_FULL_ATTENTION = 0
QWEN35_LAYER_LINEAR_ATTENTION = 1


class Qwen35Error(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({_status_string(status)})")


class qwen35_config(C.Structure):
    _fields_ = [("hidden", C.c_uint32), ("intermediate", C.c_uint32), ("num_layers", C.c_uint32),
                ("vocab", C.c_uint32), ("group_size", C.c_uint32), ("rms_eps", C.c_float),
                ("num_heads", C.c_uint32), ("num_kv_heads", C.c_uint32), ("head_dim", C.c_uint32),
                ("rope_theta", C.c_float), ("rotary_dim", C.c_uint32),
                ("num_k_heads_lin", C.c_uint32), ("num_v_heads_lin", C.c_uint32),
                ("k_head_dim_lin", C.c_uint32), ("v_head_dim_lin", C.c_uint32),
                ("conv_kernel_size", C.c_uint32)]


class qwen35_qweight(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("biases", C.c_void_p),
                ("n", C.c_uint32), ("k", C.c_uint32)]


class qwen35_fa_layer(C.Structure):
    _fields_ = [("input_ln", C.c_void_p), ("q_norm", C.c_void_p), ("k_norm", C.c_void_p),
                ("post_ln", C.c_void_p)] + \
               [(n, qwen35_qweight) for n in ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj",
                                              "up_proj", "down_proj")]


class qwen35_gdn_layer(C.Structure):
    _fields_ = [("input_ln", C.c_void_p), ("a_log", C.c_void_p), ("dt_bias", C.c_void_p),
                ("conv1d_weight", C.c_void_p), ("in_proj_a", qwen35_qweight), ("in_proj_b", qwen35_qweight),
                ("in_proj_qkv", qwen35_qweight), ("in_proj_z", qwen35_qweight), ("norm_weight", C.c_void_p),
                ("out_proj", qwen35_qweight), ("post_ln", C.c_void_p), ("gate_proj", qwen35_qweight),
                ("up_proj", qwen35_qweight), ("down_proj", qwen35_qweight)]


QWEN35_KV_BF16 = 0
QWEN35_KV_TURBO8 = 1


class qwen35_kv_cache(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("capacity", C.c_uint32), ("dtype", C.c_uint32),
                ("k_scales", C.c_void_p), ("v_scales", C.c_void_p), ("block_table", C.c_void_p),
                ("block_tokens", C.c_uint32), ("reserved", C.c_uint32)]


class qwen35_gdn_state(C.Structure):
    _fields_ = [("conv_state", C.c_void_p), ("gdn_state", C.c_void_p)]


class qwen35_layer(C.Structure):
    _fields_ = [("kind", C.c_int32), ("fa", C.POINTER(qwen35_fa_layer)), ("kv", C.POINTER(qwen35_kv_cache)),
                ("gdn", C.POINTER(qwen35_gdn_layer)), ("state", C.POINTER(qwen35_gdn_state))]


_P = C.c_void_p
_U = C.c_uint32
_SIGS = {
    "qwen35_init": (C.c_int, []),
    "qwen35_status_string": (C.c_char_p, [C.c_int]),
    "qwen35_scratch_bytes": (C.c_size_t, [C.POINTER(qwen35_config), C.c_int]),
    "qwen35_stack_scratch_bytes": (C.c_size_t, [C.POINTER(qwen35_config)]),
    "qwen35_stack_scratch_bytes_batched": (C.c_size_t, [C.POINTER(qwen35_config), _U]),
    "qwen35_scratch_init": (C.c_int, [_P, C.c_size_t, _P]),
    "qwen35_read_device_status": (C.c_int, [_P, C.POINTER(C.c_int32), _P]),
    "qwen35_forward_full_attention": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_fa_layer), _P,
                                                C.c_size_t, C.POINTER(qwen35_kv_cache), _P, _P, _U, _U, _P]),
    "qwen35_forward_full_attention_dpos": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_fa_layer), _P,
                                                     C.c_size_t, C.POINTER(qwen35_kv_cache), _P, _P, _P, _U, _P]),
    "qwen35_forward_linear_attention": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_gdn_layer), _P,
                                                  C.c_size_t, C.POINTER(qwen35_gdn_state), _P, _P, _P]),
    "qwen35_forward_linear_attention_static": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_gdn_layer),
                                                         C.POINTER(qwen35_gdn_state), _P, _P, _P]),
    "qwen35_decode_step": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_layer), _U, _P, C.c_size_t,
                                     _P, _P, _P, _U, _P]),
    "qwen35_graph_create": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_layer), _U, _P, C.c_size_t,
                                      _P, _P, _P, _U, _P, C.POINTER(C.c_void_p)]),
    "qwen35_decode_step_batched": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_layer), _U, _U, _P,
                                             C.c_size_t, _P, _P, _P, _U, _P]),
    "qwen35_graph_create_batched": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_layer), _U, _U, _P,
                                              C.c_size_t, _P, _P, _P, _U, _P, C.POINTER(C.c_void_p)]),
    "qwen35_forward_full_attention_batched": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_fa_layer), _U,
                                                        _P, C.c_size_t, C.POINTER(qwen35_kv_cache), _P, _P, _P,
                                                        _U, _P]),
    "qwen35_forward_linear_attention_batched": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_gdn_layer),
                                                          _U, _P, C.c_size_t, C.POINTER(qwen35_gdn_state), _P, _P,
                                                          _P]),
    "qwen35_graph_launch": (C.c_int, [_P, _P]),
    "qwen35_graph_destroy": (C.c_int, [_P]),
    "qwen35_gemv": (C.c_int, [C.POINTER(qwen35_qweight), _P, _P, _P, C.c_size_t, _P]),
    "qwen35_dequant": (C.c_int, [C.POINTER(qwen35_qweight), _P, _P]),
    "qwen35_lm_head_greedy": (C.c_int, [C.POINTER(qwen35_config), _P, C.POINTER(qwen35_qweight), _P, _P, _P, _P,
                                        C.c_size_t, _P]),
    "qwen35_read_static_status": (C.c_int, [C.POINTER(C.c_int32), _P]),
    "qwen35_prefill_scratch_bytes": (C.c_size_t, [C.POINTER(qwen35_config), _U]),
    "qwen35_prefill_gemm": (C.c_int, [C.POINTER(qwen35_qweight), _P, _P, _U, C.c_int, _P, C.c_size_t, _P]),
    "qwen35_prefill_full_attention": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_fa_layer), _P,
                                                C.c_size_t, C.POINTER(qwen35_kv_cache), _P, _P, _U, _U, _P]),
    "qwen35_prefill_linear_attention": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_gdn_layer), _P,
                                                  C.c_size_t, C.POINTER(qwen35_gdn_state), _P, _P, _U, _P]),
    "qwen35_prefill_step": (C.c_int, [C.POINTER(qwen35_config), C.POINTER(qwen35_layer), _U, _P, C.c_size_t,
                                      _P, _P, _U, _U, _P]),
    "qwen35_debug_scratch_offset": (C.c_size_t, [C.POINTER(qwen35_config), C.c_int, C.c_char_p]),
    "qwen35_debug_stack_scratch_offset": (C.c_size_t, [C.POINTER(qwen35_config), C.c_char_p]),
    "qwen35_debug_stage_dump": (C.c_int, [C.c_int]),
    "qwen35_debug_set_wait_limit": (C.c_int, [C.c_ulonglong]),
    "qwen35_debug_wait_probe": (C.c_int, [_P]),
    "qwen35_debug_trace": (C.c_int, [_P, C.c_uint32]),
}

_lib = None


def lib():
    """The loaded library, with prototypes declared. Raises if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing (run __graft_entry__.build())")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            if not hasattr(L, name):  # a library without this entry fails when it is called
                continue
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def _status_string(s):
    try:
        return lib().qwen35_status_string(s).decode()
    except Exception:
        return "?"


def _check(fn, status):
    if status != QWEN35_OK:
        raise Qwen35Error(fn, status)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ C calls


def qwen35_init():
    _check("qwen35_init", lib().qwen35_init())


def make_config(cfg: dict) -> qwen35_config:
    return qwen35_config(**{f: cfg[f] for f, _ in qwen35_config._fields_})


def qwen35_scratch_bytes(cfg: qwen35_config, kind: int) -> int:
    return lib().qwen35_scratch_bytes(C.byref(cfg), kind)


def qwen35_stack_scratch_bytes(cfg: qwen35_config) -> int:
    return lib().qwen35_stack_scratch_bytes(C.byref(cfg))


def qwen35_stack_scratch_bytes_batched(cfg: qwen35_config, batch: int) -> int:
    return lib().qwen35_stack_scratch_bytes_batched(C.byref(cfg), batch)


def qwen35_scratch_init(scratch, stream=None):
    _check("qwen35_scratch_init", lib().qwen35_scratch_init(_ptr(scratch), scratch.numel(), _stream(stream)))


def qwen35_read_device_status(scratch, stream=None) -> int:
    out = C.c_int32(0)
    _check("qwen35_read_device_status", lib().qwen35_read_device_status(_ptr(scratch), C.byref(out),
                                                                          _stream(stream)))
    return out.value


def qwen35_forward_full_attention(cfg, layer, scratch, kv, x_in, x_out, cache_pos, seq_len_attn, stream=None):
    return lib().qwen35_forward_full_attention(C.byref(cfg), C.byref(layer), _ptr(scratch), scratch.numel(),
                                               C.byref(kv), _ptr(x_in), _ptr(x_out), cache_pos, seq_len_attn,
                                               _stream(stream))


def qwen35_forward_full_attention_dpos(cfg, layer, scratch, kv, x_in, x_out, d_cache_pos, max_seq_len,
                                       stream=None):
    return lib().qwen35_forward_full_attention_dpos(C.byref(cfg), C.byref(layer), _ptr(scratch),
                                                    scratch.numel(), C.byref(kv), _ptr(x_in), _ptr(x_out),
                                                    _ptr(d_cache_pos), max_seq_len, _stream(stream))


def qwen35_forward_linear_attention(cfg, layer, scratch, state, x_in, x_out, stream=None):
    return lib().qwen35_forward_linear_attention(C.byref(cfg), C.byref(layer), _ptr(scratch), scratch.numel(),
                                                 C.byref(state), _ptr(x_in), _ptr(x_out), _stream(stream))


def qwen35_forward_linear_attention_static(cfg, layer, state, x_in, x_out, stream=None):
    """The linear-attention forward on the library's static scratch (nothing allocated)."""
    return lib().qwen35_forward_linear_attention_static(C.byref(cfg), C.byref(layer), C.byref(state),
                                                        _ptr(x_in), _ptr(x_out), _stream(stream))


def qwen35_read_static_status(stream=None) -> int:
    """The device status word of the static scratch (after a stream synchronise)."""
    out = C.c_int32(0)
    _check("qwen35_read_static_status", lib().qwen35_read_static_status(C.byref(out), _stream(stream)))
    return out.value


def qwen35_decode_step(cfg, layers, scratch, x_in, x_out, d_cache_pos, max_seq_len, stream=None):
    arr = (qwen35_layer * len(layers))(*layers)
    return lib().qwen35_decode_step(C.byref(cfg), arr, len(layers), _ptr(scratch), scratch.numel(), _ptr(x_in),
                                    _ptr(x_out), _ptr(d_cache_pos), max_seq_len, _stream(stream))


def qwen35_decode_step_batched(cfg, layers, batch, scratch, x_in, x_out, d_cache_pos, max_seq_len, stream=None):
    arr = (qwen35_layer * len(layers))(*layers)
    return lib().qwen35_decode_step_batched(C.byref(cfg), arr, len(layers), batch, _ptr(scratch), scratch.numel(),
                                            _ptr(x_in), _ptr(x_out), _ptr(d_cache_pos), max_seq_len,
                                            _stream(stream))


def qwen35_forward_full_attention_batched(cfg, layer, batch, scratch, kv, x_in, x_out, d_cache_pos, max_seq_len,
                                          stream=None):
    return lib().qwen35_forward_full_attention_batched(C.byref(cfg), C.byref(layer), batch, _ptr(scratch),
                                                       scratch.numel(), C.byref(kv), _ptr(x_in), _ptr(x_out),
                                                       _ptr(d_cache_pos), max_seq_len, _stream(stream))


def qwen35_forward_linear_attention_batched(cfg, layer, batch, scratch, state, x_in, x_out, stream=None):
    return lib().qwen35_forward_linear_attention_batched(C.byref(cfg), C.byref(layer), batch, _ptr(scratch),
                                                         scratch.numel(), C.byref(state), _ptr(x_in), _ptr(x_out),
                                                         _stream(stream))


class Graph:
    """A captured decode step (qwen35_graph_create, or qwen35_graph_create_batched
    for batch > 1); replay with launch()."""

    def __init__(self, cfg, layers, scratch, x_in, x_out, d_cache_pos, max_seq_len, stream=None, batch: int = 1):
        arr = (qwen35_layer * len(layers))(*layers)
        h = C.c_void_p(0)
        if batch == 1:
            _check("qwen35_graph_create",
                   lib().qwen35_graph_create(C.byref(cfg), arr, len(layers), _ptr(scratch), scratch.numel(),
                                             _ptr(x_in), _ptr(x_out), _ptr(d_cache_pos), max_seq_len,
                                             _stream(stream), C.byref(h)))
        else:
            _check("qwen35_graph_create_batched",
                   lib().qwen35_graph_create_batched(C.byref(cfg), arr, len(layers), batch, _ptr(scratch),
                                                     scratch.numel(), _ptr(x_in), _ptr(x_out), _ptr(d_cache_pos),
                                                     max_seq_len, _stream(stream), C.byref(h)))
        self.handle = h

    def launch(self, stream=None):
        _check("qwen35_graph_launch", lib().qwen35_graph_launch(self.handle, _stream(stream)))

    def close(self):
        if self.handle:
            lib().qwen35_graph_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def qwen35_prefill_gemm(w, X, Y, n_tokens, scratch, stream=None, exact: bool = True):
    return lib().qwen35_prefill_gemm(C.byref(w), _ptr(X), _ptr(Y), n_tokens, 1 if exact else 0, _ptr(scratch),
                                     scratch.numel(), _stream(stream))


def qwen35_prefill_scratch_bytes(cfg: qwen35_config, max_tokens: int) -> int:
    return lib().qwen35_prefill_scratch_bytes(C.byref(cfg), max_tokens)


def qwen35_prefill_full_attention(cfg, layer, scratch, kv, x_in, x_out, cache_pos, n_tokens, stream=None):
    return lib().qwen35_prefill_full_attention(C.byref(cfg), C.byref(layer), _ptr(scratch), scratch.numel(),
                                               C.byref(kv), _ptr(x_in), _ptr(x_out), cache_pos, n_tokens,
                                               _stream(stream))


def qwen35_prefill_linear_attention(cfg, layer, scratch, state, x_in, x_out, n_tokens, stream=None):
    return lib().qwen35_prefill_linear_attention(C.byref(cfg), C.byref(layer), _ptr(scratch), scratch.numel(),
                                                 C.byref(state), _ptr(x_in), _ptr(x_out), n_tokens,
                                                 _stream(stream))


def qwen35_prefill_step(cfg, layers, scratch, x_in, x_out, cache_pos, n_tokens, stream=None):
    arr = (qwen35_layer * len(layers))(*layers)
    return lib().qwen35_prefill_step(C.byref(cfg), arr, len(layers), _ptr(scratch), scratch.numel(), _ptr(x_in),
                                     _ptr(x_out), cache_pos, n_tokens, _stream(stream))


def qwen35_gemv(w, x, y, scratch, stream=None):
    return lib().qwen35_gemv(C.byref(w), _ptr(x), _ptr(y), _ptr(scratch), scratch.numel(), _stream(stream))


def qwen35_lm_head_greedy(cfg, final_norm, lm_head, x, logits, token, scratch, stream=None):
    return lib().qwen35_lm_head_greedy(C.byref(cfg), _ptr(final_norm), C.byref(lm_head), _ptr(x), _ptr(logits),
                                       _ptr(token), _ptr(scratch), scratch.numel(), _stream(stream))


def qwen35_debug_scratch_offset(cfg, kind, name: str) -> int:
    return lib().qwen35_debug_scratch_offset(C.byref(cfg), kind, name.encode())


def qwen35_debug_stack_scratch_offset(cfg, name: str) -> int:
    return lib().qwen35_debug_stack_scratch_offset(C.byref(cfg), name.encode())


# the fused steps' values, stored as plain bf16 while the stage dump is on; every
# other named intermediate is a 32-bit word per element with the bf16 value in its
# high half
STAGE_DUMPS = ("x_norm", "x_norm2", "qkv_smooth", "y_norm", "k_rot", "v_rot")


def scratch_view(scratch: torch.Tensor, cfg, kind, name: str, n: int, seq: int = 0, seq_stride: int = 0) -> torch.Tensor:
    """The bf16 values of intermediate `name` (n elements) inside a scratch, as int16
    bits (a copy for the tagged words, a view for the stage dumps). kind None: the
    stack's layout; seq / seq_stride: sequence `seq` of a batch."""
    off = qwen35_debug_stack_scratch_offset(cfg, name) if kind is None else qwen35_debug_scratch_offset(cfg, kind, name)
    if off == C.c_size_t(-1).value:
        raise KeyError(name)
    off += seq * seq_stride
    if name in STAGE_DUMPS:
        return scratch[off:off + 2 * n].view(torch.int16)
    words = scratch[off:off + 4 * n].view(torch.int32)
    return (words >> 16).to(torch.int16)


def qwen35_debug_stage_dump(on: bool):
    return lib().qwen35_debug_stage_dump(1 if on else 0)


def qwen35_debug_set_wait_limit(limit_ns: int):
    """Bounded waits of later launches give up after limit_ns (0: the default, 1 s)."""
    return lib().qwen35_debug_set_wait_limit(limit_ns)


def qwen35_debug_wait_probe(flag):
    """Later launches first wait (bounded) on the device word `flag` (None: off)."""
    return lib().qwen35_debug_wait_probe(_ptr(flag))


def qwen35_debug_trace(buf, max_phases: int):
    """Record the phase timeline of later launches into buf (int64 device tensor), or stop (None, 0)."""
    return lib().qwen35_debug_trace(_ptr(buf), max_phases)


def qwen35_dequant(w, out, stream=None):
    return lib().qwen35_dequant(C.byref(w), _ptr(out), _stream(stream))


# ------------------------------------------------------------------ device uploads


def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy array -> device tensor of the same bits (uint16 stays int16 storage)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    return t.to(device)


class DeviceQWeight:
    def __init__(self, qw: dict, device="cuda"):
        self.codes = to_device(qw["codes"], device)
        self.scales = to_device(qw["scales"], device)
        self.biases = to_device(qw["biases"], device)
        self.n, self.k = qw["n"], qw["k"]

    def c(self) -> qwen35_qweight:
        return qwen35_qweight(self.codes.data_ptr(), self.scales.data_ptr(), self.biases.data_ptr(), self.n, self.k)


_FA_VEC = ("input_ln", "q_norm", "k_norm", "post_ln")
_FA_MAT = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")
_GDN_VEC = ("input_ln", "a_log", "dt_bias", "conv1d_weight", "norm_weight", "post_ln")
_GDN_MAT = ("in_proj_a", "in_proj_b", "in_proj_qkv", "in_proj_z", "out_proj", "gate_proj", "up_proj",
            "down_proj")


class DeviceFaLayer:
    """Device copy of a full-attention layer's weights plus its C struct."""

    def __init__(self, layer: dict, device="cuda"):
        self.t = {n: to_device(layer[n], device) for n in _FA_VEC}
        self.m = {n: DeviceQWeight(layer[n], device) for n in _FA_MAT}
        self.struct = qwen35_fa_layer(*[self.t[n].data_ptr() for n in _FA_VEC],
                                      *[self.m[n].c() for n in _FA_MAT])


class DeviceGdnLayer:
    """Device copy of a linear-attention layer's weights plus its C struct."""

    def __init__(self, layer: dict, device="cuda"):
        self.t = {n: to_device(layer[n], device) for n in _GDN_VEC}
        self.m = {n: DeviceQWeight(layer[n], device) for n in _GDN_MAT}
        t, m = self.t, self.m
        self.struct = qwen35_gdn_layer(
            t["input_ln"].data_ptr(), t["a_log"].data_ptr(), t["dt_bias"].data_ptr(), t["conv1d_weight"].data_ptr(),
            m["in_proj_a"].c(), m["in_proj_b"].c(), m["in_proj_qkv"].c(), m["in_proj_z"].c(),
            t["norm_weight"].data_ptr(), m["out_proj"].c(), t["post_ln"].data_ptr(), m["gate_proj"].c(),
            m["up_proj"].c(), m["down_proj"].c())


class DeviceKv:
    def __init__(self, k: np.ndarray, v: np.ndarray, device="cuda"):
        self.k = to_device(k, device)
        self.v = to_device(v, device)
        self.struct = qwen35_kv_cache(self.k.data_ptr(), self.v.data_ptr(), k.shape[0])


class DeviceState:
    """A linear-attention state on the device. `ssm` is given as [Hv][Dk][Dv] and
    stored in the library's column-block layout [Hv][Dv/32][Dk][32]."""

    def __init__(self, conv: np.ndarray, ssm: np.ndarray, device="cuda"):
        hv, dk, dv = ssm.shape
        self.shape = (hv, dk, dv)
        blocked = np.ascontiguousarray(ssm.reshape(hv, dk, dv // 32, 32).transpose(0, 2, 1, 3))
        self.conv = to_device(conv, device)
        self.ssm = to_device(blocked, device)
        self.struct = qwen35_gdn_state(self.conv.data_ptr(), self.ssm.data_ptr())

    def ssm_matrix(self):
        """The state as [Hv][Dk][Dv] (a device tensor)."""
        hv, dk, dv = self.shape
        return self.ssm.view(hv, dv // 32, dk, 32).permute(0, 2, 1, 3).reshape(hv, dk, dv)


def turbo8_sstride(cfg: dict) -> int:
    """Row stride, in bf16 elements, of a Turbo8 cache's scale arrays."""
    return ((cfg["num_kv_heads"] * cfg["head_dim"] // 16 + 7) // 8) * 8


def _pad_scales(s: np.ndarray, sstride: int) -> np.ndarray:
    """[..., cap, Hkv, D/16] bf16 scales -> [..., cap, sstride] (padded rows)."""
    flat = s.reshape(s.shape[:-2] + (-1,))
    out = np.zeros(flat.shape[:-1] + (sstride,), dtype=np.uint16)
    out[..., :flat.shape[-1]] = flat
    return out


class DeviceKvTurbo8:
    """A Turbo8 cache on the device from (k_codes, k_scales, v_codes, v_scales) with
    codes [cap][Hkv][D] and scales [cap][Hkv][D/16]; the scales are stored in rows
    padded to the library's stride."""

    def __init__(self, k_codes, k_scales, v_codes, v_scales, cfg: dict, device="cuda"):
        ss = turbo8_sstride(cfg)
        self.shape = k_scales.shape
        self.k = to_device(np.ascontiguousarray(k_codes), device)
        self.v = to_device(np.ascontiguousarray(v_codes), device)
        self.ks = to_device(_pad_scales(k_scales, ss), device)
        self.vs = to_device(_pad_scales(v_scales, ss), device)
        self.struct = qwen35_kv_cache(self.k.data_ptr(), self.v.data_ptr(), k_codes.shape[-3], QWEN35_KV_TURBO8,
                                      self.ks.data_ptr(), self.vs.data_ptr())

    def scales(self, which: str) -> np.ndarray:
        """The scales back as [..., cap, Hkv, D/16] bf16 bits."""
        t = self.ks if which == "k" else self.vs
        a = t.cpu().numpy().view(np.uint16)
        n = self.shape[-2] * self.shape[-1]
        return a[..., :n].reshape(a.shape[:-1] + self.shape[-2:])


class DeviceKvBatch:
    """KV caches of a batch of sequences, [B][capacity][Hkv][D] (one capacity)."""

    def __init__(self, ks: list, vs: list, device="cuda"):
        self.k = to_device(np.stack(ks), device)
        self.v = to_device(np.stack(vs), device)
        self.struct = qwen35_kv_cache(self.k.data_ptr(), self.v.data_ptr(), ks[0].shape[0])


class DeviceKvPaged:
    """Paged bf16 caches on the device: the logical caches ks[b], vs[b] ([cap][Hkv][D]
    bf16 bits) cut into blocks of `block_tokens` rows, placed in one pool of
    `n_blocks` blocks at the blocks `table` names ([B][cap / block_tokens]); the
    pool's other blocks hold `fill`."""

    def __init__(self, ks: list, vs: list, block_tokens: int, table, n_blocks: int, fill: int = 0x7FC0,
                 device="cuda"):
        from . import synth
        self.block_tokens = block_tokens
        self.table_np = np.ascontiguousarray(np.asarray(table, dtype=np.int32).reshape(len(ks), -1))
        self.k = to_device(synth.paged_pool(ks, block_tokens, self.table_np, n_blocks, fill), device)
        self.v = to_device(synth.paged_pool(vs, block_tokens, self.table_np, n_blocks, fill), device)
        self.table = torch.from_numpy(self.table_np).to(device)
        self.capacity = ks[0].shape[0]
        self.struct = qwen35_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.capacity, QWEN35_KV_BF16, None,
                                      None, self.table.data_ptr(), block_tokens, 0)

    def pool(self, which: str) -> np.ndarray:
        t = self.k if which == "k" else self.v
        return t.cpu().numpy().view(np.uint16)

    def logical(self, which: str, b: int = 0) -> np.ndarray:
        from . import synth
        return synth.paged_gather(self.pool(which), self.table_np[b], self.block_tokens)


class DeviceStateBatch:
    """Linear-attention states of a batch: conv [B][C][Kc], ssm in the column-block
    layout [B][Hv][Dv/32][Dk][32] (given per sequence as [Hv][Dk][Dv])."""

    def __init__(self, convs: list, ssms: list, device="cuda"):
        hv, dk, dv = ssms[0].shape
        self.shape = (hv, dk, dv)
        blocked = [np.ascontiguousarray(s.reshape(hv, dk, dv // 32, 32).transpose(0, 2, 1, 3)) for s in ssms]
        self.conv = to_device(np.stack(convs), device)
        self.ssm = to_device(np.stack(blocked), device)
        self.struct = qwen35_gdn_state(self.conv.data_ptr(), self.ssm.data_ptr())

    def ssm_matrix(self, b: int):
        hv, dk, dv = self.shape
        return self.ssm[b].view(hv, dv // 32, dk, 32).permute(0, 2, 1, 3).reshape(hv, dk, dv)


def stack_layer(kind: str, dev_layer, cache) -> qwen35_layer:
    """A qwen35_layer entry; the caller keeps dev_layer and cache alive."""
    if kind == "fa":
        return qwen35_layer(QWEN35_LAYER_FULL_ATTENTION, C.pointer(dev_layer.struct), C.pointer(cache.struct),
                            None, None)
    return qwen35_layer(QWEN35_LAYER_LINEAR_ATTENTION, None, None, C.pointer(dev_layer.struct),
                        C.pointer(cache.struct))


def new_scratch(nbytes: int, device="cuda", stream=None) -> torch.Tensor:
    """A scratch buffer (uint8, 256-byte aligned by the allocator) with its status word zeroed."""
    s = torch.empty(nbytes, dtype=torch.uint8, device=device)
    qwen35_scratch_init(s, stream)
    return s


def bf16_tensor_bits(t: torch.Tensor) -> np.ndarray:
    """Device int16/bf16 tensor -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
