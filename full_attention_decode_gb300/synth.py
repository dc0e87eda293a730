"""Seeded synthetic inputs for the Qwen3.5 single-token decode layers.

This module only draws numbers: weights, KV-cache prefill, recurrent states and
per-step hidden vectors. It holds no step of the decode computation, so both the
CUDA path (through the tests and the benchmark) and the CPU oracle can take their
inputs from it without sharing any of the method's arithmetic.

Every tensor comes from its own numpy PCG64 stream keyed by (seed, tag), so any
single tensor of any layer can be regenerated on its own, bit-identically, on any
host. bf16 tensors are returned as uint16 bit patterns; fp32 tensors as float32.

Value recipe (the int8 group-64 affine format of the 4B "MLX-8bit" checkpoint
named on the module page, "Module qwen3_5"):
  codes    U{0..255}, row-major [n][k]
  scale    bf16(U(0.5, 1.5) * 0.02 / 127) per (row, group of 64 along k)
  bias     -128 * scale (exact in bf16)
  norms    bf16(1 + N(0, 0.1))
  dt_bias  bf16(N(0, 1));  A_log fp32 U(0, ln 16);  conv1d weight bf16(N(0, 0.5))
  x_in     bf16(N(0, 1)), fresh per decode step
  KV rows  bf16(N(0, 1)) for the prefilled tokens, zero above them
  GDN state fp32 N(0, std) (std 0 = zero-init), conv state zero
"""

from __future__ import annotations

import math
import zlib

import numpy as np

GROUP = 64


def gstride(k: int) -> int:
    """Row stride, in bf16 elements, of the scale and bias arrays of a [n][k] matrix.

    k/64 groups rounded up to a multiple of 8, so that every row of scales starts on
    a 16-byte boundary (the bulk-copy alignment); padding entries are zero.
    """
    return ((k // GROUP + 7) // 8) * 8


# Dimensions (the "Qwen35ForwardConfig" struct of the mod.rs page). "4b" is that
# page's qwen3_5_4b_mlx_int8 preset; "tiny" is the small correctness case;
# "tiny_alt" is a second small case with the other head dims the kernels are built
# for (attention 128 with one q-head per kv-head, linear attention 64).
CONFIGS = {
    "tiny": dict(hidden=256, intermediate=512, num_layers=2, vocab=0, group_size=64,
                 rms_eps=1e-6, num_heads=4, num_kv_heads=1, head_dim=64,
                 rope_theta=1e7, rotary_dim=16, num_k_heads_lin=2, num_v_heads_lin=4,
                 k_head_dim_lin=32, v_head_dim_lin=32, conv_kernel_size=4),
    "tiny_alt": dict(hidden=256, intermediate=512, num_layers=2, vocab=0, group_size=64,
                     rms_eps=1e-6, num_heads=3, num_kv_heads=3, head_dim=128,
                     rope_theta=1e7, rotary_dim=32, num_k_heads_lin=2, num_v_heads_lin=4,
                     k_head_dim_lin=64, v_head_dim_lin=64, conv_kernel_size=4),
    "4b": dict(hidden=2560, intermediate=9216, num_layers=32, vocab=248320, group_size=64,
               rms_eps=1e-6, num_heads=16, num_kv_heads=4, head_dim=256,
               rope_theta=1e7, rotary_dim=64, num_k_heads_lin=16, num_v_heads_lin=32,
               k_head_dim_lin=128, v_head_dim_lin=128, conv_kernel_size=4),
}


def config(name: str) -> dict:
    return dict(CONFIGS[name])


def layer_kinds(cfg: dict) -> list[str]:
    """Layer kinds of a stack: 'fa' (full attention) or 'gdn' (linear attention).

    The 4B-shape stack interleaves three GDN layers with one full-attention layer
    (layer i is full attention when i % 4 == 3). The two-layer tiny stack is
    GDN then full attention.
    """
    n = cfg["num_layers"]
    if n == 2:
        return ["gdn", "fa"]
    return ["fa" if i % 4 == 3 else "gdn" for i in range(n)]


def _rng(seed: int, *tags) -> np.random.Generator:
    tag = "/".join(str(t) for t in tags).encode()
    return np.random.default_rng(np.random.SeedSequence([seed & 0xFFFFFFFF, zlib.crc32(tag)]))


def to_bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (input generation only)."""
    b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def qweight(seed: int, tag: tuple, n: int, k: int) -> dict:
    """An int8 group-64 affine matrix [n][k]: codes, bf16 scales and biases."""
    assert k % GROUP == 0
    rng = _rng(seed, *tag)
    codes = rng.integers(0, 256, size=(n, k), dtype=np.uint8)
    g = k // GROUP
    s = to_bf16_bits(rng.uniform(0.5, 1.5, size=(n, g)) * (0.02 / 127.0))
    b = to_bf16_bits(-128.0 * bf16_bits_to_f32(s))
    gs = gstride(k)
    scales = np.zeros((n, gs), dtype=np.uint16)
    biases = np.zeros((n, gs), dtype=np.uint16)
    scales[:, :g] = s
    biases[:, :g] = b
    return {"codes": codes, "scales": scales, "biases": biases, "n": n, "k": k}


def _norm_w(seed, tag, n):
    return to_bf16_bits(1.0 + 0.1 * _rng(seed, *tag).standard_normal(n))


def fa_layer(seed: int, layer: int, cfg: dict) -> dict:
    """Weights of one full-attention layer (the FullAttentionLayer struct)."""
    E, I = cfg["hidden"], cfg["intermediate"]
    H, Hkv, D = cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    t = ("layer", layer)
    return {
        "input_ln": _norm_w(seed, t + ("input_ln",), E),
        "q_norm": _norm_w(seed, t + ("q_norm",), D),
        "k_norm": _norm_w(seed, t + ("k_norm",), D),
        "post_ln": _norm_w(seed, t + ("post_ln",), E),
        "q_proj": qweight(seed, t + ("q_proj",), 2 * H * D, E),
        "k_proj": qweight(seed, t + ("k_proj",), Hkv * D, E),
        "v_proj": qweight(seed, t + ("v_proj",), Hkv * D, E),
        "o_proj": qweight(seed, t + ("o_proj",), E, H * D),
        "gate_proj": qweight(seed, t + ("gate_proj",), I, E),
        "up_proj": qweight(seed, t + ("up_proj",), I, E),
        "down_proj": qweight(seed, t + ("down_proj",), E, I),
    }


def gdn_layer(seed: int, layer: int, cfg: dict) -> dict:
    """Weights of one linear-attention layer (the LinearAttentionLayer struct)."""
    E, I = cfg["hidden"], cfg["intermediate"]
    Hk, Hv = cfg["num_k_heads_lin"], cfg["num_v_heads_lin"]
    Dk, Dv, Kc = cfg["k_head_dim_lin"], cfg["v_head_dim_lin"], cfg["conv_kernel_size"]
    C = 2 * Hk * Dk + Hv * Dv
    t = ("layer", layer)
    return {
        "input_ln": _norm_w(seed, t + ("input_ln",), E),
        "a_log": _rng(seed, *t, "a_log").uniform(0.0, math.log(16.0), Hv).astype(np.float32),
        "dt_bias": to_bf16_bits(_rng(seed, *t, "dt_bias").standard_normal(Hv)),
        "conv1d_weight": to_bf16_bits(0.5 * _rng(seed, *t, "conv1d_weight").standard_normal((C, Kc))),
        "in_proj_a": qweight(seed, t + ("in_proj_a",), Hv, E),
        "in_proj_b": qweight(seed, t + ("in_proj_b",), Hv, E),
        "in_proj_qkv": qweight(seed, t + ("in_proj_qkv",), C, E),
        "in_proj_z": qweight(seed, t + ("in_proj_z",), Hv * Dv, E),
        "norm_weight": _norm_w(seed, t + ("norm_weight",), Dv),
        "out_proj": qweight(seed, t + ("out_proj",), E, Hv * Dv),
        "post_ln": _norm_w(seed, t + ("post_ln",), E),
        "gate_proj": qweight(seed, t + ("gate_proj",), I, E),
        "up_proj": qweight(seed, t + ("up_proj",), I, E),
        "down_proj": qweight(seed, t + ("down_proj",), E, I),
    }


def head(seed: int, cfg: dict, vocab: int | None = None) -> dict:
    """The model's output head: the final norm's weights (1 + N(0, 0.1)) and the
    lm_head matrix [vocab][hidden], int8 group-64 like every projection."""
    v = cfg["vocab"] if vocab is None else vocab
    return {"final_norm": _norm_w(seed, ("final_norm",), cfg["hidden"]),
            "lm_head": qweight(seed, ("lm_head",), v, cfg["hidden"])}


def x_in(seed: int, step: int, cfg: dict, seq: int = 0) -> np.ndarray:
    """The layer-0 hidden vector of one decode step, bf16 N(0, 1)."""
    return to_bf16_bits(_rng(seed, "x_in", seq, step).standard_normal(cfg["hidden"]))


def kv_cache(seed: int, layer: int, cfg: dict, capacity: int, n_prefill: int, seq: int = 0):
    """A bf16 KV cache [capacity][num_kv_heads][head_dim] with rows [0, n_prefill) N(0, 1)."""
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    k = np.zeros((capacity, Hkv, D), dtype=np.uint16)
    v = np.zeros((capacity, Hkv, D), dtype=np.uint16)
    if n_prefill:
        r = _rng(seed, "kv", seq, layer)
        k[:n_prefill] = to_bf16_bits(r.standard_normal((n_prefill, Hkv, D), dtype=np.float32))
        v[:n_prefill] = to_bf16_bits(r.standard_normal((n_prefill, Hkv, D), dtype=np.float32))
    return k, v


def kv_cache_turbo8(seed: int, layer: int, cfg: dict, capacity: int, n_prefill: int, seq: int = 0):
    """A Turbo8 KV cache (FP8 E4M3 codes [capacity][Hkv][D], bf16 scales
    [capacity][Hkv][D/16] for K and for V) with rows [0, n_prefill) drawn at random:
    codes U over the 254 finite E4M3 codes, scales bf16(U(0.5, 1.5) * 2 / 448) (the
    size a group of N(0, 1) values gets); zero above. Returns (k_codes, k_scales,
    v_codes, v_scales)."""
    Hkv, D = cfg["num_kv_heads"], cfg["head_dim"]
    out = []
    for part in ("k", "v"):
        codes = np.zeros((capacity, Hkv, D), dtype=np.uint8)
        scales = np.zeros((capacity, Hkv, D // 16), dtype=np.uint16)
        if n_prefill:
            r = _rng(seed, "kv_turbo8", part, seq, layer)
            c = r.integers(0, 254, size=(n_prefill, Hkv, D), dtype=np.int64)
            c = np.where(c >= 0x7F, c + 1, c)  # skip 0x7F (not a number); 0xFF is never drawn
            codes[:n_prefill] = c.astype(np.uint8)
            scales[:n_prefill] = to_bf16_bits(r.uniform(0.5, 1.5, size=(n_prefill, Hkv, D // 16)) * (2.0 / 448.0))
        out += [codes, scales]
    return tuple(out)


def gdn_state(seed: int, layer: int, cfg: dict, std: float = 0.0, seq: int = 0):
    """(conv_state fp32 [C][Kc] zero, gdn_state fp32 [Hv][Dk][Dv] N(0, std))."""
    Hk, Hv = cfg["num_k_heads_lin"], cfg["num_v_heads_lin"]
    Dk, Dv, Kc = cfg["k_head_dim_lin"], cfg["v_head_dim_lin"], cfg["conv_kernel_size"]
    C = 2 * Hk * Dk + Hv * Dv
    conv = np.zeros((C, Kc), dtype=np.float32)
    if std == 0.0:
        s = np.zeros((Hv, Dk, Dv), dtype=np.float32)
    else:
        s = (std * _rng(seed, "gdn_state", seq, layer).standard_normal((Hv, Dk, Dv))).astype(np.float32)
    return conv, s


def cache_positions(seed: int, batch: int, lo: int = 1024, hi: int = 65536) -> np.ndarray:
    """Per-sequence prefill lengths U{lo..hi} for the independent-sequences stack."""
    return _rng(seed, "cache_pos").integers(lo, hi + 1, size=batch).astype(np.int64)


# ---------------------------------------------------------------- paged KV layout


def block_table(seed: int, batch: int, n_logical: int, n_blocks: int) -> np.ndarray:
    """[batch][n_logical] distinct pool blocks drawn from [0, n_blocks), seeded (a
    shuffled placement, as a pool allocator would leave it)."""
    assert batch * n_logical <= n_blocks
    perm = _rng(seed, "block_table").permutation(n_blocks)[:batch * n_logical]
    return perm.reshape(batch, n_logical).astype(np.int32)


def paged_pool(caches: list, block_tokens: int, table: np.ndarray, n_blocks: int, fill: int) -> np.ndarray:
    """One pool [n_blocks][block_tokens][...] holding each logical cache caches[b]
    ([capacity][...], any dtype) block i at pool block table[b][i]; other blocks
    filled with `fill`."""
    c0 = np.asarray(caches[0])
    cap = c0.shape[0]
    assert cap % block_tokens == 0
    pool = np.full((n_blocks, block_tokens) + c0.shape[1:], fill, dtype=c0.dtype)
    for b, c in enumerate(caches):
        c = np.asarray(c).reshape((cap // block_tokens, block_tokens) + c0.shape[1:])
        pool[np.asarray(table[b])] = c
    return pool


def paged_gather(pool: np.ndarray, table_row, block_tokens: int) -> np.ndarray:
    """The logical cache [capacity][...] of one sequence back from a pool."""
    t = np.asarray(table_row)
    return pool[t].reshape((len(t) * block_tokens,) + pool.shape[2:])
