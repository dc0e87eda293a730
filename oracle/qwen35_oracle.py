"""CPU oracle for the single-token Qwen3.5 decoder-layer forward.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this module:
only the tests, the smoke check and the benchmark's CPU-baseline leg use it. It
shares no code with the CUDA library; its only common ground with the GPU path is
the seeded input generator (full_attention_decode_gb300.synth), which holds none
of the method's arithmetic.

What it computes is written out from the two layer forwards printed on the pages
"full_attention.rs" (forward_full_attention) and "linear_attention.rs"
(forward_linear_attention), with the data types of the structs on "mod.rs".
Arithmetic is plain numpy float64, step by step in the pages' order, with no
fusion or reordering. A value is rounded to bf16 (round to nearest even) exactly
where the pages keep it in a bf16 buffer, and to fp32 where they keep it fp32
(gate, beta, conv1d_state, gdn_state). Where the pages leave a step open, the
reading taken is named in the docstring ("Reading: ...").

Pins (see tests/test_oracle_pins.py, tests/test_oracle_composition.py and
tests/test_oracle_turbo8.py): every function below is checked against closed
forms, special cases, library routines or brute force. None is unpinned.
"""

from __future__ import annotations

import numpy as np

GROUP = 64

# ----------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), as float64.

    bf16 keeps 8 significant bits and fp32's exponent range: the spacing of
    representable values around x is 2^(e-8) with x = m * 2^e, 0.5 <= |m| < 1,
    and never below the smallest subnormal step 2^-133. np.rint rounds half to even.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    step = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(x / step) * step
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > big, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


def bf16_bits(x) -> np.ndarray:
    """float64 values that are already bf16 values -> their uint16 bit patterns."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def f32_round(x) -> np.ndarray:
    """Round float64 to the nearest fp32 value (numpy's conversion is round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Quantised weights and the GEMV family
# ----------------------------------------------------------------------------


def dequant(qw: dict) -> np.ndarray:
    """Dequantise an int8 group-64 affine matrix to float64 [n][k].

    Reading (the QuantWeights format is not printed on the pages; the module page
    names the MLX-8bit checkpoint, group_size 64 on mod.rs): element (r, c) is
    scale[r][c // 64] * code[r][c] + bias[r][c // 64]. All three factors are exact
    in float64, so this is the exact real value of each weight.
    """
    n, k = qw["n"], qw["k"]
    g = k // GROUP
    codes = np.asarray(qw["codes"], dtype=np.float64).reshape(n, k)
    s = bf16_to_f64(qw["scales"])[:, :g]
    b = bf16_to_f64(qw["biases"])[:, :g]
    return codes * np.repeat(s, GROUP, axis=1) + np.repeat(b, GROUP, axis=1)


def gemv(w, x) -> np.ndarray:
    """y = W x (QuantWeights::gemv). `w` is a quantised matrix dict or a dequantised array."""
    W = dequant(w) if isinstance(w, dict) else w
    return W @ np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------
# Elementwise and normalisation
# ----------------------------------------------------------------------------


def sigmoid(x):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    """silu(a) = a * sigmoid(a)."""
    x = np.asarray(x, dtype=np.float64)
    return x * sigmoid(x)


def softplus(x):
    """softplus(x) = log(1 + e^x); for x > 20 it equals x to far below fp32 precision."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 20.0, x, np.log1p(np.exp(np.minimum(x, 20.0))))


def rms_norm(x, w, eps) -> np.ndarray:
    """RMSNorm over the last axis: x * w / sqrt(mean(x^2) + eps).

    Reading: every rms_norm launch on the pages passes the raw weight buffer and
    rms_eps, so the weight multiplies directly (not 1 + w) and eps sits inside the
    square root. Rows are independent (the per-head q/k norm "treats each head as a
    token" in full_attention.rs).
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def l2_norm_rows(x, eps) -> np.ndarray:
    """Per-row L2 normalisation x / sqrt(sum(x^2) + eps) (the conv kernel's l2 step, eps 1e-6)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


# ----------------------------------------------------------------------------
# Full-attention pieces (full_attention.rs)
# ----------------------------------------------------------------------------


def qkv_split(q_full, H: int, D: int):
    """De-interleave the q_proj output [H][2D] into (q [H][D], gate [H][D]).

    mod.rs, q_total: each head's row of the q_proj output is [Q_h | gate_h].
    """
    qf = np.asarray(q_full).reshape(H, 2 * D)
    return qf[:, :D].copy(), qf[:, D:].copy()


def rope_inv_freq(theta: float, R: int) -> np.ndarray:
    """inv_freq[i] = theta^(-2i/R), i < R/2, computed in float64 and kept as fp32.

    Reading: the pages pass inv_freq as a device buffer without printing its
    values; this is the standard RoPE frequency table over the rotated dims.
    """
    i = np.arange(R // 2, dtype=np.float64)
    return f32_round(np.power(float(theta), -2.0 * i / R))


def rope_apply(x, pos: int, inv_freq, R: int) -> np.ndarray:
    """Rotate the first R dims of each row of x [heads][D] at position pos.

    mod.rs, rotary_dim: only the first rotary_dim elements of each head rotate; the
    rest pass through. Reading: rotate-half pairing, (x[i], x[i + R/2]) for i < R/2.
    The angle is the fp32 product fp32(pos) * inv_freq[i] (one rounding, as a
    kernel computing in fp32 forms it); its cos and sin are then taken exactly.
    """
    x = np.asarray(x, dtype=np.float64)
    half = R // 2
    ang = f32_round(np.float64(np.float32(pos)) * np.asarray(inv_freq, dtype=np.float64))
    c, s = np.cos(ang), np.sin(ang)
    out = x.copy()
    a, b = x[..., :half], x[..., half:R]
    out[..., :half] = a * c - b * s
    out[..., half:R] = b * c + a * s
    return out


def attention_decode(q, k_cache, v_cache, S: int, Hkv: int) -> np.ndarray:
    """Single-query GQA attention over cached tokens [0, S) (attention_decode).

    q [H][D]; k_cache, v_cache [>=S][Hkv][D]. Scale 1/sqrt(D) (full_attention.rs
    computes it from head_dim). Reading: q-head h reads kv-head h // (H / Hkv)
    (contiguous groups); an exact softmax, no window, no sparsity threshold.
    """
    q = np.asarray(q, dtype=np.float64)
    H, D = q.shape
    grp = H // Hkv
    scale = 1.0 / np.sqrt(np.float64(D))
    out = np.zeros((H, D))
    for h in range(H):
        g = h // grp
        K = np.asarray(k_cache[:S, g, :], dtype=np.float64)
        V = np.asarray(v_cache[:S, g, :], dtype=np.float64)
        sc = (K @ q[h]) * scale
        p = np.exp(sc - sc.max())
        out[h] = (p @ V) / p.sum()
    return out


# ----------------------------------------------------------------------------
# Linear-attention (Gated DeltaNet) pieces (linear_attention.rs)
# ----------------------------------------------------------------------------


def causal_conv1d_update(conv_state, x, w):
    """One decode step of the depthwise causal conv: returns (new_state, conv_out).

    conv_state fp32 [C][Kc] (mod.rs, LinearAttentionState), x [C], w [C][Kc].
    Reading: the state keeps the last Kc inputs in time order with the newest in
    slot Kc-1; the step shifts it left, appends x, and outputs
    sum_j w[c][j] * state[c][j]. A zeroed state is the conv's left zero padding.
    """
    st = np.asarray(conv_state, dtype=np.float64)
    new = np.concatenate([st[:, 1:], np.asarray(x, dtype=np.float64)[:, None]], axis=1)
    out = np.sum(np.asarray(w, dtype=np.float64) * new, axis=1)
    return new, out


def gdn_gate(dt_raw, dt_bias, a_log) -> np.ndarray:
    """gate = exp(softplus(dt + dt_bias) * -exp(A_log)), kept fp32 (linear_attention.rs)."""
    return f32_round(np.exp(softplus(np.asarray(dt_raw, np.float64) + np.asarray(dt_bias, np.float64))
                            * -np.exp(np.asarray(a_log, np.float64))))


def gdn_beta(b_raw) -> np.ndarray:
    """beta = sigmoid(b_raw), kept fp32 (linear_attention.rs)."""
    return f32_round(sigmoid(b_raw))


def gated_delta_rule(state, q, k, v, g, beta, Dk: int):
    """One step of the gated delta rule for all v-heads; returns (new_state, y).

    state [Hv][Dk][Dv]; q, k [Hk][Dk]; v [Hv][Dv]; g, beta [Hv].
    Reading (the kernel is only named on the pages; the published Gated DeltaNet
    recurrence): v-head h uses k-head h // (Hv / Hk); the state decays by g, the
    delta rule writes k (x) beta * (v - S^T k) against the decayed state, and the
    readout S^T q of the updated state is scaled by 1/sqrt(Dk), the query scale
    linear_attention.rs says gated_delta_rule_decode applies to its output.
    """
    S = np.asarray(state, dtype=np.float64).copy()
    Hv = S.shape[0]
    Hk = np.asarray(q).shape[0]
    grp = Hv // Hk
    y = np.zeros((Hv, S.shape[2]))
    for h in range(Hv):
        j = h // grp
        kj = np.asarray(k[j], dtype=np.float64)
        qj = np.asarray(q[j], dtype=np.float64)
        Sh = g[h] * S[h]
        u = Sh.T @ kj
        Sh = Sh + np.outer(kj, beta[h] * (np.asarray(v[h], dtype=np.float64) - u))
        S[h] = Sh
        y[h] = (Sh.T @ qj) / np.sqrt(np.float64(Dk))
    return S, y


# ----------------------------------------------------------------------------
# Turbo8 KV cache (mod.rs: MetalKvDtype::Turbo8; full_attention.rs: Turbo path)
# ----------------------------------------------------------------------------

E4M3_MAX = 448.0  # the largest finite FP8 E4M3 value, 1.75 * 2^8


def wht(x) -> np.ndarray:
    """Orthonormal Walsh-Hadamard transform along the last axis (length a power of 2).

    full_attention.rs rotates K and V before the Turbo append, Q before attention
    and the attention output back after it (wht / wht_inv). Reading: the Sylvester
    ordering H_2n = [[H, H], [H, -H]] with the orthonormal factor 1/sqrt(n), so the
    transform is its own inverse and keeps dot products (the pages name no
    normalisation; this is the one under which rotating both q and K leaves the
    scores unchanged). Written as the butterfly: each stage pairs elements h apart.
    """
    y = np.array(x, dtype=np.float64, copy=True)
    n = y.shape[-1]
    h = 1
    while h < n:
        a = y.reshape(y.shape[:-1] + (n // (2 * h), 2, h))
        lo = a[..., 0, :].copy()
        hi = a[..., 1, :].copy()
        a[..., 0, :] = lo + hi
        a[..., 1, :] = lo - hi
        h *= 2
    return y / np.sqrt(np.float64(n))


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value, ties to even, saturating at +-448.

    E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; normal values
    (1 + m/8) 2^(e-7) for e = 1..15 (e = 15, m = 7 is not a number, so 448 is the
    largest finite value), subnormal values (m/8) 2^-6. Reading (the pages print
    the format, not its rounding): round to nearest even with saturation to the
    largest finite value (no infinities or NaN from finite inputs).
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                 # a = f 2^e, 0.5 <= f < 1; the binade's step is 2^(e-4)
    step = np.ldexp(1.0, np.maximum(e - 4, -9))   # subnormal step 2^-9
    r = np.rint(a / step) * step
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def e4m3_bits(x) -> np.ndarray:
    """E4M3 values (already representable) -> their 8-bit codes."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    sign = (np.signbit(x)).astype(np.uint8) << 7
    _, e = np.frexp(a)
    exp = np.clip(e - 1 + 7, 0, 15)              # biased exponent of a normal value
    normal = (a >= 2.0 ** -6)
    mant_n = np.where(normal, np.rint((a / np.ldexp(1.0, e - 1) - 1.0) * 8), 0)
    mant_s = np.rint(a / 2.0 ** -9)              # subnormal: a = m 2^-9
    code = np.where(normal, (exp.astype(np.int64) << 3) | mant_n.astype(np.int64), mant_s.astype(np.int64))
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_value(bits) -> np.ndarray:
    """8-bit E4M3 codes -> values (code 0x7F / 0xFF, not a number, never produced here)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    return s * v


def turbo8_quantize(x):
    """Quantise rows of bf16 values in groups of 16: (E4M3 codes, bf16 scales).

    mod.rs, Turbo8: FP8 E4M3 data and a BF16 scale per group of 16 (1.125 bytes per
    element). Reading (the pages do not print the kernel): the group's scale is
    bf16(fp32(amax / 448)), so that the largest element maps to the top of the E4M3
    range, and each element's code is the E4M3 rounding of the fp32 quotient
    fp32(x / scale); a group of zeros has scale 0 and codes 0. The quotient is
    formed in fp32 because that is the precision the kernel decides the code in.
    Returns (codes uint8 [..., n], scales float64 [..., n / 16] holding bf16 values).
    """
    x = np.asarray(x, dtype=np.float64)
    g = x.reshape(x.shape[:-1] + (x.shape[-1] // 16, 16))
    amax = np.max(np.abs(g), axis=-1)
    scale = bf16_round(f32_round(amax / E4M3_MAX))
    safe = np.where(scale > 0, scale, 1.0)
    q = f32_round(g.astype(np.float32).astype(np.float64) / safe[..., None])
    q = np.where(scale[..., None] > 0, q, 0.0)
    codes = e4m3_bits(e4m3_round(q))
    return codes.reshape(x.shape), scale


def turbo8_dequantize(codes, scales) -> np.ndarray:
    """codes [..., n] and bf16 scales [..., n / 16] -> values code * scale (exact in float64)."""
    v = e4m3_value(codes)
    s = np.asarray(scales, dtype=np.float64)
    return (v.reshape(s.shape + (16,)) * s[..., None]).reshape(v.shape)


# ----------------------------------------------------------------------------
# The two layer forwards
# ----------------------------------------------------------------------------


def _W(layer: dict, name: str):
    """Dequantised matrix of a layer, cached in the layer dict (plain memoisation)."""
    key = "_deq_" + name
    if key not in layer:
        layer[key] = dequant(layer[name])
    return layer[key]


def forward_full_attention(cfg: dict, layer: dict, kv: dict, x_in, cache_pos: int,
                           seq_len_attn: int, trace: dict | None = None) -> np.ndarray:
    """Single-token full-attention decoder layer (full_attention.rs, forward_full_attention).

    kv = {"k": [cap][Hkv][D], "v": ...} float64 arrays holding bf16 values; row
    cache_pos is overwritten (the KV append). x_in holds bf16 values. Returns x_out
    (bf16 values). The steps follow the page in order; bf16 roundings sit where the
    page writes a bf16 scratch buffer.
    """
    E, eps = cfg["hidden"], cfg["rms_eps"]
    H, Hkv, D, R = cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"], cfg["rotary_dim"]
    x_in = np.asarray(x_in, dtype=np.float64)
    t = trace if trace is not None else {}

    # norm1
    x_norm = bf16_round(rms_norm(x_in, bf16_to_f64(layer["input_ln"]), eps))
    # q_proj; fused k_proj + v_proj on the same x_norm
    q_full = bf16_round(gemv(_W(layer, "q_proj"), x_norm))
    k = bf16_round(gemv(_W(layer, "k_proj"), x_norm))
    v = bf16_round(gemv(_W(layer, "v_proj"), x_norm))
    # qkv split: [Q_h | gate_h] per head
    q, gate = qkv_split(q_full, H, D)
    # per-head q/k RMSNorm
    q_n = bf16_round(rms_norm(q, bf16_to_f64(layer["q_norm"]), eps))
    k_n = bf16_round(rms_norm(k.reshape(Hkv, D), bf16_to_f64(layer["k_norm"]), eps))
    # partial RoPE at the token's position (in place on the bf16 buffers)
    inv_freq = rope_inv_freq(cfg["rope_theta"], R)
    q_r = bf16_round(rope_apply(q_n, cache_pos, inv_freq, R))
    k_r = bf16_round(rope_apply(k_n, cache_pos, inv_freq, R))
    if kv.get("dtype") == "turbo8":
        # Turbo path: K and V rotated (bf16, in place on the page) before the
        # quantising append, Q rotated before attention; the dequantising attention
        # runs in the rotated basis and its output is rotated back (bf16 each time).
        # Reading: no sparse-V gate (the page's threshold 0.0 disables it).
        k_rot = bf16_round(wht(k_r))
        v_rot = bf16_round(wht(v.reshape(Hkv, D)))
        kc, ks = turbo8_quantize(k_rot)
        vc, vs = turbo8_quantize(v_rot)
        kv["k_codes"][cache_pos], kv["k_scales"][cache_pos] = kc, ks
        kv["v_codes"][cache_pos], kv["v_scales"][cache_pos] = vc, vs
        q_rot = bf16_round(wht(q_r))
        K = turbo8_dequantize(kv["k_codes"][:seq_len_attn], kv["k_scales"][:seq_len_attn])
        V = turbo8_dequantize(kv["v_codes"][:seq_len_attn], kv["v_scales"][:seq_len_attn])
        attn_rot = bf16_round(attention_decode(q_rot, K, V, seq_len_attn, Hkv))
        attn = bf16_round(wht(attn_rot))
        t.update(k_rot=k_rot, v_rot=v_rot, q_rot=q_rot, attn_rot=attn_rot)
    else:
        # KV append at cache_pos (bf16 cache), then attention over seq_len_attn tokens
        kv["k"][cache_pos] = k_r
        kv["v"][cache_pos] = v.reshape(Hkv, D)
        attn = bf16_round(attention_decode(q_r, kv["k"], kv["v"], seq_len_attn, Hkv))
    # sigmoid gate
    gated = bf16_round(attn * sigmoid(gate))
    # o_proj
    o = bf16_round(gemv(_W(layer, "o_proj"), gated.reshape(-1)))
    # residual + post-attention RMSNorm
    x_resid = bf16_round(x_in + o)
    x_norm2 = bf16_round(rms_norm(x_resid, bf16_to_f64(layer["post_ln"]), eps))
    # gate/up dual GEMV, then down_proj with SiLU gate and residual
    g = bf16_round(gemv(_W(layer, "gate_proj"), x_norm2))
    u = bf16_round(gemv(_W(layer, "up_proj"), x_norm2))
    x_out = bf16_round(x_resid + gemv(_W(layer, "down_proj"), silu(g) * u))

    t.update(x_norm=x_norm, q_full=q_full, k=k, v=v, q_rope=q_r, k_rope=k_r, attn_out=attn,
             gated_attn=gated, o=o, x_resid=x_resid, x_norm2=x_norm2, gate_act=g, up_act=u,
             x_out=x_out)
    return x_out


def forward_linear_attention(cfg: dict, layer: dict, state: dict, x_in,
                             trace: dict | None = None) -> np.ndarray:
    """Single-token GDN decoder layer (linear_attention.rs, forward_linear_attention).

    state = {"conv": fp32 [C][Kc], "ssm": fp32 [Hv][Dk][Dv]} as float64 arrays
    holding fp32 values; both are updated in place. Returns x_out (bf16 values).
    """
    E, eps = cfg["hidden"], cfg["rms_eps"]
    Hk, Hv = cfg["num_k_heads_lin"], cfg["num_v_heads_lin"]
    Dk, Dv = cfg["k_head_dim_lin"], cfg["v_head_dim_lin"]
    x_in = np.asarray(x_in, dtype=np.float64)
    t = trace if trace is not None else {}

    x_norm = bf16_round(rms_norm(x_in, bf16_to_f64(layer["input_ln"]), eps))
    # in_proj_a / in_proj_b (dual GEMV), in_proj_qkv, in_proj_z
    dt_raw = bf16_round(gemv(_W(layer, "in_proj_a"), x_norm))
    b_raw = bf16_round(gemv(_W(layer, "in_proj_b"), x_norm))
    qkv = bf16_round(gemv(_W(layer, "in_proj_qkv"), x_norm))
    z = bf16_round(gemv(_W(layer, "in_proj_z"), x_norm))
    # causal conv update + SiLU on every channel; L2 norm per head on Q and K only
    new_conv, conv_out = causal_conv1d_update(state["conv"], qkv,
                                              bf16_to_f64(layer["conv1d_weight"]))
    state["conv"] = f32_round(new_conv)
    act = silu(conv_out)
    nqk = Hk * Dk
    qn = l2_norm_rows(act[:nqk].reshape(Hk, Dk), 1e-6)
    kn = l2_norm_rows(act[nqk:2 * nqk].reshape(Hk, Dk), 1e-6)
    qkv_smooth = bf16_round(np.concatenate([qn.reshape(-1), kn.reshape(-1), act[2 * nqk:]]))
    q = qkv_smooth[:nqk].reshape(Hk, Dk)
    k = qkv_smooth[nqk:2 * nqk].reshape(Hk, Dk)
    v = qkv_smooth[2 * nqk:].reshape(Hv, Dv)
    # decay gate and beta (fp32)
    g = gdn_gate(dt_raw, bf16_to_f64(layer["dt_bias"]), np.asarray(layer["a_log"], np.float64))
    beta = gdn_beta(b_raw)
    # gated delta rule (state read-modify-write in fp32 storage)
    S_new, y = gated_delta_rule(state["ssm"], q, k, v, g, beta, Dk)
    state["ssm"] = f32_round(S_new)
    y = bf16_round(y)
    # per-v-head RMSNorm, then out_proj(silu(z) * y_norm)
    y_norm = bf16_round(rms_norm(y, bf16_to_f64(layer["norm_weight"]), eps))
    out = bf16_round(gemv(_W(layer, "out_proj"), silu(z) * y_norm.reshape(-1)))
    # residual + post norm, MLP with residual
    x_resid = bf16_round(x_in + out)
    x_norm2 = bf16_round(rms_norm(x_resid, bf16_to_f64(layer["post_ln"]), eps))
    ga = bf16_round(gemv(_W(layer, "gate_proj"), x_norm2))
    ua = bf16_round(gemv(_W(layer, "up_proj"), x_norm2))
    x_final = bf16_round(x_resid + gemv(_W(layer, "down_proj"), silu(ga) * ua))

    t.update(x_norm=x_norm, dt_raw=dt_raw, b_raw=b_raw, qkv=qkv, z=z, qkv_smooth=qkv_smooth,
             gate=g, beta=beta, y=y.reshape(-1), y_norm=y_norm.reshape(-1), out=out,
             x_resid=x_resid, x_norm2=x_norm2, gate_act=ga, up_act=ua, x_out=x_final)
    return x_final


# ----------------------------------------------------------------------------
# Stack step
# ----------------------------------------------------------------------------


def decode_step(cfg: dict, kinds: list, layers: list, caches: list, x_in, cache_pos: int,
                layer_outputs: list | None = None) -> np.ndarray:
    """One token through a stack of layers: layer i's x_out is layer i+1's x_in.

    Reading: the pages leave the layer loop to the caller; a full-attention layer
    appends at cache_pos and attends over cache_pos + 1 tokens. caches[i] is a KV
    dict for 'fa' layers and a state dict for 'gdn' layers.
    """
    x = np.asarray(x_in, dtype=np.float64)
    for kind, layer, c in zip(kinds, layers, caches):
        if kind == "fa":
            x = forward_full_attention(cfg, layer, c, x, cache_pos, cache_pos + 1)
        else:
            x = forward_linear_attention(cfg, layer, c, x)
        if layer_outputs is not None:
            layer_outputs.append(x.copy())
    return x


# ----------------------------------------------------------------------------
# Multi-token prefill
# ----------------------------------------------------------------------------


def prefill_full_attention(cfg: dict, layer: dict, kv: dict, X, cache_pos: int,
                           traces: list | None = None) -> np.ndarray:
    """A prompt of T tokens (X [T][E], bf16 values) through a full-attention layer.

    Reading: the pages keep prefill out of the single-token path (page "Module
    qwen3_5", non-goals: multi-token prefill) and print no prefill kernel, so its
    result is fixed by the decode forward itself: token t of the prompt sits at
    position cache_pos + t, appends its K/V row there and attends over
    cache_pos + t + 1 tokens, after tokens 0 .. t-1 have done the same. The prompt
    is that forward applied token after token. Returns x_out [T][E].
    """
    X = np.asarray(X, dtype=np.float64)
    out = np.empty_like(X)
    for t in range(X.shape[0]):
        tr = {} if traces is not None else None
        out[t] = forward_full_attention(cfg, layer, kv, X[t], cache_pos + t, cache_pos + t + 1, tr)
        if traces is not None:
            traces.append(tr)
    return out


def prefill_linear_attention(cfg: dict, layer: dict, state: dict, X, traces: list | None = None) -> np.ndarray:
    """A prompt of T tokens through a linear-attention layer: the single-token forward
    token after token, the conv and delta-rule states carried from one to the next
    (the same reading as prefill_full_attention). Returns x_out [T][E]."""
    X = np.asarray(X, dtype=np.float64)
    out = np.empty_like(X)
    for t in range(X.shape[0]):
        tr = {} if traces is not None else None
        out[t] = forward_linear_attention(cfg, layer, state, X[t], tr)
        if traces is not None:
            traces.append(tr)
    return out


def prefill_step(cfg: dict, kinds: list, layers: list, caches: list, X, cache_pos: int,
                 layer_outputs: list | None = None) -> np.ndarray:
    """A prompt through a stack, layer by layer over all T tokens: layer i's outputs
    for the prompt are layer i+1's inputs. Token t of layer i depends only on token t
    of layer i-1 and tokens < t of layer i, so this equals T decode_step calls at
    positions cache_pos .. cache_pos + T - 1 (a pinned identity)."""
    x = np.asarray(X, dtype=np.float64)
    for kind, layer, c in zip(kinds, layers, caches):
        if kind == "fa":
            x = prefill_full_attention(cfg, layer, c, x, cache_pos)
        else:
            x = prefill_linear_attention(cfg, layer, c, x)
        if layer_outputs is not None:
            layer_outputs.append(x.copy())
    return x


def gated_delta_rule_chunk(state, q, k, v, g, beta, Dk: int):
    """The gated delta rule over a chunk of L tokens at once (the chunked form of the
    recurrence a prefill uses); returns (new_state, y [L][Hv][Dv]).

    q, k [L][Hk][Dk]; v [L][Hv][Dv]; g, beta [L][Hv]. Per v-head with cumulative
    decays G_t = g_1 ... g_t, the step S_t = g_t S_(t-1) + k_t d_t^T with
    d_t = beta_t (v_t - (g_t S_(t-1))^T k_t) unrolls to
    S_t = G_t S_0 + sum_(s<=t) (G_t / G_s) k_s d_s^T, so the d_t solve one
    lower-triangular system
      d_t + beta_t sum_(s<t) (G_t / G_s) (k_s . k_t) d_s = beta_t (v_t - G_t S_0^T k_t),
    and y_t = (G_t S_0^T q_t + sum_(s<=t) (G_t / G_s) (k_s . q_t) d_s) / sqrt(Dk).
    Solved here with a library linear solve, independently of gated_delta_rule's
    token loop, which it must reproduce.
    """
    S0 = np.asarray(state, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    L, Hk = q.shape[0], q.shape[1]
    Hv = S0.shape[0]
    grp = Hv // Hk
    S_new = np.empty_like(S0)
    y = np.zeros((L, Hv, S0.shape[2]))
    for h in range(Hv):
        j = h // grp
        K, Q, V = k[:, j, :], q[:, j, :], v[:, h, :]
        lg = np.cumsum(np.log(g[:, h]))
        ratio = np.exp(lg[:, None] - lg[None, :])          # G_t / G_s
        G = np.exp(lg)
        low = np.tril(np.ones((L, L)), -1)
        A = np.eye(L) + beta[:, h][:, None] * ratio * (K @ K.T) * low
        rhs = beta[:, h][:, None] * (V - G[:, None] * (K @ S0[h]))
        d = np.linalg.solve(A, rhs)
        S_new[h] = G[-1] * S0[h] + (ratio[-1][:, None] * K).T @ d
        incl = np.tril(np.ones((L, L)))
        y[:, h, :] = (G[:, None] * (Q @ S0[h]) + (ratio * (Q @ K.T) * incl) @ d) / np.sqrt(np.float64(Dk))
    return S_new, y


# ----------------------------------------------------------------------------
# Output head
# ----------------------------------------------------------------------------


def lm_head_greedy(cfg: dict, head: dict, x_in, rows_per_chunk: int = 4096) -> tuple:
    """The model's tail after the last decoder layer: final RMSNorm, the lm_head
    GEMV and the greedy token. Returns (logits, token).

    Reading: the pages stop at the decoder layers and leave the final norm, the
    lm_head and sampling to the caller (page "Module qwen3_5"); this is the plain
    tail of the model in the pages' conventions: x_norm = bf16(RMSNorm(x) * w) with
    eps = rms_eps (the same rms_norm as every other norm), logits = bf16(W_lm x_norm)
    (a bf16 GEMV output, like q_full or z), and the token is the index of the largest
    bf16 logit, the lowest such index on a tie. The matrix is dequantised a block of
    rows at a time (a full 248 320-row matrix in float64 would take 5 GB).
    """
    eps = cfg["rms_eps"]
    x_norm = bf16_round(rms_norm(np.asarray(x_in, dtype=np.float64), bf16_to_f64(head["final_norm"]), eps))
    w = head["lm_head"]
    n = w["n"]
    logits = np.empty(n, dtype=np.float64)
    for r0 in range(0, n, rows_per_chunk):
        r1 = min(n, r0 + rows_per_chunk)
        part = {"codes": w["codes"][r0:r1], "scales": w["scales"][r0:r1], "biases": w["biases"][r0:r1],
                "n": r1 - r0, "k": w["k"]}
        logits[r0:r1] = bf16_round(gemv(part, x_norm))
    token = int(np.argmax(logits))  # numpy returns the first index of the maximum
    return logits, token


def kv_from_bits(k_bits, v_bits) -> dict:
    return {"k": bf16_to_f64(k_bits), "v": bf16_to_f64(v_bits)}


def turbo8_kv(k_codes, k_scale_bits, v_codes, v_scale_bits) -> dict:
    """A Turbo8 cache for the oracle: codes uint8 [cap][Hkv][D], scales as float64
    [cap][Hkv][D / 16] (bf16 values)."""
    return {"dtype": "turbo8", "k_codes": np.array(k_codes, dtype=np.uint8), "v_codes": np.array(v_codes, dtype=np.uint8),
            "k_scales": bf16_to_f64(k_scale_bits), "v_scales": bf16_to_f64(v_scale_bits)}


def state_from_arrays(conv, ssm) -> dict:
    return {"conv": np.asarray(conv, dtype=np.float64), "ssm": np.asarray(ssm, dtype=np.float64)}
