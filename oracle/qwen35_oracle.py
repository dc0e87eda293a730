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

Pins (see tests/test_oracle_pins.py): every function below is checked against
closed forms, special cases, library routines or brute force. None is unpinned.
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


def state_from_arrays(conv, ssm) -> dict:
    return {"conv": np.asarray(conv, dtype=np.float64), "ssm": np.asarray(ssm, dtype=np.float64)}
