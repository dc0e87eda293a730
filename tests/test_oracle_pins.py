"""Pins of the CPU oracle against things other than itself.

Each test checks an oracle function against a closed form, a special case the
pages or the mathematics fix, a library routine (torch CPU in float64), or brute
force on tiny inputs, so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.
"""

import math
import struct

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O


def _bits_to_float(b):
    return struct.unpack(">f", struct.pack(">I", int(b) << 16))[0]


# ---------------------------------------------------------------- number formats

def test_bf16_round_matches_torch_conversion():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        # exact ties between two bf16 values (low 16 bits = 0x8000)
        (np.arange(1, 2001, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38], dtype=np.float32),
    ])
    ours = O.bf16_round(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_bf16_bits_roundtrip():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # finite values only
    np.testing.assert_array_equal(O.bf16_bits(O.bf16_to_f64(bits)), bits)
    for b in bits[:200]:
        assert O.bf16_to_f64(np.array([b]))[0] == _bits_to_float(b)


# ---------------------------------------------------------------- dequant / GEMV

def test_dequant_bruteforce_and_closed_form():
    qw = synth.qweight(7, ("t",), 12, 192)
    W = O.dequant(qw)
    g = qw["k"] // 64
    for r in range(qw["n"]):
        for c in range(qw["k"]):
            s = _bits_to_float(qw["scales"][r][c // 64])
            b = _bits_to_float(qw["biases"][r][c // 64])
            assert W[r, c] == s * int(qw["codes"][r][c]) + b
            # synthetic bias is -128 * scale, so the weight is scale * (code - 128) exactly
            assert W[r, c] == s * (int(qw["codes"][r][c]) - 128)
    # padding columns of the scale rows are never read
    assert qw["scales"].shape[1] == synth.gstride(192) and g == 3


def test_gemv_bruteforce_tiny():
    qw = synth.qweight(3, ("g",), 9, 128)
    rng = np.random.default_rng(0)
    # general affine: bias not tied to the scale
    qw["biases"][:, :2] = synth.to_bf16_bits(rng.standard_normal((9, 2)) * 1e-3)
    x = rng.standard_normal(128)
    y = O.gemv(qw, x)
    for r in range(9):
        acc = 0.0
        for c in range(128):
            w = _bits_to_float(qw["scales"][r][c // 64]) * int(qw["codes"][r][c]) \
                + _bits_to_float(qw["biases"][r][c // 64])
            acc += w * x[c]
        assert abs(acc - y[r]) <= 1e-12 * (1 + abs(acc))
    # and against a library matmul of the dequantised matrix
    ref = torch.from_numpy(O.dequant(qw)) @ torch.from_numpy(x)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- qkv split

def test_qkv_split_worked_example_and_roundtrip():
    # each head's row of q_proj is [Q_h | gate_h]: H=2, D=2
    q, gate = O.qkv_split(np.arange(8.0), 2, 2)
    np.testing.assert_array_equal(q, [[0, 1], [4, 5]])
    np.testing.assert_array_equal(gate, [[2, 3], [6, 7]])
    rng = np.random.default_rng(5)
    qf = O.bf16_round(rng.standard_normal(4 * 2 * 64))
    q, gate = O.qkv_split(qf, 4, 64)
    back = np.concatenate([q, gate], axis=1).reshape(-1)
    np.testing.assert_array_equal(back, qf)


# ---------------------------------------------------------------- RMSNorm

def test_rms_norm_closed_form_and_library():
    w = 1.0 + 0.1 * np.random.default_rng(2).standard_normal(64)
    c = -1.75
    y = O.rms_norm(np.full(64, c), w, 1e-6)
    np.testing.assert_allclose(y, np.sign(c) * w * abs(c) / math.sqrt(c * c + 1e-6), rtol=1e-15)
    x = np.random.default_rng(3).standard_normal((5, 64))
    ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-6), ref, rtol=1e-12)
    # scale invariance (eps negligible)
    np.testing.assert_allclose(O.rms_norm(x * 1000.0, w, 1e-6), O.rms_norm(x, w, 1e-6), rtol=2e-6)


# ---------------------------------------------------------------- RoPE

def test_rope_inv_freq_closed_form():
    inv = O.rope_inv_freq(1e7, 64)
    assert inv[0] == 1.0
    assert inv[16] == np.float32(1e7 ** -0.5)
    assert len(inv) == 32 and np.all(np.diff(inv) < 0)


@pytest.mark.parametrize("R,D", [(16, 64), (64, 256)])
def test_rope_properties(R, D):
    rng = np.random.default_rng(4)
    inv = O.rope_inv_freq(1e7, R)
    x = rng.standard_normal((4, D))
    for pos in [0, 1, 7, 511, 16383, 131071]:
        y = O.rope_apply(x, pos, inv, R)
        # dims >= rotary_dim untouched, bit for bit
        np.testing.assert_array_equal(y[:, R:], x[:, R:])
        # each rotated pair keeps its norm
        h = R // 2
        np.testing.assert_allclose(y[:, :h] ** 2 + y[:, h:R] ** 2,
                                   x[:, :h] ** 2 + x[:, h:R] ** 2, rtol=1e-12)
        # rotating by the negated angles undoes it
        ang = O.f32_round(np.float64(np.float32(pos)) * inv)
        a, b = y[:, :h], y[:, h:R]
        back = np.concatenate([a * np.cos(ang) + b * np.sin(ang), b * np.cos(ang) - a * np.sin(ang)], 1)
        np.testing.assert_allclose(back, x[:, :R], atol=1e-12)
    # position 0 is the identity
    np.testing.assert_array_equal(O.rope_apply(x, 0, inv, R), x)


def test_rope_one_hot_closed_form():
    R, D = 16, 64
    inv = O.rope_inv_freq(1e7, R)
    for i in [0, 3, 7]:
        x = np.zeros((1, D))
        x[0, i] = 1.0
        pos = 5
        ang = float(np.float32(np.float32(pos) * np.float32(inv[i])))
        y = O.rope_apply(x, pos, inv, R)
        exp = np.zeros(D)
        exp[i] = math.cos(ang)
        exp[i + R // 2] = math.sin(ang)
        np.testing.assert_allclose(y[0], exp, atol=1e-15)


def test_rope_relative_position():
    R = D = 64
    inv = O.rope_inv_freq(1e7, R)
    rng = np.random.default_rng(8)
    q, k = rng.standard_normal((1, D)), rng.standard_normal((1, D))
    for m, n in [(10, 3), (100, 40), (7, 7)]:
        a = O.rope_apply(q, m, inv, R) @ O.rope_apply(k, n, inv, R).T
        b = O.rope_apply(q, m - n, inv, R) @ k.T
        np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-5)


# ---------------------------------------------------------------- attention

def test_attention_matches_library_sdpa():
    rng = np.random.default_rng(6)
    H, Hkv, D, S = 8, 2, 64, 37
    q = rng.standard_normal((H, D))
    K = rng.standard_normal((S + 5, Hkv, D))
    V = rng.standard_normal((S + 5, Hkv, D))
    out = O.attention_decode(q, K, V, S, Hkv)
    kk = torch.from_numpy(K[:S]).permute(1, 0, 2).repeat_interleave(H // Hkv, dim=0)
    vv = torch.from_numpy(V[:S]).permute(1, 0, 2).repeat_interleave(H // Hkv, dim=0)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], kk, vv)[:, 0, :]
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    rng = np.random.default_rng(9)
    H, Hkv, D = 4, 1, 32
    q = rng.standard_normal((H, D))
    K = rng.standard_normal((10, Hkv, D))
    V = rng.standard_normal((10, Hkv, D))
    # one token: the output is that token's V row for every head
    np.testing.assert_array_equal(O.attention_decode(q, K, V, 1, Hkv), np.repeat(V[0], H, 0))
    # all keys equal: the mean of V
    K2 = np.repeat(K[:1], 10, 0)
    np.testing.assert_allclose(O.attention_decode(q, K2, V, 10, Hkv),
                               np.repeat(V[:, 0].mean(0)[None], H, 0), rtol=1e-12)
    # one key with an overwhelming logit selects its V row
    K3 = K.copy()
    K3[4, 0] = 1e4 * q[0] / np.linalg.norm(q[0])
    np.testing.assert_allclose(O.attention_decode(q[:1], K3, V, 10, 1)[0], V[4, 0], rtol=1e-12)


# ---------------------------------------------------------------- GDN pieces

def test_conv1d_update_matches_library_conv():
    rng = np.random.default_rng(10)
    C, Kc, T = 6, 4, 9
    w = rng.standard_normal((C, Kc))
    xs = rng.standard_normal((T, C))
    st = np.zeros((C, Kc))
    outs = []
    for t in range(T):
        st, o = O.causal_conv1d_update(st, xs[t], w)
        outs.append(o)
    # causal depthwise conv over the whole sequence with left zero padding
    inp = F.pad(torch.from_numpy(xs.T)[None], (Kc - 1, 0))
    ref = F.conv1d(inp, torch.from_numpy(w)[:, None, :], groups=C)[0].T.numpy()
    np.testing.assert_allclose(np.array(outs), ref, rtol=1e-13, atol=1e-14)


def test_conv1d_one_hot_taps():
    C, Kc = 3, 4
    xs = np.arange(1.0, 8.0)[:, None] * np.ones((1, C))
    for tap, delay in [(Kc - 1, 0), (0, Kc - 1)]:
        w = np.zeros((C, Kc))
        w[:, tap] = 1.0
        st = np.zeros((C, Kc))
        for t in range(len(xs)):
            st, o = O.causal_conv1d_update(st, xs[t], w)
            exp = xs[t - delay] if t - delay >= 0 else np.zeros(C)
            np.testing.assert_array_equal(o, exp)


def test_l2_norm_unit_and_library():
    x = np.random.default_rng(11).standard_normal((5, 32)) * 3
    y = O.l2_norm_rows(x, 1e-6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), 1.0, atol=1e-6)
    np.testing.assert_allclose(y, F.normalize(torch.from_numpy(x), dim=1).numpy(), rtol=1e-6)


def test_gate_beta_closed_forms():
    # dt + dt_bias = 0, A_log = 0: exp(-softplus(0)) = exp(-ln 2) = 0.5
    assert O.gdn_gate(np.array([0.5]), np.array([-0.5]), np.array([0.0]))[0] == 0.5
    # large dt: softplus(x) = x, gate = exp(-exp(A) * x)
    g = O.gdn_gate(np.array([30.0]), np.array([0.0]), np.array([math.log(0.1)]))[0]
    assert g == np.float32(math.exp(-3.0))
    assert O.gdn_beta(np.array([0.0]))[0] == 0.5
    np.testing.assert_allclose(O.softplus(np.array([-3.0, 0.0, 3.0])),
                               F.softplus(torch.tensor([-3.0, 0.0, 3.0], dtype=torch.float64)).numpy(),
                               rtol=1e-15)
    np.testing.assert_allclose(O.silu(np.array([-2.0, 0.5])),
                               F.silu(torch.tensor([-2.0, 0.5], dtype=torch.float64)).numpy(), rtol=1e-15)


def _delta_inputs(Hk=2, Hv=4, Dk=8, Dv=6, seed=12):
    rng = np.random.default_rng(seed)
    S = rng.standard_normal((Hv, Dk, Dv))
    q = rng.standard_normal((Hk, Dk))
    k = O.l2_norm_rows(rng.standard_normal((Hk, Dk)), 0)
    v = rng.standard_normal((Hv, Dv))
    return S, q, k, v


def test_delta_rule_beta0_gate1_keeps_state():
    S, q, k, v = _delta_inputs()
    Hv = S.shape[0]
    S2, y = O.gated_delta_rule(S, q, k, v, np.ones(Hv), np.zeros(Hv), 8)
    np.testing.assert_array_equal(S2, S)
    for h in range(Hv):
        np.testing.assert_allclose(y[h], S[h].T @ q[h // 2] / math.sqrt(8), rtol=1e-13)


def test_delta_rule_from_zero_and_gate0():
    S, q, k, v = _delta_inputs()
    Hv = S.shape[0]
    S2, y = O.gated_delta_rule(np.zeros_like(S), q, k, v, np.ones(Hv), np.ones(Hv), 8)
    for h in range(Hv):
        np.testing.assert_allclose(S2[h], np.outer(k[h // 2], v[h]), rtol=1e-13)
        np.testing.assert_allclose(y[h], (q[h // 2] @ k[h // 2]) * v[h] / math.sqrt(8), rtol=1e-12)
    beta = np.full(Hv, 0.3)
    S3, _ = O.gated_delta_rule(S, q, k, v, np.zeros(Hv), beta, 8)
    for h in range(Hv):
        np.testing.assert_allclose(S3[h], np.outer(k[h // 2], 0.3 * v[h]), rtol=1e-13)


def test_delta_rule_retrieves_orthonormal_keys():
    Dk, Dv, m = 8, 5, 6
    rng = np.random.default_rng(13)
    Q, _ = np.linalg.qr(rng.standard_normal((Dk, Dk)))
    keys = Q[:, :m].T
    vals = rng.standard_normal((m, Dv))
    S = np.zeros((1, Dk, Dv))
    for i in range(m):
        S, _ = O.gated_delta_rule(S, keys[i:i + 1], keys[i:i + 1], vals[i:i + 1], np.ones(1), np.ones(1), Dk)
    for i in range(m):
        _, y = O.gated_delta_rule(S, keys[i:i + 1], keys[i:i + 1], vals[i:i + 1], np.ones(1), np.zeros(1), Dk)
        np.testing.assert_allclose(y[0], vals[i] / math.sqrt(Dk), atol=1e-12)


def test_delta_rule_is_gradient_step_on_decayed_state():
    # delta rule = one step of size beta on 0.5 * ||S^T k - v||^2 from the decayed state
    S, q, k, v = _delta_inputs()
    Hv = S.shape[0]
    g = np.array([0.9, 0.5, 0.99, 0.1])
    beta = np.array([0.2, 0.7, 1.0, 0.05])
    S2, _ = O.gated_delta_rule(S, q, k, v, g, beta, 8)
    for h in range(Hv):
        Sd = torch.tensor(g[h] * S[h], requires_grad=True)
        loss = 0.5 * torch.sum((Sd.T @ torch.from_numpy(k[h // 2]) - torch.from_numpy(v[h])) ** 2)
        loss.backward()
        np.testing.assert_allclose(S2[h], (Sd - beta[h] * Sd.grad).detach().numpy(), rtol=1e-12, atol=1e-14)


def test_delta_rule_columns_independent():
    S, q, k, v = _delta_inputs()
    Hv = S.shape[0]
    perm = np.random.default_rng(14).permutation(S.shape[2])
    g, beta = np.full(Hv, 0.8), np.full(Hv, 0.6)
    S2, y = O.gated_delta_rule(S, q, k, v, g, beta, 8)
    S3, y3 = O.gated_delta_rule(S[:, :, perm], q, k, v[:, perm], g, beta, 8)
    np.testing.assert_allclose(S3, S2[:, :, perm], rtol=1e-14)
    np.testing.assert_allclose(y3, y[:, perm], rtol=1e-14)


# ---------------------------------------------------------------- whole layers

@pytest.fixture(params=["tiny", "tiny_alt"])
def CFG(request):
    return synth.config(request.param)


def _zero_matrix(qw):
    qw["codes"][:] = 128  # synthetic bias is -128 * scale, so every weight is 0


def test_fa_layer_seq1_returns_gated_v(CFG):
    lay = synth.fa_layer(0, 1, CFG)
    k, v = synth.kv_cache(0, 1, CFG, 16, 0)
    kv = O.kv_from_bits(k, v)
    x = O.bf16_to_f64(synth.x_in(0, 0, CFG))
    tr = {}
    O.forward_full_attention(CFG, lay, kv, x, 0, 1, tr)
    H, Hkv, D = CFG["num_heads"], CFG["num_kv_heads"], CFG["head_dim"]
    vh = tr["v"].reshape(Hkv, D)
    for h in range(H):
        np.testing.assert_array_equal(tr["attn_out"][h], vh[h // (H // Hkv)])
    _, gate = O.qkv_split(tr["q_full"], H, D)
    np.testing.assert_array_equal(tr["gated_attn"], O.bf16_round(tr["attn_out"] * O.sigmoid(gate)))
    # the append wrote exactly row 0: the post-RoPE k (position 0 = no rotation) and v
    np.testing.assert_array_equal(kv["k"][0], tr["k_rope"])
    np.testing.assert_array_equal(kv["v"][0], vh)
    assert not kv["k"][1:].any() and not kv["v"][1:].any()


def test_fa_layer_zero_projections_are_identity_residuals(CFG):
    lay = synth.fa_layer(0, 1, CFG)
    _zero_matrix(lay["o_proj"])
    _zero_matrix(lay["down_proj"])
    k, v = synth.kv_cache(0, 1, CFG, 16, 5)
    x = O.bf16_to_f64(synth.x_in(0, 3, CFG))
    tr = {}
    out = O.forward_full_attention(CFG, lay, O.kv_from_bits(k, v), x, 5, 6, tr)
    np.testing.assert_array_equal(tr["x_resid"], x)
    np.testing.assert_array_equal(out, x)


def test_gdn_layer_zero_projections_and_state_update(CFG):
    lay = synth.gdn_layer(0, 0, CFG)
    _zero_matrix(lay["out_proj"])
    _zero_matrix(lay["down_proj"])
    conv, ssm = synth.gdn_state(0, 0, CFG)
    st = O.state_from_arrays(conv, ssm)
    x = O.bf16_to_f64(synth.x_in(0, 0, CFG))
    tr = {}
    out = O.forward_linear_attention(CFG, lay, st, x, tr)
    np.testing.assert_array_equal(out, x)
    # zero-initialised conv state: after one step only the newest slot is filled
    np.testing.assert_array_equal(st["conv"][:, -1], tr["qkv"])
    assert not st["conv"][:, :-1].any()
    # from a zero state the new state is k (x) beta * v per head
    Hk, Hv, Dk = CFG["num_k_heads_lin"], CFG["num_v_heads_lin"], CFG["k_head_dim_lin"]
    nqk = Hk * Dk
    kk = tr["qkv_smooth"][nqk:2 * nqk].reshape(Hk, Dk)
    vv = tr["qkv_smooth"][2 * nqk:].reshape(Hv, -1)
    for h in range(Hv):
        np.testing.assert_allclose(st["ssm"][h], O.f32_round(np.outer(kk[h // (Hv // Hk)], tr["beta"][h] * vv[h])),
                                   rtol=1e-7)
    # the Q and K heads of qkv_smooth are unit vectors (up to bf16 rounding)
    qs = tr["qkv_smooth"][:2 * nqk].reshape(2 * Hk, Dk)
    np.testing.assert_allclose(np.linalg.norm(qs, axis=1), 1.0, atol=1e-2)


def test_stack_step_chains_layers(CFG):
    kinds = synth.layer_kinds(CFG)
    assert kinds == ["gdn", "fa"]
    layers = [synth.gdn_layer(0, 0, CFG), synth.fa_layer(0, 1, CFG)]
    conv, ssm = synth.gdn_state(0, 0, CFG)
    k, v = synth.kv_cache(0, 1, CFG, 16, 0)
    caches = [O.state_from_arrays(conv, ssm), O.kv_from_bits(k, v)]
    x = O.bf16_to_f64(synth.x_in(0, 0, CFG))
    outs = []
    y = O.decode_step(CFG, kinds, layers, caches, x, 0, outs)
    assert len(outs) == 2 and np.array_equal(outs[1], y)
    # the same two layers called one by one give the same result
    conv, ssm = synth.gdn_state(0, 0, CFG)
    st = O.state_from_arrays(conv, ssm)
    kv = O.kv_from_bits(k, v)
    y1 = O.forward_linear_attention(CFG, layers[0], st, x)
    y2 = O.forward_full_attention(CFG, layers[1], kv, y1, 0, 1)
    np.testing.assert_array_equal(y2, y)


# ---------------------------------------------------------------- output head

def _head_with_identical_rows(seed, cfg, vocab, winner=None, factor=1.0):
    """Every row of the lm_head a copy of row 0; row `winner` (if any) with its
    scales and biases multiplied by `factor` (a power of two: exact in bf16)."""
    h = synth.head(seed, cfg, vocab)
    w = h["lm_head"]
    for key in ("codes", "scales", "biases"):
        w[key][:] = w[key][0]
    if winner is not None:
        for key in ("scales", "biases"):
            w[key][winner] = synth.to_bf16_bits(synth.bf16_bits_to_f32(w[key][winner]) * factor)
    return h


def test_lm_head_greedy_against_library_and_brute_force(CFG):
    cfg = synth.config("tiny")
    head = synth.head(5, cfg, 300)
    x = O.bf16_to_f64(synth.x_in(5, 0, cfg)) * 3.0
    logits, tok = O.lm_head_greedy(cfg, head, x, rows_per_chunk=128)  # chunks: 128, 128, 44
    # the norm through a library routine, the GEMV as an explicit dequantised matmul
    w = torch.from_numpy(O.bf16_to_f64(head["final_norm"]))
    xn = F.rms_norm(torch.from_numpy(x), (cfg["hidden"],), w, eps=cfg["rms_eps"])
    xn = xn.to(torch.bfloat16).to(torch.float64)
    qw = head["lm_head"]
    g = qw["k"] // 64
    s = torch.from_numpy(O.bf16_to_f64(qw["scales"])[:, :g]).repeat_interleave(64, dim=1)
    b = torch.from_numpy(O.bf16_to_f64(qw["biases"])[:, :g]).repeat_interleave(64, dim=1)
    W = torch.from_numpy(qw["codes"].astype(np.float64)) * s + b
    ref = (W @ xn).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(logits, ref)
    assert tok == int(torch.argmax(torch.from_numpy(ref)))  # torch: the first maximal index
    assert logits[tok] == logits.max()


def test_lm_head_greedy_ties_and_planted_winner(CFG):
    cfg = synth.config("tiny")
    x = O.bf16_to_f64(synth.x_in(6, 0, cfg))
    base = _head_with_identical_rows(6, cfg, 64)
    logits, tok = O.lm_head_greedy(cfg, base, x)
    assert np.all(logits == logits[0]) and tok == 0  # all equal: the lowest index
    # row 37 scaled by 2 (or 1/2) so that its logit is strictly the largest
    factor = 2.0 if logits[0] > 0 else 0.5
    win = _head_with_identical_rows(6, cfg, 64, winner=37, factor=factor)
    logits2, tok2 = O.lm_head_greedy(cfg, win, x)
    assert tok2 == 37
    assert logits2[37] == logits[0] * factor
