"""Pins of how the oracle's two layer forwards compose their steps.

The per-step pins (test_oracle_pins.py) fix each piece; these fix the wiring
between them, which a whole-layer check with zeroed projections cannot see:

- which operand of the MLP takes the SiLU, and which residual the MLP adds: the
  page "full_attention.rs" (forward_full_attention, its last two steps) forms
  x_resid = x_in + o, normalises it, and returns x_resid + down(silu(gate) * up);
- the linear-attention output gate: the page "linear_attention.rs"
  (forward_linear_attention, the gemv_silu_gate step) multiplies out_proj into
  silu(z) * y_norm, y_norm being the per-head RMSNorm of the delta-rule readout;
- the order of the per-head q/k RMSNorm and the partial RoPE ("full_attention.rs":
  the q/k norms run before rope on the bf16 q/k buffers).

Each is checked two ways: against a restatement in torch library routines
(F.linear on matrices dequantised by torch ops, F.silu, F.rms_norm) from the
trace's own inputs, and against a one-hot construction whose output is a scalar
closed form in which the swapped or missing operand gives a different number.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O


@pytest.fixture(params=["tiny", "tiny_alt"])
def CFG(request):
    """The small configs: 4 q-heads of dim 64 over one kv-head and linear heads of
    dim 32, and 3 q-heads of dim 128 over 3 kv-heads and linear heads of dim 64."""
    return synth.config(request.param)


def _t(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float64))


def _bf(x):
    """Round a float64 torch tensor to bf16 values (torch's own conversion)."""
    return x.to(torch.bfloat16).to(torch.float64)


def _bits(b):
    return torch.from_numpy(synth.bf16_bits_to_f32(b).astype(np.float64))


def _torch_dequant(qw):
    """W = scale * code + bias per 64-column group, with torch ops only."""
    g = qw["k"] // 64
    s = _bits(qw["scales"][:, :g]).repeat_interleave(64, dim=1)
    b = _bits(qw["biases"][:, :g]).repeat_interleave(64, dim=1)
    return torch.from_numpy(qw["codes"].astype(np.float64)) * s + b


def _one_hot_rows(qw, col_of_row, scale=None, code=129):
    """Every weight zero except W[r][col_of_row(r)] = scale[r][group] * (code - 128)
    (the bias is -128 * scale, so code 128 is an exact zero). With `scale` given,
    every group's scale is set to it (a bf16 value) and its bias to -128 * scale."""
    if scale is not None:
        qw["scales"][:] = synth.to_bf16_bits(np.float32(scale))
        qw["biases"][:] = synth.to_bf16_bits(np.float32(-128.0 * scale))
    qw["codes"][:] = 128
    for r in range(qw["n"]):
        c = col_of_row(r)
        if c is not None:
            qw["codes"][r, c] = code


def _scale(qw, r, c):
    return float(synth.bf16_bits_to_f32(qw["scales"][r, c // 64]))


# ---------------------------------------------------------------- full attention

def _fa_run(CFG, lay, pos=5, seed=0):
    k, v = synth.kv_cache(seed, 1, CFG, 16, pos)
    kv = O.kv_from_bits(k, v)
    x = O.bf16_to_f64(synth.x_in(seed, 2, CFG))
    tr = {}
    out = O.forward_full_attention(CFG, lay, kv, x, pos, pos + 1, tr)
    return x, out, tr


def test_fa_mlp_matches_library_composition(CFG):
    """x_out = bf16(x_resid + W_down (silu(bf16(W_gate xn2)) * bf16(W_up xn2))) with
    x_resid = bf16(x_in + o) and xn2 = bf16(RMSNorm(x_resid) * post_ln); o is the
    layer's own o_proj output (nonzero, so x_in and x_resid differ)."""
    lay = synth.fa_layer(4, 1, CFG)
    x, out, tr = _fa_run(CFG, lay)
    o = _t(tr["o"])
    assert torch.count_nonzero(o) > 0
    x_resid = _bf(_t(x) + o)
    xn2 = _bf(F.rms_norm(x_resid, (CFG["hidden"],), _bits(lay["post_ln"]), eps=CFG["rms_eps"]))
    g = _bf(F.linear(xn2, _torch_dequant(lay["gate_proj"])))
    u = _bf(F.linear(xn2, _torch_dequant(lay["up_proj"])))
    ref = _bf(x_resid + F.linear(F.silu(g) * u, _torch_dequant(lay["down_proj"])))
    np.testing.assert_array_equal(tr["x_resid"], x_resid.numpy())
    np.testing.assert_array_equal(out, ref.numpy())
    # the plausible misreadings give other numbers
    swapped = _bf(x_resid + F.linear(F.silu(u) * g, _torch_dequant(lay["down_proj"])))
    from_x_in = _bf(_t(x) + F.linear(F.silu(g) * u, _torch_dequant(lay["down_proj"])))
    assert not np.array_equal(out, swapped.numpy())
    assert not np.array_equal(out, from_x_in.numpy())


def test_fa_mlp_one_hot_closed_form(CFG):
    """One-hot gate/up/down rows: gate_j = s_g,j * xn2[0], up_j = s_u,j * xn2[1], and
    x_out[j] = x_resid[j] + s_d,j * silu(gate_j) * up_j for j < hidden."""
    E, I = CFG["hidden"], CFG["intermediate"]
    lay = synth.fa_layer(5, 1, CFG)
    # distinct unit-size scales, so silu(gate) * up and silu(up) * gate differ
    _one_hot_rows(lay["gate_proj"], lambda r: 0, scale=2.0)
    _one_hot_rows(lay["up_proj"], lambda r: 1, scale=0.75)
    _one_hot_rows(lay["down_proj"], lambda r: r, scale=1.0)  # row j reads h_j (E <= I)
    assert I >= E
    x, out, tr = _fa_run(CFG, lay)
    xn2 = tr["x_norm2"]
    x_resid = tr["x_resid"]
    g = float(O.bf16_round(2.0 * xn2[0]))
    u = float(O.bf16_round(0.75 * xn2[1]))
    assert abs(g) > 0.1 and abs(u) > 0.1 and abs(g) != abs(u)
    np.testing.assert_array_equal(tr["gate_act"], np.full(I, g))
    np.testing.assert_array_equal(tr["up_act"], np.full(I, u))
    h = g / (1.0 + np.exp(-g)) * u  # silu(gate) * up
    h_swapped = u / (1.0 + np.exp(-u)) * g
    assert abs(h - h_swapped) > 0.05
    np.testing.assert_array_equal(out, O.bf16_round(x_resid + h))
    assert not np.array_equal(out, O.bf16_round(x_resid + h_swapped))
    assert not np.array_equal(out, O.bf16_round(x + h))  # the residual is x_resid, not x_in


def test_fa_qk_norm_then_rope(CFG):
    """q_rope = bf16(rope(bf16(RMSNorm_head(q) * q_norm))), with non-uniform norm
    weights at a nonzero position; the other order (rotate, then normalise) differs."""
    H, Hkv, D, R = CFG["num_heads"], CFG["num_kv_heads"], CFG["head_dim"], CFG["rotary_dim"]
    lay = synth.fa_layer(6, 1, CFG)
    pos = 7
    x, out, tr = _fa_run(CFG, lay, pos=pos)
    q = _t(tr["q_full"]).reshape(H, 2 * D)[:, :D]
    k = _t(tr["k"]).reshape(Hkv, D)
    wq, wk = _bits(lay["q_norm"]), _bits(lay["k_norm"])
    assert torch.std(wq[:R]) > 0.01  # the weights vary over the rotated dims

    # rotate-half RoPE on the first R dims at the fp32 angle pos * inv_freq (torch ops)
    inv = torch.tensor([np.float32(CFG["rope_theta"] ** (-2.0 * i / R)) for i in range(R // 2)],
                       dtype=torch.float32)
    ang = (torch.tensor(float(pos), dtype=torch.float32) * inv).to(torch.float64)
    c, s = torch.cos(ang), torch.sin(ang)

    def rope(y):
        a, b = y[:, :R // 2], y[:, R // 2:R]
        return torch.cat([a * c - b * s, b * c + a * s, y[:, R:]], dim=1)

    eps = CFG["rms_eps"]
    want_q = _bf(rope(_bf(F.rms_norm(q, (D,), wq, eps=eps))))
    want_k = _bf(rope(_bf(F.rms_norm(k, (D,), wk, eps=eps))))
    np.testing.assert_array_equal(tr["q_rope"], want_q.numpy())
    np.testing.assert_array_equal(tr["k_rope"], want_k.numpy())
    other = _bf(F.rms_norm(_bf(rope(q)), (D,), wq, eps=eps))
    assert not np.array_equal(tr["q_rope"], other.numpy())


# ---------------------------------------------------------------- linear attention

def _gdn_run(CFG, lay, seed=0, steps=2):
    conv, ssm = synth.gdn_state(seed, 0, CFG, std=0.1)
    st = O.state_from_arrays(conv, ssm)
    tr = {}
    for t in range(steps):  # a second step: a nonzero conv history
        x = O.bf16_to_f64(synth.x_in(seed, t, CFG))
        tr = {}
        out = O.forward_linear_attention(CFG, lay, st, x, tr)
    return x, out, tr


def test_gdn_output_gate_matches_library_composition(CFG):
    """out = bf16(W_out (silu(z) * y_norm)), y_norm = bf16(RMSNorm_head(y) * norm_weight),
    then x_out = bf16(x_resid + MLP) with x_resid = bf16(x_in + out)."""
    Hv, Dv = CFG["num_v_heads_lin"], CFG["v_head_dim_lin"]
    lay = synth.gdn_layer(7, 0, CFG)
    x, out, tr = _gdn_run(CFG, lay)
    y = _t(tr["y"]).reshape(Hv, Dv)
    z = _t(tr["z"])
    y_norm = _bf(F.rms_norm(y, (Dv,), _bits(lay["norm_weight"]), eps=CFG["rms_eps"])).reshape(-1)
    W = _torch_dequant(lay["out_proj"])
    want = _bf(F.linear(F.silu(z) * y_norm, W))
    np.testing.assert_array_equal(tr["y_norm"], y_norm.numpy())
    np.testing.assert_array_equal(tr["out"], want.numpy())
    x_resid = _bf(_t(x) + want)
    np.testing.assert_array_equal(tr["x_resid"], x_resid.numpy())
    xn2 = _bf(F.rms_norm(x_resid, (CFG["hidden"],), _bits(lay["post_ln"]), eps=CFG["rms_eps"]))
    g = _bf(F.linear(xn2, _torch_dequant(lay["gate_proj"])))
    u = _bf(F.linear(xn2, _torch_dequant(lay["up_proj"])))
    np.testing.assert_array_equal(out, _bf(x_resid + F.linear(F.silu(g) * u, _torch_dequant(lay["down_proj"]))).numpy())
    swapped = _bf(F.linear(F.silu(y_norm) * z, W))
    no_silu = _bf(F.linear(z * y_norm, W))
    assert not np.array_equal(tr["out"], swapped.numpy())
    assert not np.array_equal(tr["out"], no_silu.numpy())


def test_gdn_output_gate_one_hot_closed_form(CFG):
    """One-hot out_proj rows: out[j] = s_j * silu(z[c_j]) * y_norm[c_j] with c_j = j mod Z."""
    Z = CFG["num_v_heads_lin"] * CFG["v_head_dim_lin"]
    lay = synth.gdn_layer(8, 0, CFG)
    _one_hot_rows(lay["out_proj"], lambda r: r % Z, scale=1.0)
    x, out, tr = _gdn_run(CFG, lay)
    z, yn = tr["z"], tr["y_norm"]
    c = np.arange(CFG["hidden"]) % Z
    want = O.bf16_round(z[c] / (1.0 + np.exp(-z[c])) * yn[c])
    np.testing.assert_array_equal(tr["out"], want)
    other = O.bf16_round(yn[c] / (1.0 + np.exp(-yn[c])) * z[c])
    assert np.count_nonzero(other != want) > CFG["hidden"] // 4
