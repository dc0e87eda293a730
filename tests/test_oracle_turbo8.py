"""Pins of the oracle's Turbo8 KV-cache path (page "mod.rs": MetalKvDtype::Turbo8,
FP8 E4M3 data and a BF16 scale per group of 16 in the WHT-rotated basis; page
"full_attention.rs": the Turbo path that rotates K and V before the quantising
append, Q before attention, and the attention output back after it).

Each function is checked against a library routine (scipy's Hadamard matrix,
torch's float8_e4m3fn conversion), a closed form, or a special case in which a
misplaced rotation, a missing inverse, a wrong scale rule or rounding mode gives
another number.
"""

import numpy as np
import pytest
import scipy.linalg
import torch

from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O


@pytest.fixture(params=["tiny", "tiny_alt"])
def CFG(request):
    return synth.config(request.param)


# ---------------------------------------------------------------- WHT

@pytest.mark.parametrize("n", [16, 64, 128, 256])
def test_wht_is_the_orthonormal_sylvester_hadamard(n):
    x = np.random.default_rng(n).standard_normal((5, n))
    H = scipy.linalg.hadamard(n) / np.sqrt(n)  # Sylvester order: H_2n = [[H, H], [H, -H]]
    np.testing.assert_allclose(O.wht(x), x @ H.T, rtol=0, atol=1e-12)
    np.testing.assert_allclose(O.wht(O.wht(x)), x, rtol=0, atol=1e-12)  # its own inverse
    np.testing.assert_allclose(np.linalg.norm(O.wht(x), axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # the first basis vector maps to the constant vector 1/sqrt(n)
    e0 = np.zeros(n)
    e0[0] = 1.0
    np.testing.assert_allclose(O.wht(e0), np.full(n, 1 / np.sqrt(n)), rtol=1e-15)


# ---------------------------------------------------------------- E4M3

def test_e4m3_round_matches_torch_below_saturation():
    rng = np.random.default_rng(3)
    finite = np.arange(256, dtype=np.uint8)
    finite = finite[(finite & 0x7F) != 0x7F]
    vals = np.unique(O.e4m3_value(finite))
    mids = (vals[:-1] + vals[1:]) / 2  # exact ties between neighbours: to even
    x = np.concatenate([rng.standard_normal(20000) * 10, rng.standard_normal(2000) * 1e-3, mids, vals,
                        mids + 1e-9, mids - 1e-9])
    x = x[np.abs(x) < 464].astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.e4m3_round(x), ref)


def test_e4m3_saturates_and_codes_round_trip():
    x = np.array([448.0, 463.0, 464.0, 1e4, np.float32(3e38), -500.0, -1e30])
    np.testing.assert_array_equal(O.e4m3_round(x), np.array([448, 448, 448, 448, 448, -448, -448.0]))
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]
    v = O.e4m3_value(codes)
    # the decoder agrees with torch's interpretation of the same bytes
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(v, ref)
    nz = v != 0  # +0 and -0 share a value
    np.testing.assert_array_equal(O.e4m3_bits(v)[nz], codes[nz])
    assert v.max() == 448 and np.min(np.abs(v[nz])) == 2.0 ** -9


# ---------------------------------------------------------------- quantiser

def test_turbo8_quantize_scale_rule_and_error_bound():
    rng = np.random.default_rng(5)
    x = O.bf16_round(rng.standard_normal((7, 64)) * np.array([1e-3, 1, 30, 0.5, 2, 1e2, 1])[:, None])
    x[3, 16:32] = 0.0  # a group of zeros
    codes, scales = O.turbo8_quantize(x)
    assert codes.shape == x.shape and scales.shape == (7, 4)
    g = x.reshape(7, 4, 16)
    np.testing.assert_array_equal(scales, O.bf16_round(O.f32_round(np.abs(g).max(-1) / 448.0)))
    assert scales[3, 1] == 0 and not codes[3, 16:32].any()
    y = O.turbo8_dequantize(codes, scales)
    # E4M3 keeps 3 fraction bits: half a step is at most 2^-4 of the value (normal
    # range), 2^-10 of the scale in the subnormal range; the bf16 scale rounding can
    # push the largest quotient a little past 448 (saturated)
    err = np.abs(y - x).reshape(7, 4, 16)
    lim = 2.0 ** -4 * np.abs(g) + 2.0 ** -10 * scales[..., None] + 2.0 ** -7 * np.abs(g).max(-1, keepdims=True)
    assert np.all(err <= lim)


def test_turbo8_quantize_round_trips_representable_groups():
    rng = np.random.default_rng(6)
    finite = np.arange(256, dtype=np.uint8)
    finite = finite[(finite & 0x7F) != 0x7F]
    c = rng.choice(finite, size=(3, 32))
    c[:, 0] = 0x7E  # +448 in every group: the scale rule then reproduces s exactly
    c[:, 16] = 0xFE  # -448
    s = np.array([[2.0 ** -7, 0.75 * 2 ** -3], [1.0, 2.0 ** 5], [0.5, 2.0 ** -10]])
    x = O.turbo8_dequantize(c, s)
    codes, scales = O.turbo8_quantize(x)
    np.testing.assert_array_equal(scales, s)
    np.testing.assert_array_equal(O.turbo8_dequantize(codes, scales), x)


# ---------------------------------------------------------------- the layer's Turbo path

def _turbo_layer_run(CFG, pos, seed=0):
    lay = synth.fa_layer(seed, 1, CFG)
    kc, ks, vc, vs = synth.kv_cache_turbo8(seed, 1, CFG, 16, pos)
    kv = O.turbo8_kv(kc, ks, vc, vs)
    x = O.bf16_to_f64(synth.x_in(seed, 4, CFG))
    tr = {}
    out = O.forward_full_attention(CFG, lay, kv, x, pos, pos + 1, tr)
    return lay, kv, (kc, ks, vc, vs), tr, out


def test_turbo8_one_token_attention_returns_the_rotated_back_v(CFG):
    """At one token the softmax weight is 1: the rotated-basis output is the
    dequantised rotated v (bf16), and the layer's attention output is its inverse
    rotation. Without the inverse rotation, or with q rotated twice, it is not."""
    H, Hkv, D = CFG["num_heads"], CFG["num_kv_heads"], CFG["head_dim"]
    lay, kv, _, tr, _ = _turbo_layer_run(CFG, 0)
    vdeq = O.turbo8_dequantize(*O.turbo8_quantize(tr["v_rot"]))
    for h in range(H):
        np.testing.assert_array_equal(tr["attn_rot"][h], O.bf16_round(vdeq[h // (H // Hkv)]))
    np.testing.assert_array_equal(tr["attn_out"], O.bf16_round(O.wht(tr["attn_rot"])))
    assert not np.array_equal(tr["attn_out"], tr["attn_rot"])
    # the dequantised v rotated back is close to the layer's own v (E4M3 keeps ~2^-4)
    v = tr["v"].reshape(Hkv, D)
    assert np.linalg.norm(O.wht(vdeq) - v) <= 0.05 * np.linalg.norm(v)


def test_turbo8_append_writes_row_cache_pos_only(CFG):
    pos = 6
    lay, kv, before, tr, _ = _turbo_layer_run(CFG, pos)
    kc, ks, vc, vs = before
    # the rows written are the quantised rotated k (after norm and RoPE) and v
    ck, sk = O.turbo8_quantize(tr["k_rot"])
    cv, sv = O.turbo8_quantize(tr["v_rot"])
    np.testing.assert_array_equal(kv["k_codes"][pos], ck)
    np.testing.assert_array_equal(kv["k_scales"][pos], sk)
    np.testing.assert_array_equal(kv["v_codes"][pos], cv)
    np.testing.assert_array_equal(kv["v_scales"][pos], sv)
    np.testing.assert_array_equal(tr["k_rot"], O.bf16_round(O.wht(tr["k_rope"])))
    # every other row untouched
    rows = [r for r in range(16) if r != pos]
    np.testing.assert_array_equal(kv["k_codes"][rows], kc[rows])
    np.testing.assert_array_equal(kv["v_codes"][rows], vc[rows])
    np.testing.assert_array_equal(kv["k_scales"][rows], O.bf16_to_f64(ks[rows]))


def test_turbo8_attention_equals_plain_attention_on_the_rotated_back_cache(CFG):
    """Rotating q and every cached K row by the same orthonormal transform leaves the
    scores unchanged, and rotating the V-weighted sum back equals weighting the
    rotated-back V rows: the Turbo attention output (before its bf16 roundings)
    equals the plain attention on wht(dequantised rows) with the un-rotated q."""
    pos = 9
    H, Hkv, D = CFG["num_heads"], CFG["num_kv_heads"], CFG["head_dim"]
    lay, kv, _, tr, _ = _turbo_layer_run(CFG, pos)
    K = O.turbo8_dequantize(kv["k_codes"][:pos + 1], kv["k_scales"][:pos + 1])
    V = O.turbo8_dequantize(kv["v_codes"][:pos + 1], kv["v_scales"][:pos + 1])
    plain = O.attention_decode(O.wht(tr["q_rot"]), O.wht(K), O.wht(V), pos + 1, Hkv)
    rotated = O.wht(O.attention_decode(tr["q_rot"], K, V, pos + 1, Hkv))
    np.testing.assert_allclose(rotated, plain, rtol=0, atol=1e-12)
    # and the layer's values are those up to their bf16 roundings
    np.testing.assert_allclose(tr["attn_out"], plain, rtol=0, atol=2.0 ** -6 * np.abs(plain).max())
