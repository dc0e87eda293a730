"""Pins of the oracle's prefill: the chunked delta rule against the token loop, the
stack's layer-major prefill against token-major decode steps, and the prompt's
attention against a library causal attention over the whole prompt."""

import numpy as np
import pytest
import torch

from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O


def _l2n(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


@pytest.mark.parametrize("L,Hk,Hv,Dk,Dv", [(12, 2, 4, 8, 8), (1, 1, 1, 4, 4), (30, 1, 2, 16, 8)])
def test_chunked_delta_rule_equals_token_loop(L, Hk, Hv, Dk, Dv):
    """The lower-triangular-solve form over a chunk reproduces L sequential steps of
    gated_delta_rule (state and every readout), to float64 rounding."""
    r = np.random.default_rng(L * 100 + Dk)
    S0 = r.standard_normal((Hv, Dk, Dv)) * 0.3
    q = _l2n(r.standard_normal((L, Hk, Dk)))
    k = _l2n(r.standard_normal((L, Hk, Dk)))
    v = r.standard_normal((L, Hv, Dv))
    g = r.uniform(0.6, 1.0, (L, Hv))
    beta = r.uniform(0.0, 1.0, (L, Hv))
    S = S0.copy()
    ys = []
    for t in range(L):
        S, y = O.gated_delta_rule(S, q[t], k[t], v[t], g[t], beta[t], Dk)
        ys.append(y)
    Sc, yc = O.gated_delta_rule_chunk(S0, q, k, v, g, beta, Dk)
    assert np.allclose(Sc, S, rtol=1e-10, atol=1e-12)
    assert np.allclose(yc, np.stack(ys), rtol=1e-10, atol=1e-12)


def test_chunked_delta_rule_detects_a_dropped_decay():
    """A mistake planted in the token loop (no decay) is caught by the chunked form."""
    r = np.random.default_rng(7)
    L, Hk, Hv, Dk, Dv = 6, 1, 1, 4, 4
    S0 = r.standard_normal((Hv, Dk, Dv))
    q, k = _l2n(r.standard_normal((L, Hk, Dk))), _l2n(r.standard_normal((L, Hk, Dk)))
    v = r.standard_normal((L, Hv, Dv))
    g = np.full((L, Hv), 0.8)
    beta = np.full((L, Hv), 0.5)
    S = S0.copy()
    for t in range(L):
        S, _ = O.gated_delta_rule(S, q[t], k[t], v[t], np.ones(Hv), beta[t], Dk)
    Sc, _ = O.gated_delta_rule_chunk(S0, q, k, v, g, beta, Dk)
    assert not np.allclose(Sc, S, rtol=1e-3)


def _tiny_stack(cache_rows=4, capacity=32, name="tiny"):
    cfg = synth.config(name)
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(0, 0, cfg), synth.fa_layer(0, 1, cfg)]
    conv, ssm = synth.gdn_state(0, 0, cfg, 0.1)
    kb, vb = synth.kv_cache(0, 1, cfg, capacity, cache_rows)
    caches = lambda: [O.state_from_arrays(conv, ssm), O.kv_from_bits(kb, vb)]  # noqa: E731
    return cfg, kinds, layers, caches


@pytest.mark.parametrize("name", ["tiny", "tiny_alt"])
def test_prefill_stack_equals_decode_steps(name):
    """Layer-major over the prompt (prefill_step) equals token-major through the
    stack (decode_step per token at cache_pos + t): outputs, caches and states bit
    for bit."""
    cfg, kinds, layers, caches = _tiny_stack(name=name)
    T, p0 = 6, 4
    X = O.bf16_to_f64(np.stack([synth.x_in(1, t, cfg) for t in range(T)]))
    c1, c2 = caches(), caches()
    out = O.prefill_step(cfg, kinds, layers, c1, X, p0)
    ref = np.stack([O.decode_step(cfg, kinds, layers, c2, X[t], p0 + t) for t in range(T)])
    assert np.array_equal(out, ref)
    assert np.array_equal(c1[0]["ssm"], c2[0]["ssm"]) and np.array_equal(c1[0]["conv"], c2[0]["conv"])
    assert np.array_equal(c1[1]["k"], c2[1]["k"]) and np.array_equal(c1[1]["v"], c2[1]["v"])


@pytest.mark.parametrize("H,Hkv,D,R", [(4, 1, 64, 16), (3, 1, 128, 32), (6, 2, 64, 64), (2, 2, 128, 16)])
def test_prefill_attention_is_offset_causal_attention(H, Hkv, D, R):
    """Token t of a prompt at cache_pos p0 attends over cache rows [0, p0 + t]:
    every token's attention output equals a library scaled-dot-product attention
    over the final cache with the offset causal mask j <= p0 + t (GQA heads
    expanded: q-head h reads kv-head h // (H / Hkv)), rounded to bf16. Group sizes
    4, 3 and 1 and head dims 64 and 128."""
    cfg = synth.config("tiny")
    cfg.update(num_heads=H, num_kv_heads=Hkv, head_dim=D, rotary_dim=R)
    layer = synth.fa_layer(2, 1, cfg)
    T, p0, cap = 7, 5, 16
    kb, vb = synth.kv_cache(2, 1, cfg, cap, p0)
    kv = O.kv_from_bits(kb, vb)
    X = O.bf16_to_f64(np.stack([synth.x_in(2, t, cfg) for t in range(T)]))
    traces = []
    O.prefill_full_attention(cfg, layer, kv, X, p0, traces)
    H, Hkv, D = cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"]
    S = p0 + T
    q = torch.tensor(np.stack([tr["q_rope"] for tr in traces]), dtype=torch.float64)  # [T][H][D]
    K = torch.tensor(kv["k"][:S], dtype=torch.float64).repeat_interleave(H // Hkv, dim=1)  # [S][H][D]
    V = torch.tensor(kv["v"][:S], dtype=torch.float64).repeat_interleave(H // Hkv, dim=1)
    mask = torch.arange(S)[None, :] <= (p0 + torch.arange(T))[:, None]  # [T][S]
    ref = torch.nn.functional.scaled_dot_product_attention(q.transpose(0, 1), K.transpose(0, 1),
                                                           V.transpose(0, 1), attn_mask=mask)
    ref = O.bf16_round(ref.transpose(0, 1).numpy())
    got = np.stack([tr["attn_out"] for tr in traces])
    assert np.allclose(got, ref, rtol=2.0 ** -8, atol=1e-12)
    # the same library call with the plain causal mask of a prompt from position 0
    # (one row short) differs: the offset matters
    short = torch.nn.functional.scaled_dot_product_attention(q.transpose(0, 1), K.transpose(0, 1)[:, :S - 1],
                                                             V.transpose(0, 1)[:, :S - 1],
                                                             attn_mask=mask[:, :S - 1])
    assert not np.allclose(got, O.bf16_round(short.transpose(0, 1).numpy()), rtol=2.0 ** -8)
