"""Paged KV on the host: the pool layout the tests and the bench build (logical
cache blocks placed at the pool blocks a table names), and the ABI's checks of a
paged cache, which come before anything is enqueued (fake, never dereferenced
pointers)."""

import numpy as np
import pytest

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth

from test_abi import _FakeScratch, _fake_fa


def test_pool_and_gather_round_trip():
    rng = np.random.default_rng(1)
    caches = [rng.integers(0, 1 << 16, size=(48, 2, 8), dtype=np.uint16) for _ in range(3)]
    table = synth.block_table(5, 3, 48 // 16, 11)
    assert len(set(table.reshape(-1).tolist())) == 9 and table.min() >= 0 and table.max() < 11
    pool = synth.paged_pool(caches, 16, table, 11, 0x7FC0)
    assert pool.shape == (11, 16, 2, 8)
    for b in range(3):
        np.testing.assert_array_equal(synth.paged_gather(pool, table[b], 16), caches[b])
        for i, blk in enumerate(table[b]):  # block i of sequence b sits at its pool block
            np.testing.assert_array_equal(pool[blk], caches[b][16 * i:16 * (i + 1)])
    unused = sorted(set(range(11)) - set(table.reshape(-1).tolist()))
    assert len(unused) == 2 and np.all(pool[unused] == 0x7FC0)


def test_paged_cache_argument_errors_precede_launch():
    import torch
    if torch.cuda.is_available():  # fake device addresses: a lost check must not reach a real GPU
        pytest.skip("a CUDA device is present")
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    lay = _fake_fa(cfg)
    S = _FakeScratch(B.qwen35_scratch_bytes(c, 0))
    x, y, tab = 0x8000000, 0x9000000, 0xA000000
    f = B.qwen35_forward_full_attention

    def kv(**kw):
        a = dict(k=0x5000000, v=0x6000000, capacity=32, dtype=B.QWEN35_KV_BF16, k_scales=None, v_scales=None,
                 block_table=tab, block_tokens=8, reserved=0)
        a.update(kw)
        return B.qwen35_kv_cache(*a.values())

    bad = [kv(dtype=B.QWEN35_KV_TURBO8, k_scales=0xB000000, v_scales=0xC000000),  # paged is bf16 only
           kv(block_tokens=12),            # not a power of two
           kv(block_tokens=4),             # below 8 (a tile of 8 tokens must sit in one block)
           kv(capacity=36),                # capacity not a multiple of the block
           kv(block_table=tab + 2)]        # misaligned table
    for k in bad:
        assert f(c, lay, S, k, x, y, 3, 4, 0) == B.QWEN35_ERR_INVALID_ARGUMENT
    # well formed: past every check, then no device
    assert f(c, lay, S, kv(), x, y, 3, 4, 0) == B.QWEN35_ERR_CUDA
