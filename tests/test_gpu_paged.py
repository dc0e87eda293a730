"""Paged KV caches (a block table over the split-KV attention; the module page's
production decode path) against the oracle on the logical cache, through the C
ABI. The pool's blocks are placed by a shuffled table and every block no table
names holds bf16 NaN, so a read of a wrong block shows in the output.

Tolerances: the layer output within the layer tolerance (relative L2 1e-2); the
appended rows bit for bit against the same forward on a contiguous cache (the two
layouts give the kernel the same rows in the same order), and every other pool row
unchanged."""

import numpy as np
import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O

from harness import bits, f64, init, rel_l2

pytestmark = pytest.mark.gpu

TOL_X = 1e-2
NAN = 0x7FC0


class PagedFa:
    """One full-attention layer over a paged cache, beside the same layer over a
    contiguous copy of the cache (both on the GPU) and the oracle."""

    def __init__(self, cfg_name, capacity, n_prefill, bt, spare_blocks=3, seed=0):
        init()
        self.cfg = synth.config(cfg_name)
        self.c = B.make_config(self.cfg)
        self.seed = seed
        self.layer = synth.fa_layer(seed, 1, self.cfg)
        k, v = synth.kv_cache(seed, 1, self.cfg, capacity, n_prefill)
        nl = capacity // bt
        self.table = synth.block_table(seed + 7, 1, nl, nl + spare_blocks)
        self.dev = B.DeviceFaLayer(self.layer)
        self.paged = B.DeviceKvPaged([k], [v], bt, self.table, nl + spare_blocks, fill=NAN)
        self.flat = B.DeviceKv(k, v)
        self.okv = O.kv_from_bits(k, v)
        nb = B.qwen35_scratch_bytes(self.c, B.QWEN35_LAYER_FULL_ATTENTION)
        self.scratch, self.scratch2 = B.new_scratch(nb), B.new_scratch(nb)
        self.x_in = torch.empty(self.cfg["hidden"], dtype=torch.int16, device="cuda")
        self.out_p, self.out_f = torch.empty_like(self.x_in), torch.empty_like(self.x_in)

    def step(self, t, cache_pos):
        x = synth.x_in(self.seed, t, self.cfg)
        self.x_in.copy_(B.to_device(x))
        for kv, out, scr in ((self.paged, self.out_p, self.scratch), (self.flat, self.out_f, self.scratch2)):
            rc = B.qwen35_forward_full_attention(self.c, self.dev.struct, scr, kv.struct, self.x_in, out, cache_pos,
                                                 cache_pos + 1)
            assert rc == 0, rc
        ref = O.forward_full_attention(self.cfg, self.layer, self.okv, O.bf16_to_f64(x), cache_pos, cache_pos + 1)
        torch.cuda.synchronize()
        return f64(self.out_p), f64(self.out_f), ref


def check_pool(r, pos):
    """The logical cache read back from the pool equals the contiguous cache (the
    appended rows included, bit for bit); the unnamed blocks still hold NaN."""
    for w, flat in (("k", r.flat.k), ("v", r.flat.v)):
        np.testing.assert_array_equal(r.paged.logical(w)[:pos + 1], bits(flat)[:pos + 1])
        pool = r.paged.pool(w)
        unused = sorted(set(range(pool.shape[0])) - set(r.table.reshape(-1).tolist()))
        assert np.all(pool[unused] == NAN)


def test_paged_layer_tiny_16_steps():
    r = PagedFa("tiny", 32, 0, 8)
    for t in range(16):
        got, flat, ref = r.step(t, t)
        assert rel_l2(got, ref) <= TOL_X, t
        np.testing.assert_array_equal(bits(r.out_p), bits(r.out_f))  # same rows, same order
        check_pool(r, t)
    assert B.qwen35_read_device_status(r.scratch) == 0


@pytest.mark.parametrize("cache_pos", [511, 1000, 4095])
def test_paged_layer_4b(cache_pos):
    r = PagedFa("4b", (cache_pos + 1 + 15) // 16 * 16 + 16, cache_pos, 16)
    got, flat, ref = r.step(0, cache_pos)
    assert rel_l2(got, ref) <= TOL_X
    np.testing.assert_array_equal(bits(r.out_p), bits(r.out_f))
    check_pool(r, cache_pos)
    assert B.qwen35_read_device_status(r.scratch) == 0


@pytest.mark.parametrize("use_graph", [False, True])
def test_paged_tiny_stack(use_graph):
    init()
    cfg = synth.config("tiny")
    kinds = synth.layer_kinds(cfg)
    layers = [synth.gdn_layer(0, 0, cfg), synth.fa_layer(0, 1, cfg)]
    conv, ssm = synth.gdn_state(0, 0, cfg)
    kb, vb = synth.kv_cache(0, 1, cfg, 32, 0)
    table = synth.block_table(3, 1, 4, 6)
    dev = [B.DeviceGdnLayer(layers[0]), B.DeviceFaLayer(layers[1])]
    caches = [B.DeviceState(conv, ssm), B.DeviceKvPaged([kb], [vb], 8, table, 6, fill=NAN)]
    ocaches = [O.state_from_arrays(conv, ssm), O.kv_from_bits(kb, vb)]
    c = B.make_config(cfg)
    entries = [B.stack_layer(k, l, cc) for k, l, cc in zip(kinds, dev, caches)]
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes(c))
    x_in = torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    d_pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    g = None
    if use_graph:
        with torch.cuda.stream(stream):
            g = B.Graph(c, entries, scratch, x_in, x_out, d_pos, 32)
    for t in range(12):
        x = synth.x_in(0, t, cfg)
        with torch.cuda.stream(stream):
            x_in.copy_(B.to_device(x))
            if g is not None:
                g.launch()
            else:
                assert B.qwen35_decode_step(c, entries, scratch, x_in, x_out, d_pos, 32) == 0
        ref = O.decode_step(cfg, kinds, layers, ocaches, O.bf16_to_f64(x), t)
        stream.synchronize()
        assert rel_l2(f64(x_out), ref) <= TOL_X, t
    assert int(d_pos.item()) == 12
    assert B.qwen35_read_device_status(scratch, stream) == 0
    if g is not None:
        g.close()


def test_paged_batched_forward_shares_one_pool():
    """qwen35_forward_full_attention_batched on three sequences whose caches share
    one pool through disjoint tables."""
    init()
    cfg = synth.config("tiny")
    c = B.make_config(cfg)
    E = cfg["hidden"]
    positions = [0, 9, 23]
    nb, cap, bt = len(positions), 32, 8
    layer = synth.fa_layer(4, 1, cfg)
    dev = B.DeviceFaLayer(layer)
    kvs = [synth.kv_cache(60 + s, 1, cfg, cap, p) for s, p in enumerate(positions)]
    table = synth.block_table(11, nb, cap // bt, nb * cap // bt + 2)
    pkv = B.DeviceKvPaged([k for k, _ in kvs], [v for _, v in kvs], bt, table, nb * cap // bt + 2, fill=NAN)
    scratch = B.new_scratch(B.qwen35_stack_scratch_bytes_batched(c, nb))
    x_in = torch.empty(nb * E, dtype=torch.int16, device="cuda")
    x_out = torch.empty_like(x_in)
    dpos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    xs = [synth.x_in(60 + s, 0, cfg) for s in range(nb)]
    x_in.copy_(B.to_device(np.concatenate(xs)))
    assert B.qwen35_forward_full_attention_batched(c, dev.struct, nb, scratch, pkv.struct, x_in, x_out, dpos,
                                                   cap) == 0
    torch.cuda.synchronize()
    got = O.bf16_to_f64(bits(x_out).reshape(nb, E))
    for s, p in enumerate(positions):
        okv = O.kv_from_bits(*kvs[s])
        tr = {}
        ref = O.forward_full_attention(cfg, layer, okv, O.bf16_to_f64(xs[s]), p, p + 1, tr)
        assert rel_l2(got[s], ref) <= TOL_X, s
        # the appended v row, read back through the table, is the layer's v projection
        assert rel_l2(O.bf16_to_f64(pkv.logical("v", s)[p]).reshape(-1), tr["v"].reshape(-1)) <= TOL_X
        # rows other than p of sequence s unchanged
        lk = pkv.logical("k", s)
        rows = [i for i in range(cap) if i != p]
        np.testing.assert_array_equal(lk[rows], kvs[s][0][rows])
    assert B.qwen35_read_device_status(scratch) == 0
