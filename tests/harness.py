"""Helpers shared by the GPU parity tests: run layers through the C ABI and the
same steps through the CPU oracle, on the same seeded inputs."""

from __future__ import annotations

import numpy as np
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth
from oracle import qwen35_oracle as O

_inited = False


def init():
    global _inited
    if not _inited:
        torch.cuda.set_device(0)
        B.qwen35_init()
        _inited = True


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def bits(t: torch.Tensor) -> np.ndarray:
    return B.bf16_tensor_bits(t)


def f64(t: torch.Tensor) -> np.ndarray:
    """Device bf16 (int16 storage) tensor -> float64 values."""
    return O.bf16_to_f64(bits(t))


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.float64)


def bf16_ulps(got, ref) -> np.ndarray:
    """Distance in bf16 units in the last place (both arrays hold bf16 values)."""
    g = O.bf16_bits(got).astype(np.int32)
    r = O.bf16_bits(ref).astype(np.int32)
    # map sign-magnitude bit patterns to a monotonic integer line
    g = np.where(g & 0x8000, -(g & 0x7FFF), g)
    r = np.where(r & 0x8000, -(r & 0x7FFF), r)
    return np.abs(g - r)


class GdnRunner:
    """One linear-attention layer on the GPU and in the oracle, stepped together."""

    def __init__(self, cfg_name: str, seed: int = 0, layer: int = 0, state_std: float = 0.0):
        init()
        self.cfg = synth.config(cfg_name)
        self.c = B.make_config(self.cfg)
        self.seed = seed
        self.layer = synth.gdn_layer(seed, layer, self.cfg)
        conv, ssm = synth.gdn_state(seed, layer, self.cfg, state_std)
        self.dev = B.DeviceGdnLayer(self.layer)
        self.state = B.DeviceState(conv, ssm)
        self.ostate = O.state_from_arrays(conv, ssm)
        self.scratch = B.new_scratch(B.qwen35_scratch_bytes(self.c, B.QWEN35_LAYER_LINEAR_ATTENTION))
        self.x_in = torch.empty(self.cfg["hidden"], dtype=torch.int16, device="cuda")
        self.x_out = torch.empty_like(self.x_in)

    def step(self, t: int, trace=None):
        x = synth.x_in(self.seed, t, self.cfg)
        self.x_in.copy_(B.to_device(x))
        rc = B.qwen35_forward_linear_attention(self.c, self.dev.struct, self.scratch, self.state.struct,
                                               self.x_in, self.x_out)
        assert rc == 0, rc
        ref = O.forward_linear_attention(self.cfg, self.layer, self.ostate, O.bf16_to_f64(x), trace)
        torch.cuda.synchronize()
        return f64(self.x_out), ref

    def view(self, name, n):
        return O.bf16_to_f64(bits(B.scratch_view(self.scratch, self.c, 1, name, n)))


class FaRunner:
    """One full-attention layer on the GPU and in the oracle, on the same cache."""

    def __init__(self, cfg_name: str, capacity: int, n_prefill: int, seed: int = 0, layer: int = 1):
        init()
        self.cfg = synth.config(cfg_name)
        self.c = B.make_config(self.cfg)
        self.seed = seed
        self.layer = synth.fa_layer(seed, layer, self.cfg)
        k, v = synth.kv_cache(seed, layer, self.cfg, capacity, n_prefill)
        self.dev = B.DeviceFaLayer(self.layer)
        self.kv = B.DeviceKv(k, v)
        self.okv = O.kv_from_bits(k, v)
        self.scratch = B.new_scratch(B.qwen35_scratch_bytes(self.c, B.QWEN35_LAYER_FULL_ATTENTION))
        self.x_in = torch.empty(self.cfg["hidden"], dtype=torch.int16, device="cuda")
        self.x_out = torch.empty_like(self.x_in)

    def step(self, t: int, cache_pos: int, seq_len: int | None = None, trace=None, dpos=None):
        if seq_len is None:
            seq_len = cache_pos + 1
        x = synth.x_in(self.seed, t, self.cfg)
        self.x_in.copy_(B.to_device(x))
        if dpos is None:
            rc = B.qwen35_forward_full_attention(self.c, self.dev.struct, self.scratch, self.kv.struct,
                                                 self.x_in, self.x_out, cache_pos, seq_len)
        else:
            dpos.fill_(cache_pos)
            rc = B.qwen35_forward_full_attention_dpos(self.c, self.dev.struct, self.scratch, self.kv.struct,
                                                      self.x_in, self.x_out, dpos, self.kv.struct.capacity)
        assert rc == 0, rc
        ref = O.forward_full_attention(self.cfg, self.layer, self.okv, O.bf16_to_f64(x), cache_pos, seq_len,
                                       trace)
        torch.cuda.synchronize()
        return f64(self.x_out), ref

    def view(self, name, n):
        return O.bf16_to_f64(bits(B.scratch_view(self.scratch, self.c, 0, name, n)))
