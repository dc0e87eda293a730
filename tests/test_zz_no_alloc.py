"""The linear-attention forward that allocates nothing (static library scratch),
for callers that cannot call cudaMalloc, checked against the regular forward.

Both run the same kernel, in the same launch shape, on the same inputs, and every
reduction in it runs in a fixed order, so the outputs and the updated states must
agree bit for bit: any difference would point at the static array's use (an
offset, a stale word), not at rounding.

It runs in a file of its own that pytest collects last, so that a failure here
leaves every other test already run. It also passes alone in a fresh process.
"""

import numpy as np
import pytest
import torch

from full_attention_decode_gb300 import binding as B
from full_attention_decode_gb300 import synth

from harness import init

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg_name", ["tiny", "4b"])
def test_static_scratch_forward_matches_regular_forward_twice(cfg_name):
    init()
    cfg = synth.config(cfg_name)
    c = B.make_config(cfg)
    assert B.qwen35_scratch_bytes(c, B.QWEN35_LAYER_LINEAR_ATTENTION) <= 256 * 1024
    dev = B.DeviceGdnLayer(synth.gdn_layer(3, 0, cfg))
    conv, ssm = synth.gdn_state(3, 0, cfg, std=0.1)
    st_ref, st_new = B.DeviceState(conv, ssm), B.DeviceState(conv, ssm)
    scratch = B.new_scratch(B.qwen35_scratch_bytes(c, B.QWEN35_LAYER_LINEAR_ATTENTION))
    x_in = torch.empty(cfg["hidden"], dtype=torch.int16, device="cuda")
    y_ref, y_new = torch.empty_like(x_in), torch.empty_like(x_in)
    for t in range(2):  # two calls in a row: the second reuses the array and the updated state
        x_in.copy_(B.to_device(synth.x_in(3, t, cfg)))
        assert B.qwen35_forward_linear_attention(c, dev.struct, scratch, st_ref.struct, x_in, y_ref) == 0
        assert B.qwen35_forward_linear_attention_static(c, dev.struct, st_new.struct, x_in, y_new) == 0
        assert B.qwen35_read_static_status() == 0, t  # synchronises the stream
        torch.cuda.synchronize()
        assert torch.equal(y_new, y_ref), t
        assert torch.equal(st_new.ssm, st_ref.ssm), t
        assert torch.equal(st_new.conv, st_ref.conv), t
    assert B.qwen35_read_device_status(scratch) == 0


def test_static_scratch_rejects_oversized_config():
    init()
    cfg = synth.config("4b")
    cfg["hidden"] = cfg["intermediate"] = 12288  # linear-attention scratch beyond the static array
    c = B.make_config(cfg)
    assert B.qwen35_scratch_bytes(c, B.QWEN35_LAYER_LINEAR_ATTENTION) > 256 * 1024
    lay = B.qwen35_gdn_layer()
    st = B.qwen35_gdn_state(0, 0)
    assert B.qwen35_forward_linear_attention_static(c, lay, st, 0, 0) == B.QWEN35_ERR_UNSUPPORTED
