"""GPU parity on shapes that exercise every branch of the persistent unit
schedule: whole windows of grid blocks with the KV head as the slow index
(an odd KV head count, so even and odd rounds swap walkers from one window
to the next), a partial last window, many (cost class, sequence) groups
crossed inside one window, one KV head (a window per round), and the
bidirectional walk. Every output row is compared with the fp64 oracle, so a
unit that is skipped, repeated or given the wrong KV head fails.
"""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300 import binding
from long_causal_gqa_gb300.inputs import make_inputs
from oracle import causal_gqa as orc
from tests.test_gpu_parity import assert_close, full_check

pytestmark = pytest.mark.gpu

SCALE = 128 ** -0.5


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return torch.device("cuda:0")


def _windows(seqlens, hq, hkv, grid):
    """(whole windows, slots) of the schedule for a grid of `grid` CTAs."""
    unit = 2 * (128 // (hq // hkv))
    slots = sum((s + unit - 1) // unit for s in seqlens if s > 0)
    g = min(grid, slots * hkv)
    return slots // g, slots


@pytest.mark.parametrize("seqlens,hq,hkv", [
    ((5000,), 24, 3),                         # odd Hkv, one whole window + partial
    ((3000, 2500, 1700, 900, 130), 64, 8),    # many class/sequence groups per window
    ((1000,), 128, 1),                        # one KV head: every round is a window
    ((2600, 0, 2410), 48, 3),                 # odd Hkv, two sequences, two windows
])
def test_causal_schedule_shapes(dev, seqlens, hq, hkv):
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    whole, _ = _windows(seqlens, hq, hkv, sms)
    assert whole >= 1, "shape must reach at least one whole window on this GPU"
    full_check(seqlens, hq, hkv, 4000 + sum(seqlens) + hq, dev)


def test_bidirectional_schedule_odd_heads(dev):
    seqlens, hq, hkv = (5000, 377), 24, 3
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert _windows(seqlens, hq, hkv, sms)[0] >= 1
    x = make_inputs(seqlens, hq, hkv, 128, seed=4242)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse, _ = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE, causal=False)
    binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, SCALE,
                                    causal=False)
    assert_close(o.float().cpu().numpy().astype(np.float64),
                 lse.cpu().numpy().astype(np.float64), ref_o, ref_lse, "bidirectional odd Hkv")
