"""GPU parity of the Q/K prologue (RMS norm + rotary embedding) against the
fp64 oracle: the prepared keys written to k_out agree with the oracle's
within one bf16 rounding, and the attention computed on the fly from the
raw q agrees with the oracle's attention on the oracle's prepared q and k
(each rounded to bf16, as on the GPU) within the attention tolerance."""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300 import binding
from long_causal_gqa_gb300.inputs import make_inputs, norm_weights, rope_tables
from oracle import causal_gqa as orc
from tests.brute_force import bf16_bits_to_f64

pytestmark = pytest.mark.gpu
SCALE = 128 ** -0.5
EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return torch.device("cuda:0")


def _case(seqlens, seed, use_qn, use_kn, use_rope, causal, dev, in_place=False, hq=64, hkv=8):
    x = make_inputs(seqlens, hq, hkv, 128, seed)
    wq, wk = norm_weights(128, seed)
    cos, sin = rope_tables(seqlens, 128)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    k_out = k if in_place else torch.full_like(k, float("nan"))
    o, lse, _ = binding.attention_fwd(
        q, k, v, x["cu_seqlens"], SCALE, causal=causal,
        q_norm_weight=wq.to(dev) if use_qn else None,
        k_norm_weight=wk.to(dev) if use_kn else None,
        rope_cos=cos.to(dev) if use_rope else None, rope_sin=sin.to(dev) if use_rope else None,
        norm_eps=EPS, k_out=k_out)
    binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)
    rc, rs = (cos, sin) if use_rope else (None, None)
    q_ref = orc.qk_prep(x["q"], wq if use_qn else None, EPS, rc, rs)
    k_ref = orc.qk_prep(x["k"], wk if use_kn else None, EPS, rc, rs)
    if use_kn or use_rope:
        got = bf16_bits_to_f64(orc.as_bf16_bits(k_out.cpu()))
        ref = bf16_bits_to_f64(orc.as_bf16_bits(orc.to_bf16(k_ref)))
        assert np.isfinite(got).all()
        # one bf16 step of the value, plus fp32 cancellation in the rotation
        # (a*c - b*s of O(1) terms can land near 0, where fp32 and fp64 differ
        # by ~1e-7 absolute)
        assert (np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-5).all(), \
            "prepared keys off by more than one bf16 step"
        assert (got == ref).mean() > 0.99
        k_att = orc.to_bf16(k_ref)
    else:
        k_att = x["k"]
    ro, rl = orc.causal_gqa(orc.to_bf16(q_ref), k_att, x["v"], x["cu_seqlens"], hq, hkv, SCALE,
                            causal=causal)
    o64 = o.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(o64).all()
    excess = np.abs(o64 - ro) - (1e-2 + 1e-2 * np.abs(ro))
    assert excess.max() <= 0, excess.max()
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3


@pytest.mark.parametrize("use_qn,use_kn,use_rope", [(True, True, True), (False, False, True),
                                                     (True, True, False), (True, False, False)])
def test_prologue_combinations(dev, use_qn, use_kn, use_rope):
    _case((300, 0, 129, 5), 61, use_qn, use_kn, use_rope, True, dev)


def test_prologue_bidirectional_and_in_place(dev):
    _case((200, 77), 62, True, True, True, False, dev, in_place=True)


def test_prologue_long_sequence(dev):
    _case((2100,), 63, True, True, True, True, dev)


@pytest.mark.parametrize("hq,hkv,causal", [(256, 1, True), (256, 2, False), (131, 1, True)])
def test_prologue_tiles_beyond_one_group(dev, hq, hkv, causal):
    """Group sizes above 128 (a KV head's query heads span several tiles:
    G = 256 packs 128 heads x 1 token per tile, with the rotary rows staged
    beside Q) and a prime G = 131 (one head x 128 tokens per tile, rotary
    rows read from global memory), with every part of the prologue."""
    _case((70, 0, 9), 64 + hq + hkv, True, True, True, causal, dev, hq=hq, hkv=hkv)
