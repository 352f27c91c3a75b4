"""Seeded random combinations of everything h3gqa_attention_fwd takes, each
checked in full against the fp64 oracle: sequence mixes (empty and one-token
sequences included), group sizes 2..128 with 1..3 KV heads, causal or
bidirectional, head- or token-major output, bf16 or int8 codes with row
scales, and the Q/K prologue in its forms (so the rotary path that reads its
tables from global memory, used when a unit has more than 32 tokens, is
covered as well as the staged one).
"""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300 import binding
from long_causal_gqa_gb300.inputs import make_inputs, norm_weights, rope_tables
from oracle import causal_gqa as orc

pytestmark = pytest.mark.gpu

SCALE = 128 ** -0.5
EPS = 1e-6
N_CASES = 16


def _cases():
    rng = np.random.default_rng(20261202)
    out = []
    for i in range(N_CASES):
        hkv = int(rng.choice([1, 2, 3]))
        g = int(rng.choice([gg for gg in (2, 4, 8, 16, 32, 64, 128) if gg * hkv <= 128]))
        n_seqs = int(rng.integers(1, 5))
        lens = [int(v) for v in rng.integers(0, 520, n_seqs)]
        if rng.random() < 0.3:
            lens[int(rng.integers(0, n_seqs))] = int(rng.choice([0, 1]))
        if sum(lens) == 0:
            lens[0] = 37
        out.append(dict(seqlens=tuple(lens), hq=g * hkv, hkv=hkv, causal=bool(rng.random() < 0.6),
                        token_major=bool(rng.random() < 0.4), int8=bool(rng.random() < 0.3),
                        prologue=str(rng.choice(["none", "qn", "rope", "all"])), seed=3000 + i))
    return out


def _cases_any_group():
    """Group sizes that do not divide 128 (G = 1, 3, 5, 6, 7, 12, 24), whose
    tiles leave MMA rows unused and whose units may straddle two key tiles."""
    rng = np.random.default_rng(20261203)
    out = []
    for i in range(10):
        hkv = int(rng.choice([1, 2, 3]))
        g = int(rng.choice([1, 3, 5, 6, 7, 12, 24]))
        lens = [int(v) for v in rng.integers(0, 700, int(rng.integers(1, 4)))]
        if sum(lens) == 0:
            lens[0] = 301
        out.append(dict(seqlens=tuple(lens), hq=g * hkv, hkv=hkv, causal=bool(rng.random() < 0.6),
                        token_major=bool(rng.random() < 0.4), int8=bool(rng.random() < 0.3),
                        prologue=str(rng.choice(["none", "qn", "rope", "all"])), seed=3200 + i))
    return out


# the rotary path that reads its tables from global memory (G < 8), which the
# seeded draw above happens not to reach
CASES = _cases() + _cases_any_group() + [
    dict(seqlens=(333, 0, 200), hq=8, hkv=2, causal=True, token_major=False, int8=False,
         prologue="all", seed=3100),
    dict(seqlens=(1, 451), hq=4, hkv=2, causal=False, token_major=True, int8=True,
         prologue="rope", seed=3101),
    dict(seqlens=(260,), hq=24, hkv=3, causal=True, token_major=False, int8=True,
         prologue="all", seed=3102),
]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return torch.device("cuda:0")


@pytest.mark.parametrize("case", CASES, ids=["case%d" % i for i in range(len(CASES))])
def test_random_combination(dev, case):
    seqlens, hq, hkv = case["seqlens"], case["hq"], case["hkv"]
    x = make_inputs(seqlens, hq, hkv, 128, case["seed"])
    wq, wk = norm_weights(128, case["seed"])
    cos, sin = rope_tables(seqlens, 128)
    use_qn = case["prologue"] in ("qn", "all")
    use_kn = case["prologue"] == "all"
    use_rope = case["prologue"] in ("rope", "all")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    kw = {}
    if use_qn or use_kn or use_rope:
        kw = dict(q_norm_weight=wq.to(dev) if use_qn else None,
                  k_norm_weight=wk.to(dev) if use_kn else None,
                  rope_cos=cos.to(dev) if use_rope else None,
                  rope_sin=sin.to(dev) if use_rope else None,
                  norm_eps=EPS, k_out=torch.empty_like(k))
    o, lse, o_scale = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE, causal=case["causal"],
                                            token_major=case["token_major"],
                                            out_int8=case["int8"], **kw)
    binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)

    rc, rs = (cos, sin) if use_rope else (None, None)
    q_att = orc.to_bf16(orc.qk_prep(x["q"], wq if use_qn else None, EPS, rc, rs)) \
        if (use_qn or use_rope) else x["q"]
    k_att = orc.to_bf16(orc.qk_prep(x["k"], wk if use_kn else None, EPS, rc, rs)) \
        if (use_kn or use_rope) else x["k"]
    ref_o, ref_lse = orc.causal_gqa(q_att, k_att, x["v"], x["cu_seqlens"], hq, hkv, SCALE,
                                    causal=case["causal"])
    if case["token_major"]:
        ref_o = ref_o.transpose(1, 0, 2)
    if case["int8"]:
        assert o.dtype == torch.int8
        step = o_scale.cpu().numpy().astype(np.float64)[..., None]
        got = o.cpu().numpy().astype(np.float64) * step
    else:
        step = 0.0
        got = o.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    excess = np.abs(got - ref_o) - (1e-2 + 1e-2 * np.abs(ref_o) + step)
    assert excess.max() <= 0, "%s: o over tolerance by %g" % (case, excess.max())
    lerr = np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse)
    assert lerr.max() <= 1e-3, "%s: lse off by %g" % (case, lerr.max())
