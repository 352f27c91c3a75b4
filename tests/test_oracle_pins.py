"""Pins of the fp64 oracle to things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, an
off-by-one causal bound, a wrong GQA head index, a swapped operand, a missing
scale, sequences leaking into each other) fails at least one of them:

- an independent dense numpy statement (tests/brute_force.py), 1e-12;
- torch's scaled_dot_product_attention in float64 on the CPU (a library
  routine; the GQA special case uses its enable_gqa head repetition);
- closed forms: the first row of a sequence, scale = 0, a one-hot logit;
- invariants: constant V, probability rows summing to one, future keys not
  mattering, GQA == explicit KV repetition, varlen == separate calls,
  linearity in V, invariance of o to a common shift of the keys (and the
  matching LSE shift).
"""
import math

import numpy as np
import pytest
import torch

from long_causal_gqa_gb300.inputs import make_inputs, cu_seqlens_of
from oracle import causal_gqa as orc
from tests.brute_force import bf16_bits_to_f64, dense_causal_gqa


def _bits(t):
    return orc.as_bf16_bits(t)


def _f64(t):
    return bf16_bits_to_f64(_bits(t))


def _bf16_from_f64(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


SHAPES = [
    # (seqlens, Hq, Hkv, D)
    ((1,), 1, 1, 8),
    ((17,), 2, 1, 8),
    ((33,), 4, 2, 8),
    ((64,), 8, 2, 128),
    ((5, 0, 11, 1, 20), 8, 1, 8),
    ((0, 31), 4, 4, 16),
]


@pytest.mark.parametrize("seqlens,hq,hkv,d", SHAPES)
def test_oracle_matches_dense_bruteforce(seqlens, hq, hkv, d):
    x = make_inputs(seqlens, hq, hkv, d, seed=7 + hq + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, scale)
    ob, lb, _ = dense_causal_gqa(_f64(x["q"]), _f64(x["k"]), _f64(x["v"]),
                                 x["cu_seqlens"].numpy(), scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("seqlens,hq,hkv,d", [((40,), 8, 2, 16), ((64,), 8, 1, 128),
                                              ((9, 23), 4, 2, 32)])
def test_oracle_matches_torch_sdpa_float64(seqlens, hq, hkv, d):
    x = make_inputs(seqlens, hq, hkv, d, seed=99)
    scale = 0.37
    o, _ = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, scale)
    cu = x["cu_seqlens"].tolist()
    q, k, v = (torch.from_numpy(_f64(x[n])) for n in ("q", "k", "v"))
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, s:e], k[None, :, s:e], v[None, :, s:e],
            is_causal=True, scale=scale, enable_gqa=True)[0]
        np.testing.assert_allclose(o[:, s:e], ref.numpy(), rtol=0, atol=1e-12)


def test_first_row_closed_form():
    """Row 0 of every sequence sees only its own key: o = v[g, s_b] and
    lse = scale * q . k exactly (the softmax of one logit is 1)."""
    seqlens = (7, 12, 1)
    hq, hkv, d = 8, 2, 16
    x = make_inputs(seqlens, hq, hkv, d, seed=3)
    scale = 0.25
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, scale)
    q, k, v = _f64(x["q"]), _f64(x["k"]), _f64(x["v"])
    for s in x["cu_seqlens"][:-1].tolist():
        for h in range(hq):
            g = h // (hq // hkv)
            np.testing.assert_allclose(o[h, s], v[g, s], rtol=0, atol=1e-14)
            assert abs(lse[h, s] - scale * float(q[h, s] @ k[g, s])) < 1e-12


def test_zero_scale_gives_prefix_mean():
    """scale = 0 makes every visible logit 0: o[i] is the mean of v[s_b..i]
    and lse[i] = ln(i - s_b + 1)."""
    seqlens = (10, 25)
    hq, hkv, d = 4, 1, 8
    x = make_inputs(seqlens, hq, hkv, d, seed=5)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.0)
    v = _f64(x["v"])
    cu = x["cu_seqlens"].tolist()
    for b in range(len(seqlens)):
        s, e = cu[b], cu[b + 1]
        prefix_mean = np.cumsum(v[0, s:e], axis=0) / np.arange(1, e - s + 1)[:, None]
        for h in range(hq):
            np.testing.assert_allclose(o[h, s:e], prefix_mean, rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[h, s:e], np.log(np.arange(1, e - s + 1)),
                                       rtol=0, atol=1e-13)


def test_one_hot_logit_selects_its_value_row():
    """With q = c*e_0 and only key 5 having a large k[...,0], every row i >= 5
    puts (almost) all its weight on key 5; rows i < 5 do not see it."""
    T, d = 12, 8
    q = np.zeros((1, T, d)); q[0, :, 0] = 4.0
    k = np.zeros((1, T, d)); k[0, 5, 0] = 8.0
    v = np.arange(T * d, dtype=np.float64).reshape(1, T, d) / 16.0
    cu = [0, T]
    o, lse = orc.causal_gqa(_bf16_from_f64(q), _bf16_from_f64(k), _bf16_from_f64(v),
                            cu, 1, 1, 1.0)
    vb = _f64(_bf16_from_f64(v))
    for i in range(5, T):
        # logit 32 against (i) logits of 0: weight of key 5 = 1/(1 + i e^-32)
        w = 1.0 / (1.0 + i * math.exp(-32.0))
        expect = w * vb[0, 5] + (1 - w) / i * (vb[0, :i + 1].sum(0) - vb[0, 5])
        np.testing.assert_allclose(o[0, i], expect, rtol=0, atol=1e-12)
        assert abs(lse[0, i] - (32.0 + math.log1p(i * math.exp(-32.0)))) < 1e-12
    for i in range(5):
        np.testing.assert_allclose(o[0, i], vb[0, :i + 1].mean(0), rtol=0, atol=1e-12)


def test_constant_v_gives_constant_output():
    hq, hkv, d, seqlens = 8, 2, 16, (30, 3)
    x = make_inputs(seqlens, hq, hkv, d, seed=11)
    vconst = torch.full_like(x["v"], 0.0)
    vconst[0] = 1.5
    vconst[1] = -0.75
    o, _ = orc.causal_gqa(x["q"], x["k"], vconst, x["cu_seqlens"], hq, hkv, 0.3)
    np.testing.assert_allclose(o[:4], 1.5, rtol=0, atol=1e-13)
    np.testing.assert_allclose(o[4:], -0.75, rtol=0, atol=1e-13)


def test_probability_rows_sum_to_one_and_are_causal():
    hq, hkv, d, seqlens = 4, 2, 16, (9, 14)
    x = make_inputs(seqlens, hq, hkv, d, seed=13)
    cu = x["cu_seqlens"].tolist()
    _, _, probs = dense_causal_gqa(_f64(x["q"]), _f64(x["k"]), _f64(x["v"]), cu, 0.5)
    for b in range(len(seqlens)):
        for h in range(hq):
            for i in range(cu[b], cu[b + 1]):
                p = orc.attention_probs(x["q"], x["k"], x["v"], cu, hq, hkv, 0.5, h, i)
                assert len(p) == i - cu[b] + 1
                assert abs(p.sum() - 1.0) < 1e-13
                assert (p > 0).all()
                np.testing.assert_allclose(p, probs[b][h, i - cu[b], :i - cu[b] + 1],
                                           rtol=0, atol=1e-14)


def test_future_keys_do_not_matter():
    hq, hkv, d, T = 8, 2, 16, 40
    x = make_inputs((T,), hq, hkv, d, seed=17)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.3)
    cut = 23
    k2, v2 = x["k"].clone(), x["v"].clone()
    g = torch.Generator().manual_seed(1)
    k2[:, cut + 1:] = torch.randn(k2[:, cut + 1:].shape, generator=g).to(torch.bfloat16)
    v2[:, cut + 1:] = torch.randn(v2[:, cut + 1:].shape, generator=g).to(torch.bfloat16)
    o2, lse2 = orc.causal_gqa(x["q"], k2, v2, x["cu_seqlens"], hq, hkv, 0.3)
    np.testing.assert_array_equal(o[:, :cut + 1], o2[:, :cut + 1])
    np.testing.assert_array_equal(lse[:, :cut + 1], lse2[:, :cut + 1])
    assert np.abs(o[:, cut + 1:] - o2[:, cut + 1:]).max() > 1e-3


def test_gqa_equals_explicit_kv_repetition():
    hq, hkv, d, seqlens = 8, 2, 16, (21, 6)
    x = make_inputs(seqlens, hq, hkv, d, seed=19)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.4)
    k_rep = x["k"].repeat_interleave(hq // hkv, dim=0)
    v_rep = x["v"].repeat_interleave(hq // hkv, dim=0)
    o2, lse2 = orc.causal_gqa(x["q"], k_rep, v_rep, x["cu_seqlens"], hq, hq, 0.4)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_varlen_equals_separate_calls():
    hq, hkv, d, seqlens = 4, 2, 16, (13, 0, 8, 19)
    x = make_inputs(seqlens, hq, hkv, d, seed=23)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.35)
    cu = x["cu_seqlens"].tolist()
    for b in range(len(seqlens)):
        s, e = cu[b], cu[b + 1]
        if s == e:
            continue
        ob, lb = orc.causal_gqa(x["q"][:, s:e].contiguous(), x["k"][:, s:e].contiguous(),
                                x["v"][:, s:e].contiguous(), [0, e - s], hq, hkv, 0.35)
        np.testing.assert_array_equal(o[:, s:e], ob)
        np.testing.assert_array_equal(lse[:, s:e], lb)


def test_linear_in_v():
    hq, hkv, d, seqlens = 4, 1, 8, (25,)
    x = make_inputs(seqlens, hq, hkv, d, seed=29)
    y = make_inputs(seqlens, hq, hkv, d, seed=31)
    cu = x["cu_seqlens"]
    # v1 + v2 is computed in fp64 from the bf16 bits, then checked against the
    # sum of the two outputs; both v's are exact bf16, their sum may not be,
    # so compare o(v1) + o(v2) with the brute force of the fp64 sum.
    o1, _ = orc.causal_gqa(x["q"], x["k"], x["v"], cu, hq, hkv, 0.5)
    o2, _ = orc.causal_gqa(x["q"], x["k"], y["v"], cu, hq, hkv, 0.5)
    ob, _, _ = dense_causal_gqa(_f64(x["q"]), _f64(x["k"]),
                                _f64(x["v"]) + 2.0 * _f64(y["v"]), cu.numpy(), 0.5)
    np.testing.assert_allclose(o1 + 2.0 * o2, ob, rtol=0, atol=1e-12)


def test_common_key_shift():
    """Adding u to every key of a sequence adds scale*q.u to each logit of a
    row: o is unchanged and lse shifts by exactly scale*q.u."""
    hq, hkv, d, T = 2, 1, 8, 16
    x = make_inputs((T,), hq, hkv, d, seed=37)
    # keys on a 1/8 grid in [-4, 4], so that the shifted keys (grid values in
    # [-4.5, 4.5]) are exact bf16 numbers as well
    k = np.clip(np.round(_f64(x["k"]) * 8.0) / 8.0, -4.0, 4.0)
    u = np.zeros(d); u[3] = 0.5; u[6] = -0.25
    k2 = k + u
    k_bf, k2_bf = _bf16_from_f64(k), _bf16_from_f64(k2)
    assert np.array_equal(_f64(k_bf), k) and np.array_equal(_f64(k2_bf), k2)
    o, lse = orc.causal_gqa(x["q"], k_bf, x["v"], x["cu_seqlens"], hq, hkv, 0.3)
    o2, lse2 = orc.causal_gqa(x["q"], k2_bf, x["v"], x["cu_seqlens"], hq, hkv, 0.3)
    q = _f64(x["q"])
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2 - lse, 0.3 * (q @ u), rtol=0, atol=1e-12)


def test_rows_api_matches_full():
    hq, hkv, d, seqlens = 8, 2, 16, (30, 1, 17)
    x = make_inputs(seqlens, hq, hkv, d, seed=41)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.3)
    rows = np.array([[0, 0], [7, 47], [3, 30], [5, 31], [1, 12]])
    orow, lrow = orc.causal_gqa_rows(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv,
                                     0.3, rows)
    for r, (h, t) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[h, t])
        assert lrow[r] == lse[h, t]


def test_oracle_rejects_bad_arguments():
    x = make_inputs((8,), 4, 2, 8, seed=1)
    with pytest.raises(ValueError):
        orc.causal_gqa(x["q"], x["k"], x["v"], [0, 8], 4, 3, 0.3)   # shape mismatch
    with pytest.raises(ValueError):
        orc.causal_gqa_rows(x["q"], x["k"], x["v"], [0, 8], 4, 2, 0.3, [[4, 0]])
    with pytest.raises(ValueError):
        orc.causal_gqa(x["q"][:, :6], x["k"], x["v"], [0, 8], 4, 2, 0.3)


def test_input_recipe_is_deterministic_and_bf16():
    a = make_inputs((5, 3), 4, 2, 8, seed=1234, n_outlier=2)
    b = make_inputs((5, 3), 4, 2, 8, seed=1234, n_outlier=2)
    for n in ("q", "k", "v"):
        assert a[n].dtype == torch.bfloat16
        assert torch.equal(a[n], b[n])
    assert torch.equal(a["outlier_channels"], b["outlier_channels"])
    assert a["cu_seqlens"].tolist() == [0, 5, 8]
    assert cu_seqlens_of([]).tolist() == [0]


# ------------------------------------------------------- bidirectional form
@pytest.mark.parametrize("seqlens,hq,hkv,d", [((17,), 2, 1, 8), ((5, 0, 11, 1, 20), 8, 1, 8),
                                              ((64,), 8, 2, 128)])
def test_bidirectional_matches_dense_bruteforce(seqlens, hq, hkv, d):
    x = make_inputs(seqlens, hq, hkv, d, seed=70 + hq + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, scale,
                            causal=False)
    ob, lb, _ = dense_causal_gqa(_f64(x["q"]), _f64(x["k"]), _f64(x["v"]),
                                 x["cu_seqlens"].numpy(), scale, causal=False)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_bidirectional_matches_torch_sdpa_float64():
    seqlens, hq, hkv, d = (9, 23), 4, 2, 32
    x = make_inputs(seqlens, hq, hkv, d, seed=71)
    o, _ = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.37, causal=False)
    q, k, v = (torch.from_numpy(_f64(x[n])) for n in ("q", "k", "v"))
    cu = x["cu_seqlens"].tolist()
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[None, :, s:e], k[None, :, s:e], v[None, :, s:e], is_causal=False, scale=0.37,
            enable_gqa=True)[0]
        np.testing.assert_allclose(o[:, s:e], ref.numpy(), rtol=0, atol=1e-12)


def test_bidirectional_is_invariant_to_key_order():
    """Without the causal rule a row sees a set of keys: permuting the keys
    and values of a sequence together changes no output (the causal form
    does change)."""
    seqlens, hq, hkv, d = (19, 12), 4, 2, 16
    x = make_inputs(seqlens, hq, hkv, d, seed=72)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.3, causal=False)
    perm = np.concatenate([np.random.default_rng(0).permutation(19),
                           19 + np.random.default_rng(1).permutation(12)])
    k2, v2 = x["k"][:, perm].contiguous(), x["v"][:, perm].contiguous()
    o2, lse2 = orc.causal_gqa(x["q"], k2, v2, x["cu_seqlens"], hq, hkv, 0.3, causal=False)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-12)
    oc, _ = orc.causal_gqa(x["q"], k2, v2, x["cu_seqlens"], hq, hkv, 0.3)
    oc0, _ = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.3)
    assert np.abs(oc - oc0).max() > 1e-3


def test_bidirectional_zero_scale_and_last_row():
    """scale = 0: every row of a sequence is the mean of all its values and
    lse = ln(S_b); and in general the last row of a sequence is the same in
    both forms (it sees every key either way)."""
    seqlens, hq, hkv, d = (10, 25), 4, 1, 8
    x = make_inputs(seqlens, hq, hkv, d, seed=73)
    o, lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, 0.0, causal=False)
    v = _f64(x["v"])
    cu = x["cu_seqlens"].tolist()
    for b in range(len(seqlens)):
        s, e = cu[b], cu[b + 1]
        np.testing.assert_allclose(o[:, s:e], np.broadcast_to(v[0, s:e].mean(0), o[:, s:e].shape),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, s:e], math.log(e - s), rtol=0, atol=1e-13)
    ob, lb = orc.causal_gqa(x["q"], x["k"], x["v"], cu, hq, hkv, 0.4, causal=False)
    oc, lc = orc.causal_gqa(x["q"], x["k"], x["v"], cu, hq, hkv, 0.4)
    for e in cu[1:]:
        np.testing.assert_array_equal(ob[:, e - 1], oc[:, e - 1])
        np.testing.assert_array_equal(lb[:, e - 1], lc[:, e - 1])
