"""Pins of the oracle's Q/K prologue (RMS norm, rotary embedding), CPU only.

Library special case (torch rms_norm in float64), closed forms (unit mean
square, the eps shift, identity tables) and invariants of the rotation
(pair norms kept, dot products depend only on the position difference,
angles add) -- each fails for a plausible slip: wrong pairing, a sign, a
dropped weight, eps or mean.
"""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300.inputs import make_inputs, norm_weights, rope_tables
from oracle import causal_gqa as orc
from tests.brute_force import bf16_bits_to_f64

D = 128


def _f64(t):
    return bf16_bits_to_f64(orc.as_bf16_bits(t))


def _x(seed, heads=3, T=11):
    return make_inputs((T,), heads, 1, D, seed)["q"]


def test_rms_norm_matches_torch_float64():
    x = _x(1)
    w, _ = norm_weights(D, 1)
    y = orc.qk_prep(x, w, eps=1e-5)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(_f64(x)), (D,),
                                       torch.from_numpy(_f64(w)), eps=1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=0, atol=1e-12)


def test_unit_weight_gives_unit_mean_square_and_eps_shift():
    x = _x(2)
    ones = torch.ones(D, dtype=torch.bfloat16)
    y0 = orc.qk_prep(x, ones, eps=0.0)
    np.testing.assert_allclose((y0 ** 2).mean(-1), 1.0, rtol=0, atol=1e-12)
    # with eps: mean square = ms / (ms + eps)
    ms = (_f64(x) ** 2).mean(-1)
    y1 = orc.qk_prep(x, ones, eps=0.5)
    np.testing.assert_allclose((y1 ** 2).mean(-1), ms / (ms + 0.5), rtol=0, atol=1e-12)


def test_norm_is_scale_invariant():
    x = _x(3)
    w, _ = norm_weights(D, 3)
    x4 = (x.float() * 4.0).to(torch.bfloat16)          # exact power-of-two scaling
    np.testing.assert_allclose(orc.qk_prep(x4, w, 0.0), orc.qk_prep(x, w, 0.0), rtol=0, atol=1e-12)


def test_identity_tables_leave_rows_unchanged():
    x = _x(4)
    T = x.shape[1]
    c = torch.ones((T, D // 2))
    s = torch.zeros((T, D // 2))
    np.testing.assert_array_equal(orc.qk_prep(x, rope_cos=c, rope_sin=s), _f64(x))


def test_rotation_keeps_pair_norms():
    x = _x(5)
    c, s = rope_tables((x.shape[1],), D)
    y = orc.qk_prep(x, rope_cos=c, rope_sin=s)
    xf = _f64(x)
    pn_x = xf[..., :D // 2] ** 2 + xf[..., D // 2:] ** 2
    pn_y = y[..., :D // 2] ** 2 + y[..., D // 2:] ** 2
    np.testing.assert_allclose(pn_y, pn_x, rtol=1e-6, atol=1e-9)
    # and it does rotate (position 0 is the identity, later positions are not)
    np.testing.assert_allclose(y[:, 0], xf[:, 0], rtol=0, atol=1e-12)
    assert np.abs(y[:, 5] - xf[:, 5]).max() > 1e-2


def test_rotated_dot_product_depends_on_position_difference():
    """q at position m against k at position n equals q at m+d against k at
    n+d: the relative-position property of the rotary embedding."""
    T = 64
    x = _x(6, heads=2, T=T)
    c, s = rope_tables((T,), D)
    same_q = x[0:1, :1].expand(1, T, D).contiguous()      # one vector at every position
    same_k = x[1:2, :1].expand(1, T, D).contiguous()
    rq = orc.qk_prep(same_q, rope_cos=c, rope_sin=s)[0]
    rk = orc.qk_prep(same_k, rope_cos=c, rope_sin=s)[0]
    for m, n, d in ((10, 3, 20), (40, 40, 7), (5, 30, 25)):
        a = rq[m] @ rk[n]
        b = rq[m + d] @ rk[n + d]
        assert abs(a - b) <= 1e-4 * (1 + abs(a))


def test_rotation_angles_add():
    x = _x(7)
    T = x.shape[1]
    rng = np.random.default_rng(7)
    a1 = rng.uniform(-3, 3, (T, D // 2))
    a2 = rng.uniform(-3, 3, (T, D // 2))
    tab = lambda a: (torch.from_numpy(np.cos(a).astype(np.float32)),
                     torch.from_numpy(np.sin(a).astype(np.float32)))
    y1 = orc.qk_prep(x, rope_cos=tab(a1)[0], rope_sin=tab(a1)[1])
    y12 = orc.qk_prep(orc.to_bf16(y1), rope_cos=tab(a2)[0], rope_sin=tab(a2)[1])
    y3 = orc.qk_prep(x, rope_cos=tab(a1 + a2)[0], rope_sin=tab(a1 + a2)[1])
    # the intermediate bf16 rounding bounds the agreement
    np.testing.assert_allclose(y12, y3, rtol=0, atol=3e-2)
    assert np.abs(y12 - y3).mean() < 4e-3


def test_rejects_bad_tables():
    x = _x(8)
    with pytest.raises(ValueError):
        orc.qk_prep(x, rope_cos=torch.ones((3, 64)), rope_sin=torch.zeros((3, 64)))
