"""GPU parity of h3gqa_attention_fwd's options against the fp64 oracle.

- causal = 0 (bidirectional, every key of the sequence): full checks on
  small and ragged shapes, sampled rows at the 19316-row DiT size;
- token-major output: bitwise the head-major result, transposed;
- int8 output with one scale per (token, head) row: the dequantized value is
  within the attention tolerance plus one quantization step of the oracle,
  and within half a step (plus bf16 rounding) of the bf16 result.
"""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300 import binding
from long_causal_gqa_gb300.inputs import make_inputs
from oracle import causal_gqa as orc

pytestmark = pytest.mark.gpu

SCALE = 128 ** -0.5


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return torch.device("cuda:0")


def _run(x, dev, **opts):
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse, o_scale = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE, **opts)
    binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)
    return o.cpu(), lse.cpu(), (o_scale.cpu() if o_scale is not None else None)


def _check(o, lse, ref_o, ref_lse, what):
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    excess = np.abs(o - ref_o) - (1e-2 + 1e-2 * np.abs(ref_o))
    assert excess.max() <= 0, "%s: o over tolerance by %g" % (what, excess.max())
    assert np.abs(lse - ref_lse).max() <= 1e-3, "%s: lse off by %g" % (
        what, np.abs(lse - ref_lse).max())


@pytest.mark.parametrize("seqlens", [(1,), (17,), (128,), (129,), (300,), (5, 0, 129, 1, 300)])
def test_bidirectional_full(dev, seqlens):
    x = make_inputs(seqlens, 64, 8, 128, seed=300 + sum(seqlens))
    o, lse, _ = _run(x, dev, causal=False)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], 64, 8, SCALE,
                                    causal=False)
    _check(o.float().numpy(), lse.numpy(), ref_o, ref_lse, "bidirectional %s" % (seqlens,))


def test_bidirectional_dit_size_sampled(dev):
    S = 19316
    x = make_inputs((S,), 64, 8, 128, seed=19316)
    o, lse, _ = _run(x, dev, causal=False)
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, 64, 160), rng.integers(0, S, 160)], axis=1)
    rows = np.concatenate([rows, [[0, 0], [63, S - 1], [7, 128], [8, 127], [9, S - 128]]])
    ref_o, ref_lse = orc.causal_gqa_rows(x["q"], x["k"], x["v"], x["cu_seqlens"], 64, 8, SCALE,
                                         rows, causal=False)
    h, t = torch.from_numpy(rows[:, 0]), torch.from_numpy(rows[:, 1])
    _check(o[h, t].float().numpy(), lse[h, t].numpy(), ref_o, ref_lse, "S=19316 bidirectional")
    assert bool(torch.isfinite(o.float()).all())


@pytest.mark.parametrize("causal", [True, False])
def test_token_major_is_the_transposed_head_major(dev, causal):
    x = make_inputs((700, 0, 333), 64, 8, 128, seed=41)
    o_h, lse_h, _ = _run(x, dev, causal=causal)
    o_t, lse_t, _ = _run(x, dev, causal=causal, token_major=True)
    assert o_t.shape == (1033, 64, 128)
    assert torch.equal(o_t.permute(1, 0, 2), o_h)
    assert torch.equal(lse_t, lse_h)


def test_int8_rows_too_small_to_scale(dev):
    """Rows whose max|o| is at most 3.75e-37 (127 / max|o| would overflow
    fp32) are written as all-zero codes with scale max|o| / 127: no NaN or
    saturated codes. Every o row is a convex combination of v rows, so with
    |v| < 3.7e-37 every row is such a row, whatever the tensor cores do with
    the denormal products; the LSE does not depend on v."""
    x = make_inputs((300, 77), 16, 2, 128, seed=43)
    x["v"] = (x["v"].float() * 5e-38).to(torch.bfloat16)
    assert float(x["v"].float().abs().max()) < 3.7e-37
    codes, lse, scale = _run(x, dev, causal=True, token_major=False, out_int8=True)
    _, lse_bf, _ = _run(x, dev, causal=True, token_major=False)
    assert int(codes.abs().max()) == 0
    assert torch.isfinite(scale).all() and float(scale.min()) >= 0.0
    assert float(scale.max()) <= 3.75e-37 / 127.0
    assert torch.equal(lse, lse_bf)


@pytest.mark.parametrize("token_major,causal", [(False, True), (True, True), (True, False)])
def test_int8_output(dev, token_major, causal):
    x = make_inputs((640, 77), 64, 8, 128, seed=42)
    codes, lse, scale = _run(x, dev, causal=causal, token_major=token_major, out_int8=True)
    o_bf, lse_bf, _ = _run(x, dev, causal=causal, token_major=token_major)
    assert codes.dtype == torch.int8 and scale.dtype == torch.float32
    assert torch.equal(lse, lse_bf)
    assert int(codes.abs().max()) <= 127
    deq = codes.float() * scale[..., None]
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], 64, 8, SCALE,
                                    causal=causal)
    if token_major:
        ref_o = ref_o.transpose(1, 0, 2)
    step = scale.numpy().astype(np.float64)[..., None]
    # against the oracle: attention tolerance plus one quantization step
    err = np.abs(deq.numpy() - ref_o) - (1e-2 + 1e-2 * np.abs(ref_o) + step)
    assert err.max() <= 0, err.max()
    # scales: max|o| / 127 of the row
    amax = np.abs(ref_o).max(-1)
    np.testing.assert_allclose(scale.numpy(), amax / 127.0, rtol=2e-2, atol=1e-6)
    # against the bf16 output of the same kernel: half a step plus bf16 rounding
    ob = o_bf.float().numpy()
    assert (np.abs(deq.numpy() - ob) <= 0.5 * step + np.abs(ob) * 2.0 ** -8 + 1e-6).all()


@pytest.mark.parametrize("hq,hkv", [(3, 1), (131, 1), (24, 8)])
def test_epilogue_forms_with_unusual_tiles(dev, hq, hkv):
    """Token-major bf16 is bitwise the transpose of head-major, and int8 codes
    dequantize to the bf16 output within half a step (plus bf16 rounding),
    for tiles with unused rows (G = 3: 126 of 128), one head per tile
    (G = 131) and a non-power-of-two divisor (G = 3 of Hq/Hkv = 24/8)."""
    x = make_inputs((300, 0, 77), hq, hkv, 128, seed=500 + hq)
    o_h, lse_h, _ = _run(x, dev, causal=True)
    o_t, lse_t, _ = _run(x, dev, causal=True, token_major=True)
    assert torch.equal(o_t, o_h.transpose(0, 1)) and torch.equal(lse_t, lse_h)
    codes, lse_q, scale = _run(x, dev, causal=True, token_major=True, out_int8=True)
    assert torch.equal(lse_q, lse_h)
    assert int(codes.abs().max()) <= 127
    deq = codes.float() * scale[..., None]
    ob = o_t.float()
    step = scale[..., None]
    assert (np.abs((deq - ob).numpy()) <= (0.5 * step + ob.abs() * 2.0 ** -8 + 1e-6).numpy()).all()
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, SCALE)
    _check(o_h.float().numpy(), lse_h.numpy(), ref_o, ref_lse, "G=%d" % (hq // hkv))
