"""GPU parity: the sm_103a library against the fp64 oracle, element by element.

Bar (the acceptance rule of the causal GQA target): every output element
|o - ref| <= 1e-2 + 1e-2*|ref|, every LSE |lse - ref| <= 1e-3 (natural log).
Small shapes are checked in full, and so are the single-sequence full-size
workloads (S = 7700 and S = 10231: every head, every row). The packed
varlen workload and S = 32768 are checked on at least three rows of every
work unit the kernel schedules (a unit is one block of tokens of one
sequence and one head group): for every block and every query head, the
block's first and last token and one seeded random token, so a unit that
is skipped, repeated, or run with the wrong KV head, tokens or sequence
fails. Output buffers carry guard regions that must come back untouched.
"""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300 import binding
from long_causal_gqa_gb300.inputs import WORKLOADS, make_inputs, make_workload_inputs
from oracle import causal_gqa as orc

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3
GUARD = 4096
O_SENTINEL = -12345      # int16 bit pattern written around o
LSE_SENTINEL = 0x7FBADBAD  # int32 NaN pattern written around lse


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return torch.device("cuda:0")


def run_gpu(x, hq, hkv, scale, dev, stream=None, as_numpy=True, o_shift=0):
    """Runs the library with guard regions around o and lse; returns numpy
    (o fp64 [Hq,T,D], lse fp64 [Hq,T]), or the CPU tensors (o bf16, lse fp32)
    when as_numpy is False (large outputs: convert only sampled rows).
    o_shift moves o by that many bf16 elements from its 32-byte-aligned
    place (8: o is 16-byte but not 32-byte aligned)."""
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    T, d = q.shape[1], q.shape[2]
    n_o, n_l = hq * T * d, hq * T
    o_buf = torch.full((n_o + 2 * GUARD + o_shift,), O_SENTINEL, dtype=torch.int16, device=dev)
    l_buf = torch.full((n_l + 2 * GUARD,), LSE_SENTINEL, dtype=torch.int32, device=dev)
    o = o_buf[GUARD + o_shift:GUARD + o_shift + n_o].view(torch.bfloat16).view(hq, T, d)
    lse = l_buf[GUARD:GUARD + n_l].view(torch.float32).view(hq, T)
    s = stream or torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    binding.causal_gqa_fwd(q, k, v, x["cu_seqlens"], scale, o=o, lse=lse, stream=s)
    binding.h3gqa_sync_and_check(s.cuda_stream)
    ob, lb = o_buf.cpu(), l_buf.cpu()
    for name, buf, sent in (("o", ob, O_SENTINEL), ("lse", lb, LSE_SENTINEL)):
        assert (buf[:GUARD] == sent).all() and (buf[-GUARD:] == sent).all(), \
            "write outside %s" % name
    if not as_numpy:
        return o.cpu(), lse.cpu()
    return (o.float().cpu().numpy().astype(np.float64),
            lse.cpu().numpy().astype(np.float64))


def rows_of(o_t, lse_t, rows):
    """Selected (head, token) rows of CPU output tensors, as fp64 numpy."""
    h = torch.from_numpy(rows[:, 0])
    t = torch.from_numpy(rows[:, 1])
    return (o_t[h, t].float().numpy().astype(np.float64),
            lse_t[h, t].numpy().astype(np.float64))


def all_finite(o_t, lse_t):
    return bool(torch.isfinite(o_t).all()) and bool(torch.isfinite(lse_t).all())


def assert_close(o, lse, ref_o, ref_lse, what=""):
    assert np.isfinite(o).all(), "non-finite o %s" % what
    assert np.isfinite(lse).all(), "non-finite lse %s" % what
    excess = np.abs(o - ref_o) - (O_ATOL + O_RTOL * np.abs(ref_o))
    if excess.max() > 0:
        idx = np.unravel_index(np.argmax(excess), excess.shape)
        bad = (excess > 0).sum()
        raise AssertionError("o mismatch %s: %d elements over tolerance; worst at %s: got %r "
                             "want %r" % (what, bad, idx, o[idx], ref_o[idx]))
    lerr = np.abs(lse - ref_lse)
    if lerr.max() > LSE_ATOL:
        idx = np.unravel_index(np.argmax(lerr), lerr.shape)
        raise AssertionError("lse mismatch %s: %d over tolerance; worst at %s: got %r want %r"
                             % (what, (lerr > LSE_ATOL).sum(), idx, lse[idx], ref_lse[idx]))


def full_check(seqlens, hq, hkv, seed, dev, scale=None, n_outlier=0):
    x = make_inputs(seqlens, hq, hkv, 128, seed, n_outlier)
    scale = 128 ** -0.5 if scale is None else scale
    o, lse = run_gpu(x, hq, hkv, scale, dev)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, scale)
    assert_close(o, lse, ref_o, ref_lse, "seqlens=%s hq=%d hkv=%d" % (seqlens, hq, hkv))


# -------------------------------------------------------------- small, full
@pytest.mark.parametrize("S", [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257, 1000])
def test_single_sequence_sweep(dev, S):
    full_check((S,), 64, 8, 500 + S, dev)


def test_varlen_with_empty_and_unit_sequences(dev):
    full_check((5, 0, 129, 1, 1, 300, 0, 64), 64, 8, 77, dev)


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 2), (128, 1), (64, 4), (64, 32), (8, 4)])
def test_group_sizes(dev, hq, hkv):
    full_check((200, 37), hq, hkv, 900 + hq + hkv, dev)


# Group sizes whose tiles do not fill 128 rows or whose units straddle two
# key tiles: G = 1 (plain multi-head attention: 128 tokens x 1 head, 256-token
# units), G = 3, 5, 6, 7 (42 x 3, 25 x 5, 21 x 6, 18 x 7 rows), G = 96 (96 of
# 128 rows), G = 256 (two head groups per KV head) and G = 131 (a prime above
# 128: one head per tile). Lengths cross several key tiles and end ragged.
ANY_G = [(8, 8), (64, 64), (24, 8), (40, 8), (48, 8), (56, 8), (96, 1), (256, 1), (262, 2)]


@pytest.mark.parametrize("hq,hkv", ANY_G)
def test_any_group_size_causal(dev, hq, hkv):
    full_check((700, 0, 37, 1, 300), hq, hkv, 1900 + hq + hkv, dev)


@pytest.mark.parametrize("hq,hkv", ANY_G)
def test_any_group_size_bidirectional(dev, hq, hkv):
    x = make_inputs((700, 0, 37, 1, 300), hq, hkv, 128, 2900 + hq + hkv)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o, lse, _ = binding.attention_fwd(q, k, v, x["cu_seqlens"], 128 ** -0.5, causal=False)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv,
                                    128 ** -0.5, causal=False)
    assert_close(o.float().cpu().numpy().astype(np.float64),
                 lse.cpu().numpy().astype(np.float64), ref_o, ref_lse,
                 "bidirectional hq=%d hkv=%d" % (hq, hkv))


def test_o_only_16_byte_aligned(dev):
    """o 16-byte but not 32-byte aligned takes the 16-byte store path of the
    epilogue: same bits as the aligned call, within the bar of the oracle,
    guards untouched, on ragged sequences that leave partial tiles."""
    hq, hkv, scale = 16, 2, 128 ** -0.5
    x = make_inputs((300, 0, 129, 5, 700), hq, hkv, 128, 4711)
    o16, lse16 = run_gpu(x, hq, hkv, scale, dev, o_shift=8)
    o32, lse32 = run_gpu(x, hq, hkv, scale, dev)
    assert np.array_equal(o16, o32) and np.array_equal(lse16, lse32)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], hq, hkv, scale)
    assert_close(o16, lse16, ref_o, ref_lse, "(o 16-byte aligned)")


def test_workload_s512_full(dev):
    w = WORKLOADS["s512"]
    full_check(w.seqlens, w.n_q_heads, w.n_kv_heads, w.seed, dev)


def test_uniform_attention_prefix_mean(dev):
    """q = 0 makes every visible logit 0: o is the running mean of v and
    lse = ln(i+1). This isolates the P.V path from the Q.K^T path."""
    x = make_inputs((300,), 64, 8, 128, seed=3)
    x["q"] = torch.zeros_like(x["q"])
    o, lse = run_gpu(x, 64, 8, 128 ** -0.5, dev)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], 64, 8, 128 ** -0.5)
    np.testing.assert_allclose(ref_lse[0], np.log(np.arange(1, 301)), atol=1e-12)
    assert_close(o, lse, ref_o, ref_lse, "uniform")


def test_large_scale_and_outliers_small(dev):
    full_check((700,), 64, 8, 31, dev, scale=0.5)
    full_check((700,), 64, 8, 32, dev, n_outlier=4)


def test_extreme_logits_exercise_the_rescale(dev):
    """q and k scaled by 6 (logit std ~36, rows nearly one-hot): the running
    max jumps by far more than 2^8 many times per row, so the O rescale path
    runs on many tiles; causal and bidirectional, checked in full."""
    for causal in (True, False):
        x = make_inputs((900, 0, 301), 64, 8, 128, seed=606)
        x["q"] = (x["q"].float() * 6.0).to(torch.bfloat16)
        x["k"] = (x["k"].float() * 6.0).to(torch.bfloat16)
        q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
        o, lse, _ = binding.attention_fwd(q, k, v, x["cu_seqlens"], 128 ** -0.5, causal=causal)
        binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)
        ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], 64, 8,
                                        128 ** -0.5, causal=causal)
        assert_close(o.float().cpu().numpy().astype(np.float64),
                     lse.cpu().numpy().astype(np.float64), ref_o, ref_lse,
                     "extreme logits causal=%s" % causal)


def test_deterministic_and_stream(dev):
    x = make_inputs((1000, 333), 64, 8, 128, seed=8)
    o1, l1 = run_gpu(x, 64, 8, 128 ** -0.5, dev)
    s = torch.cuda.Stream(dev)
    o2, l2 = run_gpu(x, 64, 8, 128 ** -0.5, dev, stream=s)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# --------------------------------------------------------------- full size
def sample_rows(cu, hq, n_random, seed):
    """Sequence edges, both sides of every 128-token boundary (head rotated
    along the tokens), seeded random rows and every head at the last token of
    the longest sequence."""
    rows = set()
    T = int(cu[-1])
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        if s == e:
            continue
        toks = {s, s + 1, e - 1, e - 2}
        for edge in range(s + 128, e, 128):
            toks.update((edge - 1, edge))
        for t in toks:
            if s <= t < e:
                rows.add((int(t) % hq, int(t)))   # rotate heads along tokens
    rng = np.random.default_rng(seed)
    for _ in range(n_random):
        rows.add((int(rng.integers(hq)), int(rng.integers(T))))
    # every head at the last token of the longest sequence
    lens = np.diff(np.asarray(cu))
    b = int(np.argmax(lens))
    rows.update((h, int(cu[b + 1]) - 1) for h in range(hq))
    return np.array(sorted(rows), dtype=np.int64)


def unit_rows(cu, hq, hkv, seed):
    """At least three rows of every work unit, for every query head: a unit
    is one block of tokens_per_unit tokens of one sequence for the heads of
    one group; each (block, query head) pair contributes the block's first
    and last token (inside the sequence) and one seeded random token of it."""
    plan = binding.h3gqa_make_plan([int(c) for c in cu], hq, hkv)
    u = int(plan.tokens_per_unit)
    rng = np.random.default_rng(seed)
    out = []
    heads = np.arange(hq, dtype=np.int64)
    for b in range(len(cu) - 1):
        s, e = int(cu[b]), int(cu[b + 1])
        for t0 in range(s, e, u):
            t1 = min(t0 + u, e) - 1
            rand = rng.integers(t0, t1 + 1, hq)
            for toks in (np.full(hq, t0), np.full(hq, t1), rand):
                out.append(np.stack([heads, toks.astype(np.int64)], axis=1))
    rows = np.unique(np.concatenate(out), axis=0)
    return rows


@pytest.mark.parametrize("name", ["s7700", "s10231"])
def test_full_size_every_row(dev, name):
    """Every head and every row of the single-sequence full-size workloads
    against the full fp64 oracle (the call is the one the benchmark times)."""
    w = WORKLOADS[name]
    x = make_workload_inputs(w)
    o_t, lse_t = run_gpu(x, w.n_q_heads, w.n_kv_heads, w.scale, dev, as_numpy=False)
    assert all_finite(o_t, lse_t)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], w.n_q_heads,
                                    w.n_kv_heads, w.scale)
    for h0 in range(0, w.n_q_heads, 8):          # 8 heads at a time bounds the fp64 copies
        sl = slice(h0, h0 + 8)
        assert_close(o_t[sl].float().numpy().astype(np.float64),
                     lse_t[sl].numpy().astype(np.float64), ref_o[sl], ref_lse[sl],
                     "%s heads %d..%d" % (name, h0, h0 + 7))


@pytest.mark.parametrize("name", ["varlen4", "s32768_outlier"])
def test_full_size_every_unit(dev, name):
    w = WORKLOADS[name]
    x = make_workload_inputs(w)
    o_t, lse_t = run_gpu(x, w.n_q_heads, w.n_kv_heads, w.scale, dev, as_numpy=False)
    assert all_finite(o_t, lse_t)
    cu = x["cu_seqlens"].numpy()
    rows = unit_rows(cu, w.n_q_heads, w.n_kv_heads, w.seed)
    plan = binding.h3gqa_make_plan([int(c) for c in cu], w.n_q_heads, w.n_kv_heads)
    # every (unit, query head) of the schedule has its three rows
    per_unit = plan.n_units * (w.n_q_heads // w.n_kv_heads)
    assert len(rows) >= per_unit * 2
    rows = np.unique(np.concatenate([rows, sample_rows(cu, w.n_q_heads, 0, w.seed)]), axis=0)
    ref_o, ref_lse = orc.causal_gqa_rows(x["q"], x["k"], x["v"], cu, w.n_q_heads,
                                         w.n_kv_heads, w.scale, rows)
    got_o, got_l = rows_of(o_t, lse_t, rows)
    assert_close(got_o, got_l, ref_o, ref_lse, name)
    # every output row is a convex combination of value rows
    vmax = float(x["v"].float().abs().max())
    assert float(o_t.float().abs().max()) <= vmax * (1 + 1e-2)


def test_long_sequence_65536_sampled(dev):
    """A single 65536-token sequence (512 K/V tiles per unit at the end):
    index arithmetic and the online softmax over very long rows."""
    S = 65536
    x = make_inputs((S,), 64, 8, 128, seed=65536)
    o_t, lse_t = run_gpu(x, 64, 8, 128 ** -0.5, dev, as_numpy=False)
    cu = x["cu_seqlens"].numpy()
    rows = sample_rows(cu, 64, 256, 7)
    rows = rows[rows[:, 1] % 1024 < 8]                     # keep the oracle cost bounded
    rows = np.concatenate([rows, np.array([[h, S - 1] for h in range(0, 64, 9)], dtype=np.int64)])
    ref_o, ref_lse = orc.causal_gqa_rows(x["q"], x["k"], x["v"], cu, 64, 8, 128 ** -0.5, rows)
    got_o, got_l = rows_of(o_t, lse_t, rows)
    assert_close(got_o, got_l, ref_o, ref_lse, "S=65536")
    assert all_finite(o_t, lse_t)


def test_long_sequence_262144_sampled(dev):
    """A single 262144-token sequence (Hq 8, Hkv 4: 128-token units, up to
    2048 K/V tiles per unit): no length bound, sampled rows across the whole
    sequence, the last row of every head, and every output finite."""
    S, hq, hkv = 262144, 8, 4
    x = make_inputs((S,), hq, hkv, 128, seed=262144)
    o_t, lse_t = run_gpu(x, hq, hkv, 128 ** -0.5, dev, as_numpy=False)
    cu = x["cu_seqlens"].numpy()
    rng = np.random.default_rng(11)
    rows = np.stack([rng.integers(0, hq, 48), rng.integers(0, S, 48)], axis=1)
    rows = np.concatenate([rows, np.array([[h, S - 1] for h in range(hq)] +
                                          [[0, 0], [hq - 1, 127], [1, 128], [2, 131071]],
                                          dtype=np.int64)])
    ref_o, ref_lse = orc.causal_gqa_rows(x["q"], x["k"], x["v"], cu, hq, hkv, 128 ** -0.5, rows)
    got_o, got_l = rows_of(o_t, lse_t, rows)
    assert_close(got_o, got_l, ref_o, ref_lse, "S=262144")
    assert all_finite(o_t, lse_t)


def test_many_sequences_at_the_limit(dev):
    """1024 non-empty sequences (the most one call accepts) of random lengths,
    interleaved with empty ones; every row checked against the oracle."""
    rng = np.random.default_rng(1024)
    lens = []
    for i in range(1024):
        lens.append(int(rng.integers(1, 90)))
        if i % 7 == 0:
            lens.append(0)
    x = make_inputs(tuple(lens), 64, 8, 128, seed=1025)
    o, lse = run_gpu(x, 64, 8, 128 ** -0.5, dev)
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], x["cu_seqlens"], 64, 8, 128 ** -0.5)
    assert_close(o, lse, ref_o, ref_lse, "1024 sequences")
