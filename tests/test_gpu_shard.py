"""Head-sharded calls (h3gqa_options.kv_head_begin / kv_head_count).

KV heads are independent, so calls that each compute a range of KV heads
(and the query heads reading them) reassemble the whole attention with no
exchange. Run here as consecutive calls on one GPU into shared output
buffers: the union must be bitwise equal to the unsharded call (which is
checked against the fp64 oracle), each call must leave the other heads' rows
of o / lse / o_scale / k_out untouched, and the partition helper the
benchmark uses must cover every head once.
"""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300 import binding
from long_causal_gqa_gb300.inputs import make_inputs, norm_weights, rope_tables
from oracle import causal_gqa as orc
from tests.test_gpu_parity import assert_close

pytestmark = pytest.mark.gpu

SCALE = 128 ** -0.5


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return torch.device("cuda:0")


def _bits(t):
    return t.view(torch.int8).cpu() if t.dtype == torch.int8 else t.cpu().view(torch.int16) \
        if t.dtype == torch.bfloat16 else t.cpu().view(torch.int32)


def _sharded(q, k, v, cu, ranges, **kw):
    """Runs one call per (begin, count) into one set of sentinel-filled buffers."""
    hq, T, d = q.shape
    shape = (T, hq, d) if kw.get("token_major") else (hq, T, d)
    odt = torch.int8 if kw.get("out_int8") else torch.bfloat16
    o = torch.full(shape, -77, dtype=odt, device=q.device)
    lse = torch.full((hq, T), float("nan"), dtype=torch.float32, device=q.device)
    sc = (torch.full(shape[:2], -1.0, dtype=torch.float32, device=q.device)
          if kw.get("out_int8") else None)
    k_out = torch.full_like(k, 3.0) if "k_norm_weight" in kw else None
    extra = dict(kw)
    if k_out is not None:
        extra["k_out"] = k_out
    for begin, count in ranges:
        binding.attention_fwd(q, k, v, cu, SCALE, kv_heads=(begin, count), o=o, lse=lse,
                              o_scale=sc, **extra)
    return o, lse, sc, k_out


@pytest.mark.parametrize("hq,hkv,ranges", [
    (64, 8, [(0, 3), (3, 5)]),
    (64, 8, [(b, 1) for b in range(8)]),
    (64, 64, [(0, 10), (10, 7), (17, 47)]),       # G = 1
    (40, 8, [(5, 0), (0, 5)]),                    # count 0 = through the last head
    (256, 2, [(1, 1), (0, 1)]),                   # G = 128
])
def test_shards_reassemble_bitwise(dev, hq, hkv, ranges):
    x = make_inputs((900, 0, 333, 1), hq, hkv, 128, seed=5000 + hq + hkv)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    cu = x["cu_seqlens"]
    o_full, lse_full, _ = binding.attention_fwd(q, k, v, cu, SCALE)
    o, lse, _, _ = _sharded(q, k, v, cu, ranges)
    assert torch.equal(_bits(o), _bits(o_full)) and torch.equal(_bits(lse), _bits(lse_full))
    ref_o, ref_lse = orc.causal_gqa(x["q"], x["k"], x["v"], cu, hq, hkv, SCALE)
    assert_close(o.float().cpu().numpy().astype(np.float64),
                 lse.cpu().numpy().astype(np.float64), ref_o, ref_lse, "sharded")


def test_one_shard_leaves_other_heads_untouched(dev):
    hq, hkv = 64, 8
    x = make_inputs((700, 129), hq, hkv, 128, seed=5100)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    wq, wk = norm_weights(128, 5100)
    cos, sin = rope_tables((700, 129), 128)
    kw = dict(q_norm_weight=wq.to(dev), k_norm_weight=wk.to(dev), rope_cos=cos.to(dev),
              rope_sin=sin.to(dev), causal=False, token_major=True, out_int8=True)
    o, lse, sc, k_out = _sharded(q, k, v, x["cu_seqlens"], [(2, 3)], **kw)
    g = hq // hkv
    mine = torch.zeros(hq, dtype=torch.bool)
    mine[2 * g:5 * g] = True
    o_c, lse_c, sc_c, ko_c = o.cpu(), lse.cpu(), sc.cpu(), k_out.cpu()
    # token-major o / o_scale: [T][Hq]...
    assert (o_c[:, ~mine] == -77).all() and (o_c[:, mine] != -77).any()
    assert (sc_c[:, ~mine] == -1.0).all() and (sc_c[:, mine] > 0).all()
    assert torch.isnan(lse_c[~mine]).all() and torch.isfinite(lse_c[mine]).all()
    kv_mine = torch.zeros(hkv, dtype=torch.bool)
    kv_mine[2:5] = True
    assert (ko_c[~kv_mine].float() == 3.0).all() and not (ko_c[kv_mine].float() == 3.0).all()
    # the shard's rows equal those of the unsharded call with the same options
    o_f, lse_f, sc_f = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE,
                                             k_out=torch.empty_like(k), **kw)
    assert torch.equal(o_c[:, mine], o_f.cpu()[:, mine])
    assert torch.equal(sc_c[:, mine], sc_f.cpu()[:, mine])
    assert torch.equal(lse_c[mine], lse_f.cpu()[mine])


def test_benchmark_partition_reassembles(dev):
    """The ranges bench.py --shard heads gives ranks 0..N-1, run one after
    another, reproduce the unsharded output bitwise."""
    hq, hkv = 64, 8
    x = make_inputs((2048, 1000), hq, hkv, 128, seed=5200)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o_full, lse_full, _ = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE)
    for world in (2, 3, 8):
        ranges = [binding.shard_heads(hkv, world, r) for r in range(world)]
        o, lse, _, _ = _sharded(q, k, v, x["cu_seqlens"], [r for r in ranges if r[1] > 0])
        assert torch.equal(_bits(o), _bits(o_full)) and torch.equal(_bits(lse), _bits(lse_full))
