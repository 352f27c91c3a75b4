"""The C-ABI library loads, exports what include/h3gqa.h declares, and checks
its arguments on the host (CPU only: no call here reaches CUDA)."""
import ctypes
import os
import re
import subprocess

import pytest

from long_causal_gqa_gb300 import binding, build
from long_causal_gqa_gb300.binding import (H3GQA_ERR_INVALID_ARG, H3GQA_ERR_UNSUPPORTED,
                                           H3GQA_OK, H3GQAError)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "h3gqa.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared_functions():
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h3gqa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "h3gqa.h"\nint main(void){return h3gqa_version() > 0 ? 0 : 1;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", "-I",
                    os.path.join(ROOT, "include"), str(src), "-o", str(tmp_path / "use.o")],
                   check=True)


def test_version_and_status_strings(lib):
    assert binding.h3gqa_version() == 10100
    for st in range(6):
        assert binding.h3gqa_status_string(st)
    assert binding.h3gqa_status_string(99) == "unknown status"


def test_plan_headline_shape(lib):
    p = binding.h3gqa_make_plan([0, 10231], 64, 8, 128)
    assert p.total_tokens == 10231
    assert p.tokens_per_unit == 32                   # two tiles of 16 tokens x 8 heads
    assert p.n_units == 320 * 8                      # ceil(10231/32) blocks x 8 KV heads
    # block k visits floor(k/4)+1 key tiles: 8 heads * 4 * (1+...+80)
    assert p.n_kv_tiles == 8 * 4 * (80 * 81 // 2)
    assert p.max_kv_tiles == 80
    assert p.heads_per_tile == 8 and p.rows_per_tile == 128
    assert p.metric_flops == 2.0 * 10231 ** 2 * 64 * 128
    assert p.causal_flops == 2.0 * 64 * 128 * 10231 * 10232
    assert p.exp2_count == 64 * 10231 * 10232 / 2
    assert p.tensor_flops == p.n_kv_tiles * 8 * 128 ** 3
    # the MMAs do the needed work plus the masked part of the diagonal tiles
    assert 1.0 < p.tensor_flops / p.causal_flops < 1.03
    t = 10231
    assert p.algorithmic_bytes == 2 * t * 128 * (2 * 64 + 2 * 8) + 4 * t * 64


def test_plan_varlen_and_groups(lib):
    p = binding.h3gqa_make_plan([0, 8184, 16383, 24893, 35124], 64, 8)
    assert p.total_tokens == 35124
    assert p.n_units == 8 * sum((s + 31) // 32 for s in (8184, 8199, 8510, 10231))
    p2 = binding.h3gqa_make_plan([0, 0, 5, 5], 16, 8)         # G = 2: 64 tokens per tile
    assert p2.tokens_per_unit == 128 and p2.n_units == 8 and p2.max_kv_tiles == 1
    p3 = binding.h3gqa_make_plan([0, 300], 128, 1)            # G = 128: one token per tile
    assert p3.tokens_per_unit == 2 and p3.n_units == 150
    p0 = binding.h3gqa_make_plan([0], 64, 8)
    assert p0.n_units == 0 and p0.total_tokens == 0


def _units_and_tiles(lens, hq, hkv):
    """Units and key tiles counted from the tiling rule by brute force: a
    tile holds h heads (the largest divisor of G = hq/hkv up to 128) times
    floor(128/h) tokens, a unit two tiles, and a causal unit visits every key
    tile up to its last token inside the sequence."""
    g = hq // hkv
    h = max(d for d in range(1, min(g, 128) + 1) if g % d == 0)
    u = 2 * (128 // h)
    groups = hkv * (g // h)
    units = tiles = 0
    for s in lens:
        for t0 in range(0, s, u):
            last = min(t0 + u, s) - 1
            units += groups
            tiles += groups * (last // 128 + 1)
    return h, u, units, tiles


@pytest.mark.parametrize("lens,hq,hkv", [
    ((300,), 8, 8),           # G = 1 (MHA): 128 tokens x 1 head, 256-token units
    ((1000, 77), 64, 64),     # G = 1
    ((500,), 24, 8),          # G = 3: 42 tokens x 3 heads, 126 rows
    ((333, 0, 129), 40, 8),   # G = 5: 25 x 5 = 125 rows
    ((700,), 48, 8),          # G = 6: 21 x 6 = 126 rows
    ((90,), 96, 1),           # G = 96: 1 token x 96 heads
    ((90,), 256, 1),          # G = 256: two groups of 128 heads per KV head
    ((90,), 262, 2),          # G = 131 (prime): one head per tile
])
def test_plan_any_group_size(lib, lens, hq, hkv):
    cu = [0]
    for s in lens:
        cu.append(cu[-1] + s)
    p = binding.h3gqa_make_plan(cu, hq, hkv)
    h, u, units, tiles = _units_and_tiles(lens, hq, hkv)
    assert p.heads_per_tile == h and p.rows_per_tile == h * (128 // h)
    assert p.tokens_per_unit == u
    assert p.n_units == units and p.n_kv_tiles == tiles
    assert p.causal_flops == sum(2.0 * hq * 128 * s * (s + 1) for s in lens)


@pytest.mark.parametrize("cu,hq,hkv,d,status", [
    ([1, 5], 64, 8, 128, H3GQA_ERR_INVALID_ARG),       # cu[0] != 0
    ([0, 5, 3], 64, 8, 128, H3GQA_ERR_INVALID_ARG),    # decreasing
    ([0, 5], 64, 7, 128, H3GQA_ERR_INVALID_ARG),       # Hq % Hkv != 0
    ([0, 5], 0, 8, 128, H3GQA_ERR_INVALID_ARG),
    ([0, 5], 64, 8, 0, H3GQA_ERR_INVALID_ARG),
    ([0, 5], 64, 8, 64, H3GQA_ERR_UNSUPPORTED),        # head_dim
    ([0, 5], 64, -8, 128, H3GQA_ERR_INVALID_ARG),
])
def test_plan_rejects(lib, cu, hq, hkv, d, status):
    with pytest.raises(H3GQAError) as e:
        binding.h3gqa_make_plan(cu, hq, hkv, d)
    assert e.value.status == status


def test_too_many_sequences_unsupported(lib):
    cu = list(range(0, 1026))          # 1025 sequences of length 1
    with pytest.raises(H3GQAError) as e:
        binding.h3gqa_make_plan(cu, 64, 8)
    assert e.value.status == H3GQA_ERR_UNSUPPORTED
    cu2 = [0] * 3000 + list(range(1, 1025))   # zero-length ones do not count
    assert binding.h3gqa_make_plan(cu2, 64, 8).n_units == 1024 * 8


def test_forward_rejects_before_touching_cuda(lib):
    good = 1 << 20   # fake, 16-byte aligned "device" addresses; never dereferenced
    args = dict(q_ptr=good, k_ptr=good, v_ptr=good, o_ptr=good, lse_ptr=good,
                cu_seqlens=[0, 64], n_q_heads=64, n_kv_heads=8, head_dim=128, scale=0.088)
    for bad in (dict(q_ptr=0), dict(o_ptr=good + 8), dict(lse_ptr=good + 2),
                dict(scale=0.0), dict(scale=-1.0), dict(scale=float("inf")),
                dict(scale=float("nan")), dict(cu_seqlens=[0, 64, 32])):
        a = dict(args, **bad)
        st = binding.h3gqa_causal_fwd(check=False, **a)
        assert st == H3GQA_ERR_INVALID_ARG, bad
    st = binding.h3gqa_causal_fwd(check=False, **dict(args, head_dim=64))
    assert st == H3GQA_ERR_UNSUPPORTED
    # T = 0 is a no-op and needs no device
    assert binding.h3gqa_causal_fwd(check=False, **dict(args, cu_seqlens=[0, 0])) == H3GQA_OK
    assert binding.h3gqa_causal_fwd(check=False, **dict(args, cu_seqlens=[0])) == H3GQA_OK


def test_product_path_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        binding.load(str(tmp_path / "missing.so"))


def test_library_links_no_oracle():
    out = subprocess.run(["nm", "-D", binding.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    assert "oracle" not in out
    src_dir = os.path.join(ROOT, "long_causal_gqa_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    text = fh.read().lower()
                assert "oracle" not in text or f == "inputs.py", f


def test_attention_plan_bidirectional(lib):
    p = binding.h3gqa_attention_plan([0, 19316], 64, 8, causal=False)
    tiles = (19316 + 127) // 128
    assert p.n_units == 8 * ((19316 + 31) // 32)
    assert p.n_kv_tiles == p.n_units * tiles           # every unit sees every key tile
    assert p.metric_flops == 4.0 * 64 * 128 * 19316 ** 2
    assert p.causal_flops == p.metric_flops
    assert p.exp2_count == 64 * 19316 ** 2
    c = binding.h3gqa_attention_plan([0, 19316], 64, 8, causal=True)
    assert c.n_kv_tiles < p.n_kv_tiles and c.n_units == p.n_units
    assert binding.h3gqa_make_plan([0, 19316], 64, 8).n_kv_tiles == c.n_kv_tiles


def test_attention_options_rejected_before_cuda(lib):
    good = 1 << 20
    base = dict(q_ptr=good, k_ptr=good, v_ptr=good, o_ptr=good, lse_ptr=good,
                cu_seqlens=[0, 64], n_q_heads=64, n_kv_heads=8, head_dim=128, scale=0.088)
    bad_opts = [binding.make_options(out_int8=True),                       # no o_scale
                binding.make_options(out_int8=True, o_scale_ptr=good + 2),  # misaligned o_scale
                binding.make_options(out_layout=2),
                binding.make_options(kv_head_begin=8),                     # shard past the heads
                binding.make_options(kv_head_begin=-1),
                binding.make_options(kv_head_count=-1),
                binding.make_options(kv_head_count=9),
                binding.make_options(kv_head_begin=4, kv_head_count=5),
                binding.make_options(status_ptr=good + 2)]                 # misaligned status
    o = binding.make_options()
    o.causal = 2
    bad_opts.append(o)
    for opts in bad_opts:
        assert binding.h3gqa_attention_fwd(options=opts, check=False, **base) == \
            H3GQA_ERR_INVALID_ARG
    # valid options with nothing to do return OK without a device
    ok = binding.make_options(causal=False, out_layout=binding.H3GQA_LAYOUT_TOKEN_MAJOR,
                              out_int8=True, o_scale_ptr=good)
    assert binding.h3gqa_attention_fwd(options=ok, check=False,
                                       **dict(base, cu_seqlens=[0, 0])) == H3GQA_OK


def test_prologue_options_rejected_before_cuda(lib):
    good = 1 << 20
    base = dict(q_ptr=good, k_ptr=good, v_ptr=good, o_ptr=good, lse_ptr=good,
                cu_seqlens=[0, 64], n_q_heads=64, n_kv_heads=8, head_dim=128, scale=0.088)
    bad = [binding.make_options(cos_ptr=good, sin_ptr=None, k_out_ptr=good),   # cos without sin
           binding.make_options(cos_ptr=None, sin_ptr=good),                   # sin without cos
           binding.make_options(cos_ptr=good, sin_ptr=good),                   # k prepared, no k_out
           binding.make_options(k_norm_ptr=good),                              # likewise
           binding.make_options(k_norm_ptr=good, k_out_ptr=good + 8),          # misaligned k_out
           binding.make_options(q_norm_ptr=good + 2),                          # misaligned weight
           binding.make_options(cos_ptr=good + 4, sin_ptr=good, k_out_ptr=good),
           binding.make_options(q_norm_ptr=good, norm_eps=-1.0),
           binding.make_options(q_norm_ptr=good, norm_eps=float("nan"))]
    for opts in bad:
        assert binding.h3gqa_attention_fwd(options=opts, check=False, **base) == \
            H3GQA_ERR_INVALID_ARG
    ok = binding.make_options(q_norm_ptr=good, k_norm_ptr=good, cos_ptr=good, sin_ptr=good,
                              k_out_ptr=good)
    assert binding.h3gqa_attention_fwd(options=ok, check=False,
                                       **dict(base, cu_seqlens=[0])) == H3GQA_OK


def test_k_out_overlap_rejected_before_cuda(lib):
    """k_out may be k itself, but not overlap q, v or part of k (the sizes
    follow from T, the heads and head_dim: q 64*64*128*2 bytes here)."""
    q, k, v = 1 << 24, 1 << 26, 1 << 27
    base = dict(q_ptr=q, k_ptr=k, v_ptr=v, o_ptr=1 << 28, lse_ptr=1 << 29,
                cu_seqlens=[0, 64], n_q_heads=64, n_kv_heads=8, head_dim=128, scale=0.088)
    qbytes, kbytes = 64 * 64 * 128 * 2, 8 * 64 * 128 * 2
    for k_out in (q, q + qbytes - 16, v + 16, k + 16, k - kbytes + 16):
        opts = binding.make_options(k_norm_ptr=1 << 20, k_out_ptr=k_out)
        assert binding.h3gqa_attention_fwd(options=opts, check=False, **base) == \
            H3GQA_ERR_INVALID_ARG, hex(k_out)


def test_o_overlap_rejected_before_cuda(lib):
    """o may share no byte with q, k, v, lse, k_out or o_scale (it is written
    while other units still read the inputs). o is 64*64*128*2 bytes here,
    lse 64*64*4."""
    q, k, v, o, lse = 1 << 24, 1 << 26, 1 << 27, 1 << 28, 1 << 29
    base = dict(q_ptr=q, k_ptr=k, v_ptr=v, o_ptr=o, lse_ptr=lse,
                cu_seqlens=[0, 64], n_q_heads=64, n_kv_heads=8, head_dim=128, scale=0.088)
    obytes, lbytes, kbytes = 64 * 64 * 128 * 2, 64 * 64 * 4, 8 * 64 * 128 * 2
    for bad_o in (q, q + 16, k - obytes + 16, v + kbytes - 16, lse - obytes + 16, lse + lbytes - 16):
        assert binding.h3gqa_attention_fwd(check=False, **dict(base, o_ptr=bad_o)) == \
            H3GQA_ERR_INVALID_ARG, hex(bad_o)
    k_out = 1 << 25
    opts = binding.make_options(k_norm_ptr=1 << 20, k_out_ptr=k_out)
    assert binding.h3gqa_attention_fwd(options=opts, check=False,
                                       **dict(base, o_ptr=k_out + 16)) == H3GQA_ERR_INVALID_ARG
    o_scale = 1 << 30
    opts = binding.make_options(out_int8=True, o_scale_ptr=o_scale)
    assert binding.h3gqa_attention_fwd(options=opts, check=False,
                                       **dict(base, o_ptr=o_scale - 64 * 64 * 128 + 16)) == \
        H3GQA_ERR_INVALID_ARG


def test_o_overlap_rejected_in_the_binding():
    import torch
    buf = torch.zeros(4 * 40 * 128 * 4, dtype=torch.bfloat16)
    q = buf[: 8 * 40 * 128].view(8, 40, 128)
    o_bad = buf[4 * 40 * 128: 12 * 40 * 128].view(8, 40, 128)
    o_ok = buf[8 * 40 * 128: 16 * 40 * 128].view(8, 40, 128)
    with pytest.raises(ValueError):
        binding.check_output_disjoint(o_bad, q=q)
    with pytest.raises(ValueError):
        binding.check_output_disjoint(q, q=q)
    binding.check_output_disjoint(o_ok, q=q, lse=None)


def test_shard_heads_partition():
    """Contiguous head ranges: every head exactly once, sizes within one."""
    for n in (1, 3, 8, 64):
        for world in (1, 2, 3, 4, 8, 9):
            parts = [binding.shard_heads(n, world, r) for r in range(world)]
            heads = [h for b, c in parts for h in range(b, b + c)]
            assert heads == list(range(n))
            sizes = [c for _, c in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        binding.shard_heads(8, 2, 2)


def test_cu_seqlens_outside_int32_rejected_in_the_binding(lib):
    with pytest.raises(ValueError):
        binding.h3gqa_make_plan([0, 2 ** 31], 64, 8)


def test_front_end_shape_checks_on_cpu_tensors():
    import torch
    T, d = 40, 128
    q = torch.zeros(8, T, d, dtype=torch.bfloat16)
    k = torch.zeros(2, T, d, dtype=torch.bfloat16)
    v = torch.zeros(2, T, d, dtype=torch.bfloat16)
    assert binding.check_tensors(q, k, v, [0, 30, T]) == (8, 2, T, d)
    bad = [
        dict(cu_seqlens=[0, T - 1]),                                         # T mismatch
        dict(k=torch.zeros(2, T + 1, d, dtype=torch.bfloat16)),              # k's T
        dict(v=torch.zeros(2, T, d, dtype=torch.float16)),                   # dtype
        dict(q=torch.zeros(8, d, T, dtype=torch.bfloat16).transpose(1, 2)),  # not contiguous
        dict(rope_cos=torch.zeros(T - 1, d // 2)),                           # table too short
        dict(rope_sin=torch.zeros(T, d // 2, dtype=torch.float64)),
        dict(q_norm_weight=torch.zeros(d, dtype=torch.float32)),
        dict(k_out=torch.zeros(2, T, d // 2, dtype=torch.bfloat16)),
        dict(o=torch.zeros(8, T, d + 1, dtype=torch.bfloat16)),
        dict(lse=torch.zeros(8, T + 1)),
        dict(k_out=q[:2]),                                                   # overlaps q
        dict(k_out=v),                                                       # is v
        dict(lse=torch.zeros(8, T, device="meta")),                          # other device
    ]
    for b in bad:
        args = dict(q=q, k=k, v=v, cu_seqlens=[0, T])
        args.update(b)
        with pytest.raises(ValueError):
            binding.check_tensors(**args)
    assert binding.check_tensors(q, k, v, [0, T], k_out=k) == (8, 2, T, d)   # in place is fine
    with pytest.raises(ValueError):
        binding.attention_fwd(q, k, v, [0, T])          # CPU tensors never reach the library
