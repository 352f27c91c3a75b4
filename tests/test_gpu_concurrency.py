"""The library is reentrant: host threads that call it at the same time, each
on its own stream with its own buffers, get exactly the results of calls made
one after another (the kernel has no atomics and no shared scratch, so the
outputs are bitwise reproducible)."""
import threading

import pytest
import torch

from long_causal_gqa_gb300 import binding
from long_causal_gqa_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SCALE = 128 ** -0.5


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    binding.load()
    return torch.device("cuda:0")


def test_threads_on_separate_streams(dev):
    jobs = [dict(seqlens=(1500, 0, 333), causal=True, token_major=False, seed=71),
            dict(seqlens=(2049,), causal=False, token_major=True, seed=72),
            dict(seqlens=(640, 77, 1), causal=True, token_major=True, seed=73)]
    inputs = []
    for j in jobs:
        x = make_inputs(j["seqlens"], 64, 8, 128, j["seed"])
        inputs.append((x, tuple(x[n].to(dev) for n in ("q", "k", "v"))))
    # one after another on the default stream
    expected = []
    for j, (x, (q, k, v)) in zip(jobs, inputs):
        o, lse, _ = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE, causal=j["causal"],
                                          token_major=j["token_major"])
        binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)
        expected.append((o.clone(), lse.clone()))

    results = [None] * len(jobs)
    errors = []
    start = threading.Barrier(len(jobs))

    def worker(i):
        try:
            torch.cuda.set_device(dev)
            j, (x, (q, k, v)) = jobs[i], inputs[i]
            stream = torch.cuda.Stream(dev)
            outs = []
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(4):
                    o, lse, _ = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE,
                                                      causal=j["causal"],
                                                      token_major=j["token_major"],
                                                      stream=stream, check=False)
                    outs.append((o, lse))
            binding.h3gqa_sync_and_check(stream.cuda_stream)
            results[i] = outs
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for i, outs in enumerate(results):
        assert outs is not None
        for o, lse in outs:
            assert torch.equal(o, expected[i][0]) and torch.equal(lse, expected[i][1]), \
                "job %d differs from its sequential result" % i


def test_cuda_graph_capture_and_replay(dev):
    """A call captured in a CUDA graph replays to the eager result bit for bit
    (the first, eager call does the per-device setup, which is not a stream
    operation; the captured call only records the kernel launches)."""
    x = make_inputs((3000, 0, 517), 64, 8, 128, seed=81)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o_ref, lse_ref, _ = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE)
    binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    stream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        binding.h3gqa_causal_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), x["cu_seqlens"], 64, 8, 128, SCALE,
                                 torch.cuda.current_stream(dev).cuda_stream)
    for _ in range(3):
        o.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize(dev)
        assert binding.h3gqa_sync_and_check(0) == binding.H3GQA_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_cuda_graph_with_prologue_and_int8(dev):
    """The prologue's two launches (K pass, then attention) and the int8
    token-major epilogue, captured in one graph, replay to the eager result
    bit for bit: codes, scales, LSE and the prepared keys."""
    from long_causal_gqa_gb300.inputs import norm_weights, rope_tables
    seqlens = (1500, 0, 333)
    x = make_inputs(seqlens, 64, 8, 128, seed=82)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    wq, wk = (t.to(dev) for t in norm_weights(128, 82))
    cos, sin = (t.to(dev) for t in rope_tables(seqlens, 128))
    kw = dict(q_norm_weight=wq, k_norm_weight=wk, rope_cos=cos, rope_sin=sin,
              token_major=True, out_int8=True)
    o_ref, lse_ref, sc_ref = binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE, **kw)
    k_ref = torch.empty_like(k)
    binding.attention_fwd(q, k, v, x["cu_seqlens"], SCALE, k_out=k_ref, **kw)
    T = q.shape[1]
    o = torch.empty((T, 64, 128), dtype=torch.int8, device=dev)
    lse = torch.empty((64, T), dtype=torch.float32, device=dev)
    sc = torch.empty((T, 64), dtype=torch.float32, device=dev)
    k_out = torch.empty_like(k)
    opts = binding.make_options(True, binding.H3GQA_LAYOUT_TOKEN_MAJOR, True, sc.data_ptr(), 0,
                                wq.data_ptr(), wk.data_ptr(), cos.data_ptr(), sin.data_ptr(),
                                k_out.data_ptr())
    stream = torch.cuda.Stream(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        st = binding.h3gqa_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), x["cu_seqlens"], 64, 8, 128, SCALE,
                                         options=opts, stream=torch.cuda.current_stream(dev).cuda_stream,
                                         check=False)
        assert st == binding.H3GQA_OK
    for _ in range(2):
        for t in (o, lse, sc, k_out):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize(dev)
        assert binding.h3gqa_sync_and_check(0) == binding.H3GQA_OK
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref) and torch.equal(sc, sc_ref)
        assert torch.equal(k_out, k_ref)
