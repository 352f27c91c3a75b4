"""Failure detection on the GPU without a fault.

Every pipeline wait in the kernel is bounded in wall-clock time; when a bound
runs out the CTA raises a device flag, lets its in-flight copies and MMAs
finish, frees its tensor memory and exits. This test builds a copy of the
library whose bound is 200 ns, so ordinary waits (the producer waiting for
the next unit's Q buffer while a long unit runs) run out on real data. The
call must come back (no hang), report H3GQA_ERR_TIMEOUT through
h3gqa_sync_and_check, and leave the CUDA context usable: the regular library
then runs and matches the oracle in the same process.
"""
import numpy as np
import pytest
import torch

from long_causal_gqa_gb300 import binding, build
from long_causal_gqa_gb300.binding import H3GQA_ERR_TIMEOUT, H3GQA_OK, H3GQAError
from long_causal_gqa_gb300.inputs import make_inputs
from oracle import causal_gqa as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny_wait_lib(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("tinywait") / "libh3gqa_tinywait.so")
    build.build(out=out, defines=("H3GQA_WAIT_NS=200ull",))
    return binding.load(out)


def _launch(lib, x, dev, stream):
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    arr, n = binding._cu_array(x["cu_seqlens"])
    st = lib.h3gqa_causal_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), arr, n, q.shape[0], k.shape[0], 128,
                              binding.ctypes.c_float(128 ** -0.5), stream.cuda_stream)
    return st, (q, k, v, o, lse)


def test_timeout_is_reported_and_context_survives(tiny_wait_lib):
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(dev)
    # long units: the producer waits tens of microseconds for the next Q slot,
    # far past the 200 ns bound
    x = make_inputs((8000, 333), 64, 8, 128, seed=21)
    st, _ = _launch(tiny_wait_lib, x, dev, stream)
    assert st == H3GQA_OK                       # the launch itself is fine
    st = tiny_wait_lib.h3gqa_sync_and_check(stream.cuda_stream)
    assert st == H3GQA_ERR_TIMEOUT
    # the flag is cleared by the check
    assert tiny_wait_lib.h3gqa_sync_and_check(stream.cuda_stream) == H3GQA_OK

    # the regular library still works in this context
    y = make_inputs((300,), 64, 8, 128, seed=22)
    q, k, v = (y[n].to(dev) for n in ("q", "k", "v"))
    o, lse = binding.causal_gqa_fwd(q, k, v, y["cu_seqlens"], 128 ** -0.5)
    binding.h3gqa_sync_and_check(torch.cuda.current_stream(dev).cuda_stream)
    ref_o, ref_lse = orc.causal_gqa(y["q"], y["k"], y["v"], y["cu_seqlens"], 64, 8, 128 ** -0.5)
    o64 = o.float().cpu().numpy().astype(np.float64)
    assert (np.abs(o64 - ref_o) <= 1e-2 + 1e-2 * np.abs(ref_o)).all()
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3


def test_front_end_raises_on_timeout(tiny_wait_lib, monkeypatch):
    """The torch front end checks its own call by default: a call whose kernel
    gives up raises H3GQAError(H3GQA_ERR_TIMEOUT) through its per-call status
    word; with check=False the call returns and the device-wide flag still
    records the timeout."""
    dev = torch.device("cuda:0")
    x = make_inputs((8000, 333), 64, 8, 128, seed=23)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    monkeypatch.setattr(binding, "_LIB", tiny_wait_lib)
    with pytest.raises(H3GQAError) as e:
        binding.causal_gqa_fwd(q, k, v, x["cu_seqlens"], 128 ** -0.5)
    assert e.value.status == H3GQA_ERR_TIMEOUT
    with pytest.raises(H3GQAError) as e:
        binding.attention_fwd(q, k, v, x["cu_seqlens"], 128 ** -0.5, causal=False,
                              kv_heads=(1, 2))
    assert e.value.status == H3GQA_ERR_TIMEOUT
    stream = torch.cuda.current_stream(dev)
    assert tiny_wait_lib.h3gqa_sync_and_check(stream.cuda_stream) == H3GQA_ERR_TIMEOUT
    binding.causal_gqa_fwd(q, k, v, x["cu_seqlens"], 128 ** -0.5, check=False)
    assert tiny_wait_lib.h3gqa_sync_and_check(stream.cuda_stream) == H3GQA_ERR_TIMEOUT
    assert tiny_wait_lib.h3gqa_sync_and_check(stream.cuda_stream) == H3GQA_OK
    monkeypatch.undo()
    # the regular library, checked by default, reports nothing on the same inputs
    o, lse = binding.causal_gqa_fwd(q, k, v, x["cu_seqlens"], 128 ** -0.5)
    assert bool(torch.isfinite(lse).all())
