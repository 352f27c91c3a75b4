"""numpy front end of the fp64 causal GQA oracle (oracle/causal_gqa_oracle.c).

Test infrastructure only: the test suite, the smoke check and the benchmark's
CPU-baseline / reference leg call it; the GPU library never does.

The arithmetic lives in the C file (the plain definition of causal softmax
attention from antirez/h3.c issue #47, "Error" / "Suggested fix
directions"). This module only builds the library, checks shapes and passes
pointers. Tensors come in as bf16 bit patterns (numpy uint16) or as torch
bf16 tensors, in head-major layout: q [Hq][T][D], k and v [Hkv][T][D].
"""
import ctypes
import os

import numpy as np

from . import build_oracle

_LIB = None


def bind(path):
    """Load an oracle shared library from `path` and declare its signatures."""
    lib = ctypes.CDLL(path)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    f64p = ctypes.POINTER(ctypes.c_double)
    common = [u16p, u16p, u16p, i32p, ctypes.c_int, ctypes.c_int,
              ctypes.c_int, ctypes.c_int, ctypes.c_double]
    lib.oracle_causal_gqa.argtypes = common + [f64p, f64p, ctypes.c_int]
    lib.oracle_causal_gqa.restype = ctypes.c_int
    lib.oracle_causal_gqa_rows.argtypes = common + [
        i64p, ctypes.c_int64, f64p, f64p, ctypes.c_int]
    lib.oracle_causal_gqa_rows.restype = ctypes.c_int
    lib.oracle_attention_probs.argtypes = common + [
        ctypes.c_int, ctypes.c_int64, f64p]
    lib.oracle_attention_probs.restype = ctypes.c_int64
    lib.oracle_attention.argtypes = common + [ctypes.c_int, f64p, f64p, ctypes.c_int]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = common + [
        ctypes.c_int, i64p, ctypes.c_int64, f64p, f64p, ctypes.c_int]
    lib.oracle_attention_rows.restype = ctypes.c_int
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_qk_prep.argtypes = [u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, u16p,
                                   ctypes.c_double, f32p, f32p, f64p]
    lib.oracle_qk_prep.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = bind(build_oracle.build())
    return _LIB


def as_bf16_bits(x):
    """A bf16 torch tensor or a uint16 numpy array -> contiguous uint16 numpy."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be bf16 bit patterns (uint16)")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("torch inputs must be bfloat16")
    return np.ascontiguousarray(
        x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _prep(q, k, v, cu_seqlens, n_q_heads, n_kv_heads):
    q, k, v = as_bf16_bits(q), as_bf16_bits(k), as_bf16_bits(v)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T = int(cu[-1])
    D = q.shape[-1]
    if q.shape != (n_q_heads, T, D) or k.shape != (n_kv_heads, T, D) \
            or v.shape != (n_kv_heads, T, D):
        raise ValueError("shapes must be q [Hq,T,D], k/v [Hkv,T,D]; got %s %s %s"
                         % (q.shape, k.shape, v.shape))
    return q, k, v, cu, T, D


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def causal_gqa(q, k, v, cu_seqlens, n_q_heads, n_kv_heads, scale, n_threads=0, causal=True):
    """All rows. Returns (o [Hq,T,D] fp64, lse [Hq,T] fp64). causal=False gives
    the bidirectional form (every key of the sequence)."""
    q, k, v, cu, T, D = _prep(q, k, v, cu_seqlens, n_q_heads, n_kv_heads)
    o = np.zeros((n_q_heads, T, D), dtype=np.float64)
    lse = np.zeros((n_q_heads, T), dtype=np.float64)
    rc = _lib().oracle_attention(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(cu, ctypes.c_int32), len(cu) - 1, n_q_heads, n_kv_heads, D,
        float(scale), 1 if causal else 0, _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (code %d)" % rc)
    return o, lse


def causal_gqa_rows(q, k, v, cu_seqlens, n_q_heads, n_kv_heads, scale, rows,
                    n_threads=0, causal=True):
    """Selected rows: rows is an int array [n, 2] of (query head, token row).

    Returns (o [n,D] fp64, lse [n] fp64)."""
    q, k, v, cu, T, D = _prep(q, k, v, cu_seqlens, n_q_heads, n_kv_heads)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    n = rows.shape[0]
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _lib().oracle_attention_rows(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(cu, ctypes.c_int32), len(cu) - 1, n_q_heads, n_kv_heads, D,
        float(scale), 1 if causal else 0, _ptr(rows, ctypes.c_int64), n,
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), int(n_threads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (code %d)" % rc)
    return o, lse


def attention_probs(q, k, v, cu_seqlens, n_q_heads, n_kv_heads, scale, h, t):
    """Probability row of query (h, t) over keys s_b..t (fp64)."""
    q, k, v, cu, T, D = _prep(q, k, v, cu_seqlens, n_q_heads, n_kv_heads)
    p = np.zeros((max(T, 1),), dtype=np.float64)
    n = _lib().oracle_attention_probs(
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(cu, ctypes.c_int32), len(cu) - 1, n_q_heads, n_kv_heads, D,
        float(scale), int(h), int(t), _ptr(p, ctypes.c_double))
    if n < 0:
        raise ValueError("oracle rejected its arguments")
    return p[:n].copy()


def qk_prep(x, w=None, eps=1e-6, rope_cos=None, rope_sin=None):
    """Q/K prologue of every row of x [heads, T, D] (bf16): RMS norm with
    weight w (bf16 [D], optional) and rotate-half rotary embedding with fp32
    tables [T, D/2] (optional). Returns fp64 [heads, T, D] (unrounded)."""
    xb = as_bf16_bits(x)
    heads, T, D = xb.shape
    out = np.zeros((heads, T, D), dtype=np.float64)
    wb = as_bf16_bits(w) if w is not None else None
    cs = sn = None
    if rope_cos is not None:
        cs = np.ascontiguousarray(np.asarray(rope_cos, dtype=np.float32))
        sn = np.ascontiguousarray(np.asarray(rope_sin, dtype=np.float32))
        if cs.shape != (T, D // 2) or sn.shape != (T, D // 2):
            raise ValueError("rope tables must be [T, D/2]")
    rc = _lib().oracle_qk_prep(
        _ptr(xb, ctypes.c_uint16), heads * T, T, D,
        _ptr(wb, ctypes.c_uint16) if wb is not None else None, float(eps),
        _ptr(cs, ctypes.c_float) if cs is not None else None,
        _ptr(sn, ctypes.c_float) if sn is not None else None, _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (code %d)" % rc)
    return out


def to_bf16(a):
    """fp64 array -> bf16 torch tensor: rounded to fp32, then to bf16 (nearest even)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.float32))).to(torch.bfloat16)


def max_threads():
    return int(_lib().oracle_max_threads())
