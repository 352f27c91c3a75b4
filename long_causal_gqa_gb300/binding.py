"""Python binding of the h3gqa C ABI (include/h3gqa.h).

Argument marshalling only: every step of the attention runs in the CUDA
library. Importing this module does not load the library; the first call
does, and it raises if libh3gqa.so has not been built. There is no CPU
fallback.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libh3gqa.so")

H3GQA_OK = 0
H3GQA_ERR_INVALID_ARG = 1
H3GQA_ERR_UNSUPPORTED = 2
H3GQA_ERR_ARCH = 3
H3GQA_ERR_CUDA = 4
H3GQA_ERR_TIMEOUT = 5

EXPORTED = ("h3gqa_causal_fwd", "h3gqa_attention_fwd", "h3gqa_make_plan",
            "h3gqa_attention_plan", "h3gqa_sync_and_check", "h3gqa_status_string",
            "h3gqa_version")

H3GQA_LAYOUT_HEAD_MAJOR = 0
H3GQA_LAYOUT_TOKEN_MAJOR = 1


class H3GQAError(RuntimeError):
    def __init__(self, status, where):
        self.status = int(status)
        super().__init__("%s failed: %s (status %d)"
                         % (where, h3gqa_status_string(status), self.status))


class h3gqa_plan(ctypes.Structure):
    _fields_ = [
        ("total_tokens", ctypes.c_int64),
        ("n_units", ctypes.c_int64),
        ("n_kv_tiles", ctypes.c_int64),
        ("tensor_flops", ctypes.c_double),
        ("causal_flops", ctypes.c_double),
        ("metric_flops", ctypes.c_double),
        ("exp2_count", ctypes.c_double),
        ("algorithmic_bytes", ctypes.c_double),
        ("tokens_per_unit", ctypes.c_int32),
        ("max_kv_tiles", ctypes.c_int32),
        ("heads_per_tile", ctypes.c_int32),
        ("rows_per_tile", ctypes.c_int32),
    ]


class h3gqa_options(ctypes.Structure):
    _fields_ = [
        ("causal", ctypes.c_int32),
        ("out_layout", ctypes.c_int32),
        ("out_int8", ctypes.c_int32),
        ("kv_head_begin", ctypes.c_int32),
        ("o_scale", ctypes.c_void_p),
        ("q_norm_weight", ctypes.c_void_p),
        ("k_norm_weight", ctypes.c_void_p),
        ("rope_cos", ctypes.c_void_p),
        ("rope_sin", ctypes.c_void_p),
        ("k_out", ctypes.c_void_p),
        ("norm_eps", ctypes.c_float),
        ("kv_head_count", ctypes.c_int32),
        ("status", ctypes.c_void_p),
    ]


_LIB = None


def load(path: str = LIB_PATH):
    """Load the library (once) and declare the signatures of include/h3gqa.h."""
    global _LIB
    if _LIB is not None and path == LIB_PATH:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError("%s is not built; run __graft_entry__.build() (needs nvcc)" % path)
    lib = ctypes.CDLL(path)
    i32p = ctypes.POINTER(ctypes.c_int32)
    vp = ctypes.c_void_p
    lib.h3gqa_causal_fwd.argtypes = [vp, vp, vp, vp, vp, i32p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_float, vp]
    lib.h3gqa_causal_fwd.restype = ctypes.c_int
    lib.h3gqa_attention_fwd.argtypes = [vp, vp, vp, vp, vp, i32p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                        ctypes.POINTER(h3gqa_options), vp]
    lib.h3gqa_attention_fwd.restype = ctypes.c_int
    lib.h3gqa_make_plan.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.POINTER(h3gqa_plan)]
    lib.h3gqa_make_plan.restype = ctypes.c_int
    lib.h3gqa_attention_plan.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int32, ctypes.POINTER(h3gqa_plan)]
    lib.h3gqa_attention_plan.restype = ctypes.c_int
    lib.h3gqa_sync_and_check.argtypes = [vp]
    lib.h3gqa_sync_and_check.restype = ctypes.c_int
    lib.h3gqa_status_string.argtypes = [ctypes.c_int]
    lib.h3gqa_status_string.restype = ctypes.c_char_p
    lib.h3gqa_version.argtypes = []
    lib.h3gqa_version.restype = ctypes.c_int
    if path == LIB_PATH:
        _LIB = lib
    return lib


def _cu_array(cu_seqlens):
    vals = [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    # ctypes would wrap values outside int32 silently; the C ABI takes int32
    if any(v < -2 ** 31 or v >= 2 ** 31 for v in vals):
        raise ValueError("cu_seqlens values must fit in int32")
    arr = (ctypes.c_int32 * max(len(vals), 1))(*vals)
    return arr, len(vals) - 1


def h3gqa_status_string(status) -> str:
    return load().h3gqa_status_string(int(status)).decode()


def h3gqa_version() -> int:
    return int(load().h3gqa_version())


def h3gqa_make_plan(cu_seqlens, n_q_heads, n_kv_heads, head_dim=128):
    """Host-only work plan (see include/h3gqa.h). Raises H3GQAError on a bad shape."""
    arr, n = _cu_array(cu_seqlens)
    plan = h3gqa_plan()
    st = load().h3gqa_make_plan(arr, n, int(n_q_heads), int(n_kv_heads), int(head_dim),
                                ctypes.byref(plan))
    if st != H3GQA_OK:
        raise H3GQAError(st, "h3gqa_make_plan")
    return plan


def h3gqa_attention_plan(cu_seqlens, n_q_heads, n_kv_heads, head_dim=128, causal=True):
    """Host-only work plan of h3gqa_attention_fwd for the causal flag."""
    arr, n = _cu_array(cu_seqlens)
    plan = h3gqa_plan()
    st = load().h3gqa_attention_plan(arr, n, int(n_q_heads), int(n_kv_heads), int(head_dim),
                                     1 if causal else 0, ctypes.byref(plan))
    if st != H3GQA_OK:
        raise H3GQAError(st, "h3gqa_attention_plan")
    return plan


def make_options(causal=True, out_layout=H3GQA_LAYOUT_HEAD_MAJOR, out_int8=False,
                 o_scale_ptr=None, kv_head_begin=0, q_norm_ptr=None, k_norm_ptr=None,
                 cos_ptr=None, sin_ptr=None, k_out_ptr=None, norm_eps=1e-6, kv_head_count=0,
                 status_ptr=None):
    """An h3gqa_options value (pointers as ints or None; see include/h3gqa.h)."""
    return h3gqa_options(1 if causal else 0, int(out_layout), 1 if out_int8 else 0,
                         int(kv_head_begin), o_scale_ptr or None, q_norm_ptr or None,
                         k_norm_ptr or None, cos_ptr or None, sin_ptr or None,
                         k_out_ptr or None, float(norm_eps), int(kv_head_count),
                         status_ptr or None)


def h3gqa_attention_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, cu_seqlens, n_q_heads, n_kv_heads,
                        head_dim, scale, options=None, stream=0, check=True):
    """Raw call with an h3gqa_options (or None for the causal defaults)."""
    arr, n = _cu_array(cu_seqlens)
    st = load().h3gqa_attention_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, arr, n, int(n_q_heads),
                                    int(n_kv_heads), int(head_dim), ctypes.c_float(scale),
                                    ctypes.byref(options) if options is not None else None,
                                    stream or None)
    if check and st != H3GQA_OK:
        raise H3GQAError(st, "h3gqa_attention_fwd")
    return st


def h3gqa_causal_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, cu_seqlens, n_q_heads, n_kv_heads,
                     head_dim, scale, stream=0, check=True):
    """Raw call: device pointers as ints, cu_seqlens host-side, stream handle as int.
    Returns the status; raises H3GQAError on a non-zero status when check=True."""
    arr, n = _cu_array(cu_seqlens)
    st = load().h3gqa_causal_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, arr, n, int(n_q_heads),
                                 int(n_kv_heads), int(head_dim), ctypes.c_float(scale),
                                 stream or None)
    if check and st != H3GQA_OK:
        raise H3GQAError(st, "h3gqa_causal_fwd")
    return st


def h3gqa_sync_and_check(stream=0, check=True):
    st = load().h3gqa_sync_and_check(stream or None)
    if check and st != H3GQA_OK:
        raise H3GQAError(st, "h3gqa_sync_and_check")
    return st


def _cu_total(cu_seqlens):
    vals = cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else list(cu_seqlens)
    if len(vals) == 0:
        raise ValueError("cu_seqlens needs at least one entry")
    return int(vals[-1])


def shard_heads(n_kv_heads, world, rank):
    """KV heads [begin, begin + count) of rank `rank` out of `world` when the
    heads are split into contiguous, balanced ranges (sizes differ by at most
    one; a rank gets count 0 when there are more ranks than heads)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    base, extra = divmod(int(n_kv_heads), int(world))
    begin = rank * base + min(rank, extra)
    return begin, base + (1 if rank < extra else 0)


def check_tensors(q, k, v, cu_seqlens, q_norm_weight=None, k_norm_weight=None, rope_cos=None,
                  rope_sin=None, k_out=None, o=None, lse=None, o_shape=None):
    """Shape, dtype, layout and placement checks of the torch front ends. The
    C ABI takes raw pointers and cannot see sizes or devices, so a short
    table or output here would be read or written out of bounds on the
    device; these checks run first."""
    import torch
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [heads, T, head_dim]")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("%s must be a contiguous bf16 tensor" % name)
    hq, T, d = q.shape
    hkv = k.shape[0]
    if k.shape != (hkv, T, d) or v.shape != (hkv, T, d):
        raise ValueError("k and v must be [Hkv, T, D] with q's T and D")
    if _cu_total(cu_seqlens) != T:
        raise ValueError("cu_seqlens[-1] must equal T = q.shape[1]")
    for name, t, shape, dtype in (("q_norm_weight", q_norm_weight, (d,), torch.bfloat16),
                                  ("k_norm_weight", k_norm_weight, (d,), torch.bfloat16),
                                  ("rope_cos", rope_cos, (T, d // 2), torch.float32),
                                  ("rope_sin", rope_sin, (T, d // 2), torch.float32),
                                  ("k_out", k_out, tuple(k.shape), torch.bfloat16),
                                  ("lse", lse, (hq, T), torch.float32)):
        if t is not None and (tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous()):
            raise ValueError("%s must be a contiguous %s tensor of shape %s" % (name, dtype, shape))
    if o is not None and (tuple(o.shape) != tuple(o_shape or q.shape) or
                          o.dtype != torch.bfloat16 or not o.is_contiguous()):
        raise ValueError("o must be a contiguous bf16 tensor shaped like q")
    for t in (q_norm_weight, k_norm_weight, rope_cos, rope_sin, k_out, o, lse, k, v):
        if t is not None and t.device != q.device:
            raise ValueError("every tensor must be on q's device (%s); got %s" % (q.device, t.device))
    if k_out is not None and k_out.data_ptr() != k.data_ptr() and k_out.numel() > 0:
        def span(t):
            return t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()
        a0, a1 = span(k_out)
        for name, t in (("q", q), ("k", k), ("v", v)):
            b0, b1 = span(t)
            if a0 < b1 and b0 < a1:
                raise ValueError("k_out must be k itself or a buffer that does not overlap %s" % name)
    return hq, hkv, T, d


def check_output_disjoint(o, **others):
    """o is written while other units still read the inputs, so it may share
    no byte with q, k, v, lse, k_out or o_scale."""
    def span(t):
        return t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()
    if o is None or o.numel() == 0:
        return
    a0, a1 = span(o)
    for name, t in others.items():
        if t is not None and t.numel() > 0:
            b0, b1 = span(t)
            if a0 < b1 and b0 < a1:
                raise ValueError("o must not overlap %s" % name)


def _check_cuda(*tensors):
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")


def _finish(status, stream, where):
    """Waits for `stream` and raises if this call's status word is non-zero."""
    stream.synchronize()
    if int(status.item()) != 0:
        raise H3GQAError(H3GQA_ERR_TIMEOUT, where)


def attention_fwd(q, k, v, cu_seqlens, scale=None, causal=True, token_major=False,
                  out_int8=False, stream=None, q_norm_weight=None, k_norm_weight=None,
                  rope_cos=None, rope_sin=None, norm_eps=1e-6, k_out=None, kv_heads=None,
                  o=None, lse=None, o_scale=None, check=True):
    """Torch front end of h3gqa_attention_fwd. Returns (o, lse, o_scale):
    o bf16 (or int8 codes) in [Hq,T,D] or [T,Hq,D] order, lse fp32 [Hq,T],
    o_scale fp32 [Hq,T] / [T,Hq] for int8 output (else None). With the Q/K
    prologue (norm weights: bf16 [D] CUDA; rope tables: fp32 [T, D/2] CUDA)
    the prepared keys go to k_out (allocated if not given; read it back as
    the post-prologue key cache).

    kv_heads = (begin, count) computes that head shard only (rows of the other
    heads in o / lse / o_scale are left as they were; pass the buffers to
    fill them across calls). With check=True (the default) the call waits for
    its stream and raises H3GQAError(H3GQA_ERR_TIMEOUT) if the kernel gave up
    on a bounded wait, using a status word of its own; check=False returns
    at once (the work stays queued) and reports nothing."""
    import torch
    hq, hkv, T, d = check_tensors(q, k, v, cu_seqlens, q_norm_weight, k_norm_weight, rope_cos,
                                  rope_sin, k_out, lse=lse)
    _check_cuda(q, k, v, q_norm_weight, k_norm_weight, rope_cos, rope_sin, k_out, o, lse, o_scale)
    if scale is None:
        scale = d ** -0.5
    shape = (T, hq, d) if token_major else (hq, T, d)
    odt = torch.int8 if out_int8 else torch.bfloat16
    if o is None:
        o = torch.empty(shape, dtype=odt, device=q.device)
    elif tuple(o.shape) != shape or o.dtype != odt or not o.is_contiguous() or o.device != q.device:
        raise ValueError("o must be a contiguous %s tensor of shape %s on %s" % (odt, shape, q.device))
    if lse is None:
        lse = torch.empty((hq, T), dtype=torch.float32, device=q.device)
    if out_int8 and o_scale is None:
        o_scale = torch.empty(shape[:2], dtype=torch.float32, device=q.device)
    if o_scale is not None and (not out_int8 or tuple(o_scale.shape) != shape[:2] or
                                o_scale.dtype != torch.float32 or not o_scale.is_contiguous() or
                                o_scale.device != q.device):
        raise ValueError("o_scale must be a contiguous fp32 %s tensor on %s, with out_int8"
                         % (shape[:2], q.device))
    prep_k = k_norm_weight is not None or rope_cos is not None
    if prep_k and k_out is None:
        k_out = torch.empty_like(k)
    check_output_disjoint(o, q=q, k=k, v=v, lse=lse, k_out=k_out if prep_k else None,
                          o_scale=o_scale)
    kv_begin, kv_count = kv_heads if kv_heads is not None else (0, 0)
    status = torch.zeros(1, dtype=torch.int32, device=q.device) if check else None
    ptr = lambda t: t.data_ptr() if t is not None else None
    opts = make_options(causal, H3GQA_LAYOUT_TOKEN_MAJOR if token_major else
                        H3GQA_LAYOUT_HEAD_MAJOR, out_int8, ptr(o_scale), kv_begin,
                        ptr(q_norm_weight), ptr(k_norm_weight), ptr(rope_cos), ptr(rope_sin),
                        ptr(k_out) if prep_k else None, norm_eps, kv_count, ptr(status))
    with torch.cuda.device(q.device):
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        h3gqa_attention_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), cu_seqlens, hq, hkv, d, float(scale), opts,
                            stream.cuda_stream)
        if check:
            _finish(status, stream, "h3gqa_attention_fwd")
    return o, lse, o_scale


def causal_gqa_fwd(q, k, v, cu_seqlens, scale=None, o=None, lse=None, stream=None, check=True):
    """Torch front end: q [Hq,T,D], k/v [Hkv,T,D] bf16 CUDA tensors (contiguous),
    cu_seqlens host ints. Returns (o [Hq,T,D] bf16, lse [Hq,T] fp32) on q's device,
    queued on `stream` (default: torch's current stream). check=True (the
    default) waits for the stream and raises H3GQAError(H3GQA_ERR_TIMEOUT) if
    the kernel gave up on a bounded wait; check=False leaves the work queued."""
    o, lse, _ = attention_fwd(q, k, v, cu_seqlens, scale, o=o, lse=lse, stream=stream,
                              check=check)
    return o, lse
