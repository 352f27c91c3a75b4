"""Second, independent statement of causal GQA for tiny inputs (numpy, fp64).

It pins the C oracle: dense S x S logits, an explicit lower-triangular mask,
KV heads repeated in place for GQA, a log-sum-exp and a dense P @ V. It
shares nothing with the C file but the definition.
"""
import numpy as np


def bf16_bits_to_f64(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dense_causal_gqa(q, k, v, cu_seqlens, scale, causal=True):
    """q [Hq,T,D], k/v [Hkv,T,D] as float64 arrays. Returns (o, lse, P-list).
    causal=False drops the mask (every key of the sequence)."""
    hq, T, D = q.shape
    hkv = k.shape[0]
    rep = hq // hkv
    k_full = np.repeat(k, rep, axis=0)      # head h reads kv head h // rep
    v_full = np.repeat(v, rep, axis=0)
    o = np.zeros((hq, T, D))
    lse = np.zeros((hq, T))
    probs = []
    for b in range(len(cu_seqlens) - 1):
        s, e = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        n = e - s
        if n == 0:
            continue
        z = scale * np.einsum("hid,hjd->hij", q[:, s:e], k_full[:, s:e])
        mask = np.tril(np.ones((n, n), dtype=bool)) if causal else np.ones((n, n), dtype=bool)
        z = np.where(mask[None], z, -np.inf)
        m = z.max(axis=-1, keepdims=True)
        L = m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True))
        P = np.exp(z - L)
        o[:, s:e] = P @ v_full[:, s:e]
        lse[:, s:e] = L[..., 0]
        probs.append(P)
    return o, lse, probs
