"""Independent brute-force attention in numpy, for pinning the oracle on tiny inputs.

Written separately from the C oracle: storage is decoded with torch/numpy's
own type conversions, keys are gathered token by token into dense matrices,
and softmax / log-sum-exp come from scipy.  Nothing here is shared with the
oracle or with the CUDA library.
"""
from __future__ import annotations

import numpy as np
import torch
from scipy.special import logsumexp


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Storage -> float64 through the libraries' own conversions."""
    a = np.ascontiguousarray(bits)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    if dtype == "fp16":
        return a.view(np.float16).astype(np.float64)
    if dtype == "fp8":
        return torch.from_numpy(a.view(np.uint8)).view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    if dtype == "fp32":
        return a.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def dense_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, bias=None):
    """softmax(scale * K q + bias) V for one query row; returns (out, lse)."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1]), -np.inf
    s = scale * (K @ q)
    if bias is not None:
        s = s + bias
    lse = logsumexp(s)
    return np.exp(s - lse) @ V, lse


def paged_decode(case):
    """Token-by-token gather through the block table, then dense attention per row."""
    P, D, Hq, Hkv, sq = case.page_size, case.head_dim, case.num_heads, case.num_kv_heads, case.sq
    G = Hq // Hkv
    cache = decode(case.kv_cache, case.dtype)
    q = decode(case.q, case.dtype)
    B = case.batch
    out = np.zeros((B, sq, Hq, D))
    lse = np.zeros((B, sq, Hq))
    bmm1 = case.scale * case.q_scale * case.k_scale
    for b in range(B):
        L = int(case.seq_lens[b])
        for i in range(sq):
            if case.causal:
                pos = L - sq + i
                lo = max(0, pos - (case.window - 1)) if case.window > 0 else 0
                hi = pos + 1
            else:
                lo = max(0, (L - (case.window + sq - 1)) // P) * P if case.window > 0 else 0
                hi = L
            toks = list(range(lo, hi))
            K = np.zeros((len(toks), Hkv, D))
            V = np.zeros((len(toks), Hkv, D))
            for n, j in enumerate(toks):
                page = case.block_table[b, j // P]
                K[n] = cache[page, :, j % P, :D]
                V[n] = cache[page, :, j % P, D:]
            for h in range(Hq):
                o, l = dense_attention(q[b, i, h], K[:, h // G], V[:, h // G], bmm1)
                out[b, i, h] = case.v_scale * o
                lse[b, i, h] = l
    return out, lse


def segmented(case):
    """Per-segment dense attention, then the softmax-over-segments combine, in numpy."""
    q = decode(case.q, case.dtype)
    k = decode(case.k, case.dtype)
    v = decode(case.v, case.dtype)
    n, Hq, D = q.shape
    Hkv, topk, bs, local = case.num_kv_heads, case.topk, case.bs, case.local
    G = Hq // Hkv
    groups = topk + 1
    rows = topk * bs + local
    used = case.used.reshape(n, groups)
    seg_out = np.zeros((n, groups, Hq, D))
    seg_lse = np.full((n, groups, Hq), -np.inf)
    out = np.zeros((n, Hq, D))
    for i in range(n):
        for g in range(groups):
            off = i * rows + (g * bs if g < topk else topk * bs)
            u = int(used[i, g])
            for h in range(Hq):
                o, l = dense_attention(q[i, h], k[off:off + u, h // G], v[off:off + u, h // G], D ** -0.5)
                seg_out[i, g, h] = o
                seg_lse[i, g, h] = l
        live = used[i] > 0
        if not live.any():
            continue
        prior = np.concatenate([case.bias[i].astype(np.float64), [0.0]])
        for h in range(Hq):
            logits = seg_lse[i, :, h] + prior
            w = np.exp(logits[live] - logsumexp(logits[live]))
            out[i, h] = w @ seg_out[i, live, h]
    return out, seg_out, seg_lse
