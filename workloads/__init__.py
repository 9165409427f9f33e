"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws and lays out input bytes: normal samples rounded to the
storage type, page pools, block tables, lengths and masks.  It holds none of
the attention arithmetic, so both the CUDA library and the CPU oracle can be
fed from it without sharing any of the method.

Storage is returned as numpy arrays: uint16 bit patterns for bf16/fp16,
uint8 for fp8-e4m3, float32 and int32 as themselves.

Workloads (named by what they are):
  tiny_decode            B=2, sq=1, Hq=4, Hkv=2, D=64, P=16, seq_lens {37, 50},
                         8-page pool in seeded random order, the spare page NaN
  gqa_decode_b64         B=64, sq=1, Hq=32, Hkv=8, D=128, P=16, L ~ U[512, 4096]
  query_block_sq8        B=32, sq=8, Hq=32, Hkv=8, D=128, P=16, L ~ U[1024, 8192]
                         (``window=4096`` gives the windowed second pass)
  dash_segments_n256     n=256, Hq=32, Hkv=8, D=128, topk=8, bs=64, local=128
  fp8_long_b8            B=8, sq=1, Hq=64, Hkv=8, D=128, P=64, L=131072, fp8-e4m3
                         with per-tensor scales amax/448 for q, K and V
"""
from __future__ import annotations

import dataclasses
import math
import os

import numpy as np
import torch

BF16_NAN = 0x7FC0
FP16_NAN = 0x7E00
FP8_NAN = 0x7F
# fp8 power-of-two scale: just above amax/448 for N(0,1) samples of this size
# (amax ~ 6.1), so dequantisation is exact in any precision.  The fp8
# workloads use per-tensor scales amax/448 instead (paged_case, fp8_scales="amax").
FP8_SCALE = 1.0 / 64.0
E4M3_MAX = 448.0

SEED_BASE = 1000
WORKLOAD_SEEDS = {
    "tiny_decode": SEED_BASE + 0,
    "gqa_decode_b64": SEED_BASE + 1,
    "query_block_sq8": SEED_BASE + 2,
    "dash_segments_n256": SEED_BASE + 3,
    "fp8_long_b8": SEED_BASE + 4,
}


def _nan_bits(dtype: str):
    return {"bf16": BF16_NAN, "fp16": FP16_NAN, "fp8": FP8_NAN}[dtype]


def storage_dtype(dtype: str):
    return np.uint8 if dtype == "fp8" else np.uint16


def round_to(x: np.ndarray, dtype: str, scale: float = 1.0) -> np.ndarray:
    """Round float32 samples to the storage type (RNE; fp8 saturating after /scale)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp16":
        return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "fp8":
        t = torch.clamp(t / scale, -448.0, 448.0)
        return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    raise ValueError(dtype)


def normal_storage(rng: np.random.Generator, shape, dtype: str, scale: float = 1.0,
                   chunk: int = 1 << 26) -> np.ndarray:
    """N(0,1) samples rounded to ``dtype``, drawn in bounded chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=storage_dtype(dtype))
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = round_to(rng.standard_normal(e - s, dtype=np.float32), dtype, scale)
    return out.reshape(shape)


def amax_scale(amax) -> float:
    """Per-tensor fp8 scale amax / 448, as an fp32 value."""
    return float(np.float32(amax) / np.float32(E4M3_MAX))


def _parallel(fn, items, threads=None):
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=threads or min(32, os.cpu_count() or 1)) as ex:
        return list(ex.map(fn, items))


def fp8_kv_pool(seed: int, shape, chunk_rows: int = 1 << 16):
    """A pool [..., 2*D] of N(0,1) key/value rows quantised to e4m3 with
    per-tensor scales: k_scale = amax(K)/448 over every key half of the pool,
    v_scale = amax(V)/448 over every value half.

    Each block of chunk_rows rows is drawn from its own seeded stream, once to
    find the two maxima and again to quantise, so the pool is never held in
    fp32.  Returns (uint8 storage, k_scale, v_scale).
    """
    twoD = int(shape[-1])
    D = twoD // 2
    rows = int(np.prod(shape[:-1]))
    starts = list(range(0, rows, chunk_rows))
    seeds = np.random.SeedSequence([int(seed), 0xF8]).spawn(len(starts))

    def draw(i):
        n = min(chunk_rows, rows - starts[i])
        return np.random.default_rng(seeds[i]).standard_normal((n, twoD), dtype=np.float32)

    def maxima(i):
        x = np.abs(draw(i))
        return float(x[:, :D].max()), float(x[:, D:].max())

    m = _parallel(maxima, range(len(starts)))
    k_scale = amax_scale(max(a for a, _ in m))
    v_scale = amax_scale(max(b for _, b in m))
    out = np.empty((rows, twoD), np.uint8)

    def fill(i):
        x = draw(i)
        s = starts[i]
        out[s:s + x.shape[0], :D] = round_to(x[:, :D], "fp8", k_scale)
        out[s:s + x.shape[0], D:] = round_to(x[:, D:], "fp8", v_scale)

    _parallel(fill, range(len(starts)))
    return out.reshape(shape), k_scale, v_scale


def fp8_quantised(rng: np.random.Generator, shape):
    """N(0,1) samples quantised to e4m3 with the per-tensor scale amax/448.
    Returns (uint8 storage, scale)."""
    x = rng.standard_normal(int(np.prod(shape)), dtype=np.float32)
    scale = amax_scale(np.abs(x).max()) if x.size else 1.0
    return round_to(x, "fp8", scale).reshape(shape), scale


@dataclasses.dataclass
class PagedCase:
    """One paged-decode problem: raw storage plus the scalars of the call."""
    name: str
    q: np.ndarray            # [B, sq, Hq, D] storage
    kv_cache: np.ndarray     # [num_pages, Hkv, P, 2*D] storage
    block_table: np.ndarray  # int32 [B, W]
    seq_lens: np.ndarray     # int32 [B]
    dtype: str               # storage type of q and the cache
    sq: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    scale: float
    q_scale: float = 1.0
    k_scale: float = 1.0
    v_scale: float = 1.0
    window: int = 0
    causal: bool = False
    poison_page: int = -1
    chunk_tokens: int = 0    # Split-KV chunk the configuration fixes (0: the library's plan)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_kv_len(self) -> int:
        return int(self.seq_lens.max()) if self.batch else 0

    def oracle_kwargs(self):
        return dict(sq=self.sq, num_heads=self.num_heads, num_kv_heads=self.num_kv_heads,
                    head_dim=self.head_dim, page_size=self.page_size, scale=self.scale,
                    q_scale=self.q_scale, k_scale=self.k_scale, v_scale=self.v_scale,
                    window=self.window, causal=self.causal)


def paged_case(*, name="paged", seq_lens, sq=1, num_heads=32, num_kv_heads=8, head_dim=128,
               page_size=16, dtype="bf16", seed=0, pool_factor=1.25, window=0, causal=False,
               poison_tail=True, table_width=None, scale=None, fp8_scale=FP8_SCALE,
               spare_pages=1, fp8_scales="amax", scales=None) -> PagedCase:
    """Build a paged-decode problem.

    The pool holds ceil(pool_factor * sum ceil(L/P)) data pages plus one
    NaN page; every request takes its pages without replacement from a seeded
    permutation of the pool, so pages are scattered and out of order.  Table
    columns past a request's last page point at the NaN page, and (with
    ``poison_tail``) the slots past L in a request's last page are NaN too, so
    any read outside the visible keys shows up in the output.

    fp8 caches: with fp8_scales="amax" (default) K, V and the pre-quantised q
    each get their own per-tensor scale amax/448 (three distinct scales that
    are not powers of two); with "pow2" all three share the power of two
    ``fp8_scale``.  ``scales=(q_scale, k_scale, v_scale)`` sets the three
    scalars of a 16-bit case (1.0 each by default).
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(seq_lens, dtype=np.int32).reshape(-1)
    B, P, D, Hkv = lens.shape[0], int(page_size), int(head_dim), int(num_kv_heads)
    pages_needed = [int(math.ceil(int(L) / P)) for L in lens]
    total = sum(pages_needed)
    n_data = max(int(math.ceil(pool_factor * total)), total + spare_pages - 1, 1)
    num_pages = n_data + 1
    poison = n_data  # the last page of the pool is all NaN
    W = table_width or max(1, max(pages_needed) if B else 1)
    per_tensor = dtype == "fp8" and fp8_scales == "amax"
    if dtype == "fp8" and fp8_scales not in ("amax", "pow2"):
        raise ValueError(fp8_scales)
    scale_kv = fp8_scale if dtype == "fp8" else 1.0
    q_scale = k_scale = v_scale = scale_kv
    if scales is not None:
        if dtype == "fp8":
            raise ValueError("fp8 scales come from the data (fp8_scales)")
        q_scale, k_scale, v_scale = (float(x) for x in scales)

    if per_tensor:
        cache, k_scale, v_scale = fp8_kv_pool(seed, (num_pages, Hkv, P, 2 * D))
    else:
        cache = normal_storage(rng, (num_pages, Hkv, P, 2 * D), dtype, scale_kv)
    cache[poison] = _nan_bits(dtype)
    perm = rng.permutation(n_data).astype(np.int32)
    table = np.full((B, W), poison, dtype=np.int32)
    cursor = 0
    for b in range(B):
        k = pages_needed[b]
        table[b, :k] = perm[cursor:cursor + k]
        cursor += k
        if poison_tail and k > 0 and lens[b] % P:
            cache[table[b, k - 1], :, lens[b] % P:, :] = _nan_bits(dtype)
    if per_tensor:
        q, q_scale = fp8_quantised(rng, (B, sq, num_heads, D))
    else:
        q = normal_storage(rng, (B, sq, num_heads, D), dtype, scale_kv)
    return PagedCase(
        name=name, q=q, kv_cache=cache, block_table=table, seq_lens=lens, dtype=dtype, sq=int(sq),
        num_heads=int(num_heads), num_kv_heads=Hkv, head_dim=D, page_size=P,
        scale=float(scale if scale is not None else D ** -0.5),
        q_scale=q_scale, k_scale=k_scale, v_scale=v_scale,
        window=int(window), causal=bool(causal), poison_page=poison)


def uniform_lens(rng_seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """Integer lengths drawn uniformly from [lo, hi] (both ends included)."""
    return np.random.default_rng(rng_seed).integers(lo, hi + 1, size=B).astype(np.int32)


def tiny_decode() -> PagedCase:
    """B=2, sq=1, Hq=4, Hkv=2, D=64, P=16, L={37, 50}; 3 + 4 pages of an 8-page pool."""
    seed = WORKLOAD_SEEDS["tiny_decode"]
    rng = np.random.default_rng(seed)
    P, D, Hkv, Hq = 16, 64, 2, 4
    lens = np.array([37, 50], np.int32)
    cache = normal_storage(rng, (8, Hkv, P, 2 * D), "bf16")
    perm = rng.permutation(8).astype(np.int32)
    table = np.empty((2, 4), np.int32)
    table[0, :3] = perm[0:3]
    table[0, 3] = perm[7]          # padding column: the spare page
    table[1, :4] = perm[3:7]
    cache[perm[7]] = BF16_NAN      # the spare page is NaN
    cache[table[0, 2], :, 37 % P:, :] = BF16_NAN
    cache[table[1, 3], :, 50 % P:, :] = BF16_NAN
    q = normal_storage(rng, (2, 1, Hq, D), "bf16")
    return PagedCase(name="tiny_decode", q=q, kv_cache=cache, block_table=table, seq_lens=lens,
                     dtype="bf16", sq=1, num_heads=Hq, num_kv_heads=Hkv, head_dim=D, page_size=P,
                     scale=1.0 / 8.0, poison_page=int(perm[7]))


def gqa_decode_b64() -> PagedCase:
    seed = WORKLOAD_SEEDS["gqa_decode_b64"]
    return paged_case(name="gqa_decode_b64", seq_lens=uniform_lens(seed, 64, 512, 4096), sq=1,
                      num_heads=32, num_kv_heads=8, head_dim=128, page_size=16, dtype="bf16",
                      seed=seed + 100)


def query_block_sq8(window: int = 0) -> PagedCase:
    seed = WORKLOAD_SEEDS["query_block_sq8"]
    name = "query_block_sq8" + (f"_w{window}" if window else "")
    return paged_case(name=name, seq_lens=uniform_lens(seed, 32, 1024, 8192), sq=8,
                      num_heads=32, num_kv_heads=8, head_dim=128, page_size=16, dtype="bf16",
                      seed=seed + 100, window=window)


def fp8_long_b8(seq_len: int = 131072, batch: int = 8) -> PagedCase:
    seed = WORKLOAD_SEEDS["fp8_long_b8"]
    case = paged_case(name="fp8_long_b8", seq_lens=np.full(batch, seq_len, np.int32), sq=1,
                      num_heads=64, num_kv_heads=8, head_dim=128, page_size=64, dtype="fp8",
                      seed=seed + 100)
    case.chunk_tokens = 4096  # the configuration's Split-KV: 32 chunks of 4096 keys per sequence
    return case


@dataclasses.dataclass
class SegmentCase:
    """One DASH segmented-attention problem."""
    name: str
    q: np.ndarray      # [n, Hq, D] storage
    k: np.ndarray      # [n*(topk*bs+local), Hkv, D] storage
    v: np.ndarray      # same
    used: np.ndarray   # int32 [n*(topk+1)]
    bias: np.ndarray   # float32 [n, topk]
    dtype: str
    num_kv_heads: int
    topk: int
    bs: int
    local: int

    @property
    def n(self):
        return int(self.q.shape[0])


def segment_case(*, name="segments", n=256, num_heads=32, num_kv_heads=8, head_dim=128, topk=8,
                 bs=64, local=128, dtype="bf16", seed=0, p_empty=0.1, poison_unused=True,
                 used=None) -> SegmentCase:
    """Segments of bs rows (topk per query) plus one local segment per query.

    used: 0 with probability p_empty, else uniform on [1, bs]; local used is
    uniform on [1, local].  Rows past a segment's used prefix are NaN when
    ``poison_unused`` is set.  bias ~ N(0, 1) in float32.
    """
    rng = np.random.default_rng(seed)
    rows = topk * bs + local
    k = normal_storage(rng, (n * rows, num_kv_heads, head_dim), dtype)
    v = normal_storage(rng, (n * rows, num_kv_heads, head_dim), dtype)
    q = normal_storage(rng, (n, num_heads, head_dim), dtype)
    if used is None:
        u = np.empty((n, topk + 1), np.int32)
        if topk:
            u[:, :topk] = rng.integers(1, bs + 1, size=(n, topk))
            u[:, :topk][rng.random((n, topk)) < p_empty] = 0
        u[:, topk] = rng.integers(1, local + 1, size=n) if local else 0
    else:
        u = np.asarray(used, np.int32).reshape(n, topk + 1)
    bias = rng.standard_normal((n, topk), dtype=np.float32)
    if poison_unused:
        nan = _nan_bits(dtype)
        for i in range(n):
            for g in range(topk + 1):
                off = i * rows + (g * bs if g < topk else topk * bs)
                cap = bs if g < topk else local
                k[off + u[i, g]: off + cap] = nan
                v[off + u[i, g]: off + cap] = nan
    return SegmentCase(name=name, q=q, k=k, v=v, used=u.reshape(-1).copy(), bias=bias, dtype=dtype,
                       num_kv_heads=num_kv_heads, topk=topk, bs=bs, local=local)


@dataclasses.dataclass
class PagedSegmentCase:
    """DASH segments as key ranges of each query's request in a paged cache."""
    name: str
    q: np.ndarray            # [n, Hq, D] storage
    kv_cache: np.ndarray     # [num_pages, Hkv, P, 2D] storage
    block_table: np.ndarray  # int32 [n, W]
    seq_lens: np.ndarray     # int32 [n]
    seg_start: np.ndarray    # int32 [n, topk+1]
    used: np.ndarray         # int32 [n, topk+1]
    bias: np.ndarray         # float32 [n, topk]
    dtype: str
    num_kv_heads: int
    page_size: int
    topk: int
    bs: int
    local: int

    @property
    def n(self):
        return int(self.q.shape[0])


def paged_segment_case(*, name="paged_segments", n=16, seq_lens=None, num_heads=32, num_kv_heads=8, head_dim=128,
                       page_size=16, topk=8, bs=64, local=128, dtype="bf16", seed=0, p_empty=0.1,
                       seq_range=(1024, 4096)) -> PagedSegmentCase:
    """Each query is one request: its gathered segments are topk distinct
    bs-aligned blocks of its history (a random used prefix, 0 with p_empty),
    and its local segment is the last `used` keys (used ~ U[1, local])."""
    rng = np.random.default_rng(seed)
    lens = (np.asarray(seq_lens, np.int32) if seq_lens is not None
            else rng.integers(seq_range[0], seq_range[1] + 1, size=n).astype(np.int32))
    base = paged_case(name=name, seq_lens=lens, sq=1, num_heads=num_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, page_size=page_size, dtype=dtype, seed=seed + 1)
    groups = topk + 1
    seg_start = np.zeros((n, groups), np.int32)
    used = np.zeros((n, groups), np.int32)
    for i in range(n):
        L = int(lens[i])
        u_loc = int(rng.integers(1, min(local, L) + 1))
        seg_start[i, topk] = L - u_loc
        used[i, topk] = u_loc
        nblocks = max(1, (L - u_loc) // bs)
        blocks = rng.choice(nblocks, size=topk, replace=nblocks < topk)
        for g in range(topk):
            seg_start[i, g] = int(blocks[g]) * bs
            room = max(0, min(bs, L - seg_start[i, g]))
            used[i, g] = 0 if (rng.random() < p_empty or room == 0) else int(rng.integers(1, room + 1))
    bias = rng.standard_normal((n, topk), dtype=np.float32)
    q = normal_storage(rng, (n, num_heads, head_dim), dtype)
    return PagedSegmentCase(name=name, q=q, kv_cache=base.kv_cache, block_table=base.block_table, seq_lens=lens,
                            seg_start=seg_start, used=used, bias=bias, dtype=dtype, num_kv_heads=num_kv_heads,
                            page_size=page_size, topk=topk, bs=bs, local=local)


def dash_paged_n256() -> PagedSegmentCase:
    """256 decode queries, each attending 8 gathered blocks of 64 keys plus the
    last up-to-128 keys of its own request (L ~ U[1024, 4096]) in a paged cache."""
    return paged_segment_case(name="dash_paged_n256", n=256, seed=SEED_BASE + 6)


def dash_segments_n256() -> SegmentCase:
    return segment_case(name="dash_segments_n256", seed=WORKLOAD_SEEDS["dash_segments_n256"])


@dataclasses.dataclass
class CacheWriteCase:
    """A batch of new key/value rows and the paged cache they are written into."""
    name: str
    key: np.ndarray        # [T, Hkv, D] storage (in_dtype)
    value: np.ndarray      # [T, Hkv, D]
    slots: np.ndarray      # int64 [T]; -1 marks a padding token
    kv_cache: np.ndarray   # [num_pages, Hkv, P, 2*D] storage (kv_dtype)
    in_dtype: str
    kv_dtype: str
    page_size: int
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def num_tokens(self):
        return int(self.slots.shape[0])


def cache_write_case(*, name="cache_write", num_tokens, num_kv_heads=8, head_dim=128, page_size=16,
                     in_dtype="bf16", kv_dtype="fp8", seed=0, pool_factor=1.25, pad_every=0) -> CacheWriteCase:
    """num_tokens new rows written to distinct slots of whole pages drawn in
    seeded random order from a pool pool_factor times larger than needed."""
    rng = np.random.default_rng(seed)
    pages_needed = -(-num_tokens // page_size)
    num_pages = max(1, int(math.ceil(pool_factor * pages_needed)))
    pages = rng.permutation(num_pages)[:pages_needed].astype(np.int64)
    t = np.arange(num_tokens)
    slots = pages[t // page_size] * page_size + t % page_size
    if pad_every:
        slots[::pad_every] = -1
    key = normal_storage(rng, (num_tokens, num_kv_heads, head_dim), in_dtype)
    value = normal_storage(rng, (num_tokens, num_kv_heads, head_dim), in_dtype)
    cache = np.zeros((num_pages, num_kv_heads, page_size, 2 * head_dim), dtype=storage_dtype(kv_dtype))
    scale = FP8_SCALE if kv_dtype == "fp8" else 1.0
    return CacheWriteCase(name=name, key=key, value=value, slots=slots, kv_cache=cache, in_dtype=in_dtype,
                          kv_dtype=kv_dtype, page_size=page_size, k_scale=scale, v_scale=scale)


def kv_write_32k() -> CacheWriteCase:
    """32768 new tokens (a prefill chunk), Hkv=8, D=128, bf16 rows into an fp8 cache, P=16."""
    return cache_write_case(name="kv_write_32k", num_tokens=32768, seed=SEED_BASE + 5)


def to_torch(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Storage array -> torch tensor on `device` (bf16/fp16 as themselves, fp8 as uint8)."""
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif dtype == "fp16":
        t = torch.from_numpy(a.view(np.int16)).view(torch.float16)
    elif dtype == "fp8":
        t = torch.from_numpy(a.view(np.uint8))
    elif dtype == "int32":
        t = torch.from_numpy(a.astype(np.int32))
    elif dtype == "fp32":
        t = torch.from_numpy(a.astype(np.float32))
    else:
        raise ValueError(dtype)
    return t.to(device)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "gqa_decode_b64": gqa_decode_b64,
    "query_block_sq8": query_block_sq8,
    "query_block_sq8_w4096": lambda: query_block_sq8(window=4096),
    "dash_segments_n256": dash_segments_n256,
    "fp8_long_b8": fp8_long_b8,
    "kv_write_32k": kv_write_32k,
    "dash_paged_n256": dash_paged_n256,
}
