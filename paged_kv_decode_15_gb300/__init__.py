"""Attention over a paged KV cache on GB300 (sm_103a): Python binding of libpkd.

Argument marshalling only.  Every step runs in the library's CUDA kernels;
torch supplies device memory and the current stream.  There is no CPU path:
if libpkd.so is missing or a GPU is absent, the calls raise.

Entry points (same names as the C ABI in include/pkd.h, without the prefix):
  paged_decode(q, kv_cache, block_table, seq_lens, scale, window, out, lse, ...)
  segmented_attention(q, k, v, used, bias, bs, local, out, ...)
  lse_merge(part_out, part_lse, prior=None, live=None, out=None, lse_out=None)
  workspace_size(...), workspace_init(ws), workspace_check(ws)
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkd.so")

OK, EINVAL, EUNSUPPORTED, ECUDA, EDEVICE_BOUNDS, ETIMEOUT = range(6)
BF16, FP16, FP8_E4M3, FP32 = 0, 1, 2, 3
FLAG_CAUSAL, FLAG_MMA_SMALL_M, FLAG_FMA, FLAG_GRID, FLAG_FLAT, FLAG_BALANCED = 1, 2, 4, 8, 16, 32
FLAG_TEST_TIMEOUT = 64
FLAG_HOST_IO = 128

SYMBOLS = ("pkd_version", "pkd_last_error", "pkd_paged_decode_workspace_size", "pkd_paged_decode_kernel_name",
           "pkd_workspace_init",
           "pkd_workspace_check", "pkd_paged_decode", "pkd_paged_decode_static", "pkd_paged_decode_static_check",
           "pkd_cache_write",
           "pkd_segmented_attention", "pkd_segmented_attention_paged", "pkd_lse_merge")


class PkdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkd status {status}: {message}")
        self.status = status


_lib = None


def build(force: bool = False) -> str:
    """Compile libpkd.so in-tree for sm_103a."""
    from . import _build
    return _build.build(force=force)


def load_library(path: str = LIB_PATH):
    """Load libpkd.so and declare its C signatures (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with paged_kv_decode_15_gb300.build() "
                          "(nvcc for sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    P, I, I64, F, U, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_uint,
                           ctypes.c_size_t)
    lib.pkd_version.restype = I
    lib.pkd_last_error.restype = ctypes.c_char_p
    lib.pkd_paged_decode_workspace_size.argtypes = [I, I, I, I, I, I, I, I, I, I, U]
    lib.pkd_paged_decode_workspace_size.restype = SZ
    lib.pkd_paged_decode_kernel_name.argtypes = [I, I, I, I, I, I, I, I, I, I, U]
    lib.pkd_paged_decode_kernel_name.restype = ctypes.c_char_p
    lib.pkd_workspace_init.argtypes = [P, SZ, P]
    lib.pkd_workspace_check.argtypes = [P, SZ, P]
    lib.pkd_paged_decode.argtypes = [P, I, P, I, I64, P, I64, P, I, I, I, I, I, I, I, F, F, F, F, I,
                                     P, I, P, P, SZ, I, U, P]
    lib.pkd_paged_decode_static.argtypes = [P, I, P, I, I64, P, I64, P, I, I, I, I, I, I, I, F, F, F, F, I,
                                            P, I, P, I, U, P]
    lib.pkd_paged_decode_static_check.argtypes = [P]
    lib.pkd_cache_write.argtypes = [P, P, I, I64, I64, P, I64, I, I, I, I64, P, I, F, F, P]
    lib.pkd_segmented_attention.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, P, P, P, P]
    lib.pkd_segmented_attention_paged.argtypes = [P, I, P, I64, P, I64, P, P, P, I, I, I, I, I, I, I, I, I,
                                                  P, P, P, P]
    lib.pkd_lse_merge.argtypes = [P, P, P, P, I, I, I, I, P, I, P, P]
    for name in ("pkd_workspace_init", "pkd_workspace_check", "pkd_paged_decode", "pkd_paged_decode_static",
                 "pkd_paged_decode_static_check", "pkd_cache_write", "pkd_segmented_attention", "pkd_segmented_attention_paged", "pkd_lse_merge"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def _check(status: int):
    if status != OK:
        raise PkdError(status, load_library().pkd_last_error().decode())


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return BF16
    if t == torch.float16:
        return FP16
    if t in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return FP8_E4M3
    if t == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _cuda(t, name):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t


def version() -> int:
    return load_library().pkd_version()


def workspace_size(batch, sq, num_heads, num_kv_heads, head_dim, page_size, max_kv_len, kv_dtype, window=0,
                   chunk_tokens=0, flags=0) -> int:
    n = load_library().pkd_paged_decode_workspace_size(batch, sq, num_heads, num_kv_heads, head_dim, page_size,
                                                       max_kv_len, int(kv_dtype), int(window), int(chunk_tokens),
                                                       int(flags))
    if n == 0:
        raise PkdError(EINVAL, load_library().pkd_last_error().decode())
    return n


def kernel_name(batch, sq, num_heads, num_kv_heads, head_dim, page_size, max_kv_len, kv_dtype, window=0,
                chunk_tokens=0, flags=0) -> str:
    """The kernel paged_decode launches for these shapes and flags."""
    name = load_library().pkd_paged_decode_kernel_name(batch, sq, num_heads, num_kv_heads, head_dim, page_size,
                                                       max_kv_len, int(kv_dtype), int(window), int(chunk_tokens),
                                                       int(flags))
    if name is None:
        raise PkdError(EINVAL, load_library().pkd_last_error().decode())
    return name.decode()


def workspace_init(ws: torch.Tensor, stream=None):
    _check(load_library().pkd_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def workspace_check(ws: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the workspace status word; returns the status code."""
    return load_library().pkd_workspace_check(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


_ws_cache: dict = {}


def _workspace(nbytes: int, device) -> torch.Tensor:
    key = (str(device), nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        workspace_init(ws)
        _ws_cache[key] = ws
    return ws


def paged_decode(q, kv_cache, block_table, seq_lens, scale, window=0, out=None, lse=None, *, q_scale=1.0,
                 k_scale=1.0, v_scale=1.0, max_kv_len=None, workspace=None, chunk_tokens=0, causal=False,
                 mma_small_m=False, force_fma=False, grid=False, flat=False, balanced=False, out_dtype=None,
                 test_timeout=False, host_io=False, stream=None):
    """Attention of each request's query block over its paged keys.

    q [B, sq, Hq, D]; kv_cache [num_pages, Hkv, P, 2*D] (bf16, fp16, or uint8 /
    float8_e4m3fn for fp8, with q of the same type); block_table int32 [B, W];
    seq_lens int32 [B].  Returns (out [B, sq, Hq, D], lse fp32 [B, sq, Hq]).
    max_kv_len defaults to the table's capacity W * P (no host sync).
    test_timeout sets the diagnostic PKD_FLAG_TEST_TIMEOUT.  host_io sets
    PKD_FLAG_HOST_IO: q, block_table, seq_lens (and out, lse, allocated pinned
    when not given) are pinned host tensors that the kernels read and write in
    place; kv_cache and the workspace stay on the device.
    """
    lib = load_library()
    _cuda(kv_cache, "kv_cache")
    io = ((q, "q"), (block_table, "block_table"), (seq_lens, "seq_lens"), (out, "out"), (lse, "lse"))
    for t, n in io:
        if host_io:
            if t is not None and (t.is_cuda or not t.is_pinned()):
                raise ValueError(f"{n} must be a pinned host tensor with host_io")
        else:
            _cuda(t, n)
    B, sq, Hq, D = q.shape
    num_pages, Hkv, P, twoD = kv_cache.shape
    if twoD != 2 * D:
        raise ValueError(f"kv_cache last dim {twoD} != 2 * head_dim {2 * D}")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if not (q.is_contiguous() and kv_cache.is_contiguous() and seq_lens.is_contiguous()):
        raise ValueError("q, kv_cache and seq_lens must be contiguous")
    if block_table.stride(1) != 1:
        raise ValueError("block_table rows must be contiguous")
    kv_dt = dtype_code(kv_cache.dtype)
    q_dt = dtype_code(q.dtype)
    place = dict(pin_memory=True) if host_io else dict(device=q.device)
    if out is None:
        odt = out_dtype or (torch.bfloat16 if kv_dt == FP8_E4M3 else q.dtype)
        out = torch.empty((B, sq, Hq, D), dtype=odt, **place)
    if lse is None:
        lse = torch.empty((B, sq, Hq), dtype=torch.float32, **place)
    if max_kv_len is None:
        max_kv_len = block_table.shape[1] * P
    flags = (FLAG_CAUSAL if causal else 0) | (FLAG_MMA_SMALL_M if mma_small_m else 0) | \
        (FLAG_FMA if force_fma else 0) | (FLAG_GRID if grid else 0) | (FLAG_FLAT if flat else 0) | \
        (FLAG_BALANCED if balanced else 0) | (FLAG_TEST_TIMEOUT if test_timeout else 0) | \
        (FLAG_HOST_IO if host_io else 0)
    need = workspace_size(B, sq, Hq, Hkv, D, P, max_kv_len, kv_dt, window, chunk_tokens, flags)
    if workspace is None:
        workspace = _workspace(need, kv_cache.device)
    _check(lib.pkd_paged_decode(
        _ptr(q), q_dt, _ptr(kv_cache), kv_dt, num_pages, _ptr(block_table), block_table.stride(0), _ptr(seq_lens),
        B, sq, Hq, Hkv, D, P, int(max_kv_len), float(scale), float(q_scale), float(k_scale), float(v_scale),
        int(window), _ptr(out), dtype_code(out.dtype), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), int(chunk_tokens), flags, _stream(stream)))
    return out, lse


def segmented_attention(q, k, v, used, bias, bs, local, out=None, *, seg_out=None, seg_lse=None,
                        return_segments=False, stream=None):
    """DASH segmented attention + combine.

    q [n, Hq, D]; k, v [n*(topk*bs+local), Hkv, D]; used int32 [n*(topk+1)];
    bias fp32 [n, topk].  Returns out [n, Hq, D] (and the per-segment fp32
    (seg_out [n, topk+1, Hq, D], seg_lse [n, topk+1, Hq]) when asked).
    """
    lib = load_library()
    n, Hq, D = q.shape
    Hkv = k.shape[1]
    topk = bias.shape[1] if bias is not None else 0
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (used, "used"), (bias, "bias")):
        _cuda(t, name)
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if used.dtype != torch.int32 or (bias is not None and bias.dtype != torch.float32):
        raise TypeError("used must be int32 and bias float32")
    if out is None:
        out = torch.empty_like(q)
    if return_segments and seg_out is None:
        seg_out = torch.empty((n, topk + 1, Hq, D), dtype=torch.float32, device=q.device)
        seg_lse = torch.empty((n, topk + 1, Hq), dtype=torch.float32, device=q.device)
    _check(lib.pkd_segmented_attention(
        _ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(used), _ptr(bias), n, Hq, Hkv, D, topk, int(bs),
        int(local), _ptr(out), _ptr(seg_out), _ptr(seg_lse), _stream(stream)))
    return (out, seg_out, seg_lse) if return_segments else out


def segmented_attention_paged(q, kv_cache, block_table, seg_start, used, bias, bs, local, out=None, *,
                              max_kv_len=None, return_segments=False, stream=None):
    """DASH segmented attention over key ranges of each query's request in a paged cache.

    q [n, Hq, D]; kv_cache [num_pages, Hkv, P, 2D]; block_table int32 [n, W];
    seg_start, used int32 [n, topk+1]; bias fp32 [n, topk].
    """
    lib = load_library()
    n, Hq, D = q.shape
    num_pages, Hkv, P, _ = kv_cache.shape
    topk = bias.shape[1] if bias is not None else 0
    for t, name in ((q, "q"), (kv_cache, "kv_cache"), (block_table, "block_table"), (seg_start, "seg_start"),
                    (used, "used"), (bias, "bias")):
        _cuda(t, name)
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty_like(q)
    seg_out = seg_lse = None
    if return_segments:
        seg_out = torch.empty((n, topk + 1, Hq, D), dtype=torch.float32, device=q.device)
        seg_lse = torch.empty((n, topk + 1, Hq), dtype=torch.float32, device=q.device)
    if max_kv_len is None:
        max_kv_len = block_table.shape[1] * P
    _check(lib.pkd_segmented_attention_paged(
        _ptr(q), dtype_code(q.dtype), _ptr(kv_cache), num_pages, _ptr(block_table), block_table.stride(0),
        _ptr(seg_start), _ptr(used), _ptr(bias), n, Hq, Hkv, D, P, topk, int(bs), int(local), int(max_kv_len),
        _ptr(out), _ptr(seg_out), _ptr(seg_lse), _stream(stream)))
    return (out, seg_out, seg_lse) if return_segments else out


def lse_merge(part_out, part_lse, prior=None, live=None, out=None, lse_out=None, out_dtype=torch.float32,
              stream=None):
    """Merge partials part_out [N, S, H, D] fp32 by their LSE [N, S, H]."""
    lib = load_library()
    N, S, H, D = part_out.shape
    for t, name in ((part_out, "part_out"), (part_lse, "part_lse"), (prior, "prior"), (live, "live")):
        _cuda(t, name)
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty((N, H, D), dtype=out_dtype, device=part_out.device)
    if lse_out is None:
        lse_out = torch.empty((N, H), dtype=torch.float32, device=part_out.device)
    _check(lib.pkd_lse_merge(_ptr(part_out), _ptr(part_lse), _ptr(prior), _ptr(live), N, S, H, D, _ptr(out),
                             dtype_code(out.dtype), _ptr(lse_out), _stream(stream)))
    return out, lse_out


def cache_write(key, value, slot_mapping, kv_cache, k_scale=1.0, v_scale=1.0, stream=None):
    """Write key/value rows [T, Hkv, D] (bf16/fp16) into their slots of kv_cache
    [num_pages, Hkv, P, 2D] (same dtype, or uint8 / float8_e4m3fn for fp8)."""
    lib = load_library()
    for t, n in ((key, "key"), (value, "value"), (slot_mapping, "slot_mapping"), (kv_cache, "kv_cache")):
        _cuda(t, n)
    T, Hkv, D = key.shape
    num_pages, Hkv2, P, twoD = kv_cache.shape
    if Hkv2 != Hkv or twoD != 2 * D:
        raise ValueError("kv_cache shape does not match key")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if key.stride(2) != 1 or key.stride(1) != D or value.stride(2) != 1 or value.stride(1) != D:
        raise ValueError("rows of one token must be contiguous")
    _check(lib.pkd_cache_write(_ptr(key), _ptr(value), dtype_code(key.dtype), key.stride(0), value.stride(0),
                               _ptr(slot_mapping), T, Hkv, D, P, num_pages, _ptr(kv_cache), dtype_code(kv_cache.dtype),
                               float(k_scale), float(v_scale), _stream(stream)))
    return kv_cache
