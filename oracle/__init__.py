"""fp64 CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

This package states, in plain fp64 C (``oracle.c``), what the hot path
computes: the page gather through a block table, the page-aligned sliding
window, softmax(QK^T)V with its natural-log LSE, the DASH segment combine and
the LSE merge.  It shares no code with the CUDA library and the library never
imports it.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may load it.

Sources: the vLLM API pages ``vllm.v1.attention.backends.flashinfer_ts``
(FlashInferTSImpl.forward, _kv_views, FlashInferTSMetadataBuilder.build and
_restrict_to_window), ``vllm.v1.attention.ops.dash_attention``
(flash_dash_attention) and ``vllm.v1.attention.backends.fa_utils``
(FlashAttentionCuTeDSLCompileSpec: Split-KV and return_softmax_lse).

The wrappers take raw storage (uint16 bits for bf16/fp16, uint8 for fp8-e4m3,
float32) as numpy arrays and return float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")

BF16, FP16, FP8_E4M3, FP32 = 0, 1, 2, 3
DTYPES = {"bf16": BF16, "fp16": FP16, "fp8": FP8_E4M3, "fp8_e4m3": FP8_E4M3, "fp32": FP32}

_lib = None


def _compile(openmp: bool) -> bool:
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    if openmp:
        cmd.insert(1, "-fopenmp")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        os.unlink(tmp)
        return False
    shutil.move(tmp, _LIB_PATH)
    return True


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_liboracle.so`` beside it (OpenMP if available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    if not _compile(openmp=True) and not _compile(openmp=False):
        raise RuntimeError("could not compile the oracle with gcc")
    return _LIB_PATH


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_double
    lib.orc_decode.argtypes = [P, I, L, P]
    lib.orc_window_start_page.argtypes = [L, L, L, L]
    lib.orc_window_start_page.restype = L
    lib.orc_restrict_to_window.argtypes = [P, P, I, I, I, I, I, I, P, P]
    lib.orc_paged_decode.argtypes = [P, I, P, I, L, P, L, P, I, I, I, I, I, I,
                                     D, D, D, D, I, I, P, P, I]
    lib.orc_segmented_attention.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, P, P, P, I]
    lib.orc_lse_merge.argtypes = [P, P, P, P, I, I, I, I, P, P]
    lib.orc_segmented_paged.argtypes = [P, I, P, L, P, L, P, P, P, I, I, I, I, I, I, I, I, P, P, P, I]
    lib.orc_encode_e4m3.argtypes = [ctypes.c_float]
    lib.orc_encode_e4m3.restype = ctypes.c_uint8
    lib.orc_cache_write.argtypes = [P, P, I, P, L, I, I, I, L, P, I, ctypes.c_float, ctypes.c_float]
    for f in ("orc_decode", "orc_restrict_to_window", "orc_paged_decode",
              "orc_segmented_attention", "orc_lse_merge", "orc_cache_write", "orc_segmented_paged"):
        getattr(lib, f).restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _dt(dt) -> int:
    return DTYPES[dt] if isinstance(dt, str) else int(dt)


def _storage(a, dt):
    code = _dt(dt)
    want = {BF16: np.uint16, FP16: np.uint16, FP8_E4M3: np.uint8, FP32: np.float32}[code]
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        a = a.view(want) if a.dtype.itemsize == np.dtype(want).itemsize else a.astype(want)
    return a, code


def decode(bits, dt) -> np.ndarray:
    """Decode raw storage to float64, element by element from the format's definition."""
    a, code = _storage(bits, dt)
    out = np.empty(a.shape, dtype=np.float64)
    if _load().orc_decode(_ptr(a), code, a.size, _ptr(out)) != 0:
        raise ValueError("unknown dtype")
    return out


def window_start_page(L: int, window: int, sq: int, page_size: int) -> int:
    """First visible page of a request under the page-aligned window (0 without one)."""
    return int(_load().orc_window_start_page(int(L), int(window), int(sq), int(page_size)))


def restrict_to_window(seq_lens, block_table, window, sq, page_size, width_out):
    """Table form of the window restriction: (new seq_lens, new block_table)."""
    lens = _c(seq_lens, np.int32)
    bt = _c(block_table, np.int32)
    B, width_in = bt.shape
    out_lens = np.empty(B, np.int32)
    out_bt = np.empty((B, width_out), np.int32)
    rc = _load().orc_restrict_to_window(_ptr(lens), _ptr(bt), B, width_in, int(window), int(sq),
                                        int(page_size), int(width_out), _ptr(out_lens), _ptr(out_bt))
    if rc != 0:
        raise ValueError("restrict_to_window: invalid arguments")
    return out_lens, out_bt


def paged_decode(q, q_dt, kv_cache, kv_dt, block_table, seq_lens, *, sq, num_heads, num_kv_heads,
                 head_dim, page_size, scale, q_scale=1.0, k_scale=1.0, v_scale=1.0, window=0,
                 causal=False, threads=1):
    """Attention of each query block over its request's paged keys.

    q: storage of [B, sq, Hq, D]; kv_cache: storage of [num_pages, Hkv, P, 2*D];
    block_table int32 [B, W]; seq_lens int32 [B].
    Returns (out float64 [B, sq, Hq, D], lse float64 [B, sq, Hq]).
    """
    qa, qc = _storage(q, q_dt)
    ca, cc = _storage(kv_cache, kv_dt)
    bt = _c(block_table, np.int32)
    lens = _c(seq_lens, np.int32)
    B = lens.shape[0]
    D = int(head_dim)
    num_pages = ca.size // (int(num_kv_heads) * int(page_size) * 2 * D)
    out = np.zeros((B, sq, num_heads, D), np.float64)
    lse = np.zeros((B, sq, num_heads), np.float64)
    rc = _load().orc_paged_decode(
        _ptr(qa), qc, _ptr(ca), cc, num_pages, _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0,
        _ptr(lens), B, int(sq), int(num_heads), int(num_kv_heads), D, int(page_size),
        float(scale), float(q_scale), float(k_scale), float(v_scale), int(window), 1 if causal else 0,
        _ptr(out), _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError(f"paged_decode oracle rejected its input (code {rc})")
    return out, lse


def segmented_attention(q, k, v, dt, used, bias, *, topk, bs, local, num_kv_heads,
                        return_segments=False, threads=1):
    """DASH segmented attention and combine.

    q: storage of [n, Hq, D]; k, v: storage of [n*(topk*bs+local), Hkv, D];
    used int32 [n*(topk+1)]; bias [n, topk].  Returns out float64 [n, Hq, D]
    and, if asked, (seg_out [n, topk+1, Hq, D], seg_lse [n, topk+1, Hq]).
    """
    qa, code = _storage(q, dt)
    ka, _ = _storage(k, dt)
    va, _ = _storage(v, dt)
    n, Hq, D = qa.shape
    u = _c(used, np.int32).reshape(-1)
    bi = _c(bias, np.float64).reshape(-1) if topk > 0 else np.zeros(1, np.float64)
    out = np.zeros((n, Hq, D), np.float64)
    seg_out = np.zeros((n, topk + 1, Hq, D), np.float64) if return_segments else None
    seg_lse = np.zeros((n, topk + 1, Hq), np.float64) if return_segments else None
    rc = _load().orc_segmented_attention(
        _ptr(qa), _ptr(ka), _ptr(va), code, _ptr(u), _ptr(bi), n, Hq, int(num_kv_heads), D,
        int(topk), int(bs), int(local), _ptr(out), _ptr(seg_out), _ptr(seg_lse), int(threads))
    if rc != 0:
        raise ValueError(f"segmented_attention oracle rejected its input (code {rc})")
    return (out, seg_out, seg_lse) if return_segments else out


def lse_merge(part_out, part_lse, prior=None, live=None):
    """Merge partials [N, S, H, D] / [N, S, H] by LSE; returns (out [N, H, D], lse [N, H])."""
    po = _c(part_out, np.float64)
    pl = _c(part_lse, np.float64)
    N, S, H, D = po.shape
    pr = _c(prior, np.float64)
    lv = _c(live, np.int32)
    out = np.zeros((N, H, D), np.float64)
    lse = np.zeros((N, H), np.float64)
    rc = _load().orc_lse_merge(_ptr(po), _ptr(pl), _ptr(pr), _ptr(lv), N, S, H, D, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("lse_merge oracle rejected its input")
    return out, lse


def encode_e4m3(x) -> np.ndarray:
    """fp32 values -> e4m3fn codes: round to nearest even, saturating to +-448."""
    a = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    lib = _load()
    return np.array([lib.orc_encode_e4m3(float(v)) for v in a], dtype=np.uint8).reshape(np.shape(x))


def cache_write(key, value, in_dt, slot_mapping, kv_cache, kv_dt, *, num_kv_heads, head_dim, page_size,
                k_scale=1.0, v_scale=1.0):
    """Write key/value rows [T, Hkv, D] into a copy of kv_cache at slot_mapping; returns the new cache."""
    ka, code = _storage(key, in_dt)
    va, _ = _storage(value, in_dt)
    cache = np.array(kv_cache, copy=True)
    ca, cc = _storage(cache, kv_dt)
    sm = _c(slot_mapping, np.int64).reshape(-1)
    num_pages = ca.size // (int(num_kv_heads) * int(page_size) * 2 * int(head_dim))
    rc = _load().orc_cache_write(_ptr(ka), _ptr(va), code, _ptr(sm), sm.size, int(num_kv_heads), int(head_dim),
                                 int(page_size), num_pages, _ptr(ca), cc, float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError(f"cache_write oracle rejected its input (code {rc})")
    return ca.reshape(np.shape(kv_cache))


def segmented_paged(q, dt, kv_cache, block_table, seg_start, used, bias, *, num_kv_heads, page_size, topk, bs,
                    local, return_segments=False, threads=1):
    """DASH segmented attention over key ranges of each query's request in a paged cache.

    q: storage [n, Hq, D]; kv_cache: storage [num_pages, Hkv, P, 2D];
    block_table int32 [n, W]; seg_start, used int32 [n, topk+1]; bias [n, topk].
    """
    qa, code = _storage(q, dt)
    ca, _ = _storage(kv_cache, dt)
    n, Hq, D = qa.shape
    bt = _c(block_table, np.int32)
    ss = _c(seg_start, np.int32).reshape(-1)
    u = _c(used, np.int32).reshape(-1)
    bi = _c(bias, np.float64).reshape(-1) if topk > 0 else np.zeros(1, np.float64)
    num_pages = ca.size // (int(num_kv_heads) * int(page_size) * 2 * D)
    out = np.zeros((n, Hq, D), np.float64)
    seg_out = np.zeros((n, topk + 1, Hq, D), np.float64) if return_segments else None
    seg_lse = np.zeros((n, topk + 1, Hq), np.float64) if return_segments else None
    rc = _load().orc_segmented_paged(
        _ptr(qa), code, _ptr(ca), num_pages, _ptr(bt), bt.shape[1], _ptr(ss), _ptr(u), _ptr(bi), n, Hq,
        int(num_kv_heads), D, int(page_size), int(topk), int(bs), int(local), _ptr(out), _ptr(seg_out),
        _ptr(seg_lse), int(threads))
    if rc != 0:
        raise ValueError(f"segmented_paged oracle rejected its input (code {rc})")
    return (out, seg_out, seg_lse) if return_segments else out
