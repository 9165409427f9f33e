"""Paged decode with PKD_FLAG_HOST_IO: q, the block table, the lengths, out
and lse in pinned host memory, read and written by the kernels in place.

Every kernel that takes the flag must give the bits of the same call on
device memory; pointers that are not pinned host memory are refused before
any launch.
"""
import ctypes
import zlib

import numpy as np
import pytest
import torch

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    import paged_kv_decode_15_gb300 as pkd
    pkd.build()
    pkd.load_library()


LENS = [1, 15, 16, 17, 200, 1000, 777, 64, 0, 333]
B50_LENS = [1000 + (i * 397) % 1049 for i in range(50)]

CASES = {
    # name: paged_case kwargs, call kwargs (the same for both calls)
    "bf16_g4": (dict(seq_lens=LENS), dict()),
    "bf16_g4_flat": (dict(seq_lens=LENS), dict(flat=True)),
    "bf16_g4_balanced": (dict(seq_lens=LENS), dict(balanced=True)),
    "bf16_g4_fma": (dict(seq_lens=LENS), dict(force_fma=True)),
    "bf16_causal_sq4_window50": (dict(seq_lens=LENS, sq=4, causal=True, window=50), dict(chunk_tokens=32)),
    "fp16_d64_p32_scales": (dict(seq_lens=LENS, dtype="fp16", head_dim=64, page_size=32, scales=(1.3, 0.7, 0.9)),
                            dict(chunk_tokens=64)),
    "fp8_g8": (dict(seq_lens=LENS, dtype="fp8", num_heads=64, num_kv_heads=8), dict(chunk_tokens=64)),
    "fp8_sq8_m32_flat": (dict(seq_lens=LENS, dtype="fp8", sq=8), dict()),
    # a tcgen05 shape: with host memory it runs on the chunked grid, so the
    # device call forces the grid to compare the same kernel
    "bf16_sq8_b50_m32": (dict(seq_lens=B50_LENS, sq=8), dict(grid=True)),
}


def _pinned(t):
    return torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu())


@pytest.mark.parametrize("name", sorted(CASES))
def test_host_io_gives_the_bits_of_the_device_call(name):
    import paged_kv_decode_15_gb300 as pkd
    ckw, kw = CASES[name]
    case = wl.paged_case(name=name, seed=zlib.crc32(name.encode()) % 1000, **ckw)
    q = gu.to_dev(case.q, case.dtype)
    cache = gu.to_dev(case.kv_cache, case.dtype)
    bt = gu.to_dev(case.block_table, "int32")
    lens = gu.to_dev(case.seq_lens, "int32")
    common = dict(q_scale=case.q_scale, k_scale=case.k_scale, v_scale=case.v_scale, causal=case.causal,
                  max_kv_len=int(case.block_table.shape[1] * case.page_size))
    out_d, lse_d = pkd.paged_decode(q, cache, bt, lens, case.scale, case.window, **common, **kw)
    host_kw = {k: v for k, v in kw.items() if k != "grid"}
    out_h, lse_h = pkd.paged_decode(_pinned(q), cache, _pinned(bt), _pinned(lens), case.scale, case.window,
                                    host_io=True, **common, **host_kw)
    torch.cuda.synchronize()
    assert not out_h.is_cuda and not lse_h.is_cuda
    assert torch.equal(out_h, out_d.cpu()), f"{name}: out differs from the device call"
    assert torch.equal(lse_h, lse_d.cpu()), f"{name}: lse differs from the device call"
    # and the device call itself against the oracle
    ref, rlse = gu.oracle_paged(case)
    tol = gu.TOL_OUT_FP8 if case.dtype == "fp8" else gu.TOL_OUT
    gu.assert_close(out_h.double().numpy(), ref, tol, f"{name} out")
    gu.assert_close(lse_h.double().numpy(), rlse, gu.TOL_LSE, f"{name} lse")


def test_host_io_refuses_device_and_pageable_memory():
    import paged_kv_decode_15_gb300 as pkd
    lib = pkd.load_library()
    case = wl.paged_case(name="refuse", seq_lens=[40, 70], seed=3)
    q = gu.to_dev(case.q, case.dtype)
    cache = gu.to_dev(case.kv_cache, case.dtype)
    bt = gu.to_dev(case.block_table, "int32")
    lens = gu.to_dev(case.seq_lens, "int32")
    with pytest.raises(ValueError):
        pkd.paged_decode(q, cache, _pinned(bt), _pinned(lens), case.scale, host_io=True)
    B, sq, Hq, D = q.shape
    num_pages, Hkv, P, _ = cache.shape
    max_kv_len = int(case.block_table.shape[1] * P)
    ws = torch.zeros(pkd.workspace_size(B, sq, Hq, Hkv, D, P, max_kv_len, pkd.BF16, flags=pkd.FLAG_HOST_IO),
                     dtype=torch.uint8, device="cuda")
    hq, hbt, hlens = _pinned(q), _pinned(bt), _pinned(lens)
    hout = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    pageable_q = np.empty(q.numel() * 2 + 64, np.uint8)
    pq = ctypes.c_void_p((pageable_q.ctypes.data + 63) // 64 * 64)
    sentinel = torch.full(q.shape, 7.0, dtype=q.dtype, pin_memory=True)
    hout.copy_(sentinel)

    def call(qp, outp):
        return lib.pkd_paged_decode(qp, pkd.BF16, pkd._ptr(cache), pkd.BF16, num_pages, pkd._ptr(hbt),
                                    hbt.stride(0), pkd._ptr(hlens), B, sq, Hq, Hkv, D, P, max_kv_len,
                                    float(case.scale), 1.0, 1.0, 1.0, 0, outp, pkd.BF16, None, pkd._ptr(ws),
                                    ws.numel(), 0, pkd.FLAG_HOST_IO, pkd._stream())

    assert call(pkd._ptr(q), pkd._ptr(hout)) == pkd.EINVAL            # q in device memory
    assert b"q is not pinned host memory" in lib.pkd_last_error()
    assert call(pq, pkd._ptr(hout)) == pkd.EINVAL                      # q in pageable host memory
    assert call(pkd._ptr(hq), pkd._ptr(torch.empty_like(q))) == pkd.EINVAL  # out in device memory
    assert b"out is not pinned host memory" in lib.pkd_last_error()
    torch.cuda.synchronize()
    assert torch.equal(hout, sentinel), "a refused call launched a kernel"
    assert call(pkd._ptr(hq), pkd._ptr(hout)) == pkd.OK
    torch.cuda.synchronize()
    ref, _ = gu.oracle_paged(case)
    gu.assert_close(hout.double().numpy(), ref, gu.TOL_OUT, "host_io out")
