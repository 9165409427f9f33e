"""pkd_paged_decode_static: paged decode for callers that cannot allocate.

Callers inside a runtime that owns all device memory, serving loops that
must not allocate once their memory budget is fixed, and C callers without
an allocator cannot hand the library a workspace.
The static entry point uses a scratch array compiled into the library
instead.  This checks it through the C ABI against pkd_paged_decode (with a
caller workspace) on two calls in a row, the second with different lengths,
so that what the first call left in the shared scratch cannot leak into the
second.  It lives in its own file, collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _args(case, d, out, lse, dt):
    return [_ptr(d["q"]), dt, _ptr(d["cache"]), dt, case.num_pages, _ptr(d["bt"]),
            d["bt"].stride(0), _ptr(d["lens"]), case.batch, case.sq, case.num_heads, case.num_kv_heads,
            case.head_dim, case.page_size, d["max_kv_len"], case.scale, case.q_scale, case.k_scale, case.v_scale,
            case.window, _ptr(out), 0, _ptr(lse)]


# (cache type, Split-KV chunk, flags name): the bf16 chunked grid with a fixed
# chunk, the persistent per-CTA partition, and the e4m3 grid with its own plan
PLANS = [("bf16", 256, None), ("bf16", 0, "FLAG_BALANCED"), ("fp8", 0, None)]


@pytest.mark.parametrize("dtype,chunk,flag", PLANS)
def test_static_scratch_matches_caller_workspace_twice(dtype, chunk, flag):
    import paged_kv_decode_15_gb300 as pkd
    pkd.build()
    lib = pkd.load_library()
    flags = getattr(pkd, flag) if flag else 0
    dt = {"bf16": pkd.BF16, "fp8": pkd.FP8_E4M3}[dtype]
    case = wl.paged_case(name="static", seq_lens=[4000, 700, 2600, 33, 4096, 1500], seed=77, table_width=256,
                         dtype=dtype)
    d = dict(q=gu.to_dev(case.q, dtype), cache=gu.to_dev(case.kv_cache, dtype),
             bt=gu.to_dev(case.block_table, "int32"), lens=gu.to_dev(case.seq_lens, "int32"), max_kv_len=4096)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    shape = case.q.shape
    ws = torch.empty(pkd.workspace_size(case.batch, 1, 32, 8, 128, 16, 4096, dt, chunk_tokens=chunk, flags=flags),
                     dtype=torch.uint8, device="cuda")
    pkd.workspace_init(ws)
    free = []
    for lens in ([4000, 700, 2600, 33, 4096, 1500], [64, 4096, 17, 3000, 0, 2222]):
        d["lens"].copy_(torch.tensor(lens, dtype=torch.int32))
        ref = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty(shape[:3], dtype=torch.float32, device="cuda")
        got = torch.empty_like(ref)
        got_lse = torch.empty_like(ref_lse)
        st = lib.pkd_paged_decode(*_args(case, d, ref, ref_lse, dt), _ptr(ws), ws.numel(), chunk, flags, stream)
        assert st == pkd.OK, lib.pkd_last_error()
        torch.cuda.synchronize()
        before = torch.cuda.mem_get_info()[0]
        st = lib.pkd_paged_decode_static(*_args(case, d, got, got_lse, dt), chunk, flags, stream)
        assert st == pkd.OK, lib.pkd_last_error()
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0] - before)
        tol = gu.TOL_OUT_FP8 if dtype == "fp8" else gu.TOL_OUT
        gu.assert_close(got.double().cpu().numpy(), ref.double().cpu().numpy(), tol, "static out")
        gu.assert_close(got_lse.double().cpu().numpy(), ref_lse.double().cpu().numpy(), gu.TOL_LSE, "static lse")
    # the first static call on a device may load the library's module (and
    # with it the scratch array); the second call allocates nothing at all
    assert free[1] == 0, f"device memory changed by {free[1]} bytes across a static call"


def test_static_scratch_rejects_plans_above_its_size():
    import paged_kv_decode_15_gb300 as pkd
    lib = pkd.load_library()
    # 4096 requests x 8 kv heads x 128 chunks of 16 keys needs far more than 32 MiB
    st = lib.pkd_paged_decode_static(None, pkd.BF16, None, pkd.BF16, 1, None, 128, None, 4096, 1, 32, 8, 128, 16,
                                     2048, 0.1, 1.0, 1.0, 1.0, 0, None, pkd.BF16, None, 16, 0, None)
    assert st == pkd.EUNSUPPORTED
    assert b"static" in lib.pkd_last_error()


def test_static_check_reports_and_clears_the_status_word():
    """The static call's status word is read back by its companion check: a
    length above max_kv_len is clamped and reported, then the word is clear."""
    import paged_kv_decode_15_gb300 as pkd
    lib = pkd.load_library()
    case = wl.paged_case(name="static_bad", seq_lens=[100, 50], seed=9, table_width=8)
    d = dict(q=gu.to_dev(case.q, "bf16"), cache=gu.to_dev(case.kv_cache, "bf16"),
             bt=gu.to_dev(case.block_table, "int32"), lens=gu.to_dev(case.seq_lens, "int32"), max_kv_len=128)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty(case.q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
    assert lib.pkd_paged_decode_static(*_args(case, d, out, lse, pkd.BF16), 0, 0, stream) == pkd.OK
    assert lib.pkd_paged_decode_static_check(stream) == pkd.OK
    d["lens"][0] = 500  # above max_kv_len: clamped and reported
    assert lib.pkd_paged_decode_static(*_args(case, d, out, lse, pkd.BF16), 0, 0, stream) == pkd.OK
    assert lib.pkd_paged_decode_static_check(stream) == pkd.EDEVICE_BOUNDS
    assert lib.pkd_paged_decode_static_check(stream) == pkd.OK  # the word was cleared
    assert torch.isfinite(out.float()).all()
