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


def _args(case, d, out, lse):
    import paged_kv_decode_15_gb300 as pkd
    return [_ptr(d["q"]), pkd.BF16, _ptr(d["cache"]), pkd.BF16, case.num_pages, _ptr(d["bt"]),
            d["bt"].stride(0), _ptr(d["lens"]), case.batch, case.sq, case.num_heads, case.num_kv_heads,
            case.head_dim, case.page_size, d["max_kv_len"], case.scale, 1.0, 1.0, 1.0, case.window,
            _ptr(out), pkd.BF16, _ptr(lse)]


def test_static_scratch_matches_caller_workspace_twice():
    import paged_kv_decode_15_gb300 as pkd
    pkd.build()
    lib = pkd.load_library()
    case = wl.paged_case(name="static", seq_lens=[4000, 700, 2600, 33, 4096, 1500], seed=77, table_width=256)
    d = dict(q=gu.to_dev(case.q, "bf16"), cache=gu.to_dev(case.kv_cache, "bf16"),
             bt=gu.to_dev(case.block_table, "int32"), lens=gu.to_dev(case.seq_lens, "int32"), max_kv_len=4096)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    shape = case.q.shape
    ws = torch.empty(pkd.workspace_size(case.batch, 1, 32, 8, 128, 16, 4096, pkd.BF16), dtype=torch.uint8,
                     device="cuda")
    pkd.workspace_init(ws)
    for lens in ([4000, 700, 2600, 33, 4096, 1500], [64, 4096, 17, 3000, 0, 2222]):
        d["lens"].copy_(torch.tensor(lens, dtype=torch.int32))
        ref = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.empty(shape[:3], dtype=torch.float32, device="cuda")
        got = torch.empty_like(ref)
        got_lse = torch.empty_like(ref_lse)
        st = lib.pkd_paged_decode(*_args(case, d, ref, ref_lse), _ptr(ws), ws.numel(), 256, 0, stream)
        assert st == pkd.OK, lib.pkd_last_error()
        st = lib.pkd_paged_decode_static(*_args(case, d, got, got_lse), 256, 0, stream)
        assert st == pkd.OK, lib.pkd_last_error()
        torch.cuda.synchronize()
        gu.assert_close(got.double().cpu().numpy(), ref.double().cpu().numpy(), gu.TOL_OUT, "static out")
        gu.assert_close(got_lse.double().cpu().numpy(), ref_lse.double().cpu().numpy(), gu.TOL_LSE, "static lse")


def test_static_scratch_rejects_plans_above_its_size():
    import paged_kv_decode_15_gb300 as pkd
    lib = pkd.load_library()
    # 4096 requests x 8 kv heads x 128 chunks of 16 keys needs far more than 32 MiB
    st = lib.pkd_paged_decode_static(None, pkd.BF16, None, pkd.BF16, 1, None, 128, None, 4096, 1, 32, 8, 128, 16,
                                     2048, 0.1, 1.0, 1.0, 1.0, 0, None, pkd.BF16, None, 16, 0, None)
    assert st == pkd.EUNSUPPORTED
    assert b"static" in lib.pkd_last_error()
