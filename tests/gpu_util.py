"""Helpers for the GPU parity tests: move workload storage to the device, run
the library, and compare with the oracle element by element."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import workloads as wl
import paged_kv_decode_15_gb300 as pkd

# tolerances: max |gpu - oracle| on outputs (bf16/fp16 storage, fp8 caches)
# and on the natural-log LSE
TOL_OUT = 1e-2
TOL_OUT_FP8 = 4e-2
TOL_LSE = 1e-3

THREADS = os.cpu_count() or 1


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    return wl.to_torch(a, dtype, "cuda")


def run_paged(case, **kw):
    """Run the library on a PagedCase; returns (out float64 numpy, lse float64 numpy)."""
    q = to_dev(case.q, case.dtype)
    cache = to_dev(case.kv_cache, case.dtype)
    bt = to_dev(case.block_table, "int32")
    lens = to_dev(case.seq_lens, "int32")
    kw.setdefault("max_kv_len", int(case.block_table.shape[1] * case.page_size))
    out, lse = pkd.paged_decode(q, cache, bt, lens, case.scale, case.window, q_scale=case.q_scale,
                                k_scale=case.k_scale, v_scale=case.v_scale, causal=case.causal, **kw)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_paged(case, batch_index=None):
    """Oracle result, optionally on a subset of requests (their own rows only)."""
    if batch_index is None:
        return oracle.paged_decode(case.q, case.dtype, case.kv_cache, case.dtype, case.block_table,
                                   case.seq_lens, threads=THREADS, **case.oracle_kwargs())
    idx = np.asarray(batch_index)
    return oracle.paged_decode(case.q[idx], case.dtype, case.kv_cache, case.dtype, case.block_table[idx],
                               case.seq_lens[idx], threads=THREADS, **case.oracle_kwargs())


def assert_close(got, ref, tol, what):
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    inf_r = np.isinf(r)
    assert np.array_equal(np.isinf(g), inf_r), f"{what}: infinities differ"
    assert np.array_equal(g[inf_r], r[inf_r]), f"{what}: infinities differ in sign"
    assert not np.isnan(g).any(), f"{what}: NaN in the GPU result"
    fin = ~inf_r
    err = np.abs(g[fin] - r[fin]).max() if fin.any() else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3g} > {tol}"
    return err
