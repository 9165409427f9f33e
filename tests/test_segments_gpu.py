"""GPU parity of DASH segmented attention (+ combine) and of the LSE merge."""
import zlib

import numpy as np
import pytest
import torch

import oracle
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


def _dev(s):
    return (gu.to_dev(s.q, s.dtype), gu.to_dev(s.k, s.dtype), gu.to_dev(s.v, s.dtype),
            gu.to_dev(s.used, "int32"), gu.to_dev(s.bias, "fp32") if s.topk else None)


def _run(s, segments=False):
    import paged_kv_decode_15_gb300 as pkd
    q, k, v, used, bias = _dev(s)
    if bias is None:
        bias = torch.zeros((s.n, 0), dtype=torch.float32, device="cuda")
    r = pkd.segmented_attention(q, k, v, used, bias, s.bs, s.local, return_segments=segments)
    torch.cuda.synchronize()
    if segments:
        out, so, sl = r
        return out.double().cpu().numpy(), so.double().cpu().numpy(), sl.double().cpu().numpy()
    return r.double().cpu().numpy()


def _oracle(s, segments=False):
    return oracle.segmented_attention(s.q, s.k, s.v, s.dtype, s.used, s.bias, topk=s.topk, bs=s.bs,
                                      local=s.local, num_kv_heads=s.num_kv_heads, return_segments=segments,
                                      threads=gu.THREADS)


SMALL = {
    "g4_topk3_bs16": dict(n=7, num_heads=8, num_kv_heads=2, topk=3, bs=16, local=32),
    "g4_topk5_bs8_odd": dict(n=5, num_heads=8, num_kv_heads=2, topk=5, bs=8, local=24),
    "g8_d64": dict(n=6, num_heads=16, num_kv_heads=2, head_dim=64, topk=4, bs=24, local=40),
    "g16": dict(n=3, num_heads=32, num_kv_heads=2, topk=2, bs=32, local=16),
    "mha_g1_fp16": dict(n=4, num_heads=4, num_kv_heads=4, topk=3, bs=40, local=8, dtype="fp16"),
    "local_only": dict(n=5, num_heads=8, num_kv_heads=2, topk=0, bs=16, local=48),
    "many_empty": dict(n=9, num_heads=8, num_kv_heads=2, topk=6, bs=16, local=16, p_empty=0.7),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_segments_fused(name):
    s = wl.segment_case(name=name, seed=zlib.crc32(name.encode()) % 997, **SMALL[name])
    gu.assert_close(_run(s), _oracle(s), gu.TOL_OUT, name)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_segments_with_per_segment_results(name):
    s = wl.segment_case(name=name, seed=zlib.crc32(name.encode()) % 991, **SMALL[name])
    out, so, sl = _run(s, segments=True)
    ro, rso, rsl = _oracle(s, segments=True)
    gu.assert_close(out, ro, gu.TOL_OUT, name + " out")
    gu.assert_close(so, rso, gu.TOL_OUT, name + " seg_out")
    gu.assert_close(sl, rsl, gu.TOL_LSE, name + " seg_lse")


def test_all_segments_empty_gives_zero():
    used = np.zeros((3, 4), np.int32)
    used[1] = [0, 5, 0, 9]
    s = wl.segment_case(name="dead", n=3, num_heads=8, num_kv_heads=2, topk=3, bs=16, local=16, used=used)
    out = _run(s)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    gu.assert_close(out, _oracle(s), gu.TOL_OUT, "dead")


def test_full_segments_at_capacity():
    n, topk, bs, local = 4, 3, 16, 32
    used = np.tile(np.array([bs] * topk + [local], np.int32), (n, 1))
    s = wl.segment_case(name="cap", n=n, num_heads=8, num_kv_heads=2, topk=topk, bs=bs, local=local, used=used)
    gu.assert_close(_run(s), _oracle(s), gu.TOL_OUT, "cap")


def test_dash_segments_n256_full():
    s = wl.dash_segments_n256()
    gu.assert_close(_run(s), _oracle(s), gu.TOL_OUT, "dash fused")
    out, so, sl = _run(s, segments=True)
    ro, rso, rsl = _oracle(s, segments=True)
    gu.assert_close(out, ro, gu.TOL_OUT, "dash out")
    gu.assert_close(so, rso, gu.TOL_OUT, "dash seg_out")
    gu.assert_close(sl, rsl, gu.TOL_LSE, "dash seg_lse")


@pytest.mark.parametrize("with_prior,with_live", [(False, False), (True, False), (False, True), (True, True)])
def test_lse_merge_matches_oracle(with_prior, with_live):
    import paged_kv_decode_15_gb300 as pkd
    rng = np.random.default_rng(42)
    N, S, H, D = 37, 11, 4, 128
    po = rng.standard_normal((N, S, H, D)).astype(np.float32)
    pl = (rng.standard_normal((N, S, H)) * 3).astype(np.float32)
    pl[0, 3] = -np.inf                       # an empty part
    prior = rng.standard_normal((N, S)).astype(np.float32) if with_prior else None
    live = (rng.random((N, S)) > 0.3).astype(np.int32) if with_live else None
    if with_live:
        live[5] = 0                          # a row with no live part
        po[live == 0] = np.nan               # dead parts are never read
    out, lse = pkd.lse_merge(gu.to_dev(po, "fp32"), gu.to_dev(pl, "fp32"),
                             None if prior is None else gu.to_dev(prior, "fp32"),
                             None if live is None else gu.to_dev(live, "int32"))
    torch.cuda.synchronize()
    ro, rl = oracle.lse_merge(po.astype(np.float64), pl.astype(np.float64),
                              None if prior is None else prior.astype(np.float64), live)
    gu.assert_close(out.double().cpu().numpy(), ro, 1e-5, "merge out")
    gu.assert_close(lse.double().cpu().numpy(), rl, 1e-5, "merge lse")


# ------------------------------------------------ segments from the paged cache
def _run_paged(s, segments=False):
    import paged_kv_decode_15_gb300 as pkd
    bias = gu.to_dev(s.bias, "fp32") if s.topk else torch.zeros((s.n, 0), dtype=torch.float32, device="cuda")
    r = pkd.segmented_attention_paged(gu.to_dev(s.q, s.dtype), gu.to_dev(s.kv_cache, s.dtype),
                                      gu.to_dev(s.block_table, "int32"), gu.to_dev(s.seg_start, "int32"),
                                      gu.to_dev(s.used, "int32"), bias, s.bs, s.local, return_segments=segments)
    torch.cuda.synchronize()
    if segments:
        return tuple(t.double().cpu().numpy() for t in r)
    return r.double().cpu().numpy()


def _oracle_paged(s, segments=False):
    return oracle.segmented_paged(s.q, s.dtype, s.kv_cache, s.block_table, s.seg_start, s.used, s.bias,
                                  num_kv_heads=s.num_kv_heads, page_size=s.page_size, topk=s.topk, bs=s.bs,
                                  local=s.local, return_segments=segments, threads=gu.THREADS)


PAGED = {
    "g4_topk3_bs24": dict(n=7, num_heads=8, num_kv_heads=2, topk=3, bs=24, local=40, seq_range=(60, 400)),
    "g8_d64_p32": dict(n=6, num_heads=16, num_kv_heads=2, head_dim=64, page_size=32, topk=4, bs=16, local=48,
                       seq_range=(100, 300)),
    "fp16_mha": dict(n=5, num_heads=4, num_kv_heads=4, topk=2, bs=64, local=16, dtype="fp16",
                     seq_range=(200, 600)),
    "local_only": dict(n=4, num_heads=8, num_kv_heads=2, topk=0, bs=16, local=72, seq_range=(80, 200)),
    "many_empty": dict(n=9, num_heads=8, num_kv_heads=2, topk=6, bs=32, local=24, p_empty=0.7,
                       seq_range=(100, 500)),
}


@pytest.mark.parametrize("name", sorted(PAGED))
def test_paged_segments_match_oracle(name):
    s = wl.paged_segment_case(name=name, seed=zlib.crc32(name.encode()) % 983, **PAGED[name])
    gu.assert_close(_run_paged(s), _oracle_paged(s), gu.TOL_OUT, name)
    out, so, sl = _run_paged(s, segments=True)
    ro, rso, rsl = _oracle_paged(s, segments=True)
    gu.assert_close(out, ro, gu.TOL_OUT, name + " out")
    gu.assert_close(so, rso, gu.TOL_OUT, name + " seg_out")
    gu.assert_close(sl, rsl, gu.TOL_LSE, name + " seg_lse")


def test_dash_paged_n256_full():
    s = wl.dash_paged_n256()
    gu.assert_close(_run_paged(s), _oracle_paged(s), gu.TOL_OUT, "dash paged")


def test_paged_segments_at_any_start_read_no_row_outside():
    """Segments start at any key (a page's last key, inside one 16-key stage,
    across a page boundary), and every cache row of a request that no segment
    of its query covers holds NaN: a stage the segments cover in part must not
    let those rows into the result (they are not copied, or are masked with
    their V zeroed)."""
    import dataclasses
    s = wl.paged_segment_case(name="any_start", n=12, num_heads=8, num_kv_heads=2, topk=5, bs=40, local=24,
                              seed=77, seq_range=(60, 300))
    P, caps = s.page_size, [s.bs] * s.topk + [s.local]
    rng = np.random.default_rng(5)
    seg_start, used = s.seg_start.copy(), s.used.copy()
    for i in range(s.n):
        L = int(s.seq_lens[i])
        for g in range(s.topk + 1):
            st = int(rng.integers(0, L))
            seg_start[i, g], used[i, g] = st, int(rng.integers(0, min(caps[g], L - st) + 1))
    # query 0: one key at a page's last row, five keys inside one stage, ten
    # keys across a page boundary, a full-capacity block, the local segment at
    # an odd offset
    for g, (st, u) in enumerate([(P - 1, 1), (3 + P, 5), (2 * P - 3, 10), (7, s.bs), (0, 0), (33, s.local)]):
        seg_start[0, g], used[0, g] = st, u
    assert int(s.seq_lens[0]) >= 33 + s.local
    cache = s.kv_cache.copy()
    owner = {}
    for i in range(s.n):
        L = int(s.seq_lens[i])
        covered = np.zeros(L, bool)
        for g in range(s.topk + 1):
            covered[seg_start[i, g]:seg_start[i, g] + used[i, g]] = True
        for t in np.flatnonzero(~covered):
            pg = int(s.block_table[i, t // P])
            assert owner.setdefault(pg, i) == i, "pages are not shared between requests"
            cache[pg, :, t % P, :] = wl.BF16_NAN if s.dtype == "bf16" else wl.FP16_NAN
    s = dataclasses.replace(s, kv_cache=cache, seg_start=seg_start, used=used)
    out = _run_paged(s)
    assert np.isfinite(out).all()
    gu.assert_close(out, _oracle_paged(s), gu.TOL_OUT, "any start")
    out2, so, sl = _run_paged(s, segments=True)
    ro, rso, rsl = _oracle_paged(s, segments=True)
    gu.assert_close(out2, ro, gu.TOL_OUT, "any start out")
    gu.assert_close(so, rso, gu.TOL_OUT, "any start seg_out")
    gu.assert_close(sl, rsl, gu.TOL_LSE, "any start seg_lse")
