"""GPU parity of the KV-cache write (bit-exact against the oracle), and a
write-then-decode round trip."""
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


def _case(T, Hkv, D, P, num_pages, in_dt, kv_dt, seed, pad=(3, 11)):
    rng = np.random.default_rng(seed)
    key = wl.normal_storage(rng, (T, Hkv, D), in_dt)
    value = wl.normal_storage(rng, (T, Hkv, D), in_dt)
    # scale up some values so fp8 saturation is exercised
    big = rng.random((T, Hkv, D)) < 0.01
    kf = torch.from_numpy(key.view(np.int16)).view(torch.bfloat16 if in_dt == "bf16" else torch.float16).float()
    kf[torch.from_numpy(big)] *= 100.0
    key = wl.round_to(kf.numpy(), in_dt)
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    for i in pad:
        if i < T:
            slots[i] = -1
    cache = wl.normal_storage(rng, (num_pages, Hkv, P, 2 * D), kv_dt)
    return key, value, slots, cache


@pytest.mark.parametrize("in_dt,kv_dt,D,P", [("bf16", "bf16", 128, 16), ("fp16", "fp16", 64, 32),
                                             ("bf16", "fp8", 128, 16), ("fp16", "fp8", 128, 64),
                                             ("bf16", "fp8", 64, 16)])
def test_cache_write_is_bit_exact(in_dt, kv_dt, D, P):
    import paged_kv_decode_15_gb300 as pkd
    T, Hkv, num_pages = 333, 4, 40
    key, value, slots, cache = _case(T, Hkv, D, P, num_pages, in_dt, kv_dt, seed=D + P)
    ks, vs = (1.0 / 64, 1.0 / 32) if kv_dt == "fp8" else (1.0, 1.0)
    ref = oracle.cache_write(key, value, in_dt, slots, cache, kv_dt, num_kv_heads=Hkv, head_dim=D, page_size=P,
                             k_scale=ks, v_scale=vs)
    dev_cache = gu.to_dev(cache, kv_dt)
    pkd.cache_write(gu.to_dev(key, in_dt), gu.to_dev(value, in_dt), torch.from_numpy(slots).cuda(), dev_cache,
                    k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    got = dev_cache.cpu().view(torch.uint8 if kv_dt == "fp8" else torch.int16).numpy()
    assert np.array_equal(got.view(ref.dtype), ref)


@pytest.mark.parametrize("in_dt,D,P,ks,vs", [("bf16", 128, 16, 0.0137, 0.021), ("fp16", 64, 32, 0.0091, 1.0 / 64)])
def test_cache_write_fp8_scales_that_are_not_powers_of_two(in_dt, D, P, ks, vs):
    """The quotient then takes an IEEE division on both sides (no exact reciprocal)."""
    import paged_kv_decode_15_gb300 as pkd
    T, Hkv, num_pages = 257, 2, 40
    key, value, slots, cache = _case(T, Hkv, D, P, num_pages, in_dt, "fp8", seed=D + P + 7)
    ref = oracle.cache_write(key, value, in_dt, slots, cache, "fp8", num_kv_heads=Hkv, head_dim=D, page_size=P,
                             k_scale=ks, v_scale=vs)
    dev_cache = gu.to_dev(cache, "fp8")
    pkd.cache_write(gu.to_dev(key, in_dt), gu.to_dev(value, in_dt), torch.from_numpy(slots).cuda(), dev_cache,
                    k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert np.array_equal(dev_cache.cpu().numpy().view(np.uint8), ref.view(np.uint8))


def test_cache_write_strided_rows():
    """key/value as slices of a fused [T, 3, Hkv, D] projection output."""
    import paged_kv_decode_15_gb300 as pkd
    T, Hkv, D, P, num_pages = 100, 2, 128, 16, 10
    rng = np.random.default_rng(3)
    fused = wl.normal_storage(rng, (T, 3, Hkv, D), "bf16")
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    cache = wl.normal_storage(rng, (num_pages, Hkv, P, 2 * D), "bf16")
    ref = oracle.cache_write(np.ascontiguousarray(fused[:, 1]), np.ascontiguousarray(fused[:, 2]), "bf16", slots,
                             cache, "bf16", num_kv_heads=Hkv, head_dim=D, page_size=P)
    dev = gu.to_dev(fused, "bf16")
    dev_cache = gu.to_dev(cache, "bf16")
    pkd.cache_write(dev[:, 1], dev[:, 2], torch.from_numpy(slots).cuda(), dev_cache)
    torch.cuda.synchronize()
    assert np.array_equal(dev_cache.cpu().view(torch.int16).numpy().view(np.uint16), ref)


def test_write_then_decode_matches_oracle():
    """Fill a cache through the write kernel (fp8), then decode it."""
    import paged_kv_decode_15_gb300 as pkd
    case = wl.paged_case(name="wd", seq_lens=[300, 1000, 77], dtype="fp8", num_heads=32, num_kv_heads=8, seed=12)
    rng = np.random.default_rng(5)
    P, D, Hkv = case.page_size, case.head_dim, case.num_kv_heads
    dev_cache = gu.to_dev(case.kv_cache, "fp8")
    host_cache = case.kv_cache
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        toks = np.arange(L)
        slots = case.block_table[b, toks // P].astype(np.int64) * P + toks % P
        k = wl.normal_storage(rng, (L, Hkv, D), "bf16")
        v = wl.normal_storage(rng, (L, Hkv, D), "bf16")
        host_cache = oracle.cache_write(k, v, "bf16", slots, host_cache, "fp8", num_kv_heads=Hkv, head_dim=D,
                                        page_size=P, k_scale=case.k_scale, v_scale=case.v_scale)
        pkd.cache_write(gu.to_dev(k, "bf16"), gu.to_dev(v, "bf16"), torch.from_numpy(slots).cuda(), dev_cache,
                        k_scale=case.k_scale, v_scale=case.v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(dev_cache.cpu().numpy(), host_cache)
    case.kv_cache = host_cache
    out, lse = pkd.paged_decode(gu.to_dev(case.q, "fp8"), dev_cache, gu.to_dev(case.block_table, "int32"),
                                gu.to_dev(case.seq_lens, "int32"), case.scale, 0, q_scale=case.q_scale,
                                k_scale=case.k_scale, v_scale=case.v_scale)
    torch.cuda.synchronize()
    ref, rlse = gu.oracle_paged(case)
    gu.assert_close(out.double().cpu().numpy(), ref, gu.TOL_OUT_FP8, "write+decode out")
    gu.assert_close(lse.double().cpu().numpy(), rlse, gu.TOL_LSE, "write+decode lse")
