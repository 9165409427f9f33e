"""GPU parity of paged decode against the fp64 oracle, through the C ABI.

Small cases span several 16-key stages, several Split-KV chunks and ragged
tails; full-size workloads are compared on every request.  The
probes check the page gather bit-exactly.
"""
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


def _check(case, tol=None, batch_index=None, **kw):
    out, lse = gu.run_paged(case, **kw)
    ref, rlse = gu.oracle_paged(case, batch_index)
    if batch_index is not None:
        out, lse = out[batch_index], lse[batch_index]
    tol = tol or (gu.TOL_OUT_FP8 if case.dtype == "fp8" else gu.TOL_OUT)
    e1 = gu.assert_close(out, ref, tol, f"{case.name} out")
    e2 = gu.assert_close(lse, rlse, gu.TOL_LSE, f"{case.name} lse")
    return e1, e2


LENS = [1, 15, 16, 17, 200, 1000, 777, 64, 0, 333]
B50_LENS = [1000 + (i * 397) % 1049 for i in range(50)]
SHORT40 = [(i * 211) % 900 for i in range(40)]  # 0-899 keys, one empty request

SMALL = {
    # name: paged_case kwargs, call kwargs
    "bf16_g4": (dict(seq_lens=LENS), dict()),
    "bf16_g4_chunk16": (dict(seq_lens=LENS), dict(chunk_tokens=16)),
    "bf16_g4_chunk32": (dict(seq_lens=LENS), dict(chunk_tokens=32)),
    "fp16_g4": (dict(seq_lens=LENS, dtype="fp16"), dict(chunk_tokens=64)),
    "fp16_g4_chunk128": (dict(seq_lens=LENS, dtype="fp16"), dict(chunk_tokens=128)),
    "bf16_d64_p32": (dict(seq_lens=LENS, head_dim=64, page_size=32), dict(chunk_tokens=64)),
    "bf16_d64_p32_auto": (dict(seq_lens=LENS, head_dim=64, page_size=32), dict()),
    "bf16_p48_not_power_of_two": (dict(seq_lens=LENS, page_size=48, window=300), dict()),
    "bf16_sq8_p48_not_power_of_two": (dict(seq_lens=LENS, sq=8, page_size=48), dict()),
    "bf16_sq8_p48_chunk96": (dict(seq_lens=LENS, sq=8, page_size=48), dict(chunk_tokens=96)),
    # warp pairs over 50 requests of 1000-2048 keys
    "bf16_sq8_b50": (dict(seq_lens=B50_LENS, sq=8), dict()),
    "bf16_sq8_b50_window300_causal": (dict(seq_lens=B50_LENS, sq=8, window=300, causal=True), dict()),
    # tcgen05 kernel with more chunks than SMs: equal tile shares that cut
    # chunks (also one-chunk units), a chunk that is not a whole number of
    # tiles, short and empty requests
    "bf16_sq8_b50_window700_share": (dict(seq_lens=B50_LENS, sq=8, window=700), dict()),
    "bf16_sq8_b50_chunk480_share": (dict(seq_lens=B50_LENS, sq=8), dict(chunk_tokens=480)),
    "fp16_sq8_b40_short_chunk256_share": (dict(seq_lens=SHORT40, sq=8, dtype="fp16", scales=(1.3, 0.7, 0.9)),
                                          dict(chunk_tokens=256)),
    # causal blocks of 32 rows on the tcgen05 kernel: per-row masks across
    # shares and runs, with and without a window
    "fp16_sq8_b50_causal_share": (dict(seq_lens=B50_LENS, sq=8, dtype="fp16", causal=True), dict()),
    "bf16_sq8_b50_causal_window700_chunk480": (dict(seq_lens=B50_LENS, sq=8, causal=True, window=700),
                                               dict(chunk_tokens=480)),
    "bf16_mha_g1": (dict(seq_lens=LENS, num_heads=8, num_kv_heads=8), dict(chunk_tokens=48)),
    "bf16_g2_sq1": (dict(seq_lens=LENS, num_heads=4, num_kv_heads=2), dict()),
    "bf16_g8": (dict(seq_lens=LENS, num_heads=64, num_kv_heads=8), dict(chunk_tokens=96)),
    "bf16_g8_auto": (dict(seq_lens=LENS, num_heads=64, num_kv_heads=8), dict()),
    "bf16_sq3_g4_m12": (dict(seq_lens=LENS, sq=3), dict(chunk_tokens=64)),
    "bf16_sq8_g4_m32": (dict(seq_lens=LENS, sq=8), dict(chunk_tokens=128)),
    "bf16_sq8_g4_m32_auto": (dict(seq_lens=LENS, sq=8), dict()),
    "bf16_sq5_g4_m20": (dict(seq_lens=LENS, sq=5, head_dim=64), dict(chunk_tokens=64)),
    "bf16_sq8_window100": (dict(seq_lens=LENS, sq=8, window=100), dict(chunk_tokens=32)),
    "bf16_sq1_window40": (dict(seq_lens=LENS, window=40), dict()),
    "bf16_p64_window300": (dict(seq_lens=LENS, page_size=64, window=300), dict(chunk_tokens=128)),
    "bf16_causal_sq4_m16": (dict(seq_lens=LENS, sq=4, causal=True), dict(chunk_tokens=64)),
    "bf16_causal_sq4_window50": (dict(seq_lens=LENS, sq=4, causal=True, window=50), dict(chunk_tokens=32)),
    "bf16_causal_sq2_g2": (dict(seq_lens=LENS, sq=2, num_heads=4, num_kv_heads=2, causal=True, window=30), dict()),
    "bf16_causal_sq8_m32_window": (dict(seq_lens=LENS, sq=8, causal=True, window=200), dict(chunk_tokens=64)),
    "bf16_causal_sq8_m32_auto": (dict(seq_lens=LENS, sq=8, causal=True), dict()),
    "fp16_sq6_g4_m24_p32": (dict(seq_lens=LENS, sq=6, dtype="fp16", page_size=32), dict(chunk_tokens=96)),
    # q_scale, k_scale and v_scale all different and not powers of two: a
    # kernel that swapped two of them, or dropped or squared one, fails here
    # (bf16 keeps v_scale < 1 so that |out| stays where a bf16 ulp is < 1e-2)
    "bf16_scales_qkv": (dict(seq_lens=LENS, scales=(0.731, 1.377, 0.589)), dict()),
    "bf16_sq4_causal_scales_qkv": (dict(seq_lens=LENS, sq=4, causal=True, scales=(1.9, 0.53, 0.77)),
                                   dict(chunk_tokens=64)),
    "fp16_sq8_m32_scales_qkv": (dict(seq_lens=LENS, sq=8, dtype="fp16", scales=(1.7, 0.45, 2.3)), dict()),
    "bf16_g8_window_scales_qkv": (dict(seq_lens=LENS, num_heads=64, window=100, scales=(0.61, 0.83, 0.97)),
                                  dict(chunk_tokens=32)),
    # fp8 caches: q, K and V with their own per-tensor scales amax/448 (the
    # default of the generator), and the power-of-two shared scale
    "fp8_g8": (dict(seq_lens=LENS, dtype="fp8", num_heads=64, num_kv_heads=8), dict(chunk_tokens=64)),
    "fp8_g8_pow2": (dict(seq_lens=LENS, dtype="fp8", num_heads=64, num_kv_heads=8, fp8_scales="pow2"),
                    dict(chunk_tokens=64)),
    "fp8_sq4_pow2": (dict(seq_lens=LENS, dtype="fp8", sq=4, fp8_scales="pow2"), dict()),
    "fp8_g4_p64": (dict(seq_lens=LENS, dtype="fp8", page_size=64), dict()),
    "fp8_g2_window": (dict(seq_lens=LENS, dtype="fp8", num_heads=16, num_kv_heads=8, window=100), dict()),
    "fp8_sq4_g4_m16": (dict(seq_lens=LENS, dtype="fp8", sq=4), dict()),
    "fp8_sq8_g4_m32_causal": (dict(seq_lens=LENS, dtype="fp8", sq=8, causal=True, window=200), dict()),
}

# kernel variants: persistent flat partition / one CTA per chunk; tensor / CUDA cores
VARIANTS = {"auto": dict(), "flat": dict(flat=True), "grid": dict(grid=True), "balanced": dict(balanced=True),
            "flat_fma": dict(force_fma=True), "grid_fma": dict(grid=True, force_fma=True)}


def _m(ckw):
    return ckw.get("sq", 1) * ckw.get("num_heads", 32) // ckw.get("num_kv_heads", 8)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_cases_match_oracle(name, variant):
    ckw, kw = SMALL[name]
    vkw = VARIANTS[variant]
    if vkw.get("force_fma") and _m(ckw) > 8:
        pytest.skip("the CUDA-core kernel takes M <= 8")
    if vkw.get("grid") and ckw.get("dtype") == "fp8" and _m(ckw) > 16:
        pytest.skip("fp8 with more than 16 rows runs on the flat partition only")
    if vkw.get("balanced") and ckw.get("dtype") == "fp8":
        pytest.skip("the per-CTA partition runs 16-bit caches only")
    case = wl.paged_case(name=name, seed=zlib.crc32(name.encode()) % 1000, **ckw)
    _check(case, **kw, **vkw)


def test_tiny_workload_all_variants():
    case = wl.tiny_decode()
    for vkw in VARIANTS.values():
        _check(case, **vkw)
    _check(case, chunk_tokens=16, grid=True)


def test_results_are_deterministic():
    case = wl.paged_case(name="det", seq_lens=[900, 4000, 33], seed=3)
    a = gu.run_paged(case, chunk_tokens=256)
    b = gu.run_paged(case, chunk_tokens=256)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_argmax_probe_gathers_bit_exactly(variant):
    """q equal to one visible key and a huge scale: every other weight underflows
    to 0 and the output must be that key's V row, bit for bit."""
    case = wl.paged_case(name="probe", seq_lens=[37, 300, 129], num_heads=8, num_kv_heads=2, window=64,
                         seed=21, table_width=24)
    rng = np.random.default_rng(0)
    P, D = case.page_size, case.head_dim
    targets = {}
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        start = max(0, (L - 64) // P) * P
        cands = [start, L - 1] + list(rng.integers(start, L, size=2))
        for h in range(case.num_heads):
            t = int(cands[h % len(cands)])
            page = case.block_table[b, t // P]
            case.q[b, 0, h] = case.kv_cache[page, h // 4, t % P, :D]
            targets[(b, h)] = (page, h // 4, t % P)
    case.scale = 100.0
    out, _ = gu.run_paged(case, chunk_tokens=32, **VARIANTS[variant])
    got_bits = torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for (b, h), (page, hk, slot) in targets.items():
        assert np.array_equal(got_bits[b, 0, h], case.kv_cache[page, hk, slot, D:]), (b, h)


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_constant_v_is_exact_and_nan_pages_are_never_read(variant):
    case = wl.paged_case(name="constv", seq_lens=[37, 300, 1, 129, 700], seed=5)
    one = 0x3F80
    P, D = case.page_size, case.head_dim
    for b in range(case.batch):
        for j in range(int(case.seq_lens[b])):
            case.kv_cache[case.block_table[b, j // P], :, j % P, D:] = one
    out, lse = gu.run_paged(case, chunk_tokens=64, **VARIANTS[variant])
    assert np.all(out == 1.0)
    assert np.all(np.isfinite(lse))


def test_out_dtypes_and_no_lse():
    import paged_kv_decode_15_gb300 as pkd
    case = wl.paged_case(name="dt", seq_lens=[100, 513], seed=8)
    q = gu.to_dev(case.q, "bf16")
    cache = gu.to_dev(case.kv_cache, "bf16")
    bt = gu.to_dev(case.block_table, "int32")
    lens = gu.to_dev(case.seq_lens, "int32")
    ref, _ = gu.oracle_paged(case)
    for odt in (torch.float32, torch.float16, torch.bfloat16):
        out = torch.empty(q.shape, dtype=odt, device="cuda")
        pkd.paged_decode(q, cache, bt, lens, case.scale, 0, out=out)
        torch.cuda.synchronize()
        gu.assert_close(out.double().cpu().numpy(), ref, gu.TOL_OUT, str(odt))


def test_bad_lengths_and_pages_raise_the_status_word():
    import paged_kv_decode_15_gb300 as pkd
    case = wl.paged_case(name="bad", seq_lens=[100, 50], seed=9, table_width=8)
    q = gu.to_dev(case.q, "bf16")
    cache = gu.to_dev(case.kv_cache, "bf16")
    bt = gu.to_dev(case.block_table, "int32")
    lens = gu.to_dev(case.seq_lens, "int32")
    ws = torch.zeros(pkd.workspace_size(2, 1, 32, 8, 128, 16, 128, pkd.BF16), dtype=torch.uint8, device="cuda")
    out, lse = pkd.paged_decode(q, cache, bt, lens, case.scale, 0, max_kv_len=128, workspace=ws)
    assert pkd.workspace_check(ws) == pkd.OK
    lens[0] = 500  # above max_kv_len: clamped and reported
    pkd.paged_decode(q, cache, bt, lens, case.scale, 0, max_kv_len=128, workspace=ws)
    assert pkd.workspace_check(ws) == pkd.EDEVICE_BOUNDS
    assert pkd.workspace_check(ws) == pkd.OK  # the word was cleared
    lens[0] = 100
    bt[1, 1] = case.num_pages + 7  # a page outside the pool: its keys are skipped and reported
    out, lse = pkd.paged_decode(q, cache, bt, lens, case.scale, 0, max_kv_len=128, workspace=ws)
    assert pkd.workspace_check(ws) == pkd.EDEVICE_BOUNDS
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("variant", ["auto", "pair", "flat", "balanced", "grid_fma"])
def test_wait_timeout_is_reported_and_the_workspace_recovers(variant):
    """With the diagnostic flag every wait on a stage's copy tests its barrier
    once, so copies still in flight count as lost: the call must report
    PKD_ETIMEOUT through the status word, leave a finite output, and (after
    the workspace is zeroed again) a normal call must match the oracle.  No
    copy is withheld: the kernels let every issued copy land before leaving."""
    import paged_kv_decode_15_gb300 as pkd
    sq = 8 if variant == "pair" else 1
    vkw = {} if variant == "pair" else VARIANTS[variant]
    lens = wl.uniform_lens(41, 48, 512, 4096)
    case = wl.paged_case(name="timeout", seq_lens=lens, sq=sq, seed=42)
    q = gu.to_dev(case.q, "bf16")
    cache = gu.to_dev(case.kv_cache, "bf16")
    bt = gu.to_dev(case.block_table, "int32")
    dl = gu.to_dev(case.seq_lens, "int32")
    flags = (pkd.FLAG_FLAT if vkw.get("flat") else 0) | (pkd.FLAG_BALANCED if vkw.get("balanced") else 0) | \
        (pkd.FLAG_GRID if vkw.get("grid") else 0) | (pkd.FLAG_FMA if vkw.get("force_fma") else 0)
    W = case.block_table.shape[1] * case.page_size
    ws = torch.empty(pkd.workspace_size(case.batch, sq, 32, 8, 128, 16, W, pkd.BF16, flags=flags),
                     dtype=torch.uint8, device="cuda")
    pkd.workspace_init(ws)
    out = torch.zeros(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(q.shape[:3], dtype=torch.float32, device="cuda")
    status = pkd.OK
    for _ in range(3):  # a copy that lands before its first test is not a timeout: try again
        pkd.paged_decode(q, cache, bt, dl, case.scale, 0, out=out, lse=lse, workspace=ws, test_timeout=True, **vkw)
        status = pkd.workspace_check(ws)
        if status == pkd.ETIMEOUT:
            break
    assert status == pkd.ETIMEOUT
    assert torch.isfinite(out.float()).all()
    pkd.workspace_init(ws)
    out, lse = pkd.paged_decode(q, cache, bt, dl, case.scale, 0, workspace=ws, **vkw)
    assert pkd.workspace_check(ws) == pkd.OK
    ref, rlse = gu.oracle_paged(case)
    gu.assert_close(out.double().cpu().numpy(), ref, gu.TOL_OUT, "after timeout out")
    gu.assert_close(lse.double().cpu().numpy(), rlse, gu.TOL_LSE, "after timeout lse")


def test_cuda_graph_replay_follows_new_lengths():
    """The call records no host state: a captured graph replays correctly when
    the lengths and the table change in place."""
    import paged_kv_decode_15_gb300 as pkd
    # pages are allocated for the longest lengths either pass uses
    case = wl.paged_case(name="graph", seq_lens=[2000, 1200, 1024, 2048], seed=10, table_width=160)
    case.seq_lens = np.array([500, 1200, 64, 2048], np.int32)
    q = gu.to_dev(case.q, "bf16")
    cache = gu.to_dev(case.kv_cache, "bf16")
    bt = gu.to_dev(case.block_table, "int32")
    lens = gu.to_dev(case.seq_lens, "int32")
    out = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    ws = torch.empty(pkd.workspace_size(4, 1, 32, 8, 128, 16, 2560, pkd.BF16), dtype=torch.uint8, device="cuda")
    pkd.workspace_init(ws)
    kw = dict(out=out, lse=lse, workspace=ws, max_kv_len=2560)
    pkd.paged_decode(q, cache, bt, lens, case.scale, 0, **kw)  # warm-up outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pkd.paged_decode(q, cache, bt, lens, case.scale, 0, **kw)
    new_lens = np.array([2000, 17, 1024, 2048], np.int32)
    lens.copy_(torch.from_numpy(new_lens))
    g.replay()
    torch.cuda.synchronize()
    case.seq_lens = new_lens
    ref, rlse = gu.oracle_paged(case)
    gu.assert_close(out.double().cpu().numpy(), ref, gu.TOL_OUT, "graph out")
    gu.assert_close(lse.double().cpu().numpy(), rlse, gu.TOL_LSE, "graph lse")


# ------------------------------------------------------ full-size workloads
def test_gqa_decode_b64_full():
    case = wl.gqa_decode_b64()
    _check(case)


@pytest.mark.parametrize("variant", ["flat", "balanced", "flat_fma"])
def test_gqa_decode_b64_other_variants(variant):
    case = wl.gqa_decode_b64()
    _check(case, **VARIANTS[variant])


_FULL = {}


def _full_case(name, make):
    """A full-size workload and its oracle result, made once per module."""
    if name not in _FULL:
        case = make()
        _FULL[name] = (case, gu.oracle_paged(case))
    return _FULL[name]


def _check_full(case, ref, **kw):
    out, lse = gu.run_paged(case, **kw)
    tol = gu.TOL_OUT_FP8 if case.dtype == "fp8" else gu.TOL_OUT
    gu.assert_close(out, ref[0], tol, f"{case.name} out")
    gu.assert_close(lse, ref[1], gu.TOL_LSE, f"{case.name} lse")


@pytest.mark.parametrize("variant", ["auto", "grid", "balanced"])
@pytest.mark.parametrize("window", [0, 4096])
def test_query_block_sq8_full(window, variant):
    """Every request of the query-block workload, both passes."""
    case, ref = _full_case(f"qb{window}", lambda: wl.query_block_sq8(window=window))
    _check_full(case, ref, **VARIANTS[variant])


@pytest.mark.parametrize("variant", ["auto", "grid", "flat_fma", "configured_chunks"])
def test_fp8_long_b8_full(variant):
    """Every request of the long fp8 workload, whose q, K and V carry three
    distinct per-tensor scales amax/448."""
    case, ref = _full_case("fp8_long", wl.fp8_long_b8)
    assert len({case.q_scale, case.k_scale, case.v_scale}) == 3
    if variant == "configured_chunks":  # 32 chunks of 4096 keys, as the workload fixes
        _check_full(case, ref, chunk_tokens=case.chunk_tokens)
    else:
        _check_full(case, ref, **VARIANTS[variant])


@pytest.mark.parametrize("hkv,window", [(1, 0), (2, 0), (2, 70000)])
def test_tcgen05_units_over_many_ctas(hkv, window):
    """One 300,000-key request, 32 query heads per kv head (M = 32).  With one
    kv head its 147 chunks each get a CTA (147 pieces); with two, CTAs take tile
    shares of about 31 tiles, so each unit is cut into about 76 pieces.  Either
    way the CTA completing a unit's last piece merges its pieces in blocks of
    32."""
    import paged_kv_decode_15_gb300 as pkd
    case = wl.paged_case(name="long_units", seq_lens=[300_000], sq=1, num_heads=32 * hkv, num_kv_heads=hkv,
                         seed=91, window=window)
    assert pkd.kernel_name(1, 1, 32 * hkv, hkv, 128, 16, 300_000, pkd.BF16, window=window) == \
        "persistent tcgen05 kernel, TMEM accumulators"
    _check(case)


def _check_fp32_then_rounding(case, what):
    """Short requests put many outputs near |4|, where half a bf16 ulp alone is
    0.0078: the arithmetic is compared on the fp32 output (at the bf16
    tolerance) and the 16-bit output is checked to be that fp32 output rounded
    to nearest even, bit for bit."""
    import paged_kv_decode_15_gb300 as pkd
    ref, rlse = gu.oracle_paged(case)
    q = gu.to_dev(case.q, case.dtype)
    cache = gu.to_dev(case.kv_cache, case.dtype)
    bt = gu.to_dev(case.block_table, "int32")
    dl = gu.to_dev(case.seq_lens, "int32")
    kw = dict(q_scale=case.q_scale, k_scale=case.k_scale, v_scale=case.v_scale)
    o32, lse = pkd.paged_decode(q, cache, bt, dl, case.scale, case.window, out_dtype=torch.float32, **kw)
    o16, lse16 = pkd.paged_decode(q, cache, bt, dl, case.scale, case.window, out_dtype=torch.bfloat16, **kw)
    torch.cuda.synchronize()
    tol = gu.TOL_OUT_FP8 if case.dtype == "fp8" else gu.TOL_OUT
    gu.assert_close(o32.double().cpu().numpy(), ref, tol, f"{what} out (fp32)")
    gu.assert_close(lse.double().cpu().numpy(), rlse, gu.TOL_LSE, f"{what} lse")
    assert torch.equal(o16.cpu().view(torch.int16), o32.cpu().to(torch.bfloat16).view(torch.int16))
    assert torch.equal(lse16.cpu(), lse.cpu())


def test_tcgen05_largest_batch():
    """512 requests (the tcgen05 kernel's batch limit) of 0-300 keys, 32 rows
    per kv head: more units than CTAs, many cut by shares, some empty."""
    import paged_kv_decode_15_gb300 as pkd
    lens = np.random.default_rng(93).integers(0, 301, size=512).astype(np.int32)
    lens[::37] = 0
    case = wl.paged_case(name="b512", seq_lens=lens, sq=8, seed=94)
    assert pkd.kernel_name(512, 8, 32, 8, 128, 16, 300, pkd.BF16) == "persistent tcgen05 kernel, TMEM accumulators"
    _check_fp32_then_rounding(case, "b512")


@pytest.mark.parametrize("sq", [1, 8])
def test_long_slices_reload_the_page_list(sq):
    """One 2M-key request on the per-CTA partition: every CTA streams more keys
    than its page list holds at once, so it reloads the list inside the unit."""
    case = wl.paged_case(name="long", seq_lens=[2_000_000], sq=sq, num_heads=4, num_kv_heads=1, head_dim=64,
                         pool_factor=1.0, seed=31 + sq)
    _check(case, balanced=True)


@pytest.mark.parametrize("dtype,sq", [("fp8", 1), ("bf16", 8)])
def test_batch_above_the_flat_table_limit(dtype, sq):
    """1500 short requests (0-69 keys): the chunked grid (e4m3 warp, or warp
    pairs for 32 rows)."""
    lens = np.random.default_rng(77).integers(0, 70, size=1500).astype(np.int32)
    case = wl.paged_case(name="wide", seq_lens=lens, sq=sq, dtype=dtype, seed=78)
    _check_fp32_then_rounding(case, "wide")
