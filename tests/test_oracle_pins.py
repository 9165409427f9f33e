"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics.

Each test checks the oracle against something other than itself: worked
examples under tests/golden/, library conversions, closed forms, invariants,
and an independent numpy brute force on tiny inputs (tests/brute.py).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append([float(x) for x in line.split()])
    return rows


def _run(case, **over):
    kw = case.oracle_kwargs()
    kw.update(over)
    return oracle.paged_decode(case.q, case.dtype, case.kv_cache, case.dtype, case.block_table,
                               case.seq_lens, **kw)


# ----------------------------------------------------------------- decoders
def test_decode_bf16_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(codes, "bf16")
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_decode_fp16_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(codes, "fp16")
    ref = codes.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_decode_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode(codes, "fp8")
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.nanmax(got) == 448.0 and np.isnan(got[0x7F]) and np.isnan(got[0xFF])


# ------------------------------------------------------------------ window
def test_window_start_matches_hand_worked_rows():
    for L, w, sq, P, sp, new_len in _rows("window_restriction.txt"):
        got = oracle.window_start_page(int(L), int(w), int(sq), int(P))
        assert got == sp, (L, w, sq, P)
        assert L - got * P == new_len


def test_restrict_to_window_table_form():
    # request 0: L=100, w=32, sq=1, P=16 -> start page 4; request 1: L=30 -> 0
    bt = np.arange(20, dtype=np.int32).reshape(2, 10) + np.array([[0], [100]], np.int32)
    lens, table = oracle.restrict_to_window(np.array([100, 30]), bt, 32, 1, 16, 3)
    assert lens.tolist() == [36, 30]
    assert table.tolist() == [[4, 5, 6], [110, 111, 112]]
    # columns past the old table clamp to its last column
    lens, table = oracle.restrict_to_window(np.array([160]), bt[:1], 16, 1, 16, 4)
    assert lens.tolist() == [16] and table.tolist() == [[9, 9, 9, 9]]


def test_no_window_is_start_zero():
    assert oracle.window_start_page(10 ** 6, 0, 8, 16) == 0
    assert oracle.window_start_page(10 ** 6, -1, 1, 16) == 0


# ------------------------------------------------------------- worked examples
def test_two_key_worked_example():
    (lse_ref, o0, o1), = _rows("two_key_attention.txt")
    one, zero = 0x3F80, 0x0000
    # cache [1 page, 1 head, P=2, 2*D=4]: row t = [K_t | V_t]
    cache = np.array([[[[one, zero, one, zero], [zero, zero, zero, one]]]], np.uint16)
    q = np.array([[[[one, zero]]]], np.uint16)
    out, lse = oracle.paged_decode(q, "bf16", cache, "bf16", np.zeros((1, 1), np.int32),
                                   np.array([2], np.int32), sq=1, num_heads=1, num_kv_heads=1,
                                   head_dim=2, page_size=2, scale=1.0)
    assert abs(lse[0, 0, 0] - lse_ref) < 1e-15
    assert np.allclose(out[0, 0, 0], [o0, o1], atol=1e-15, rtol=0)


def test_lse_merge_worked_example():
    po = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])          # [N=1, S=2, H=1, D=2]
    pl = np.array([[[0.0], [math.log(3.0)]]])               # [1, 2, 1]
    for p1, p2, lse_ref, o0, o1 in _rows("lse_merge_two_parts.txt"):
        out, lse = oracle.lse_merge(po, pl, prior=np.array([[p1, p2]]))
        assert abs(lse[0, 0] - lse_ref) < 1e-14
        assert np.allclose(out[0, 0], [o0, o1], atol=1e-14, rtol=0)


# ---------------------------------------------------------- closed forms
def _small_case(**kw):
    base = dict(name="t", seq_lens=[37, 50, 16, 1], sq=1, num_heads=4, num_kv_heads=2, head_dim=16,
                page_size=16, seed=7)
    base.update(kw)
    return wl.paged_case(**base)


def test_single_key_returns_its_value():
    c = _small_case(seq_lens=[1, 1])
    out, lse = _run(c)
    cache = brute.decode(c.kv_cache, c.dtype)
    q = brute.decode(c.q, c.dtype)
    for b in range(2):
        page = c.block_table[b, 0]
        for h in range(c.num_heads):
            k0 = cache[page, h // 2, 0, :16]
            v0 = cache[page, h // 2, 0, 16:]
            assert np.array_equal(out[b, 0, h], v0)
            assert abs(lse[b, 0, h] - c.scale * float(q[b, 0, h] @ k0)) < 1e-12


def test_constant_v_returns_v_and_reads_nothing_else():
    c = _small_case()
    one = 0x3F80
    for b in range(c.batch):
        L = int(c.seq_lens[b])
        for j in range(L):
            c.kv_cache[c.block_table[b, j // 16], :, j % 16, 16:] = one
    out, lse = _run(c)
    assert np.all(np.isfinite(lse))
    # NaN tail slots and the NaN page are never read; the weights sum to one
    assert np.all(np.abs(out - 1.0) < 1e-14)


def test_zero_query_gives_log_count_and_mean():
    c = _small_case()
    c.q[:] = 0
    out, lse = _run(c)
    cache = brute.decode(c.kv_cache, c.dtype)
    for b in range(c.batch):
        L = int(c.seq_lens[b])
        V = np.stack([cache[c.block_table[b, j // 16], :, j % 16, 16:] for j in range(L)])
        for h in range(c.num_heads):
            assert abs(lse[b, 0, h] - math.log(L)) < 1e-12
            assert np.allclose(out[b, 0, h], V[:, h // 2].mean(0), atol=1e-12, rtol=0)


def test_empty_request_is_zero_and_minus_inf():
    c = _small_case(seq_lens=[0, 20])
    out, lse = _run(c)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# ----------------------------------------------------------- invariants
def test_page_permutation_invariance():
    c = _small_case(seq_lens=[37, 50, 64, 5])
    out, lse = _run(c)
    perm = np.random.default_rng(3).permutation(c.num_pages)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(c.num_pages)
    moved = c.kv_cache[perm]                  # new page p holds old page perm[p]
    table = inv[c.block_table].astype(np.int32)
    out2, lse2 = oracle.paged_decode(c.q, c.dtype, moved, c.dtype, table, c.seq_lens, **c.oracle_kwargs())
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_gqa_equals_mha_with_repeated_heads():
    c = _small_case(num_heads=8, num_kv_heads=2)
    out, lse = _run(c)
    rep = np.repeat(c.kv_cache, 4, axis=1)    # kv head h//4 copied to heads h
    out2, lse2 = oracle.paged_decode(c.q, c.dtype, rep, c.dtype, c.block_table, c.seq_lens,
                                     **dict(c.oracle_kwargs(), num_kv_heads=8))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_block_rows_equal_single_token_decode():
    c = _small_case(sq=4)
    out, lse = _run(c)
    for i in range(4):
        qi = np.ascontiguousarray(c.q[:, i:i + 1])
        o1, l1 = oracle.paged_decode(qi, c.dtype, c.kv_cache, c.dtype, c.block_table, c.seq_lens,
                                     **dict(c.oracle_kwargs(), sq=1))
        assert np.array_equal(out[:, i:i + 1], o1) and np.array_equal(lse[:, i:i + 1], l1)


def test_split_merge_equals_whole_sequence():
    c = _small_case(seq_lens=[80, 47], page_size=16)
    out, lse = _run(c)
    # split request b at page boundaries into parts of 1..2 pages and merge by LSE
    for b in range(2):
        L = int(c.seq_lens[b])
        cuts = sorted({0, 16, min(48, L), L})
        po, pl = [], []
        for a, e in zip(cuts[:-1], cuts[1:]):
            table = c.block_table[b:b + 1, a // 16:]
            o, l = oracle.paged_decode(c.q[b:b + 1], c.dtype, c.kv_cache, c.dtype,
                                       np.ascontiguousarray(table), np.array([e - a], np.int32),
                                       **c.oracle_kwargs())
            po.append(o[0, 0])
            pl.append(l[0, 0])
        mo, ml = oracle.lse_merge(np.stack(po)[None], np.stack(pl)[None])
        assert np.allclose(mo[0], out[b, 0], atol=1e-13, rtol=0)
        assert np.allclose(ml[0], lse[b, 0], atol=1e-13, rtol=0)


def test_windowed_equals_restricted_table_and_wide_window_is_none():
    c = _small_case(seq_lens=[100, 37, 64, 17], sq=2, window=20, table_width=8)
    out, lse = _run(c)
    lens, table = oracle.restrict_to_window(c.seq_lens, c.block_table, 20, 2, 16, 4)
    out2, lse2 = oracle.paged_decode(c.q, c.dtype, c.kv_cache, c.dtype, table, lens,
                                     **dict(c.oracle_kwargs(), window=0))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    wide, wl_ = _run(c, window=10 ** 6)
    none, nl = _run(c, window=0)
    assert np.array_equal(wide, none) and np.array_equal(wl_, nl)


def test_fp8_power_of_two_scales_equal_bf16_on_dequantised_values():
    c = _small_case(dtype="fp8", seq_lens=[40, 64, 3], fp8_scales="pow2")
    out, lse = _run(c)
    deq_cache = wl.round_to((brute.decode(c.kv_cache, "fp8") * c.k_scale).astype(np.float32), "bf16")
    deq_q = wl.round_to((brute.decode(c.q, "fp8") * c.q_scale).astype(np.float32), "bf16")
    # the dequantised values are exact in bf16 (3 mantissa bits, small exponents)
    assert np.array_equal(brute.decode(deq_cache, "bf16")[~np.isnan(brute.decode(deq_cache, "bf16"))],
                          (brute.decode(c.kv_cache, "fp8") * c.k_scale)[~np.isnan(brute.decode(c.kv_cache, "fp8"))])
    out2, lse2 = oracle.paged_decode(deq_q, "bf16", deq_cache, "bf16", c.block_table, c.seq_lens,
                                     **dict(c.oracle_kwargs(), q_scale=1.0, k_scale=1.0, v_scale=1.0))
    assert np.allclose(out, out2, atol=1e-13, rtol=0) and np.allclose(lse, lse2, atol=1e-13, rtol=0)


# ------------------------------------------------------- brute force (tiny)
@pytest.mark.parametrize("kw", [
    dict(),
    dict(sq=3),
    dict(sq=3, window=20),
    dict(sq=3, causal=True),
    dict(sq=3, causal=True, window=10),
    dict(dtype="fp16"),
    dict(dtype="fp8"),                       # q, K, V with three per-tensor scales amax/448
    dict(dtype="fp8", fp8_scales="pow2"),
    dict(scales=(0.731, 1.377, 0.589)),      # 16-bit storage with distinct q, k, v scales
    dict(dtype="fp16", sq=3, scales=(1.7, 0.45, 2.3), causal=True),
    dict(head_dim=64, page_size=32, seq_lens=[70, 1, 33]),
])
def test_paged_decode_matches_brute_force(kw):
    c = _small_case(**kw)
    out, lse = _run(c)
    bo, bl = brute.paged_decode(c)
    assert np.allclose(out, bo, atol=1e-12, rtol=1e-12)
    assert np.allclose(lse, bl, atol=1e-12, rtol=1e-12)


def test_tiny_workload_matches_brute_force():
    c = wl.tiny_decode()
    out, lse = _run(c)
    bo, bl = brute.paged_decode(c)
    assert np.all(np.isfinite(out))
    assert np.allclose(out, bo, atol=1e-12, rtol=1e-12) and np.allclose(lse, bl, atol=1e-12, rtol=1e-12)


# ----------------------------------------------------------- segments
def _seg(**kw):
    base = dict(n=5, num_heads=4, num_kv_heads=2, head_dim=16, topk=3, bs=8, local=16, seed=11)
    base.update(kw)
    return wl.segment_case(**base)


def _seg_run(s, **kw):
    return oracle.segmented_attention(s.q, s.k, s.v, s.dtype, s.used, s.bias, topk=s.topk, bs=s.bs,
                                      local=s.local, num_kv_heads=s.num_kv_heads, **kw)


def test_segments_match_brute_force():
    used = np.array([[8, 0, 3, 16], [0, 0, 0, 1], [1, 8, 8, 16], [0, 0, 0, 0], [5, 0, 0, 7]])
    s = _seg(used=used)
    out, so, sl = _seg_run(s, return_segments=True)
    bo, bso, bsl = brute.segmented(s)
    assert np.allclose(out, bo, atol=1e-12, rtol=1e-12)
    assert np.allclose(so, bso, atol=1e-12, rtol=1e-12)
    assert np.array_equal(np.isneginf(sl), np.isneginf(bsl))
    fin = np.isfinite(bsl)
    assert np.allclose(sl[fin], bsl[fin], atol=1e-12, rtol=1e-12)
    assert np.all(out[3] == 0)                       # no live segment -> 0


def test_segments_combine_equals_union_attention_with_bias():
    """softmax over segments of (lse_g + bias_g) weighting o_g is plain attention
    over the union of live keys whose logits carry their segment's bias."""
    s = _seg(n=3)
    out = _seg_run(s)
    q = brute.decode(s.q, s.dtype)
    k = brute.decode(s.k, s.dtype)
    v = brute.decode(s.v, s.dtype)
    used = s.used.reshape(3, 4)
    rows = 3 * 8 + 16
    for i in range(3):
        idx, bias = [], []
        for g in range(4):
            off = i * rows + (g * 8 if g < 3 else 24)
            idx += list(range(off, off + used[i, g]))
            bias += [float(s.bias[i, g]) if g < 3 else 0.0] * int(used[i, g])
        for h in range(4):
            o, _ = brute.dense_attention(q[i, h], k[idx, h // 2], v[idx, h // 2], 16 ** -0.5, np.array(bias))
            assert np.allclose(out[i, h], o, atol=1e-12, rtol=1e-12)


def test_zero_length_segments_contribute_nothing():
    used = np.array([[0, 4, 0, 9], [3, 0, 0, 2]])
    s = _seg(n=2, used=used)
    out = _seg_run(s)
    # rewrite the dead segments' rows with arbitrary finite values: output is unchanged
    s2 = _seg(n=2, used=used)
    for i, g in [(0, 0), (0, 2), (1, 1), (1, 2)]:
        off = i * 40 + g * 8
        s2.k[off:off + 8] = 0x4000   # 2.0
        s2.v[off:off + 8] = 0xC040   # -3.0
    assert np.array_equal(out, _seg_run(s2))
    assert np.all(np.isfinite(out))


def test_segments_arbitrary_split_merges_to_whole():
    """One query's keys cut at arbitrary (not page-aligned) points into segments:
    with zero bias the combine equals attention over all of them."""
    s = _seg(n=1, topk=3, bs=8, local=16, used=np.array([[5, 8, 2, 13]]))
    s.bias[:] = 0
    out = _seg_run(s)
    q = brute.decode(s.q, s.dtype)
    k = brute.decode(s.k, s.dtype)
    v = brute.decode(s.v, s.dtype)
    idx = list(range(0, 5)) + list(range(8, 16)) + list(range(16, 18)) + list(range(24, 37))
    for h in range(4):
        o, _ = brute.dense_attention(q[0, h], k[idx, h // 2], v[idx, h // 2], 16 ** -0.5)
        assert np.allclose(out[0, h], o, atol=1e-12, rtol=1e-12)


def test_segments_reject_used_above_capacity():
    s = _seg(n=1, used=np.array([[9, 0, 0, 1]]), poison_unused=False)
    with pytest.raises(ValueError):
        _seg_run(s)


# ----------------------------------------------------------- lse merge
def test_lse_merge_dead_parts_and_all_dead():
    rng = np.random.default_rng(5)
    po = rng.standard_normal((3, 4, 2, 8))
    pl = rng.standard_normal((3, 4, 2))
    live = np.array([[1, 0, 1, 1], [0, 0, 0, 0], [1, 1, 1, 1]], np.int32)
    po[0, 1] = np.nan                                  # dead part: never read
    out, lse = oracle.lse_merge(po, pl, live=live)
    ref, rl = oracle.lse_merge(po[:1, [0, 2, 3]], pl[:1, [0, 2, 3]])
    assert np.array_equal(out[0], ref[0]) and np.array_equal(lse[0], rl[0])
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    # closed form for row 2: weights softmax(lse)
    w = np.exp(pl[2] - np.log(np.exp(pl[2]).sum(0)))
    assert np.allclose(out[2], np.einsum("sh,shd->hd", w, po[2]), atol=1e-13)


# ----------------------------------------------------------- cache write
def _all_finite_e4m3():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    return codes, torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()


def test_encode_e4m3_exact_values_round_trip():
    codes, vals = _all_finite_e4m3()
    got = oracle.encode_e4m3(vals)
    # -0.0 and +0.0 keep their sign; every finite code maps back to itself
    assert np.array_equal(got, codes)


def test_encode_e4m3_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(12)
    mags = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(440.0), 200_000)).astype(np.float32)
    x = mags * rng.choice([-1.0, 1.0], mags.size).astype(np.float32)
    # ties: midpoints between neighbouring finite codes (round half to even decides)
    _, vals = _all_finite_e4m3()
    pos = np.unique(vals[vals >= 0])
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.encode_e4m3(x), ref)


def test_encode_e4m3_saturates():
    got = oracle.encode_e4m3(np.array([448.0, 463.9, 464.0, 1e6, np.inf, -500.0, -np.inf], np.float32))
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def _cache_write_case(dtype_in="bf16", kv="bf16", T=37, Hkv=2, D=16, P=16, num_pages=9, seed=4):
    rng = np.random.default_rng(seed)
    key = wl.normal_storage(rng, (T, Hkv, D), dtype_in)
    value = wl.normal_storage(rng, (T, Hkv, D), dtype_in)
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    slots[[3, 11]] = -1                                   # padding tokens
    cache = wl.normal_storage(rng, (num_pages, Hkv, P, 2 * D), kv)
    return key, value, slots, cache


def test_cache_write_16bit_places_rows_by_slot():
    key, value, slots, cache = _cache_write_case()
    out = oracle.cache_write(key, value, "bf16", slots, cache, "bf16", num_kv_heads=2, head_dim=16, page_size=16)
    expect = cache.copy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        expect[s // 16, :, s % 16, :16] = key[t]
        expect[s // 16, :, s % 16, 16:] = value[t]
    assert np.array_equal(out, expect)


def test_cache_write_fp8_quantises_each_element():
    key, value, slots, cache = _cache_write_case(kv="fp8")
    ks, vs = 1.0 / 64, 1.0 / 32
    out = oracle.cache_write(key, value, "bf16", slots, cache, "fp8", num_kv_heads=2, head_dim=16, page_size=16,
                             k_scale=ks, v_scale=vs)
    kf = brute.decode(key, "bf16").astype(np.float32)
    vf = brute.decode(value, "bf16").astype(np.float32)
    kq = torch.from_numpy(np.clip(kf / np.float32(ks), -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vq = torch.from_numpy(np.clip(vf / np.float32(vs), -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    expect = cache.copy()
    for t, s in enumerate(slots):
        if s >= 0:
            expect[s // 16, :, s % 16, :16] = kq[t]
            expect[s // 16, :, s % 16, 16:] = vq[t]
    assert np.array_equal(out, expect)


def test_cache_write_then_decode_reads_what_was_written():
    """A cache filled through cache_write decodes the same as one laid out directly."""
    P, D, Hkv = 16, 16, 2
    c = _small_case(seq_lens=[40, 17], num_heads=4, num_kv_heads=Hkv, head_dim=D, page_size=P)
    keys = {}
    blank = np.zeros_like(c.kv_cache)
    blank[c.poison_page] = c.kv_cache[c.poison_page]
    written = blank
    for b in range(c.batch):
        L = int(c.seq_lens[b])
        toks = np.arange(L)
        slots = (c.block_table[b, toks // P].astype(np.int64) * P + toks % P)
        k = np.stack([c.kv_cache[c.block_table[b, t // P], :, t % P, :D] for t in toks])
        v = np.stack([c.kv_cache[c.block_table[b, t // P], :, t % P, D:] for t in toks])
        written = oracle.cache_write(k, v, "bf16", slots, written, "bf16", num_kv_heads=Hkv, head_dim=D, page_size=P)
    o1, l1 = _run(c)
    o2, l2 = oracle.paged_decode(c.q, c.dtype, written, c.dtype, c.block_table, c.seq_lens, **c.oracle_kwargs())
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ------------------------------------------------------ paged segments
def test_paged_segments_equal_contiguous_segments_after_gathering():
    """Gathering each segment's keys into contiguous rows (by a plain loop over
    the block table) and running the contiguous-segment oracle gives the same."""
    s = wl.paged_segment_case(n=5, num_heads=4, num_kv_heads=2, head_dim=16, page_size=16, topk=3, bs=24,
                              local=32, seed=9, seq_range=(40, 200))
    out, so, sl = oracle.segmented_paged(s.q, s.dtype, s.kv_cache, s.block_table, s.seg_start, s.used, s.bias,
                                         num_kv_heads=2, page_size=16, topk=3, bs=24, local=32,
                                         return_segments=True)
    rows = 3 * 24 + 32
    k = np.zeros((5 * rows, 2, 16), np.uint16)
    v = np.zeros_like(k)
    for i in range(5):
        for g in range(4):
            off = i * rows + (g * 24 if g < 3 else 72)
            for t in range(int(s.used[i, g])):
                j = int(s.seg_start[i, g]) + t
                page = s.block_table[i, j // 16]
                k[off + t] = s.kv_cache[page, :, j % 16, :16]
                v[off + t] = s.kv_cache[page, :, j % 16, 16:]
    ref, rso, rsl = oracle.segmented_attention(s.q, k, v, s.dtype, s.used, s.bias, topk=3, bs=24, local=32,
                                               num_kv_heads=2, return_segments=True)
    assert np.array_equal(out, ref) and np.array_equal(so, rso) and np.array_equal(sl, rsl)


def test_paged_segments_single_segment_is_window_decode():
    """One local segment covering the last w keys equals paged decode of that
    key range (a table sliced to start there, with the length renumbered)."""
    c = _small_case(seq_lens=[64, 96], num_heads=4, num_kv_heads=2)
    w = 32
    seg_start = (c.seq_lens - w).reshape(2, 1).astype(np.int32)
    used = np.full((2, 1), w, np.int32)
    q3 = np.ascontiguousarray(c.q[:, 0])
    out = oracle.segmented_paged(q3, c.dtype, c.kv_cache, c.block_table, seg_start, used, np.zeros((2, 0)),
                                 num_kv_heads=2, page_size=16, topk=0, bs=0, local=w)
    for b in range(2):
        start = int(c.seq_lens[b]) - w       # a page boundary here
        table = np.ascontiguousarray(c.block_table[b:b + 1, start // 16:])
        o, _ = oracle.paged_decode(c.q[b:b + 1], c.dtype, c.kv_cache, c.dtype, table, np.array([w], np.int32),
                                   **dict(c.oracle_kwargs(), scale=16 ** -0.5))
        assert np.allclose(out[b], o[0, 0], atol=1e-13, rtol=0)
