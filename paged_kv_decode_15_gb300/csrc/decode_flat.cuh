// Persistent paged decode with a flat partition of the key stream.
//
// All (request, kv head) units are laid end to end as one sequence of
// 16-key stages (unit u = b*Hkv + hk holds ceil(visible_b / 16) stages).  A
// fixed set of workers -- every warp of a grid sized to fill the GPU once --
// takes equal, contiguous slices of that sequence, so every warp streams the
// same number of bytes and the launch ends without a tail of unequal CTAs.
// A slice may start inside one unit and end inside another:
//   - a unit covered by one worker alone is finished and written directly;
//   - a unit shared by several workers gets one partial (O / l, LSE) per
//     worker, in the worker's own slot; the last worker to arrive on the
//     unit's counter merges the partials by LSE and resets the counter.
// No worker ever waits on another, so the kernel needs no co-residency.
//
// Each warp runs its own TMA ring of NBUF stages; the page index of every
// stage is looked up 32 stages ahead (one per lane) so a TMA issue never
// waits on the block table.
#pragma once

#include "fma_warp.cuh"
#include "fp8_warp.cuh"
#include "mma_warp.cuh"

namespace pkd {

constexpr int kFlatMinStages = 4;     // a worker streams at least this many stages

template <int D, int ELT, int NBUF, int SCR = 0>
struct FlatShape {
    static constexpr int HALF = (D * ELT / 128) * 2048;
    static constexpr int STAGE = 2 * HALF;
    static constexpr int RING = kNW * NBUF * STAGE;
    static constexpr int OFF_SCR = RING;                     // per-warp scratch (1 KiB aligned)
    static constexpr int OFF_BARS = OFF_SCR + kNW * SCR;
    static constexpr int OFF_PRE = OFF_BARS + kNW * NBUF * 8;
    static constexpr int OFF_LEN = OFF_PRE + (kFlatMaxBatch + 1) * 4;
    static constexpr int OFF_SCAN = OFF_LEN + kFlatMaxBatch * 4;
    static constexpr int OFF_MERGE = OFF_SCAN + 64;             // per-warp row stats of a merge
    static constexpr int SMEM = OFF_MERGE + kNW * 3 * 32 * 4 + 1024;
};

struct StageMeta {
    int b, hk, s, page;
};

// Merge the partials of unit (b, hk) left by workers wf..wl (the caller is the
// last to arrive).  Two passes of independent loads: per-row max and sum of
// weights, then float4 sums.  Out of line: it runs once per shared unit.
template <int D>
__device__ __noinline__ void merge_unit(const DecodeParams& p, int b, int hk, long long wf, long long wl,
                                        long long Stot, long long Weff, long long E, float* mstat, int lane) {
    auto slot = [&](long long v) { return v * 2 + ((v + 1) * Stot / Weff < E ? 1 : 0); };
    float* smx = mstat;
    float* sinv = mstat + 32;
    for (int r = lane; r < p.M; r += 32) {
        float mx = -INFINITY;
#pragma unroll 4
        for (long long v = wf; v <= wl; ++v) mx = fmaxf(mx, __ldcg(p.part_lse + slot(v) * p.M + r));
        float ws = 0.f;
        if (mx != -INFINITY) {
#pragma unroll 4
            for (long long v = wf; v <= wl; ++v) {
                const float lc = __ldcg(p.part_lse + slot(v) * p.M + r);
                ws += lc == -INFINITY ? 0.f : fast_exp2(lc - mx);
            }
        }
        smx[r] = mx;
        sinv[r] = ws > 0.f ? 1.f / ws : 0.f;
        if (p.lse) {
            const int i = r / p.G, g = r % p.G;
            p.lse[(static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g] =
                ws > 0.f ? (mx + __log2f(ws)) * kLn2 : -INFINITY;
        }
    }
    __syncwarp();
    for (int q4 = lane; q4 < p.M * D / 4; q4 += 32) {
        const int r = (q4 * 4) / D, d = (q4 * 4) % D;
        const float mx = smx[r], inv = sinv[r];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (inv > 0.f) {
#pragma unroll 4
            for (long long v = wf; v <= wl; ++v) {
                const long long sl2 = slot(v);
                const float lc = __ldcg(p.part_lse + sl2 * p.M + r);
                const float4 o = __ldcg(reinterpret_cast<const float4*>(p.part_out + sl2 * p.M * D) + q4);
                const float w = lc == -INFINITY ? 0.f : fast_exp2(lc - mx) * inv;  // empty partials hold 0
                acc.x = fmaf(w, o.x, acc.x);
                acc.y = fmaf(w, o.y, acc.y);
                acc.z = fmaf(w, o.z, acc.z);
                acc.w = fmaf(w, o.w, acc.w);
            }
        }
        const long long oi = out_index(p, b, hk, r, d, D);
        store_out(p.out, oi, acc.x * p.v_scale, p.out_dtype);
        store_out(p.out, oi + 1, acc.y * p.v_scale, p.out_dtype);
        store_out(p.out, oi + 2, acc.z * p.v_scale, p.out_dtype);
        store_out(p.out, oi + 3, acc.w * p.v_scale, p.out_dtype);
    }
}

// RT > 1: the query rows of a unit are split into RT tiles of 16, held by RT
// consecutive warps that walk the same slice of keys (each with its own ring;
// the repeated loads of a stage are served by L2).
template <class W, int D, int ELT, int NBUF, int RT>
__global__ void __launch_bounds__(kNW * 32)
decode_flat_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    using S = FlatShape<D, ELT, NBUF, W::kScratchBytes>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
    int* pre = reinterpret_cast<int*>(smem + S::OFF_PRE);   // stage prefix over requests (per kv head)
    int* lens = reinterpret_cast<int*>(smem + S::OFF_LEN);  // clamped lengths
    int* scan = reinterpret_cast<int*>(smem + S::OFF_SCAN);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B;
    if (tid == 0) {
        prefetch_tmap(&tmap);
        for (int i = 0; i < kNW * NBUF; ++i) mbar_init(smem_u32(bars + i), 1);
        fence_barrier_init();
    }

    // ---- per-request stage counts and their prefix (block-wide scan)
    const int per = (B + blockDim.x - 1) / blockDim.x;
    const int b_begin = tid * per, b_end = min(B, b_begin + per);
    int local = 0;
    for (int b = b_begin; b < b_end; ++b) {
        const int L = clamp_len(p, b, blockIdx.x == 0);
        lens[b] = L;
        const int vis = L - visible_lo(p, L);
        local += (vis + kStageTok - 1) / kStageTok;
    }
    int incl = local;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, m);
        if (lane >= m) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int k = 0; k < warp; ++k) base += scan[k];
    int run = base + incl - local;
    for (int b = b_begin; b < b_end; ++b) {
        pre[b] = run;
        const int L = lens[b];
        run += (L - visible_lo(p, L) + kStageTok - 1) / kStageTok;
    }
    if (tid == blockDim.x - 1) pre[B] = base + incl;
    __syncthreads();

    const long long Hkv = p.Hkv;
    const long long Stot = static_cast<long long>(pre[B]) * Hkv;

    // ---- requests with no visible key: out = 0, lse = -inf
    for (int b = blockIdx.x; b < B; b += gridDim.x)
        if (pre[b + 1] == pre[b]) write_empty_request<D>(p, b);

    // ---- this warp's slice of the flat stage sequence
    static_assert(kNW % RT == 0, "row-tile groups must not straddle CTAs");
    const int rt = warp % RT;
    const long long Wtot = static_cast<long long>(gridDim.x) * (kNW / RT);
    long long Weff = Stot / kFlatMinStages;
    if (Weff > Wtot) Weff = Wtot;
    if (Weff < 1) Weff = 1;
    const long long wid = (static_cast<long long>(blockIdx.x) * kNW + warp) / RT;
    if (Stot == 0 || wid >= Weff) return;
    const long long f0 = wid * Stot / Weff, f1 = (wid + 1) * Stot / Weff;
    const int n = static_cast<int>(f1 - f0);
    if (n == 0) return;

    // stage -> (request, kv head, stage in unit, page); one stage per lane
    auto fetch = [&](long long f) {
        StageMeta m;
        m.b = -1;
        m.hk = 0;
        m.s = 0;
        m.page = -1;
        if (f < f1) {
            int lo = 0, hi = B;  // largest b with Hkv * pre[b] <= f
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (Hkv * pre[mid] <= f) lo = mid; else hi = mid;
            }
            const int b = lo;
            const int cnt = pre[b + 1] - pre[b];
            const long long loc = f - Hkv * pre[b];
            m.b = b;
            m.hk = static_cast<int>(loc / cnt);
            m.s = static_cast<int>(loc % cnt);
            const int tok = visible_lo(p, lens[b]) + m.s * kStageTok;
            int pg = p.block_table[static_cast<long long>(b) * p.bt_stride + page_col(p, tok)];
            if (pg < 0 || pg >= p.num_pages) {
                raise_status(p, kErrBounds);
                pg = -1;
            }
            m.page = pg;
        }
        return m;
    };
    auto shfl_meta = [&](const StageMeta& m, int src) {
        StageMeta r;
        r.b = __shfl_sync(kFull, m.b, src);
        r.hk = __shfl_sync(kFull, m.hk, src);
        r.s = __shfl_sync(kFull, m.s, src);
        r.page = __shfl_sync(kFull, m.page, src);
        return r;
    };

    float* mstat = reinterpret_cast<float*>(smem + S::OFF_MERGE) + warp * 3 * 32;
    uint8_t* ring_gen = smem + warp * NBUF * S::STAGE;
    const uint32_t ring = smem_u32(ring_gen);
    const uint32_t bar0 = smem_u32(bars + warp * NBUF);
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int k, const StageMeta& m) {  // lane 0 only
        const uint32_t buf = ring + (k % NBUF) * S::STAGE;
        const uint32_t bar = bar0 + 8 * (k % NBUF);
        if (m.page < 0) {
            mbar_arrive(bar);
            return;
        }
        const int tok = visible_lo(p, lens[m.b]) + m.s * kStageTok;
        const int row = (m.page * p.Hkv + m.hk) * p.P + page_slot(p, tok);
        mbar_arrive_expect_tx(bar, S::STAGE);
        tma_load_3d(buf, &tmap, 0, row, 0, bar, pol);
    };

    StageMeta cur = fetch(f0 + lane), nxt = fetch(f0 + 32 + lane);
    for (int k = 0; k < NBUF && k < n; ++k) {
        const StageMeta m = shfl_meta(cur, k);
        if (lane == 0) issue(k, m);
    }

    W wp;
    wp.init(lane);
    wp.setup(smem + S::OFF_SCR + warp * W::kScratchBytes);
    wp.row0 = rt * 16;
    const int row0 = wp.row0;
    int ub = -1, uh = -1, uL = 0, ulo = 0, ucnt = 0;

    // finish unit (ub, uh): direct write, or partial + last-arriver merge
    auto finalize = [&]() {
        wp.finish();
        const long long F = Hkv * pre[ub] + static_cast<long long>(uh) * ucnt, E = F + ucnt;
        auto owner = [&](long long f) { return ((f + 1) * Weff - 1) / Stot; };
        const long long wf = owner(F), wl = owner(E - 1);
        const int b = ub, hk = uh;
        if (wf == wl) {
            wp.emit([&](int r, int d, float v) {
                r += row0;
                if (r < p.M) store_out(p.out, out_index(p, b, hk, r, d, D), v * p.v_scale, p.out_dtype);
            }, lane);
            if (p.lse)
                wp.emit_lse([&](int r, float l2) {
                    r += row0;
                    if (r < p.M) {
                        const int i = r / p.G, g = r % p.G;
                        p.lse[(static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g] = l2 * kLn2;
                    }
                }, lane);
            return;
        }
        const int side = f1 < E ? 1 : 0;  // 1: the unit continues past this slice
        float* so = p.part_out + (wid * 2 + side) * p.M * D;
        float* sl = p.part_lse + (wid * 2 + side) * p.M;
        wp.emit([&](int r, int d, float v) { r += row0; if (r < p.M) __stcg(so + r * D + d, v); }, lane);
        wp.emit_lse([&](int r, float l2) { r += row0; if (r < p.M) __stcg(sl + r, l2); }, lane);
        // the warp's stores, then one arrival with acquire-release semantics at
        // GPU scope; the warp barrier after it passes the acquire on to every lane
        __syncwarp();
        const int u = b * p.Hkv + hk;
        int last = 0;
        if (lane == 0) {
            const int prev = atom_add_acq_rel_gpu(p.counters + u);
            last = prev == static_cast<int>((wl - wf + 1) * RT - 1);
            if (last) atomicExch(p.counters + u, 0);  // ready for the next call
        }
        last = __shfl_sync(kFull, last, 0);
        if (!last) return;
        __syncwarp();
        merge_unit<D>(p, b, hk, wf, wl, Stot, Weff, E, mstat, lane);
        __syncwarp();
    };

    for (int k = 0; k < n; ++k) {
        if (__builtin_expect(k > 0 && (k & 31) == 0, 0)) {
            cur = nxt;
            nxt = fetch(f0 + k + 32 + lane);
        }
        const StageMeta mk = shfl_meta(cur, k & 31);
        if (__builtin_expect(mk.b != ub || mk.hk != uh, 0)) {
            if (ub >= 0) finalize();
            ub = mk.b;
            uh = mk.hk;
            uL = lens[ub];
            ulo = visible_lo(p, uL);
            ucnt = pre[ub + 1] - pre[ub];
            wp.reset();
            wp.load_q(p, ub, uh, lane);
        }
        const int buf = k % NBUF;
        if (__builtin_expect(!mbar_wait(bar0 + 8 * buf, (k / NBUF) & 1, p.status, p.wait_ns), 0)) {
            // let the issued copies (stages k .. k + NBUF - 1) land first
            if (lane == 0) raise_status(p, kErrTimeout);
            for (int j = k; j < n && j < k + NBUF; ++j) mbar_wait(bar0 + 8 * (j % NBUF), (j / NBUF) & 1);
            return;
        }
        const int tok0 = ulo + mk.s * kStageTok;
        int nvalid = min(kStageTok, uL - tok0);
        if (mk.page < 0) nvalid = 0;
        uint8_t* st_gen = ring_gen + buf * S::STAGE;
        if (nvalid < kStageTok) zero_tail_v<D, ELT>(st_gen, nvalid, lane);
        const int L = uL;
        auto visible = [&](int row, int kt) { return row_sees(p, L, row0 + row, tok0 + kt); };
        if constexpr (W::kTensor)
            wp.consume(ring + buf * S::STAGE, S::HALF, nvalid, nvalid < kStageTok || p.causal, p.scale_log2, 0.f,
                       visible, lane);
        else
            wp.consume(st_gen, nvalid, visible, lane);
        __syncwarp();
        const int j = k + NBUF;
        if (j < n) {
            const StageMeta mj = shfl_meta((j >> 5) == (k >> 5) ? cur : nxt, j & 31);
            if (lane == 0) {
                fence_proxy_async();
                issue(j, mj);
            }
        }
    }
    finalize();
}

}  // namespace pkd
