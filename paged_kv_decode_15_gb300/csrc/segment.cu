// DASH segmented attention and the LSE merge.
//
// Segmented attention: query i attends topk gathered segments of bs rows and
// one local segment of `local` rows, each cut to its used prefix; each
// segment's softmax result (o_g, lse_g) is then combined by a softmax over
// segments of lse_g + prior_g.  Because
//     sum_g softmax_g(lse_g + b_g) o_g  =  sum_j exp(s_j + b_g(j) - LSE) V_j,
// the fused kernel runs ONE online softmax over the union of the live keys
// with each key's logit shifted by its segment's prior; dead (empty) segments
// contribute no key at all.  One CTA per (query, kv head); its four warps
// take 16-key stages round-robin from a TMA ring, as in paged decode.
// When the per-segment results are asked for, each warp instead owns whole
// segments, writes (o_g, lse_g), and the combine runs as a separate LSE merge.
#include "launch.h"
#include "mma_warp.cuh"
#include "segment.cuh"

namespace pkd {

constexpr int kSegNbuf = 2;
constexpr int kMaxGroups = 64;
constexpr int kMaxSegStages = 512;  // paged segments: page index of every stage of a CTA

template <int D, int NT>
struct SegShape {
    static constexpr int HALF = (D * 2 / 128) * 2048;
    static constexpr int STAGE = 2 * HALF;
    static constexpr int MROWS = 16;
    static constexpr int QSTRIDE = D * 2 + 16;
    static constexpr int OSTRIDE = D + 4;
    static constexpr int RING = kNW * kSegNbuf * STAGE;
    static constexpr int MERGE = kNW * MROWS * OSTRIDE * 4;
    static constexpr int BIG = RING > MERGE ? RING : MERGE;
    static constexpr int OFF_BARS = BIG;
    static constexpr int OFF_Q = OFF_BARS + kNW * kSegNbuf * 8;
    static constexpr int OFF_ML = OFF_Q + MROWS * QSTRIDE;
    static constexpr int OFF_SEG = OFF_ML + 2 * kNW * MROWS * 4;  // used, prefix, bias2, start, aligned start
    static constexpr int OFF_PAGE = OFF_SEG + 5 * (kMaxGroups + 1) * 4;
    static constexpr int SMEM = OFF_PAGE + kMaxSegStages * 4 + 1024;
};

// tok / P by a magic-number multiply (exact for 0 <= tok < 2^31)
__device__ __forceinline__ int seg_page_col(const SegmentParams& p, int tok) {
    return page_div(tok, p.pmagic, p.pmshift);
}

// One 16-byte copy into shared memory that completes asynchronously; with
// `nbytes` = 0 it reads nothing and writes 16 zero bytes.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int nbytes, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst), "l"(src), "r"(nbytes),
                 "l"(policy)
                 : "memory");
}

// An arrive on `bar` once this thread's earlier cp.async copies have landed;
// it raises the barrier's pending count first, so the phase still waits for
// its ordinary arrivals as well.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

template <int D, bool kBF16, int NT, bool kSegOut, bool kPaged>
__global__ void __launch_bounds__(kNW * 32)
segmented_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                 const SegmentParams p) {
    using S = SegShape<D, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
    uint8_t* qs = smem + S::OFF_Q;
    float* wm = reinterpret_cast<float*>(smem + S::OFF_ML);
    float* wl = wm + kNW * S::MROWS;
    int* su = reinterpret_cast<int*>(smem + S::OFF_SEG);    // used, clamped
    int* pre = su + (kMaxGroups + 1);                       // stage prefix (fused mode)
    float* sb = reinterpret_cast<float*>(pre + (kMaxGroups + 1));  // prior, log2 domain
    int* ss = reinterpret_cast<int*>(sb + (kMaxGroups + 1));       // paged: first key of the segment
    int* sa = ss + (kMaxGroups + 1);                               // paged: first key of its first stage
    int* spage = reinterpret_cast<int*>(smem + S::OFF_PAGE);       // paged: page of every stage

    const int i = blockIdx.x, hk = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int groups = p.topk + 1;
    const long long row_base = static_cast<long long>(i) * (static_cast<long long>(p.topk) * p.bs + p.local);
    const int M = p.G;

    if (warp == 0) {
        // segments g = lane and lane + 32: used, prior, start; then their
        // stage counts, scanned across the warp into the stage prefix
        int cnt[2], incl[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int g = lane + 32 * h;
            cnt[h] = 0;
            if (g < groups) {
                const int cap = g < p.topk ? p.bs : p.local;
                int u = p.used[static_cast<long long>(i) * groups + g];
                u = u < 0 ? 0 : (u > cap ? cap : u);
                sb[g] = g < p.topk ? p.bias[static_cast<long long>(i) * p.topk + g] * kLog2e : 0.f;
                if constexpr (kPaged) {
                    // keys [start, start + used) of request row i; stages start on 16-key boundaries
                    int st = p.seg_start[static_cast<long long>(i) * groups + g];
                    st = st < 0 ? 0 : st;
                    if (st > p.max_kv_len) st = p.max_kv_len;
                    if (u > p.max_kv_len - st) u = p.max_kv_len - st;
                    const int a = st / kStageTok * kStageTok;
                    ss[g] = st;
                    sa[g] = a;
                    cnt[h] = u > 0 ? (st + u - a + kStageTok - 1) / kStageTok : 0;
                } else {
                    cnt[h] = (u + kStageTok - 1) / kStageTok;
                }
                su[g] = u;
            }
            incl[h] = cnt[h];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl[h], o);
                if (lane >= o) incl[h] += v;
            }
        }
        const int total0 = __shfl_sync(0xffffffffu, incl[0], 31);
        incl[1] += total0;
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (lane + 32 * h < groups) pre[lane + 32 * h] = incl[h] - cnt[h];
        const int total = __shfl_sync(0xffffffffu, incl[1], 31);
        if (lane == 0) pre[groups] = total < kMaxSegStages || !kPaged ? total : kMaxSegStages;
    }
    if (tid == 0) {
        for (int k = 0; k < kNW * kSegNbuf; ++k) mbar_init(smem_u32(bars + k), 1);
        fence_barrier_init();
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    {
        constexpr int VPR = D * 2 / 16;
        const uint4* qg = reinterpret_cast<const uint4*>(p.q);
        for (int e = tid; e < S::MROWS * VPR; e += blockDim.x) {
            const int r = e / VPR, v = e % VPR;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (r < M) val = __ldg(qg + (static_cast<long long>(i) * p.Hq + hk * p.G + r) * VPR + v);
            *reinterpret_cast<uint4*>(qs + r * S::QSTRIDE + v * 16) = val;
        }
    }
    __syncthreads();  // segments, stage prefix, q rows and barriers are in place

    // stage list of this warp: fused mode takes stages round-robin over the
    // union; segment-output mode takes whole segments g = warp, warp + 4, ...
    // A cursor per walk (the copies issued ahead, the stages consumed) that
    // only moves forward: fused mode tracks the group of stage s (the union's
    // stages in order); segment-output mode the warp's current group and how
    // many of the warp's stages precede it.
    struct StageCursor {
        int g, before;
    };
    auto stage_of = [&](StageCursor& c, int k, int& g, int& sidx) {
        if constexpr (!kSegOut) {
            const int s = warp + k * kNW;
            while (c.g + 1 < groups && pre[c.g + 1] <= s) ++c.g;
            g = c.g;
            sidx = s - pre[g];
        } else {
            while (c.g < groups && k - c.before >= pre[c.g + 1] - pre[c.g]) {
                c.before += pre[c.g + 1] - pre[c.g];
                c.g += kNW;
            }
            g = c.g;
            sidx = k - c.before;
        }
    };
    StageCursor issue_cur{kSegOut ? warp : 0, 0}, use_cur{kSegOut ? warp : 0, 0};
    int my_n = 0;
    if constexpr (!kSegOut) {
        const int total = pre[groups];
        my_n = total > warp ? (total - warp + kNW - 1) / kNW : 0;
    } else {
        for (int g = warp; g < groups; g += kNW) my_n += pre[g + 1] - pre[g];
    }

    // Contiguous segments: the last stage of a segment longer than one stage
    // whose length is not a multiple of 16 is moved back to end at the
    // segment's last used row; its first rows (read again, from L2) are masked
    // as already consumed.  No row past the used prefix is then read from
    // DRAM.  A segment shorter than a stage copies its used rows only.
    auto shifted = [&](int g, int sidx) {
        const int u = su[g];
        return !kPaged && u > kStageTok && (u % kStageTok) != 0 && sidx == (u - 1) / kStageTok;
    };
    auto stage_row = [&](int g, int sidx) { return shifted(g, sidx) ? su[g] - kStageTok : sidx * kStageTok; };

    uint8_t* ring_gen = smem + warp * kSegNbuf * S::STAGE;
    const uint32_t ring = smem_u32(ring_gen);
    const uint32_t bar0 = smem_u32(bars + warp * kSegNbuf);
    const uint64_t pol = policy_evict_first();
    // Rows [r0, r1) of a stage copied row-exactly by the warp's 32 lanes, 16
    // bytes a lane, into the layout the 128-byte-swizzled copies give (16-byte
    // piece j of row r at ((j ^ (r & 7)) << 4) in its 128-byte chunk, the K
    // chunks then the V chunks); the other rows are zero-filled without a read.
    // The lanes' copies signal the stage's barrier on landing, lane 0 arrives.
    auto copy_rows = [&](uint32_t buf, uint32_t bar, const uint8_t* kb, const uint8_t* vb, long long rstride, int r0,
                         int r1) {
        constexpr int HP = D * 2 / 16;  // 16-byte pieces of a K (or V) row
        constexpr int PR = 2 * HP;      // of a stage row, K then V
        constexpr int RPP = 32 / PR;    // rows per pass of the warp
        const int pc = lane % PR, j = pc & 7;
        const uint8_t* src = (pc < HP ? kb : vb) + (pc % HP) * 16;
        const uint32_t dst = buf + (pc >> 3) * 2048;
#pragma unroll
        for (int it = 0; it < kStageTok / RPP; ++it) {
            const int row = it * RPP + lane / PR;
            const bool in = row >= r0 && row < r1;
            cp_async_16(dst + row * 128 + ((j ^ (row & 7)) << 4), src + (in ? row : r0) * rstride, in ? 16 : 0, pol);
        }
        cp_async_mbar_arrive(bar);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
    };
    // Called by all 32 lanes.  A stage the segment covers whole is one TMA copy
    // (two per half in the contiguous mode) issued by lane 0; a stage it covers
    // in part is copied row-exactly: in the paged mode a segment's first or
    // last stage, in the contiguous mode a segment shorter than a stage.
    auto issue = [&](int k) {
        int g, sidx;
        stage_of(issue_cur, k, g, sidx);
        const uint32_t buf = ring + (k % kSegNbuf) * S::STAGE;
        const uint32_t bar = bar0 + 8 * (k % kSegNbuf);
        if constexpr (kPaged) {
            const int pg = spage[pre[g] + sidx];
            if (pg < 0) {
                if (lane == 0) mbar_arrive(bar);
                return;
            }
            const int tok0 = sa[g] + sidx * kStageTok;
            const int crow = (pg * p.Hkv + hk) * p.P + (tok0 - seg_page_col(p, tok0) * p.P);
            const int r0 = max(0, ss[g] - tok0), r1 = min(kStageTok, ss[g] + su[g] - tok0);
            if (r0 > 0 || r1 < kStageTok) {
                const uint8_t* kb = static_cast<const uint8_t*>(p.k) + static_cast<long long>(crow) * (D * 4);
                copy_rows(buf, bar, kb, kb + D * 2, D * 4, r0, r1);  // a cache row: K then V
                return;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, S::STAGE);
                tma_load_3d(buf, &kmap, 0, crow, 0, bar, pol);
            }
            return;
        }
        const long long row = row_base + (g < p.topk ? static_cast<long long>(g) * p.bs : static_cast<long long>(p.topk) * p.bs) +
                              stage_row(g, sidx);
        if (su[g] < kStageTok) {
            const long long off = (row * p.Hkv + hk) * (D * 2);
            copy_rows(buf, bar, static_cast<const uint8_t*>(p.k) + off, static_cast<const uint8_t*>(p.v) + off,
                      static_cast<long long>(p.Hkv) * D * 2, 0, su[g]);
            return;
        }
        if (lane != 0) return;
        mbar_arrive_expect_tx(bar, S::STAGE);
#pragma unroll
        for (int bx = 0; bx < D * 2 / 128; ++bx) {
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(buf + bx * 2048),
                "l"(reinterpret_cast<uint64_t>(&kmap)), "r"(bx * 64), "r"(hk), "r"(static_cast<int>(row)), "r"(bar),
                "l"(pol)
                : "memory");
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
                " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(buf + S::HALF + bx * 2048),
                "l"(reinterpret_cast<uint64_t>(&vmap)), "r"(bx * 64), "r"(hk), "r"(static_cast<int>(row)), "r"(bar),
                "l"(pol)
                : "memory");
        }
    };
    if constexpr (kPaged) {
        // page of each of this warp's stages, looked up once so that no TMA
        // issue waits on the table; a warp reads only its own stages' pages
        for (int k = lane; k < my_n; k += 32) {
            int g, sidx;
            if constexpr (!kSegOut) {
                const int s2 = warp + k * kNW;
                g = 0;
                while (g + 1 < groups && pre[g + 1] <= s2) ++g;
                sidx = s2 - pre[g];
            } else {
                int before = 0;
                g = warp;
                while (g < groups && k - before >= pre[g + 1] - pre[g]) {
                    before += pre[g + 1] - pre[g];
                    g += kNW;
                }
                sidx = k - before;
            }
            const int tok0 = sa[g] + sidx * kStageTok;
            const int pg = p.block_table[static_cast<long long>(i) * p.bt_stride + seg_page_col(p, tok0)];
            spage[pre[g] + sidx] = (pg < 0 || pg >= p.num_pages) ? -1 : pg;
        }
        __syncwarp();
    }
    for (int k = 0; k < kSegNbuf && k < my_n; ++k) issue(k);

    MmaWarp<D, kBF16, 1, NT> wp;
    wp.load_q(smem_u32(qs), S::QSTRIDE, lane);
    wp.reset();
    const int g_lane = lane >> 2, tg = lane & 3;

    // segment-output mode: write (o_g, lse_g) of the segment the warp just finished
    auto emit_segment = [&](int g) {
        wp.reduce_l();
        float lcol[NT][2];
        wp.column_rows_stat(wp.l_run, lcol, lane);
        const long long sbase = (static_cast<long long>(i) * groups + g) * p.Hq + hk * p.G;
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int r = n * 8 + 2 * tg + (c & 1);
                    const int d = dt * 16 + g_lane + (c >> 1) * 8;
                    const float l = lcol[n][c & 1];
                    if (r < M && p.seg_out) p.seg_out[(sbase + r) * D + d] = l > 0.f ? wp.oacc[dt][n][c] / l : 0.f;
                }
        if (tg == 0 && p.seg_lse)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = h * 8 + g_lane;
                const float l = wp.l_run[0][h];
                if (r < M) p.seg_lse[sbase + r] = l > 0.f ? (wp.m_run[0][h] + __log2f(l)) * kLn2 : -INFINITY;
            }
        wp.reset();
    };

    int timed_out = 0, consumed = 0;
    for (int k = 0; k < my_n; ++k) {
        const int buf = k % kSegNbuf;
        if (!mbar_wait(bar0 + 8 * buf, (k / kSegNbuf) & 1)) {
            timed_out = 1;
            break;
        }
        consumed = k + 1;
        int g, sidx;
        stage_of(use_cur, k, g, sidx);
        // keys [lo, nvalid) of this stage belong to the segment
        int nvalid, lo = 0;
        if constexpr (kPaged) {
            const int tok0 = sa[g] + sidx * kStageTok;
            nvalid = min(kStageTok, ss[g] + su[g] - tok0);
            lo = ss[g] - tok0;
            if (spage[pre[g] + sidx] < 0) nvalid = 0;
        } else if (shifted(g, sidx)) {
            nvalid = kStageTok;
            lo = sidx * kStageTok - stage_row(g, sidx);  // rows the previous stage already took
        } else {
            nvalid = min(kStageTok, su[g] - sidx * kStageTok);
        }
        const uint32_t st = ring + buf * S::STAGE;
        // a stage of a missing page holds stale values: P.V must not meet them
        // (masked keys weigh 0, and 0 * NaN is not 0); a partial stage's rows
        // outside the segment were zero-filled by its copies
        if (nvalid == 0) zero_tail_v<D, 2>(ring_gen + buf * S::STAGE, 0, lane);
        {
            // Q.K^T in two accumulation chains (kSplitQK)
            const float bias2 = kSegOut ? 0.f : sb[g];
            auto visible = [&](int row, int kt) { return row < M && kt >= lo; };
            if (nvalid < kStageTok || lo > 0)
                wp.template consume<true, true>(st, S::HALF, nvalid, p.scale_log2, bias2, visible, lane);
            else
                wp.template consume<false, true>(st, S::HALF, nvalid, p.scale_log2, bias2, visible, lane);
        }
        __syncwarp();
        if (k + kSegNbuf < my_n) {
            fence_proxy_async();
            issue(k + kSegNbuf);
        }
        if constexpr (kSegOut) {
            if (sidx + 1 >= pre[g + 1] - pre[g]) emit_segment(g);
        }
    }
    if (timed_out) {
        // this ABI has no status word: the warp stops, lets its other copies land
        // and leaves its share of the result incomplete
        for (int k = consumed; k < my_n && k < consumed + kSegNbuf; ++k)
            mbar_wait(bar0 + 8 * (k % kSegNbuf), (k / kSegNbuf) & 1);
    }

    if constexpr (kSegOut) {
        // empty segments of this warp: o = 0, lse = -inf
        for (int g = warp; g < groups; g += kNW) {
            if (su[g] > 0) continue;
            const long long sbase = (static_cast<long long>(i) * groups + g) * p.Hq + hk * p.G;
            if (p.seg_out)
                for (int e = lane; e < M * D; e += 32) p.seg_out[sbase * D + e] = 0.f;
            if (p.seg_lse)
                for (int r = lane; r < M; r += 32) p.seg_lse[sbase + r] = -INFINITY;
        }
        return;
    } else {
        wp.reduce_l();
        __syncthreads();
        float* O = reinterpret_cast<float*>(smem);
        wp.store(O + warp * S::MROWS * S::OSTRIDE, wm + warp * S::MROWS, wl + warp * S::MROWS, S::OSTRIDE, lane);
        __syncthreads();
        for (int e = tid; e < M * D; e += blockDim.x) {
            const int r = e / D, d = e % D;
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < kNW; ++k) mx = fmaxf(mx, wm[k * S::MROWS + r]);
            float lsum = 0.f, o = 0.f;
            if (mx != -INFINITY) {
#pragma unroll
                for (int k = 0; k < kNW; ++k) {
                    const float s = fast_exp2(wm[k * S::MROWS + r] - mx);
                    lsum += wl[k * S::MROWS + r] * s;
                    o += O[(k * S::MROWS + r) * S::OSTRIDE + d] * s;
                }
            }
            const float v = lsum > 0.f ? o / lsum : 0.f;
            const long long idx = (static_cast<long long>(i) * p.Hq + hk * p.G + r) * D + d;
            if (kBF16)
                reinterpret_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
            else
                reinterpret_cast<__half*>(p.out)[idx] = __float2half_rn(v);
        }
    }
}

// One warp per (row n, head h): out = sum over live parts of
// exp(lse_p + prior_p - lse) * part_out_p, lse = ln sum exp(lse_p + prior_p).
__global__ void __launch_bounds__(128) lse_merge_kernel(const MergeParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long rowid = static_cast<long long>(blockIdx.x) * 4 + warp;
    if (rowid >= static_cast<long long>(p.n) * p.heads) return;
    const long long nn = rowid / p.heads;
    const int h = static_cast<int>(rowid % p.heads);
    auto logit = [&](int s) -> float {
        if (p.live && p.live[nn * p.parts + s] <= 0) return -INFINITY;
        float v = p.part_lse[(nn * p.parts + s) * p.heads + h];
        if (p.prior && s < p.prior_cols) v += p.prior[nn * p.prior_cols + s];
        return v;
    };
    float mx = -INFINITY;
    for (int s = lane; s < p.parts; s += 32) mx = fmaxf(mx, logit(s));
    mx = warp_max(mx);
    constexpr int KD = 8;  // D <= 256
    float acc[KD];
#pragma unroll
    for (int k = 0; k < KD; ++k) acc[k] = 0.f;
    float total = -INFINITY;
    if (mx != -INFINITY) {
        float sum = 0.f;
        for (int s = lane; s < p.parts; s += 32) {
            const float lg = logit(s);
            if (lg != -INFINITY) sum += fast_exp2((lg - mx) * kLog2e);
        }
        sum = warp_sum(sum);
        total = mx + __logf(sum);
        for (int s = 0; s < p.parts; ++s) {
            const float lg = logit(s);
            if (lg == -INFINITY) continue;
            const float wgt = fast_exp2((lg - total) * kLog2e);
            const float* src = p.part_out + ((nn * p.parts + s) * p.heads + h) * p.D;
#pragma unroll
            for (int k = 0; k < KD; ++k) {
                const int d = lane + 32 * k;
                if (d < p.D) acc[k] = fmaf(wgt, src[d], acc[k]);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < KD; ++k) {
        const int d = lane + 32 * k;
        if (d < p.D) store_out(p.out, (nn * p.heads + h) * p.D + d, acc[k], p.out_dtype);
    }
    if (lane == 0 && p.lse_out) p.lse_out[nn * p.heads + h] = total;
}

template <int D, bool kBF16, int NT, bool kSegOut, bool kPaged>
static cudaError_t launch_seg_paged(const SegmentParams& p, cudaStream_t stream) {
    using S = SegShape<D, NT>;
    auto kern = segmented_kernel<D, kBF16, NT, kSegOut, kPaged>;
    static PerDevice state;
    cudaError_t e = kernel_setup(state, kern, kNW * 32, S::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<dim3(p.n, p.Hkv), kNW * 32, S::SMEM, stream>>>(p.kmap, p.vmap, p);
    return cudaGetLastError();
}

template <int D, bool kBF16, int NT, bool kSegOut>
static cudaError_t launch_seg_one(const SegmentParams& p, cudaStream_t stream) {
    return p.paged ? launch_seg_paged<D, kBF16, NT, kSegOut, true>(p, stream)
                   : launch_seg_paged<D, kBF16, NT, kSegOut, false>(p, stream);
}

template <int D, bool kBF16, bool kSegOut>
static cudaError_t launch_seg_nt(const SegmentParams& p, cudaStream_t stream) {
    return p.G <= 8 ? launch_seg_one<D, kBF16, 1, kSegOut>(p, stream) : launch_seg_one<D, kBF16, 2, kSegOut>(p, stream);
}

template <bool kSegOut>
static cudaError_t launch_seg_mode(const SegmentParams& p, cudaStream_t stream) {
    if (p.D == 128)
        return p.bf16 ? launch_seg_nt<128, true, kSegOut>(p, stream) : launch_seg_nt<128, false, kSegOut>(p, stream);
    return p.bf16 ? launch_seg_nt<64, true, kSegOut>(p, stream) : launch_seg_nt<64, false, kSegOut>(p, stream);
}

cudaError_t launch_segmented(const SegmentParams& p, cudaStream_t stream) {
    if (p.topk + 1 > kMaxGroups) return cudaErrorInvalidValue;
    if (!p.seg_out && !p.seg_lse) return launch_seg_mode<false>(p, stream);
    // per-segment results, then the combine as an LSE merge over segments
    cudaError_t e = launch_seg_mode<true>(p, stream);
    if (e != cudaSuccess) return e;
    MergeParams m;
    m.part_out = p.seg_out;
    m.part_lse = p.seg_lse;
    m.prior = p.bias;
    m.prior_cols = p.topk;
    m.live = p.used;
    m.n = p.n;
    m.parts = p.topk + 1;
    m.heads = p.Hq;
    m.D = p.D;
    m.out = p.out;
    m.out_dtype = p.bf16 ? 0 : 1;
    m.lse_out = nullptr;
    return launch_lse_merge(m, stream);
}

cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.n) * p.heads;
    if (rows == 0) return cudaSuccess;
    lse_merge_kernel<<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkd
