// CUDA-core paged decode for small M (M = sq * Hq/Hkv <= 8), fp32 FMA.
//
// Same TMA stage ring as the tensor-core kernel.  Inside a warp, LPT lanes
// share one key: each lane owns EPL elements of the head dimension (whole
// 16-byte chunks of the swizzled stage, or halves of them), so
//   q.k  is EPL FMAs per row followed by a reduce-scatter over the LPT lanes
//        (each lane ends with the full logit of one row),
//   p*V  accumulates into a per-lane [M][EPL] slice with no reduction until
//        the very end (the 32/LPT keys in flight are summed once per CTA).
// Softmax runs per 16-key stage in fp32 (exp2 domain, scale folded into q).
#pragma once

#include "fma_warp.cuh"

namespace pkd {

template <int D, int KVT, int LPT, int MR, int NBUF>
struct FmaShape {
    using G = FmaGeom<D, KVT, LPT, MR>;
    static constexpr int STAGE = G::STAGE;
    static constexpr int OSTRIDE = D + 4;
    static constexpr int RING = kNW * NBUF * STAGE;
    static constexpr int MERGE = kNW * MR * OSTRIDE * 4;
    static constexpr int BIG = RING > MERGE ? RING : MERGE;
    static constexpr int OFF_BARS = BIG;
    static constexpr int OFF_PAGES = OFF_BARS + kNW * NBUF * 8;
    static constexpr int OFF_ML = OFF_PAGES + kMaxCtaPages * 4;
    static constexpr int OFF_FLAG = OFF_ML + 2 * kNW * MR * 4;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;
};

// One CTA per (request, kv head, Split-KV chunk); four warps take the chunk's
// stages round-robin and merge in shared memory at the end.
template <int D, int KVT, int LPT, int MR, int NBUF>
__global__ void __launch_bounds__(kNW * 32)
decode_fma_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    using S = FmaShape<D, KVT, LPT, MR, NBUF>;
    constexpr int ELT = S::G::ELT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
    int* pages = reinterpret_cast<int*>(smem + S::OFF_PAGES);
    float* wm = reinterpret_cast<float*>(smem + S::OFF_ML);
    float* wl = wm + kNW * MR;
    int* flag = reinterpret_cast<int*>(smem + S::OFF_FLAG);

    CtaWork w;
    if (!cta_setup<D>(p, w)) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        prefetch_tmap(&tmap);
        for (int i = 0; i < kNW * NBUF; ++i) mbar_init(smem_u32(bars + i), 1);
        fence_barrier_init();
    }
    load_cta_pages(p, w, pages);
    __syncthreads();

    const int nst = (w.t1 - w.t0 + kStageTok - 1) / kStageTok;
    const int my_n = nst > warp ? (nst - warp + kNW - 1) / kNW : 0;
    uint8_t* ring_gen = smem + warp * NBUF * S::STAGE;
    const uint32_t ring = smem_u32(ring_gen);
    const uint32_t bar0 = smem_u32(bars + warp * NBUF);
    const uint64_t pol = policy_evict_first();
    if (lane == 0)
        for (int k = 0; k < NBUF && k < my_n; ++k)
            issue_stage<D, ELT>(&tmap, p, w, pages, warp + k * kNW, ring + k * S::STAGE, bar0 + 8 * k, pol);

    FmaWarp<D, KVT, LPT, MR> wp;
    wp.init(lane);
    wp.load_q(p, w.b, w.hk, lane);
    wp.reset();
    const int L = w.L;

    int timed_out = 0, consumed = 0;
    for (int k = 0; k < my_n; ++k) {
        const int buf = k % NBUF;
        if (!mbar_wait(bar0 + 8 * buf, (k / NBUF) & 1, p.status, p.wait_ns)) {
            timed_out = 1;
            break;
        }
        consumed = k + 1;
        const int stage = warp + k * kNW;
        const int tok0 = w.t0 + stage * kStageTok;
        int nvalid = min(kStageTok, w.t1 - tok0);
        if (page_of(p, w, pages, tok0) < 0) nvalid = 0;
        uint8_t* st = ring_gen + buf * S::STAGE;
        if (nvalid < kStageTok) zero_tail_v<D, ELT>(st, nvalid, lane);
        wp.consume(st, nvalid, [&](int row, int kt) { return row_sees(p, L, row, tok0 + kt); }, lane);
        __syncwarp();
        if (lane == 0 && k + NBUF < my_n) {
            fence_proxy_async();
            issue_stage<D, ELT>(&tmap, p, w, pages, warp + (k + NBUF) * kNW, ring + buf * S::STAGE,
                                bar0 + 8 * buf, pol);
        }
    }
    if (timed_out) {
        if (lane == 0) raise_status(p, kErrTimeout);
        for (int k = consumed; k < my_n && k < consumed + NBUF; ++k)
            mbar_wait(bar0 + 8 * (k % NBUF), (k / NBUF) & 1);
    }

    wp.finish();
    __syncthreads();
    float* O = reinterpret_cast<float*>(smem);
    wp.store(O + warp * MR * S::OSTRIDE, wm + warp * MR, wl + warp * MR, S::OSTRIDE, lane);
    __syncthreads();
    cta_finish<D, S::OSTRIDE>(p, w, O, wm, wl, MR, flag);
}

}  // namespace pkd
