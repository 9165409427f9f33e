// Tensor-core paged decode (mma.sync m16n8k16, fp32 accumulate).
//
// The GQA group and the query block are folded into one M dimension of
// M = sq * Hq/Hkv query rows per (request, kv head).  Per 16-key stage:
//   S   = Q K^T     A = Q (M padded to 16-row tiles, fragments from shared
//                   memory), B = K straight from the swizzled TMA stage
//   P   = online-softmax(S) in fp32, rounded to the operand type
//   O^T += V^T P^T  "swapped" so that M sits in the 8-wide N dimension: A = V^T
//                   (ldmatrix.trans of the stage), B = P^T, which is exactly
//                   the accumulator layout of S -- no shuffles between the
//                   two products, and rows only pad to a multiple of 8.
// Keys arrive through a per-warp ring of NBUF stages filled by 2-D TMA tile
// loads (128-byte swizzle) addressed by the block table, so K and V are read
// from the cache's own [pages, Hkv, P, 2*D] layout without any repacking.
#pragma once

#include "fp8_warp.cuh"
#include "mma_warp.cuh"

namespace pkd {

// Shared memory of a grid CTA: NW rings of NBUF stages (reused for the warps'
// O at the end), barriers, the page list, the q rows staged for the warps
// (W::kCtaQ), per-warp row statistics and per-warp scratch (W::kScratchBytes).
template <class W, int D, int ELT, int NBUF, int NW = kNW>
struct MmaShape {
    static constexpr int KBOX = D * ELT / 128;
    static constexpr int HALF = KBOX * 2048;
    static constexpr int STAGE = 2 * HALF;
    static constexpr int MROWS = W::MROWS;
    static constexpr int QSTRIDE = D * 2 + 16;           // bytes per staged q row
    static constexpr int OSTRIDE = D + 4;                // floats per merge row
    static constexpr int RING = NW * NBUF * STAGE;
    static constexpr int MERGE = NW * MROWS * OSTRIDE * 4;
    static constexpr int BIG = RING > MERGE ? RING : MERGE;
    static constexpr int OFF_SCR = BIG;                  // per-warp scratch, 1 KiB granules
    static constexpr int OFF_BARS = OFF_SCR + NW * W::kScratchBytes;
    static constexpr int OFF_PAGES = OFF_BARS + NW * NBUF * 8;
    static constexpr int OFF_Q = OFF_PAGES + kMaxCtaPages * 4;
    static constexpr int OFF_ML = OFF_Q + (W::kCtaQ ? MROWS * QSTRIDE : 0);
    static constexpr int OFF_FLAG = OFF_ML + 2 * NW * MROWS * 4;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;    // + slack to align the base to 1 KiB
};

// Without a window a chunk's first key is split * chunk whatever the
// request's length, so the chunk's block-table entries can be read while the
// length itself is read: the page list is then ready one memory round trip
// earlier.  Entries are validated once the length is known; columns at or
// past ceil(max_kv_len / P) are never read.
template <int NTHREADS>
struct SpecPages {
    static constexpr int PER = (kMaxCtaPages + NTHREADS - 1) / NTHREADS;
    int ent[PER];
    bool on = false;
    __device__ __forceinline__ void load(const DecodeParams& p) {
        on = p.window <= 0;
        if (!on) return;
        const int b = blockIdx.z, col0 = blockIdx.x * (p.chunk / p.P);
        const int cols = (p.max_kv_len + p.P - 1) / p.P;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int i = threadIdx.x + j * NTHREADS;
            ent[j] = (i < p.chunk / p.P && col0 + i < cols)
                         ? p.block_table[static_cast<long long>(b) * p.bt_stride + col0 + i] : -1;
        }
    }
    // the page list of [w.t0, w.t1) (w.t0 = split * chunk here)
    __device__ __forceinline__ void store(const DecodeParams& p, const CtaWork& w, int* pages) const {
        const int npages = (w.t1 - 1) / p.P - w.t0 / p.P + 1;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int i = threadIdx.x + j * NTHREADS;
            if (i < npages) {
                int pg = ent[j];
                if (pg < 0 || pg >= p.num_pages) {
                    raise_status(p, kErrBounds);
                    pg = -1;
                }
                pages[i] = pg;
            }
        }
    }
};

// W: MmaWarp (16-bit caches; q rows staged once for the CTA's warps) or
// Fp8MmaWarp (e4m3 caches; q fragments loaded by each warp, V widened in the
// warp's scratch).
template <class W, int D, int ELT, int NBUF, int NW = kNW>
__global__ void __launch_bounds__(NW * 32, W::kMinBlocks)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    using S = MmaShape<W, D, ELT, NBUF, NW>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
    int* pages = reinterpret_cast<int*>(smem + S::OFF_PAGES);
    uint8_t* qs = smem + S::OFF_Q;
    float* wm = reinterpret_cast<float*>(smem + S::OFF_ML);
    float* wl = wm + NW * S::MROWS;
    int* flag = reinterpret_cast<int*>(smem + S::OFF_FLAG);

    // Start-up in one memory round trip: the chunk's table entries (no
    // window), the q rows and the request's length are read at once; each
    // warp then sets up its own barriers and issues its first copies before
    // the CTA barrier that publishes the page list and q.
    constexpr int VPR = D * 2 / 16;  // 16-byte vectors per q row
    constexpr int QPER = W::kCtaQ ? (S::MROWS * VPR + NW * 32 - 1) / (NW * 32) : 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    SpecPages<NW * 32> spec;
    spec.load(p);
    uint4 qv[QPER];
    if constexpr (W::kCtaQ) {
        const uint4* qg = reinterpret_cast<const uint4*>(p.q);
        const int b = blockIdx.z, hk = blockIdx.y;
#pragma unroll
        for (int j = 0; j < QPER; ++j) {
            const int e = tid + j * NW * 32, r = e / VPR, v = e % VPR;
            qv[j] = make_uint4(0u, 0u, 0u, 0u);
            if (e < S::MROWS * VPR && r < p.M) {
                const int i = r / p.G, g = r % p.G;
                qv[j] = __ldg(qg + ((static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g) * VPR + v);
            }
        }
    }
    CtaWork w;
    if (!cta_setup<D>(p, w)) return;

    const int nst = (w.t1 - w.t0 + kStageTok - 1) / kStageTok;
    const int my_n = nst > warp ? (nst - warp + NW - 1) / NW : 0;
    uint8_t* ring_gen = smem + warp * NBUF * S::STAGE;
    const uint32_t ring = smem_u32(ring_gen);
    const uint32_t bar0 = smem_u32(bars + warp * NBUF);
    const uint64_t pol = policy_evict_first();
    if (lane == 0) {
        // a warp's barriers serve its own ring only
        if (warp == 0) prefetch_tmap(&tmap);
        for (int k = 0; k < NBUF; ++k) mbar_init(bar0 + 8 * k, 1);
        fence_barrier_init();
        for (int k = 0; k < NBUF && k < my_n; ++k) {
            const int tok = w.t0 + (warp + k * NW) * kStageTok;
            const int pg = p.block_table[static_cast<long long>(w.b) * p.bt_stride + page_col(p, tok)];
            const uint32_t bar = bar0 + 8 * k;
            if (pg < 0 || pg >= p.num_pages) {  // skipped; reported when the page list is built
                mbar_arrive(bar);
                continue;
            }
            mbar_arrive_expect_tx(bar, S::STAGE);
            tma_load_3d(ring + k * S::STAGE, &tmap, 0, (pg * p.Hkv + w.hk) * p.P + page_slot(p, tok), 0, bar, pol);
        }
    }
    if (spec.on)
        spec.store(p, w, pages);
    else
        load_cta_pages(p, w, pages);
    if constexpr (W::kCtaQ) {
#pragma unroll
        for (int j = 0; j < QPER; ++j) {
            const int e = tid + j * NW * 32, r = e / VPR, v = e % VPR;
            if (e < S::MROWS * VPR) *reinterpret_cast<uint4*>(qs + r * S::QSTRIDE + v * 16) = qv[j];
        }
    }
    __syncthreads();

    W wp;
    wp.setup(smem + S::OFF_SCR + warp * W::kScratchBytes);
    if constexpr (W::kCtaQ)
        wp.load_q(smem_u32(qs), S::QSTRIDE, lane);
    else
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
        const int stage = warp + k * NW;
        const int tok0 = w.t0 + stage * kStageTok;
        int nvalid = min(kStageTok, w.t1 - tok0);
        if (page_of(p, w, pages, tok0) < 0) nvalid = 0;
        const uint32_t st = ring + buf * S::STAGE;
        if (nvalid < kStageTok) zero_tail_v<D, ELT>(ring_gen + buf * S::STAGE, nvalid, lane);
        wp.consume(st, S::HALF, nvalid, nvalid < kStageTok || p.causal, p.scale_log2, 0.f,
                   [&](int row, int kt) { return row_sees(p, L, row, tok0 + kt); }, lane);
        __syncwarp();
        if (lane == 0 && k + NBUF < my_n) {
            fence_proxy_async();
            issue_stage<D, ELT>(&tmap, p, w, pages, warp + (k + NBUF) * NW, st, bar0 + 8 * buf, pol);
        }
    }
    if (timed_out) {
        // let this warp's copies land before the CTA leaves or reuses the ring:
        // stages consumed .. consumed + NBUF - 1 were issued (the first is the
        // one whose wait gave up)
        if (lane == 0) raise_status(p, kErrTimeout);
        for (int k = consumed; k < my_n && k < consumed + NBUF; ++k)
            mbar_wait(bar0 + 8 * (k % NBUF), (k / NBUF) & 1);
    }

    // ---- per-warp state to shared memory (the ring is reused for O)
    wp.reduce_l();
    __syncthreads();
    float* O = reinterpret_cast<float*>(smem);
    wp.store(O + warp * S::MROWS * S::OSTRIDE, wm + warp * S::MROWS, wl + warp * S::MROWS, S::OSTRIDE, lane);
    __syncthreads();
    cta_finish<D, S::OSTRIDE, NW>(p, w, O, wm, wl, S::MROWS, flag);
}

// Query blocks of 17..32 rows (M = sq * Hq/Hkv).  One warp holding both
// 16-row tiles needs two CTAs' worth of registers per SM and twice the tensor
// work per stage; instead the four warps form two pairs.  The warps of a pair
// hold rows [0, 16) and [16, 32) and consume the same stages from one shared
// ring (pair p takes stages p, p + 2, ...), so every stage is loaded once and
// each warp does half the tensor work.  A buffer is refilled once both warps
// of its pair have arrived on its "empty" barrier (count 2); the pair's first
// warp issues the copies.  The pairs' states are merged like the warps' of
// the one-warp kernel.
template <int D, int NBUF>
struct PairShape {
    static constexpr int KBOX = D * 2 / 128;
    static constexpr int HALF = KBOX * 2048;
    static constexpr int STAGE = 2 * HALF;
    static constexpr int PAIRS = kNW / 2;
    static constexpr int MROWS = 32;
    static constexpr int QSTRIDE = D * 2 + 16;
    static constexpr int OSTRIDE = D + 4;
    static constexpr int RING = PAIRS * NBUF * STAGE;
    static constexpr int MERGE = PAIRS * MROWS * OSTRIDE * 4;
    static constexpr int BIG = RING > MERGE ? RING : MERGE;
    static constexpr int OFF_BARS = BIG;                        // full[PAIRS][NBUF], then empty[PAIRS][NBUF]
    static constexpr int OFF_PAGES = OFF_BARS + 2 * PAIRS * NBUF * 8;
    static constexpr int OFF_Q = 0;                             // q rows staged in the ring before any copy
    static constexpr int OFF_ML = OFF_PAGES + kMaxCtaPages * 4;
    static constexpr int OFF_FLAG = OFF_ML + 2 * PAIRS * MROWS * 4;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;           // three CTAs per SM
    static_assert(MROWS * QSTRIDE <= RING, "q rows fit the ring");
};

template <int D, bool kBF16, int NBUF>
__global__ void __launch_bounds__(kNW * 32, 3)  // three CTAs per SM fit the shared memory
decode_mma_pair_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    using S = PairShape<D, NBUF>;
    using W = MmaWarp<D, kBF16, 1, 2>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
    int* pages = reinterpret_cast<int*>(smem + S::OFF_PAGES);
    uint8_t* qs = smem + S::OFF_Q;
    float* wm = reinterpret_cast<float*>(smem + S::OFF_ML);
    float* wl = wm + S::PAIRS * S::MROWS;
    int* flag = reinterpret_cast<int*>(smem + S::OFF_FLAG);

    SpecPages<kNW * 32> spec;
    spec.load(p);
    CtaWork w;
    if (!cta_setup<D>(p, w)) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pair = warp >> 1, half = warp & 1;
    if (tid == 0) {
        prefetch_tmap(&tmap);
        for (int i = 0; i < S::PAIRS * NBUF; ++i) {
            mbar_init(smem_u32(bars + i), 1);                         // full: the copy's bytes
            mbar_init(smem_u32(bars + S::PAIRS * NBUF + i), 2);       // empty: both warps of the pair
        }
        fence_barrier_init();
    }
    if (spec.on)
        spec.store(p, w, pages);
    else
        load_cta_pages(p, w, pages);
    {
        constexpr int VPR = D * 2 / 16;
        const uint4* qg = reinterpret_cast<const uint4*>(p.q);
        for (int e = tid; e < S::MROWS * VPR; e += blockDim.x) {
            const int r = e / VPR, v = e % VPR;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (r < p.M) {
                const int i = r / p.G, g = r % p.G;
                const long long row = (static_cast<long long>(w.b) * p.sq + i) * p.Hq + w.hk * p.G + g;
                val = __ldg(qg + row * VPR + v);
            }
            *reinterpret_cast<uint4*>(qs + r * S::QSTRIDE + v * 16) = val;
        }
    }
    __syncthreads();

    const int nst = (w.t1 - w.t0 + kStageTok - 1) / kStageTok;
    const int my_n = nst > pair ? (nst - pair + S::PAIRS - 1) / S::PAIRS : 0;
    uint8_t* ring_gen = smem + pair * NBUF * S::STAGE;
    const uint32_t ring = smem_u32(ring_gen);
    const uint32_t full0 = smem_u32(bars + pair * NBUF);
    const uint32_t empty0 = smem_u32(bars + S::PAIRS * NBUF + pair * NBUF);
    const bool producer = half == 0 && lane == 0;
    const uint64_t pol = policy_evict_first();

    W wp;
    wp.row0 = half * 16;
    wp.load_q(smem_u32(qs) + half * 16 * S::QSTRIDE, S::QSTRIDE, lane);  // into registers
    wp.reset();
    fence_proxy_async();  // the q rows were written (generic proxy) where the copies land
    __syncthreads();      // every warp has its q fragments: the ring may be filled
    if (producer) {
        for (int k = 0; k < NBUF && k < my_n; ++k)
            issue_stage<D, 2>(&tmap, p, w, pages, pair + k * S::PAIRS, ring + k * S::STAGE, full0 + 8 * k, pol);
    }
    const int L = w.L, row0 = half * 16;

    int timed_out = 0, consumed = 0;
    for (int k = 0; k < my_n; ++k) {
        const int buf = k % NBUF;
        const uint32_t parity = (k / NBUF) & 1;
        if (!mbar_wait(full0 + 8 * buf, parity, p.status, p.wait_ns)) {
            timed_out = 1;
            break;
        }
        consumed = k + 1;
        const int tok0 = w.t0 + (pair + k * S::PAIRS) * kStageTok;
        int nvalid = min(kStageTok, w.t1 - tok0);
        if (page_of(p, w, pages, tok0) < 0) nvalid = 0;
        const uint32_t st = ring + buf * S::STAGE;
        // both warps zero the same tail rows (the same zeros: benign)
        if (nvalid < kStageTok) zero_tail_v<D, 2>(ring_gen + buf * S::STAGE, nvalid, lane);
        wp.consume(st, S::HALF, nvalid, nvalid < kStageTok || p.causal, p.scale_log2, 0.f,
                   [&](int row, int kt) { return row_sees(p, L, row0 + row, tok0 + kt); }, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * buf);
        if (producer && k + NBUF < my_n) {
            // both warps are done with this buffer: refill it
            if (!mbar_wait(empty0 + 8 * buf, parity, p.status)) {
                timed_out = 1;
            } else {
                fence_proxy_async();
                issue_stage<D, 2>(&tmap, p, w, pages, pair + (k + NBUF) * S::PAIRS, st, full0 + 8 * buf, pol);
            }
        }
        if (__shfl_sync(kFull, timed_out, 0)) break;
    }
    if (timed_out) {
        // let this pair's other copies land before the CTA leaves or reuses the ring
        if (lane == 0) raise_status(p, kErrTimeout);
        for (int k = consumed; k < my_n && k < consumed + NBUF; ++k)
            mbar_wait(full0 + 8 * (k % NBUF), (k / NBUF) & 1);
    }

    // ---- per-pair states to shared memory (the ring is reused for O)
    wp.reduce_l();
    __syncthreads();
    float* O = reinterpret_cast<float*>(smem);
    wp.store(O + (pair * S::MROWS + row0) * S::OSTRIDE, wm + pair * S::MROWS + row0, wl + pair * S::MROWS + row0,
             S::OSTRIDE, lane);
    __syncthreads();
    cta_finish<D, S::OSTRIDE, S::PAIRS>(p, w, O, wm, wl, S::MROWS, flag);
}

}  // namespace pkd
