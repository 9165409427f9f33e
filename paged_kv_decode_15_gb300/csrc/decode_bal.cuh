// Persistent paged decode with an equal share of the key stream per CTA.
//
// All (request, kv head) units are laid end to end as one sequence of 16-key
// stages (unit (b, hk) holds ceil(visible_b / 16) stages, b-major).  The grid
// fills the GPU once and CTA c takes the contiguous slice
// [c*Stot/C, (c+1)*Stot/C), so every CTA streams the same bytes and the launch
// has no tail of unequal CTAs.  A slice is cut at unit boundaries into pieces;
// a piece is run like a chunk of the chunked grid (its stages are shared by
// the CTA's warps, whose states are merged in shared memory), and a unit
// shared by several CTAs is merged by LSE by the last of them to arrive, from
// two partial slots per CTA (one for the unit its slice starts in, one for the
// unit that continues past its end).  No CTA waits on another.
//
// Two bodies run a piece:
//   WarpsBody  M <= 16: four warps with a ring of two stages each, stage j of
//              the piece to warp j % 4;
//   PairBody   17..32 rows: two warp pairs, each with one ring of four stages
//              that both warps read (rows 0-15 and 16-31); a buffer is
//              refilled once both have arrived on its "empty" barrier.
#pragma once

#include "mma_warp.cuh"

namespace pkd {

constexpr int kBalMinStages = 16;                   // a CTA streams at least this many stages
constexpr int kBalMaxCtas = kFlatMaxWorkers / kNW;  // two partial slots per CTA in the workspace

template <int D, int NBUF, int MROWS_, int NS_, int NBARS, bool kQInRing>
struct BalShape {
    static constexpr int KBOX = D * 2 / 128;
    static constexpr int HALF = KBOX * 2048;
    static constexpr int STAGE = 2 * HALF;
    static constexpr int MROWS = MROWS_;
    static constexpr int NS = NS_;
    static constexpr int QSTRIDE = D * 2 + 16;
    static constexpr int OSTRIDE = D + 4;
    static constexpr int RING = NS * NBUF * STAGE;
    static constexpr int MERGE = NS * MROWS * OSTRIDE * 4;
    static constexpr int BIG = RING > MERGE ? RING : MERGE;
    static constexpr int OFF_BARS = BIG;
    static constexpr int OFF_PAGES = OFF_BARS + NBARS * 8;
    static constexpr int OFF_Q = kQInRing ? 0 : OFF_PAGES + kMaxCtaPages * 4;
    static constexpr int OFF_ML = kQInRing ? OFF_PAGES + kMaxCtaPages * 4 : OFF_Q + MROWS * QSTRIDE;
    static constexpr int OFF_FLAG = OFF_ML + 2 * NS * MROWS * 4;
    static constexpr int OFF_SCAN = OFF_FLAG + 16;  // [0..3] warp sums, [4..5] start, [6] abort
    static constexpr int SMEM = OFF_SCAN + 64 + 1024;
    static_assert(!kQInRing || MROWS * QSTRIDE <= RING, "q rows fit the ring");
};

// M <= 16: four warps, each its own ring; stage j of a piece goes to warp j % 4.
template <int D, bool kBF16, int NT>
struct WarpsBody {
    static constexpr int NBUF = 2;
    static constexpr bool kQInRing = false;
    using S = BalShape<D, NBUF, 16, kNW, kNW * NBUF, false>;
    MmaWarp<D, kBF16, 1, NT> wp;
    uint32_t uses = 0;  // this warp's ring uses so far (buffer and phase of the next)
    int warp, lane;

    __device__ WarpsBody(int w, int l) : warp(w), lane(l) {}
    static __device__ void init_barriers(uint64_t* bars) {
        for (int i = 0; i < kNW * NBUF; ++i) mbar_init(smem_u32(bars + i), 1);
    }
    __device__ void load_q(uint32_t qs) {
        wp.load_q(qs, S::QSTRIDE, lane);
        wp.reset();
    }

    // Fold keys [w.t0, w.t1) into this warp's state.  False if a wait timed out.
    __device__ bool stream(const CUtensorMap* tmap, const DecodeParams& p, const CtaWork& w, const int* pages,
                           uint8_t* smem, uint64_t* bars, uint64_t pol) {
        uint8_t* ring_gen = smem + warp * NBUF * S::STAGE;
        const uint32_t ring = smem_u32(ring_gen), bar0 = smem_u32(bars + warp * NBUF);
        const int nst = (w.t1 - w.t0 + kStageTok - 1) / kStageTok;
        const int my_n = nst > warp ? (nst - warp + kNW - 1) / kNW : 0;
        const uint32_t u0 = uses;
        uses = u0 + my_n;
        if (lane == 0) {
            fence_proxy_async();  // earlier generic accesses of the ring come before the copies
            for (int k = 0; k < NBUF && k < my_n; ++k) {
                const uint32_t buf = (u0 + k) % NBUF;
                issue_stage<D, 2>(tmap, p, w, pages, warp + k * kNW, ring + buf * S::STAGE, bar0 + 8 * buf, pol);
            }
        }
        const int L = w.L;
        for (int k = 0; k < my_n; ++k) {
            const uint32_t u = u0 + k, buf = u % NBUF;
            if (!mbar_wait(bar0 + 8 * buf, (u / NBUF) & 1, p.status, p.wait_ns)) {
                // let the issued copies (stages k .. k + NBUF - 1) land first
                if (lane == 0) raise_status(p, kErrTimeout);
                for (int j = k; j < my_n && j < k + NBUF; ++j)
                    mbar_wait(bar0 + 8 * ((u0 + j) % NBUF), ((u0 + j) / NBUF) & 1);
                return false;
            }
            const int tok0 = w.t0 + (warp + k * kNW) * kStageTok;
            int nvalid = min(kStageTok, w.t1 - tok0);
            if (page_of(p, w, pages, tok0) < 0) nvalid = 0;
            const uint32_t st = ring + buf * S::STAGE;
            if (nvalid < kStageTok) zero_tail_v<D, 2>(ring_gen + buf * S::STAGE, nvalid, lane);
            wp.consume(st, S::HALF, nvalid, nvalid < kStageTok || p.causal, p.scale_log2, 0.f,
                       [&](int row, int kt) { return row_sees(p, L, row, tok0 + kt); }, lane);
            __syncwarp();
            if (lane == 0 && k + NBUF < my_n) {
                fence_proxy_async();
                issue_stage<D, 2>(tmap, p, w, pages, warp + (k + NBUF) * kNW, st, bar0 + 8 * buf, pol);
            }
        }
        return true;
    }

    __device__ void store(float* O, float* wm, float* wl) {
        wp.reduce_l();
        wp.store(O + warp * S::MROWS * S::OSTRIDE, wm + warp * S::MROWS, wl + warp * S::MROWS, S::OSTRIDE, lane);
    }
};

// 17..32 rows: two warp pairs, each with one shared ring; pair p takes the
// piece's stages p, p + 2, ...; warp `half` of a pair holds rows 16*half..+15.
template <int D, bool kBF16>
struct PairBody {
    static constexpr int NBUF = 4;
    static constexpr int PAIRS = kNW / 2;
    static constexpr bool kQInRing = true;  // q rows are read into registers before any copy lands
    using S = BalShape<D, NBUF, 32, PAIRS, 2 * PAIRS * NBUF, true>;
    MmaWarp<D, kBF16, 1, 2> wp;
    uint32_t uses = 0;  // this pair's ring uses so far
    int warp, lane, pair, half;

    __device__ PairBody(int w, int l) : warp(w), lane(l), pair(w >> 1), half(w & 1) {}
    static __device__ void init_barriers(uint64_t* bars) {
        for (int i = 0; i < PAIRS * NBUF; ++i) {
            mbar_init(smem_u32(bars + i), 1);                 // full: the copy's bytes
            mbar_init(smem_u32(bars + PAIRS * NBUF + i), 2);  // empty: both warps of the pair
        }
    }
    __device__ void load_q(uint32_t qs) {
        wp.row0 = half * 16;
        wp.load_q(qs + half * 16 * S::QSTRIDE, S::QSTRIDE, lane);
        wp.reset();
    }

    __device__ bool stream(const CUtensorMap* tmap, const DecodeParams& p, const CtaWork& w, const int* pages,
                           uint8_t* smem, uint64_t* bars, uint64_t pol) {
        uint8_t* ring_gen = smem + pair * NBUF * S::STAGE;
        const uint32_t ring = smem_u32(ring_gen);
        const uint32_t full0 = smem_u32(bars + pair * NBUF);
        const uint32_t empty0 = smem_u32(bars + PAIRS * NBUF + pair * NBUF);
        const bool producer = half == 0 && lane == 0;
        const int nst = (w.t1 - w.t0 + kStageTok - 1) / kStageTok;
        const int my_n = nst > pair ? (nst - pair + PAIRS - 1) / PAIRS : 0;
        const uint32_t u0 = uses;
        uses = u0 + my_n;
        // every earlier use of these buffers was consumed by both warps before
        // the CTA barrier that precedes this call: no wait on "empty" here
        if (producer) {
            fence_proxy_async();
            for (int k = 0; k < NBUF && k < my_n; ++k) {
                const uint32_t buf = (u0 + k) % NBUF;
                issue_stage<D, 2>(tmap, p, w, pages, pair + k * PAIRS, ring + buf * S::STAGE, full0 + 8 * buf, pol);
            }
        }
        const int L = w.L, row0 = half * 16;
        int failed = 0;
        for (int k = 0; k < my_n; ++k) {
            const uint32_t u = u0 + k, buf = u % NBUF, parity = (u / NBUF) & 1;
            if (!mbar_wait(full0 + 8 * buf, parity, p.status, p.wait_ns)) {
                failed = 1;
            } else {
                const int tok0 = w.t0 + (pair + k * PAIRS) * kStageTok;
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
                    if (!mbar_wait(empty0 + 8 * buf, parity, p.status)) {
                        failed = 1;
                    } else {
                        fence_proxy_async();
                        issue_stage<D, 2>(tmap, p, w, pages, pair + (k + NBUF) * PAIRS, st, full0 + 8 * buf, pol);
                    }
                }
            }
            if (__shfl_sync(kFull, failed, 0)) {
                if (lane == 0) raise_status(p, kErrTimeout);
                for (int j = k; j < my_n && j < k + NBUF; ++j)
                    mbar_wait(full0 + 8 * ((u0 + j) % NBUF), ((u0 + j) / NBUF) & 1);
                return false;
            }
        }
        return true;
    }

    __device__ void store(float* O, float* wm, float* wl) {
        wp.reduce_l();
        const int r0 = pair * S::MROWS + half * 16;
        wp.store(O + r0 * S::OSTRIDE, wm + r0, wl + r0, S::OSTRIDE, lane);
    }
};

// Number of 16-key stages of a request of length L.
__device__ __forceinline__ int request_stages(const DecodeParams& p, int L) {
    return (L - visible_lo(p, L) + kStageTok - 1) / kStageTok;
}

// Stage the M query rows of (b, hk) (zero padding rows) for ldmatrix.
template <int D>
__device__ __forceinline__ void stage_q_rows_cta(const DecodeParams& p, int b, int hk, uint8_t* qs, int mrows,
                                                 int qstride) {
    constexpr int VPR = D * 2 / 16;  // 16-byte vectors per row
    const uint4* qg = reinterpret_cast<const uint4*>(p.q);
    for (int e = threadIdx.x; e < mrows * VPR; e += blockDim.x) {
        const int r = e / VPR, v = e % VPR;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.M) {
            const int i = r / p.G, g = r % p.G;
            val = __ldg(qg + ((static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g) * VPR + v);
        }
        *reinterpret_cast<uint4*>(qs + r * qstride + v * 16) = val;
    }
}

template <class Body, int D>
__global__ void __launch_bounds__(kNW * 32, 3)  // three CTAs per SM fit the shared memory
decode_bal_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    using S = typename Body::S;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BARS);
    int* pages = reinterpret_cast<int*>(smem + S::OFF_PAGES);
    uint8_t* qs = smem + S::OFF_Q;
    float* wm = reinterpret_cast<float*>(smem + S::OFF_ML);
    float* wl = wm + S::NS * S::MROWS;
    int* flag = reinterpret_cast<int*>(smem + S::OFF_FLAG);
    int* scan = reinterpret_cast<int*>(smem + S::OFF_SCAN);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B;
    if (tid == 0) {
        prefetch_tmap(&tmap);
        Body::init_barriers(bars);
        fence_barrier_init();
        scan[4] = -1;
        scan[6] = 0;
    }

    // ---- stages per request, block-wide exclusive scan
    const int per = (B + blockDim.x - 1) / blockDim.x;
    const int bb = min(B, tid * per), be = min(B, bb + per);
    int local = 0;
    for (int b = bb; b < be; ++b) local += request_stages(p, clamp_len(p, b, blockIdx.x == 0));
    int incl = local;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, m);
        if (lane >= m) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int k = 0; k < kNW; ++k) {
        base += k < warp ? scan[k] : 0;
        total += scan[k];
    }
    const int excl = base + incl - local;

    // ---- requests with no visible key: out = 0, lse = -inf
    for (int b = blockIdx.x; b < B; b += gridDim.x)
        if (request_stages(p, clamp_len(p, b, false)) == 0) write_empty_request<D>(p, b);

    // ---- this CTA's slice [f0, f1)
    const long long Hkv = p.Hkv;
    const long long Stot = static_cast<long long>(total) * Hkv;
    long long C = Stot / kBalMinStages;
    if (C > gridDim.x) C = gridDim.x;
    if (C < 1) C = 1;
    const long long c = blockIdx.x;
    if (Stot == 0 || c >= C) return;
    const long long f0 = c * Stot / C, f1 = (c + 1) * Stot / C;
    if (local > 0 && Hkv * excl <= f0 && f0 < Hkv * (excl + local)) {
        int run = excl;
        for (int b = bb; b < be; ++b) {
            const int cnt = request_stages(p, clamp_len(p, b, false));
            if (f0 < Hkv * (run + cnt)) {
                scan[4] = b;
                scan[5] = run;
                break;
            }
            run += cnt;
        }
    }
    __syncthreads();
    int b = scan[4];
    if (b < 0) {  // unreachable: the scan covers [0, Stot)
        if (tid == 0) raise_status(p, kErrBounds);
        return;
    }
    long long Fb = Hkv * scan[5];  // first stage of request b
    int L = clamp_len(p, b, false), lo = visible_lo(p, L), cnt = request_stages(p, L);
    auto owner = [&](long long f) { return ((f + 1) * C - 1) / Stot; };  // the CTA whose slice holds f

    Body body(warp, lane);
    const uint64_t pol = policy_evict_first();
    const int win = (kMaxCtaPages - 1) * p.P;  // keys whose pages always fit the page list

    for (long long f = f0; f < f1;) {
        while (f >= Fb + Hkv * cnt && b + 1 < B) {  // next request (skips requests with no stage)
            Fb += Hkv * cnt;
            ++b;
            L = clamp_len(p, b, false);
            lo = visible_lo(p, L);
            cnt = request_stages(p, L);
        }
        if (f >= Fb + Hkv * cnt) {  // unreachable: f < Stot
            if (tid == 0) raise_status(p, kErrBounds);
            return;
        }
        const int hk = static_cast<int>((f - Fb) / cnt);
        const int s0 = static_cast<int>((f - Fb) % cnt);
        const long long F = Fb + static_cast<long long>(hk) * cnt, E = F + cnt;
        const int s1 = static_cast<int>(f1 - F < cnt ? f1 - F : cnt);
        const long long wf = owner(F), wl_ = owner(E - 1);

        CtaWork w;
        w.b = b;
        w.hk = hk;
        w.L = L;
        w.split = static_cast<int>(c - wf);
        w.nsplit = static_cast<int>(wl_ - wf + 1);
        const int t0 = lo + s0 * kStageTok, t1 = min(lo + s1 * kStageTok, L);

        __syncthreads();  // the previous piece is done with q, the page list and the merge area
        stage_q_rows_cta<D>(p, b, hk, qs, S::MROWS, S::QSTRIDE);
        bool ok = true;
        for (int wt0 = t0; wt0 < t1; wt0 += win) {
            w.t0 = wt0;
            w.t1 = min(t1, wt0 + win);
            if (wt0 != t0) __syncthreads();  // every warp is done with the previous window's pages
            load_cta_pages(p, w, pages);
            if (wt0 == t0 && Body::kQInRing) fence_proxy_async();  // q rows sit where copies will land
            __syncthreads();
            if (wt0 == t0) {
                body.load_q(smem_u32(qs));
                if (Body::kQInRing) __syncthreads();  // every warp holds its q fragments: the ring is free
            }
            if (ok) ok = body.stream(&tmap, p, w, pages, smem, bars, pol);
        }
        if (!ok && lane == 0) scan[6] = 1;
        w.t0 = t0;
        w.t1 = t1;
        __syncthreads();  // every stage of the piece consumed: the ring is free for O
        if (scan[6]) return;  // a copy was lost (reported in the status word)
        float* O = reinterpret_cast<float*>(smem);
        body.store(O, wm, wl);
        __syncthreads();
        // split j of the unit is CTA wf+j's piece; a CTA's second slot holds
        // the unit that continues past the end of its slice
        cta_finish_parts<D, S::OSTRIDE, S::NS>(p, w, O, wm, wl, S::MROWS, flag, [&](int j) {
            const long long v = wf + j;
            return 2 * v + ((v + 1) * Stot / C < E ? 1 : 0);
        });
        fence_proxy_async();  // O and q were written through the generic proxy where the next copies land
        f = F + s1;
    }
}

}  // namespace pkd
