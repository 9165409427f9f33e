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

#include "decode_common.cuh"

namespace pkd {

template <int KVT>
struct KvType;
template <>
struct KvType<0> { static constexpr int ELT = 2; };  // bf16
template <>
struct KvType<1> { static constexpr int ELT = 2; };  // fp16
template <>
struct KvType<2> { static constexpr int ELT = 1; };  // fp8 e4m3

// Convert `SEG` bytes of stored elements (one 32-bit word at a time) to floats.
template <int KVT, int SEG>
__device__ __forceinline__ void load_seg(const uint8_t* src, float* out) {
    uint32_t wds[SEG / 4];
    if constexpr (SEG == 16) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        wds[0] = v.x; wds[1] = v.y; wds[2] = v.z; wds[3] = v.w;
    } else {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        wds[0] = v.x; wds[1] = v.y;
    }
#pragma unroll
    for (int i = 0; i < SEG / 4; ++i) {
        if constexpr (KVT == 0) {
            bf16x2_to_f32(wds[i], out[2 * i], out[2 * i + 1]);
        } else if constexpr (KVT == 1) {
            f16x2_to_f32(wds[i], out[2 * i], out[2 * i + 1]);
        } else {
            e4m3x2_to_f32(wds[i], out[4 * i], out[4 * i + 1]);
            e4m3x2_to_f32(wds[i] >> 16, out[4 * i + 2], out[4 * i + 3]);
        }
    }
}

template <int D, int KVT, int LPT, int MR, int NBUF>
struct FmaShape {
    static constexpr int ELT = KvType<KVT>::ELT;
    static constexpr int ROWB = D * ELT;                       // bytes of one K (or V) row
    static constexpr int KBOX = ROWB / 128;
    static constexpr int HALF = KBOX * 2048;
    static constexpr int STAGE = 2 * HALF;
    static constexpr int SEG = ROWB / LPT >= 16 ? 16 : 8;      // bytes per lane segment
    static constexpr int SPL = ROWB / (LPT * SEG);             // segments per lane
    static constexpr int EPS = SEG / ELT;                      // elements per segment
    static constexpr int EPL = SPL * EPS;                      // elements per lane
    static constexpr int TPP = 32 / LPT;                       // keys per pass
    static constexpr int NPASS = kStageTok / TPP;
    static constexpr int OSTRIDE = D + 4;
    static constexpr int RING = kNW * NBUF * STAGE;
    static constexpr int MERGE = kNW * MR * OSTRIDE * 4;
    static constexpr int BIG = RING > MERGE ? RING : MERGE;
    static constexpr int OFF_BARS = BIG;
    static constexpr int OFF_PAGES = OFF_BARS + kNW * NBUF * 8;
    static constexpr int OFF_ML = OFF_PAGES + kMaxCtaPages * 4;
    static constexpr int OFF_FLAG = OFF_ML + 2 * kNW * MR * 4;
    static constexpr int SMEM = OFF_FLAG + 16 + 1024;
    static_assert(MR <= LPT, "one row per lane after the reduce-scatter");
    static_assert(SPL >= 1 && ROWB % (LPT * SEG) == 0, "segments must tile a row");
};

// element index (within the head dim) of lane segment s, element e
template <int LPT, int SEG, int ELT>
__device__ __forceinline__ int seg_dim(int j, int s, int e) {
    return (j + LPT * s) * (SEG / ELT) + e;
}

template <int D, int KVT, int LPT, int MR, int NBUF>
__global__ void __launch_bounds__(kNW * 32)
decode_fma_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    using S = FmaShape<D, KVT, LPT, MR, NBUF>;
    constexpr int EPL = S::EPL, SEG = S::SEG, SPL = S::SPL, EPS = S::EPS, ELT = S::ELT;
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

    const int grp = lane / LPT, j = lane % LPT;
    const int gbase = grp * LPT;

    // q rows in fp32 with the logit scale folded in (log2 domain)
    float qf[MR][EPL];
#pragma unroll
    for (int r = 0; r < MR; ++r) {
        if (r < p.M) {
            const int i = r / p.G, g = r % p.G;
            const long long row = (static_cast<long long>(w.b) * p.sq + i) * p.Hq + w.hk * p.G + g;
            const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q) + row * S::ROWB;
#pragma unroll
            for (int s = 0; s < SPL; ++s) {
                float tmp[EPS];
                load_seg<KVT, SEG>(qrow + (j + LPT * s) * SEG, tmp);
#pragma unroll
                for (int e = 0; e < EPS; ++e) qf[r][s * EPS + e] = tmp[e] * p.scale_log2;
            }
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) qf[r][e] = 0.f;
        }
    }

    // which row this lane holds after the reduce-scatter
    int myrow = 0;
    {
        int cnt = MR;
#pragma unroll
        for (int m = LPT / 2; m >= 1; m >>= 1)
            if (cnt > 1) {
                if (lane & m) myrow += cnt / 2;
                cnt /= 2;
            }
    }
    constexpr int ROWSTEP = LPT / MR;  // lane distance between row owners in a group

    float acc[MR][EPL];
#pragma unroll
    for (int r = 0; r < MR; ++r)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[r][e] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    int timed_out = 0, consumed = 0;
    for (int k = 0; k < my_n; ++k) {
        const int buf = k % NBUF;
        if (!mbar_wait(bar0 + 8 * buf, (k / NBUF) & 1, p.status)) {
            timed_out = 1;
            break;
        }
        consumed = k + 1;
        const int stage = warp + k * kNW;
        const int tok0 = w.t0 + stage * kStageTok;
        int nvalid = min(kStageTok, w.t1 - tok0);
        if (pages[(tok0 - w.t0) / p.P] < 0) nvalid = 0;
        uint8_t* st = ring_gen + buf * S::STAGE;
        if (nvalid < kStageTok) zero_tail_v<D, ELT>(st, nvalid, lane);

        // ---- logits for the stage's 16 keys
        float sc[S::NPASS];
#pragma unroll
        for (int pass = 0; pass < S::NPASS; ++pass) {
            const int t = pass * S::TPP + grp;
            float kf[EPL];
#pragma unroll
            for (int s = 0; s < SPL; ++s) load_seg<KVT, SEG>(st + swz(t, (j + LPT * s) * SEG), kf + s * EPS);
            float v[MR];
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) a = fmaf(qf[r][e], kf[e], a);
                v[r] = a;
            }
            // reduce-scatter over the LPT lanes of this key
            int cnt = MR;
#pragma unroll
            for (int m = LPT / 2; m >= 1; m >>= 1) {
                if (cnt > 1) {
                    const int half = cnt / 2;
                    const bool up = lane & m;
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const float send = up ? v[i] : v[i + half];
                        const float keep = up ? v[i + half] : v[i];
                        v[i] = keep + __shfl_xor_sync(kFull, send, m);
                    }
                    cnt = half;
                } else {
                    v[0] += __shfl_xor_sync(kFull, v[0], m);
                }
            }
            const bool ok = t < nvalid && row_sees(p, w.L, myrow, tok0 + t);
            sc[pass] = ok ? v[0] : -INFINITY;
        }

        // ---- online softmax for this lane's row
        float mx = sc[0];
#pragma unroll
        for (int pass = 1; pass < S::NPASS; ++pass) mx = fmaxf(mx, sc[pass]);
#pragma unroll
        for (int m = LPT; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m_run - m_use);
        m_run = m_new;
        float ls = 0.f;
#pragma unroll
        for (int pass = 0; pass < S::NPASS; ++pass) {
            sc[pass] = fast_exp2(sc[pass] - m_use);
            ls += sc[pass];
        }
        l_run = l_run * alpha + ls;
        if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                const float ar = __shfl_sync(kFull, alpha, gbase + r * ROWSTEP);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[r][e] *= ar;
            }
        }

        // ---- acc += p * V
#pragma unroll
        for (int pass = 0; pass < S::NPASS; ++pass) {
            const int t = pass * S::TPP + grp;
            float vf[EPL];
#pragma unroll
            for (int s = 0; s < SPL; ++s)
                load_seg<KVT, SEG>(st + S::HALF + swz(t, (j + LPT * s) * SEG), vf + s * EPS);
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                const float pr = __shfl_sync(kFull, sc[pass], gbase + r * ROWSTEP);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[r][e] = fmaf(pr, vf[e], acc[r][e]);
            }
        }

        __syncwarp();
        if (lane == 0 && k + NBUF < my_n) {
            fence_proxy_async();
            issue_stage<D, ELT>(&tmap, p, w, pages, warp + (k + NBUF) * kNW, ring + buf * S::STAGE,
                                bar0 + 8 * buf, pol);
        }
    }
    if (timed_out) {
        if (lane == 0) raise_status(p, kErrTimeout);
        for (int k = consumed + 1; k < my_n && k < consumed + NBUF; ++k)
            mbar_wait(bar0 + 8 * (k % NBUF), (k / NBUF) & 1, p.status);
    }

    // ---- sum the keys-in-flight groups, then hand the warp state to the CTA
#pragma unroll
    for (int m = LPT; m < 32; m <<= 1) {
        l_run += __shfl_xor_sync(kFull, l_run, m);
#pragma unroll
        for (int r = 0; r < MR; ++r)
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[r][e] += __shfl_xor_sync(kFull, acc[r][e], m);
    }
    __syncthreads();
    float* O = reinterpret_cast<float*>(smem);
    if (grp == 0) {
        if (j % ROWSTEP == 0) {
            wm[warp * MR + myrow] = m_run;
            wl[warp * MR + myrow] = l_run;
        }
#pragma unroll
        for (int r = 0; r < MR; ++r)
#pragma unroll
            for (int s = 0; s < SPL; ++s)
#pragma unroll
                for (int e = 0; e < EPS; ++e)
                    O[(warp * MR + r) * S::OSTRIDE + seg_dim<LPT, SEG, ELT>(j, s, e)] = acc[r][s * EPS + e];
    }
    __syncthreads();
    cta_finish<D, S::OSTRIDE>(p, w, O, wm, wl, MR, flag);
}

}  // namespace pkd
