// One warp's share of CUDA-core attention over 16-key stages (M <= 8 rows).
//
// LPT lanes share one key: each lane owns EPL elements of the head dimension
// (whole 16-byte chunks of the swizzled stage, or halves of them), so
//   q.k  is EPL FMAs per row followed by a reduce-scatter over the LPT lanes
//        (each lane ends with the full logit of one row),
//   p*V  accumulates into a per-lane [MR][EPL] slice with no reduction until
//        finish(), which sums the 32/LPT keys-in-flight groups once.
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

template <int D, int KVT, int LPT, int MR>
struct FmaGeom {
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
    static constexpr int ROWSTEP = LPT / MR;                   // lane distance between row owners
    static_assert(MR <= LPT, "one row per lane after the reduce-scatter");
    static_assert(SPL >= 1 && ROWB % (LPT * SEG) == 0, "segments must tile a row");
};

template <int D, int KVT, int LPT, int MR>
struct FmaWarp {
    using S = FmaGeom<D, KVT, LPT, MR>;
    static constexpr int EPL = S::EPL, SEG = S::SEG, SPL = S::SPL, EPS = S::EPS, ELT = S::ELT;
    static constexpr int MROWS = MR;
    static constexpr bool kTensor = false;
    static constexpr int kScratchBytes = 0;  // per-warp shared memory beyond the ring
    static constexpr int kNbuf = 3;

    __device__ __forceinline__ void setup(uint8_t*) {}

    float qf[MR][EPL];
    float acc[MR][EPL];
    float m_run, l_run;
    int myrow;
    int row0 = 0;  // row tiles are never split across CUDA-core warps (M <= 8)

    // head-dimension index of lane segment s, element e
    __device__ __forceinline__ static int dim_of(int j, int s, int e) { return (j + LPT * s) * EPS + e; }

    __device__ __forceinline__ void init(int lane) {
        myrow = 0;
        int cnt = MR;
#pragma unroll
        for (int m = LPT / 2; m >= 1; m >>= 1)
            if (cnt > 1) {
                if (lane & m) myrow += cnt / 2;
                cnt /= 2;
            }
    }

    // q rows of (b, hk) in fp32 with the logit scale folded in (log2 domain)
    __device__ __forceinline__ void load_q(const DecodeParams& p, int b, int hk, int lane) {
        const int j = lane % LPT;
#pragma unroll
        for (int r = 0; r < MR; ++r) {
            if (r < p.M) {
                const int i = r / p.G, g = r % p.G;
                const long long row = (static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g;
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
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int r = 0; r < MR; ++r)
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[r][e] = 0.f;
        m_run = -INFINITY;
        l_run = 0.f;
    }

    // Fold one stage (generic pointer to its swizzled tile) into the state.
    // Key kt (0..15) is used by row `row` iff kt < nvalid and visible(row, kt).
    template <class Visible>
    __device__ __forceinline__ void consume(const uint8_t* st, int nvalid, Visible visible, int lane) {
        const int grp = lane / LPT, j = lane % LPT, gbase = grp * LPT;
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
            const bool ok = t < nvalid && visible(myrow, t);
            sc[pass] = ok ? v[0] : -INFINITY;
        }

        // online softmax for this lane's row
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
                const float ar = __shfl_sync(kFull, alpha, gbase + r * S::ROWSTEP);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[r][e] *= ar;
            }
        }

        // acc += p * V
#pragma unroll
        for (int pass = 0; pass < S::NPASS; ++pass) {
            const int t = pass * S::TPP + grp;
            float vf[EPL];
#pragma unroll
            for (int s = 0; s < SPL; ++s)
                load_seg<KVT, SEG>(st + S::HALF + swz(t, (j + LPT * s) * SEG), vf + s * EPS);
#pragma unroll
            for (int r = 0; r < MR; ++r) {
                const float pr = __shfl_sync(kFull, sc[pass], gbase + r * S::ROWSTEP);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[r][e] = fmaf(pr, vf[e], acc[r][e]);
            }
        }
    }

    // Sum the keys-in-flight groups: afterwards every group holds the warp's
    // totals (acc per row, l for this lane's row).
    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int m = LPT; m < 32; m <<= 1) {
            l_run += __shfl_xor_sync(kFull, l_run, m);
#pragma unroll
            for (int r = 0; r < MR; ++r)
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc[r][e] += __shfl_xor_sync(kFull, acc[r][e], m);
        }
    }

    // After finish(): f(row, d, o / l) for every (row < MR, d) once (group 0 lanes).
    template <class F>
    __device__ __forceinline__ void emit(F&& f, int lane) const {
        const int j = lane % LPT;
        float lr[MR];
#pragma unroll
        for (int r = 0; r < MR; ++r) lr[r] = __shfl_sync(kFull, l_run, r * S::ROWSTEP);
        if (lane < LPT) {
#pragma unroll
            for (int r = 0; r < MR; ++r)
#pragma unroll
                for (int s = 0; s < SPL; ++s)
#pragma unroll
                    for (int e = 0; e < EPS; ++e)
                        f(r, dim_of(j, s, e), lr[r] > 0.f ? acc[r][s * EPS + e] / lr[r] : 0.f);
        }
    }

    // After finish(): f(row, lse in log2 units, or -inf) once per row.
    template <class F>
    __device__ __forceinline__ void emit_lse(F&& f, int lane) const {
        if (lane < LPT && (lane % S::ROWSTEP) == 0)
            f(myrow, l_run > 0.f ? m_run + __log2f(l_run) : -INFINITY);
    }

    // After finish(): unnormalised state to shared memory for a CTA merge.
    __device__ __forceinline__ void store(float* O, float* wm, float* wl, int ostride, int lane) const {
        const int j = lane % LPT;
        if (lane < LPT) {
            if (j % S::ROWSTEP == 0) {
                wm[myrow] = m_run;
                wl[myrow] = l_run;
            }
#pragma unroll
            for (int r = 0; r < MR; ++r)
#pragma unroll
                for (int s = 0; s < SPL; ++s)
#pragma unroll
                    for (int e = 0; e < EPS; ++e) O[r * ostride + dim_of(j, s, e)] = acc[r][s * EPS + e];
        }
    }
};

}  // namespace pkd
