// One warp's share of tensor-core attention over 16-key stages.
//
// The warp keeps M query rows (M padded to MT 16-row tiles for Q K^T and to
// NT 8-wide tiles for the swapped V^T P^T) and an online-softmax state per
// row.  Stages are the swizzled [16 keys x (K | V)] tiles that the TMA loads
// produce: K at byte 0, V at byte `half`.
//   S   = Q K^T          A = Q fragments (registers), B = K (ldmatrix)
//   O^T += V^T P^T       A = V^T (ldmatrix.trans), B = P^T, which is the
//                        accumulator layout of S, so no data moves between them.
#pragma once

#include "decode_common.cuh"

namespace pkd {

template <int D, bool kBF16, int MT, int NT>
struct MmaWarp {
    uint32_t qa[MT][D / 16][4];
    float m_run[MT][2], l_run[MT][2];
    float oacc[D / 16][NT][4];

    // Q fragments from rows staged in shared memory (row stride qstride bytes).
    __device__ __forceinline__ void load_q(uint32_t qs, int qstride, int lane) {
        const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int row = mt * 16 + (mi & 1) * 8 + ri;
                const int chunk = 2 * kk + (mi >> 1);
                ldsm_x4(qs + row * qstride + chunk * 16, qa[mt][kk][0], qa[mt][kk][1], qa[mt][kk][2],
                        qa[mt][kk][3]);
            }
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                m_run[mt][h] = -INFINITY;
                l_run[mt][h] = 0.f;
            }
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) oacc[dt][n][c] = 0.f;
    }

    // Fold one stage into the state.  Logits are scale2 * q.k + bias2 (log2
    // domain); key kt (0..15) is used by row `row` iff kt < nvalid and
    // visible(row, kt).  V rows at or past nvalid must be finite (zeroed).
    template <class Visible>
    __device__ __forceinline__ void consume(uint32_t st, int half, int nvalid, float scale2, float bias2,
                                            Visible visible, int lane) {
        const int g = lane >> 2, tg = lane & 3;
        const int mi = lane >> 3, ri = lane & 7;
        float sacc[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) sacc[mt][n][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t b00, b01, b10, b11;
            ldsm_x4(st + swz((mi >> 1) * 8 + ri, (2 * kk + (mi & 1)) * 16), b00, b01, b10, b11);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                mma16816<kBF16>(sacc[mt][0], qa[mt][kk], b00, b01);
                mma16816<kBF16>(sacc[mt][1], qa[mt][kk], b10, b11);
            }
        }

        float alpha[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = mt * 16 + h * 8 + g;
                float mx = -INFINITY;
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int kt = n * 8 + 2 * tg + e;
                        const bool ok = kt < nvalid && visible(row, kt);
                        const float s = ok ? fmaf(sacc[mt][n][2 * h + e], scale2, bias2) : -INFINITY;
                        sacc[mt][n][2 * h + e] = s;
                        mx = fmaxf(mx, s);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                const float m_new = fmaxf(m_run[mt][h], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                alpha[mt][h] = fast_exp2(m_run[mt][h] - m_use);
                m_run[mt][h] = m_new;
                float ls = 0.f;
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        // l sums the fp32 weights; P.V uses them rounded to the operand
                        // type (relative error <= 2^-9 for bf16, so a constant V still
                        // comes back exactly after the final rounding)
                        const float pe = fast_exp2(sacc[mt][n][2 * h + e] - m_use);
                        sacc[mt][n][2 * h + e] = pe;
                        ls += pe;
                    }
                l_run[mt][h] = l_run[mt][h] * alpha[mt][h] + ls;
            }

        uint32_t pb[NT][2];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int mt = n >> 1, h = n & 1;
            const float a0 = __shfl_sync(kFull, alpha[mt][h], 4 * (2 * tg));
            const float a1 = __shfl_sync(kFull, alpha[mt][h], 4 * (2 * tg + 1));
#pragma unroll
            for (int dt = 0; dt < D / 16; ++dt) {
                oacc[dt][n][0] *= a0;
                oacc[dt][n][1] *= a1;
                oacc[dt][n][2] *= a0;
                oacc[dt][n][3] *= a1;
            }
            pb[n][0] = pack2<kBF16>(sacc[mt][0][2 * h], sacc[mt][0][2 * h + 1]);
            pb[n][1] = pack2<kBF16>(sacc[mt][1][2 * h], sacc[mt][1][2 * h + 1]);
        }
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
            uint32_t va[4];
            ldsm_x4_t(st + half + swz((mi >> 1) * 8 + ri, (2 * dt + (mi & 1)) * 16), va[0], va[1], va[2], va[3]);
#pragma unroll
            for (int n = 0; n < NT; ++n) mma16816<kBF16>(oacc[dt][n], va, pb[n][0], pb[n][1]);
        }
    }

    // Sum each row's l over the four lanes that share it.
    __device__ __forceinline__ void reduce_l() {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                l_run[mt][h] += __shfl_xor_sync(kFull, l_run[mt][h], 1);
                l_run[mt][h] += __shfl_xor_sync(kFull, l_run[mt][h], 2);
            }
    }

    // Row stats of the accumulator columns this lane holds: rows 8n + 2tg + e.
    __device__ __forceinline__ void column_rows_stat(const float (&v)[MT][2], float (&out)[NT][2], int lane) const {
        const int tg = lane & 3;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            out[n][0] = __shfl_sync(kFull, v[n >> 1][n & 1], 4 * (2 * tg));
            out[n][1] = __shfl_sync(kFull, v[n >> 1][n & 1], 4 * (2 * tg + 1));
        }
    }

    // Store m, l (rows 0..16*MT) and the unnormalised O (rows 0..8*NT) of this
    // warp to shared memory: wm[row], wl[row], O[row * ostride + d].
    __device__ __forceinline__ void store(float* O, float* wm, float* wl, int ostride, int lane) const {
        const int g = lane >> 2, tg = lane & 3;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (tg == 0) {
                    wm[mt * 16 + h * 8 + g] = m_run[mt][h];
                    wl[mt * 16 + h * 8 + g] = l_run[mt][h];
                }
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    O[(n * 8 + 2 * tg + (c & 1)) * ostride + dt * 16 + g + (c >> 1) * 8] = oacc[dt][n][c];
    }
};

}  // namespace pkd
