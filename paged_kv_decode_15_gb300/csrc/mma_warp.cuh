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

// kPairRows: the P.V accumulator rows hold head-dim pairs (row r < 8 of a
// 16-row tile is dim 2r, row 8 + r is dim 2r + 1), the layout the e4m3 warp's
// register-widened V fragments give; otherwise row r is dim r.
template <int D, bool kBF16, int MT, int NT, bool kPairRows = false>
struct MmaWarp {
    // With two row tiles the Q fragments would not fit in registers next to
    // the accumulators: they are then staged in shared memory and re-read.
    static constexpr bool kQSmem = MT > 1;
    static constexpr int QSTRIDE = D * 2 + 16;  // bytes per staged q row (conflict-free ldmatrix)
    uint32_t qa[kQSmem ? 1 : MT][D / 16][4];
    uint32_t qs = 0;
    uint8_t* qs_gen = nullptr;
    int row0 = 0;  // first query row of (b, hk) this warp holds (row tiles split across warps)
    float m_run[MT][2], l_run[MT][2];
    float oacc[D / 16][NT][4];

    // A fragment of Q for row tile mt, k-step kk
    __device__ __forceinline__ void q_frag(int mt, int kk, uint32_t (&a)[4], int lane) const {
        if constexpr (kQSmem) {
            const int mi = lane >> 3, ri = lane & 7;
            const int row = mt * 16 + (mi & 1) * 8 + ri;
            ldsm_x4(qs + row * QSTRIDE + (2 * kk + (mi >> 1)) * 16, a[0], a[1], a[2], a[3]);
        } else {
            a[0] = qa[mt][kk][0];
            a[1] = qa[mt][kk][1];
            a[2] = qa[mt][kk][2];
            a[3] = qa[mt][kk][3];
        }
    }

    // Q fragments from rows staged in shared memory (row stride qstride bytes).
    __device__ __forceinline__ void load_q(uint32_t qsm, int qstride, int lane) {
        if constexpr (kQSmem) {
            qs = qsm;  // re-read at every stage; the caller keeps the rows in place
            return;
        }
        const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int row = mt * 16 + (mi & 1) * 8 + ri;
                const int chunk = 2 * kk + (mi >> 1);
                ldsm_x4(qsm + row * qstride + chunk * 16, qa[mt][kk][0], qa[mt][kk][1], qa[mt][kk][2],
                        qa[mt][kk][3]);
            }
    }

    static constexpr int MROWS = MT * 16;
    static constexpr bool kTensor = true;
    // per-warp shared memory beyond the ring: the staged q rows (1 KiB granules)
    static constexpr int kScratchBytes = kQSmem ? (MROWS * QSTRIDE + 1023) / 1024 * 1024 : 0;
    static constexpr int kNbuf = 2;  // ring depth per warp (three CTAs of four warps fit an SM)
    static constexpr bool kCtaQ = true;  // grid kernels stage q once for the CTA's warps
    static constexpr int kMinBlocks = 1;  // CTAs per SM the grid kernel's register budget aims for

    __device__ __forceinline__ void setup(uint8_t* scratch) {
        qs_gen = scratch;
        qs = smem_u32(scratch);
    }

    // stage q rows r < M of (b, hk) (16-bit storage) in this warp's scratch
    __device__ __forceinline__ void stage_q_rows(const DecodeParams& p, int b, int hk, int lane) {
        constexpr int VPR = D * 2 / 16;
        const uint4* q = reinterpret_cast<const uint4*>(p.q);
        for (int e = lane; e < MROWS * VPR; e += 32) {
            const int r = e / VPR, v = e % VPR;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (r < p.M) {
                const int i = r / p.G, g = r % p.G;
                val = __ldg(q + ((static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g) * VPR + v);
            }
            *reinterpret_cast<uint4*>(qs_gen + r * QSTRIDE + v * 16) = val;
        }
        __syncwarp();
    }

    __device__ __forceinline__ void init(int) {}
    __device__ __forceinline__ void load_q(const DecodeParams& p, int b, int hk, int lane) {
        if constexpr (kQSmem)
            stage_q_rows(p, b, hk, lane);
        else
            load_q_global(p, b, hk, lane);
    }

    // Q fragments straight from global memory: rows r < M of (b, hk), zero padding.
    __device__ __forceinline__ void load_q_global(const DecodeParams& p, int b, int hk, int lane) {
        static_assert(!kQSmem, "register Q fragments only for one row tile");
        const int g = lane >> 2, tg = lane & 3;
        const uint16_t* q = reinterpret_cast<const uint16_t*>(p.q);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = row0 + mt * 16 + h * 8 + g;
                const uint32_t* row = nullptr;
                if (r < p.M) {
                    const int i = r / p.G, gg = r % p.G;
                    row = reinterpret_cast<const uint32_t*>(
                        q + ((static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + gg) * D);
                }
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    qa[mt][kk][h] = row ? __ldg(row + kk * 8 + tg) : 0u;
                    qa[mt][kk][2 + h] = row ? __ldg(row + kk * 8 + 4 + tg) : 0u;
                }
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

    // Row half h of row tile mt feeds P.V n-tile 2*mt + h; halves past NT
    // hold only padding rows and are skipped.
    static __device__ __forceinline__ constexpr bool half_used(int mt, int h) { return 2 * mt + h < NT; }

    // Fold one stage into the state.  Logits are scale2 * q.k + bias2 (log2
    // domain).  kMasked: key kt (0..15) is used by row `row` iff kt < nvalid
    // and visible(row, kt), and V rows at or past nvalid must be finite
    // (zeroed); otherwise all 16 keys are used by every row.  kSplitQK: see qk.
    template <bool kMasked, bool kSplitQK = false, class Visible>
    __device__ __forceinline__ void consume(uint32_t st, int half, int nvalid, float scale2, float bias2,
                                            Visible visible, int lane) {
        float sacc[MT][2][4];
        qk<kSplitQK>(st, sacc, lane);
        softmax_pv<kMasked>(sacc, st + half, nvalid, scale2, bias2, visible, lane);
    }

    // S = Q K^T for the 16 keys of the K tile at `st`.  kSplit (one row tile
    // only): the k-steps accumulate in two chains, even and odd, summed at the
    // end, which halves the dependent MMA chain of a stage.  It pays where a
    // warp's wait-to-refill chain per stage is the limit (segments: 66.5 ->
    // 65.9 us on dash_paged_n256); elsewhere it gains nothing and its
    // registers spill.
    template <bool kSplit = false>
    __device__ __forceinline__ void qk(uint32_t st, float (&sacc)[MT][2][4], int lane) const {
        static_assert(!kSplit || MT == 1, "two chains for one row tile only");
        const int mi = lane >> 3, ri = lane & 7;
        float sodd[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) sacc[mt][n][c] = sodd[mt][n][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t b00, b01, b10, b11;
            ldsm_x4(st + swz((mi >> 1) * 8 + ri, (2 * kk + (mi & 1)) * 16), b00, b01, b10, b11);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                q_frag(mt, kk, a, lane);
                float (&acc)[2][4] = (kSplit && (kk & 1)) ? sodd[mt] : sacc[mt];
                mma16816<kBF16>(acc[0], a, b00, b01);
                mma16816<kBF16>(acc[1], a, b10, b11);
            }
        }
        if constexpr (kSplit)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) sacc[0][n][c] += sodd[0][n][c];
    }

    // Head dim of accumulator element c of d-tile dt held by lane group g.
    static __device__ __forceinline__ int d_of(int dt, int g, int c) {
        return kPairRows ? dt * 16 + 2 * g + (c >> 1) : dt * 16 + g + (c >> 1) * 8;
    }

    // Online softmax of S (scaled here), then O^T += V^T P^T with the V tile at `vt`.
    template <bool kMasked, class Visible>
    __device__ __forceinline__ void softmax_pv(float (&sacc)[MT][2][4], uint32_t vt, int nvalid, float scale2,
                                               float bias2, Visible visible, int lane) {
        uint32_t pb[NT][2];
        softmax<kMasked>(sacc, pb, nvalid, scale2, bias2, visible, lane);
        pv(vt, pb, lane);
    }

    // Online softmax of S: updates the row statistics, rescales O when a
    // row's maximum moved, and returns P^T (rounded to the operand type) as
    // the B fragments of the P.V product.
    template <bool kMasked, class Visible>
    __device__ __forceinline__ void softmax(float (&sacc)[MT][2][4], uint32_t (&pb)[NT][2], int nvalid,
                                            float scale2, float bias2, Visible visible, int lane) {
        const int g = lane >> 2, tg = lane & 3;
        float alpha[MT][2];
        bool grew = false;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                alpha[mt][h] = 1.f;
                if (!half_used(mt, h)) continue;
                const int row = mt * 16 + h * 8 + g;
                float mx = -INFINITY;
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float s = fmaf(sacc[mt][n][2 * h + e], scale2, bias2);
                        if constexpr (kMasked) {
                            const int kt = n * 8 + 2 * tg + e;
                            if (!(kt < nvalid && visible(row, kt))) s = -INFINITY;
                        }
                        sacc[mt][n][2 * h + e] = s;
                        mx = fmaxf(mx, s);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                const float m_new = fmaxf(m_run[mt][h], mx);
                const float m_use = (kMasked && m_new == -INFINITY) ? 0.f : m_new;
                grew |= m_new > m_run[mt][h];
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

        // rescale O^T columns (rows 8n + 2tg + e) only when some row's max moved
        if (__any_sync(kFull, grew)) {
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
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int mt = n >> 1, h = n & 1;
            pb[n][0] = pack2<kBF16>(sacc[mt][0][2 * h], sacc[mt][0][2 * h + 1]);
            pb[n][1] = pack2<kBF16>(sacc[mt][1][2 * h], sacc[mt][1][2 * h + 1]);
        }
    }

    // O^T += V^T P^T for the 16-bit V tile at `vt` (A = V^T by ldmatrix.trans).
    __device__ __forceinline__ void pv(uint32_t vt, const uint32_t (&pb)[NT][2], int lane) {
        const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt) {
            uint32_t va[4];
            ldsm_x4_t(vt + swz((mi >> 1) * 8 + ri, (2 * dt + (mi & 1)) * 16), va[0], va[1], va[2], va[3]);
#pragma unroll
            for (int n = 0; n < NT; ++n) mma16816<kBF16>(oacc[dt][n], va, pb[n][0], pb[n][1]);
        }
    }

    // Full or masked stage, chosen per call (the choice is warp-uniform).
    template <class Visible>
    __device__ __forceinline__ void consume(uint32_t st, int half, int nvalid, bool masked, float scale2,
                                            float bias2, Visible visible, int lane) {
        if (masked)
            consume<true>(st, half, nvalid, scale2, bias2, visible, lane);
        else
            consume<false>(st, half, nvalid, scale2, bias2, visible, lane);
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

    __device__ __forceinline__ void finish() { reduce_l(); }

    // After finish(): f(row, d, o / l) for every element this lane holds.
    template <class F>
    __device__ __forceinline__ void emit(F&& f, int lane) const {
        const int g = lane >> 2, tg = lane & 3;
        float lcol[NT][2];
        column_rows_stat(l_run, lcol, lane);
#pragma unroll
        for (int dt = 0; dt < D / 16; ++dt)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float l = lcol[n][c & 1];
                    f(n * 8 + 2 * tg + (c & 1), d_of(dt, g, c), l > 0.f ? oacc[dt][n][c] / l : 0.f);
                }
    }

    // After finish(): f(row, lse in log2 units, or -inf) once per row.
    template <class F>
    __device__ __forceinline__ void emit_lse(F&& f, int lane) const {
        const int g = lane >> 2, tg = lane & 3;
        if (tg == 0)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float l = l_run[mt][h];
                    f(mt * 16 + h * 8 + g, l > 0.f ? m_run[mt][h] + __log2f(l) : -INFINITY);
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
                    O[(n * 8 + 2 * tg + (c & 1)) * ostride + d_of(dt, g, c)] = oacc[dt][n][c];
    }
};

}  // namespace pkd
