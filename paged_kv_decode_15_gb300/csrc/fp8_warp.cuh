// Tensor-core warp for fp8-e4m3 caches.
//
// S = Q K^T runs directly on e4m3 operands (mma m16n8k32): q arrives already
// quantised and the K tile is used as the TMA delivered it.  O^T += V^T P^T
// runs on fp16 operands (every e4m3 value is exact in fp16), with V widened
// in registers, fragment by fragment, straight from the e4m3 stage:
//   ldmatrix.trans of 16-bit units -- each unit a pair of e4m3 values of one
//   key at dims (2j, 2j+1) -- gives lane (g, tg) the bytes
//   V[2tg][2j], V[2tg][2j+1], V[2tg+1][2j], V[2tg+1][2j+1] with j = j0 + g;
//   a byte permute pairs the two keys of one dim and cvt.f16x2.e4m3x2 widens
//   them, which is an A fragment of V^T whose 16 rows are the dims
//   2j0 .. 2j0+15 in the order (2j0, 2j0+2, ..., 2j0+14, 2j0+1, ..., 2j0+15).
// The accumulator rows then hold dim pairs (MmaWarp's kPairRows layout), and
// no V tile goes through shared memory twice.  P is rounded only to fp16;
// the q/k scales stay in the logit scale and v_scale in the epilogue.
#pragma once

#include "mma_warp.cuh"

namespace pkd {

template <int MT, int NT>
struct Fp8MmaWarp : MmaWarp<128, false, MT, NT, true> {
    using Base = MmaWarp<128, false, MT, NT, true>;
    static constexpr int kScratchBytes = 0;  // V is widened in registers
    static constexpr bool kCtaQ = false;     // e4m3 q fragments come straight from global memory
    // five CTAs per SM (96 registers): fp8_long_b8 at 32 chunks 363 us against 377 us with four
    static constexpr int kMinBlocks = 5;
    uint32_t q8[MT][4][4];                   // e4m3 A fragments, 4 k-steps of 32

    __device__ __forceinline__ void setup(uint8_t*) {}

    // e4m3 q rows of (b, hk) as m16n8k32 A fragments (zero padding rows)
    __device__ __forceinline__ void load_q(const DecodeParams& p, int b, int hk, int lane) {
        const int g = lane >> 2, tg = lane & 3;
        const uint8_t* q = reinterpret_cast<const uint8_t*>(p.q);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = this->row0 + mt * 16 + h * 8 + g;
                const uint32_t* row = nullptr;
                if (r < p.M) {
                    const int i = r / p.G, gg = r % p.G;
                    row = reinterpret_cast<const uint32_t*>(
                        q + ((static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + gg) * 128);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    // bytes kk*32 + 4tg .. +3 and kk*32 + 16 + 4tg .. +3
                    q8[mt][kk][h] = row ? __ldg(row + kk * 8 + tg) : 0u;
                    q8[mt][kk][2 + h] = row ? __ldg(row + kk * 8 + 4 + tg) : 0u;
                }
            }
    }

    // O^T += V^T P^T with the e4m3 V tile at `vt` (16 keys x 128 bytes, 128-byte
    // swizzle).  Load i covers the 16-byte chunks 2i and 2i+1 (dims 32i ..
    // 32i+31) for keys 0-7 and 8-15: four 8x8 blocks of 16-bit units.
    __device__ __forceinline__ void pv_e4m3(uint32_t vt, const uint32_t (&pb)[NT][2], int lane) {
        const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t r[4];
            ldsm_x4_t(vt + swz((mi & 1) * 8 + ri, (2 * i + (mi >> 1)) * 16), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // r[2h]: keys 2tg, 2tg+1; r[2h+1]: keys 8+2tg, 8+2tg+1 (of chunk 2i+h)
                uint32_t va[4];
                va[0] = e4m3x2_to_f16x2(__byte_perm(r[2 * h], 0u, 0x0020));      // row g: dim 2j
                va[1] = e4m3x2_to_f16x2(__byte_perm(r[2 * h], 0u, 0x0031));      // row g+8: dim 2j+1
                va[2] = e4m3x2_to_f16x2(__byte_perm(r[2 * h + 1], 0u, 0x0020));
                va[3] = e4m3x2_to_f16x2(__byte_perm(r[2 * h + 1], 0u, 0x0031));
#pragma unroll
                for (int n = 0; n < NT; ++n) mma16816<false>(this->oacc[2 * i + h][n], va, pb[n][0], pb[n][1]);
            }
        }
    }

    template <class Visible>
    __device__ __forceinline__ void consume(uint32_t st, int half, int nvalid, bool masked, float scale2,
                                            float bias2, Visible visible, int lane) {
        // S = Q K^T on e4m3: the K tile is one 128-byte box per key row
        const int mi = lane >> 3, ri = lane & 7;
        float sacc[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int c = 0; c < 4; ++c) sacc[mt][n][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t b00, b01, b10, b11;
            ldsm_x4(st + swz((mi >> 1) * 8 + ri, (2 * kk + (mi & 1)) * 16), b00, b01, b10, b11);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                mma16832_e4m3(sacc[mt][0], q8[mt][kk], b00, b01);
                mma16832_e4m3(sacc[mt][1], q8[mt][kk], b10, b11);
            }
        }
        uint32_t pb[NT][2];
        if (masked)
            Base::template softmax<true>(sacc, pb, nvalid, scale2, bias2, visible, lane);
        else
            Base::template softmax<false>(sacc, pb, nvalid, scale2, bias2, visible, lane);
        pv_e4m3(st + half, pb, lane);
    }
};

}  // namespace pkd
