// Tensor-core warp for fp8-e4m3 caches.
//
// S = Q K^T runs directly on e4m3 operands (mma m16n8k32): q arrives already
// quantised and the K tile is used as the TMA delivered it.  For O^T += V^T P^T
// the V tile is widened once, in shared memory, to an fp16 tile of the same
// swizzled layout (every e4m3 value is exact in fp16) and the fp16 warp runs
// the softmax and P.V unchanged, so P is rounded only to fp16.  The q/k scales
// stay in the logit scale and v_scale in the epilogue; all products are exact.
#pragma once

#include "mma_warp.cuh"

namespace pkd {

template <int MT, int NT>
struct Fp8MmaWarp : MmaWarp<128, false, MT, NT> {
    using Base = MmaWarp<128, false, MT, NT>;
    static constexpr int kWide = 2 * 2048;  // one fp16 V tile: two 128-byte boxes of 16 rows
    static constexpr int kScratchBytes = kWide;
    static constexpr bool kCtaQ = false;  // e4m3 q fragments come straight from global memory
    uint32_t q8[MT][4][4];                  // e4m3 A fragments, 4 k-steps of 32
    uint32_t wide = 0;
    uint8_t* wide_gen = nullptr;

    __device__ __forceinline__ void setup(uint8_t* scratch) {
        wide_gen = scratch;
        wide = smem_u32(scratch);
    }

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
        // widen the V tile to fp16
        const uint8_t* src = static_cast<const uint8_t*>(__cvta_shared_to_generic(st + half));
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int c = it * 32 + lane;  // 128 chunks of 16 e4m3: row, chunk
            const int row = c >> 3, chunk = c & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(src + swz(row, chunk * 16));
            const uint4 w0 = make_uint4(e4m3x2_to_f16x2(v.x & 0xffffu), e4m3x2_to_f16x2(v.x >> 16),
                                        e4m3x2_to_f16x2(v.y & 0xffffu), e4m3x2_to_f16x2(v.y >> 16));
            const uint4 w1 = make_uint4(e4m3x2_to_f16x2(v.z & 0xffffu), e4m3x2_to_f16x2(v.z >> 16),
                                        e4m3x2_to_f16x2(v.w & 0xffffu), e4m3x2_to_f16x2(v.w >> 16));
            *reinterpret_cast<uint4*>(wide_gen + swz(row, chunk * 32)) = w0;
            *reinterpret_cast<uint4*>(wide_gen + swz(row, chunk * 32 + 16)) = w1;
        }
        __syncwarp();
        if (masked)
            Base::template softmax_pv<true>(sacc, wide, nvalid, scale2, bias2, visible, lane);
        else
            Base::template softmax_pv<false>(sacc, wide, nvalid, scale2, bias2, visible, lane);
        __syncwarp();
    }
};

}  // namespace pkd
