// Instantiations of the tensor-core decode kernel.
#include "decode_mma.cuh"
#include "launch.h"

namespace pkd {

constexpr int kMmaNbuf = 2;
constexpr int kGridWarps = 4;  // warps per CTA of the one-tile kernel
constexpr int kPairNbuf = 4;  // per warp pair: the same 64 KiB of ring per CTA as four rings of two

template <int D, bool kBF16, int MT, int NT>
static cudaError_t launch_one(const CUtensorMap& tmap, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    using S = MmaShape<D, MT, NT, kMmaNbuf, kGridWarps>;
    auto kern = decode_mma_kernel<D, kBF16, MT, NT, kMmaNbuf, kGridWarps>;
    static bool configured = false;  // benign race: the attribute call is idempotent
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, kGridWarps * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}

template <int D, bool kBF16>
static cudaError_t launch_pair(const CUtensorMap& tmap, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    using S = PairShape<D, kPairNbuf>;
    auto kern = decode_mma_pair_kernel<D, kBF16, kPairNbuf>;
    static bool configured = false;  // benign race: the attribute call is idempotent
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, kNW * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}

int decode_mma_smem(int D, int MT, int NT) {
#define PKD_MMA_SMEM(d, mt, nt) \
    if (D == d && MT == mt && NT == nt) return MmaShape<d, mt, nt, kMmaNbuf>::SMEM;
    PKD_MMA_SMEM(128, 1, 1) PKD_MMA_SMEM(128, 1, 2) PKD_MMA_SMEM(64, 1, 1) PKD_MMA_SMEM(64, 1, 2)
    if (MT == 2) return D == 128 ? PairShape<128, kPairNbuf>::SMEM : D == 64 ? PairShape<64, kPairNbuf>::SMEM : -1;
#undef PKD_MMA_SMEM
    return -1;
}

cudaError_t launch_decode_mma(int D, bool bf16, int MT, int NT, const CUtensorMap& tmap,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream) {
#define PKD_MMA_CASE(d, mt, nt)                                                              \
    if (D == d && MT == mt && NT == nt)                                                      \
        return bf16 ? launch_one<d, true, mt, nt>(tmap, p, grid, stream)                     \
                    : launch_one<d, false, mt, nt>(tmap, p, grid, stream);
    PKD_MMA_CASE(128, 1, 1) PKD_MMA_CASE(128, 1, 2) PKD_MMA_CASE(64, 1, 1) PKD_MMA_CASE(64, 1, 2)
    // 17..32 rows: warp pairs sharing one ring, 16 rows per warp
    if (MT == 2 && D == 128) return bf16 ? launch_pair<128, true>(tmap, p, grid, stream)
                                         : launch_pair<128, false>(tmap, p, grid, stream);
    if (MT == 2 && D == 64) return bf16 ? launch_pair<64, true>(tmap, p, grid, stream)
                                        : launch_pair<64, false>(tmap, p, grid, stream);
#undef PKD_MMA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkd
