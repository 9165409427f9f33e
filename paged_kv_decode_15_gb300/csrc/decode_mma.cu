// Instantiations of the tensor-core decode kernel.
#include "decode_mma.cuh"
#include "launch.h"

namespace pkd {

constexpr int kMmaNbuf = 2;
constexpr int kGridWarps = 4;  // warps per CTA of the one-tile kernel
constexpr int kPairNbuf = 4;  // per warp pair: the same 64 KiB of ring per CTA as four rings of two
constexpr int kFp8Nbuf = 2;   // 4 KiB e4m3 stages: two per warp keep four CTAs on an SM (fp8_long_b8: 438 us, three stages 481 us)

template <class W, int D, int ELT, int NBUF>
static cudaError_t launch_one(const CUtensorMap& tmap, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    using S = MmaShape<W, D, ELT, NBUF, kGridWarps>;
    auto kern = decode_mma_kernel<W, D, ELT, NBUF, kGridWarps>;
    static PerDevice state;
    cudaError_t e = kernel_setup(state, kern, kGridWarps * 32, S::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kGridWarps * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}

template <int D, bool kBF16>
static cudaError_t launch_pair(const CUtensorMap& tmap, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    using S = PairShape<D, kPairNbuf>;
    auto kern = decode_mma_pair_kernel<D, kBF16, kPairNbuf>;
    static PerDevice state;
    cudaError_t e = kernel_setup(state, kern, kNW * 32, S::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kNW * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}


cudaError_t launch_decode_mma_fp8(int D, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p, dim3 grid,
                                  cudaStream_t stream) {
    if (D == 128 && MT == 1 && NT == 1) return launch_one<Fp8MmaWarp<1, 1>, 128, 1, kFp8Nbuf>(tmap, p, grid, stream);
    if (D == 128 && MT == 1 && NT == 2) return launch_one<Fp8MmaWarp<1, 2>, 128, 1, kFp8Nbuf>(tmap, p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_mma(int D, bool bf16, int MT, int NT, const CUtensorMap& tmap,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream) {
#define PKD_MMA_CASE(d, mt, nt)                                                                          \
    if (D == d && MT == mt && NT == nt)                                                                  \
        return bf16 ? launch_one<MmaWarp<d, true, mt, nt>, d, 2, kMmaNbuf>(tmap, p, grid, stream)         \
                    : launch_one<MmaWarp<d, false, mt, nt>, d, 2, kMmaNbuf>(tmap, p, grid, stream);
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
