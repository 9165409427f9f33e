// Instantiations of the CUDA-core decode kernel.
#include "decode_fma.cuh"
#include "launch.h"

namespace pkd {

constexpr int kFmaNbuf = 2;

template <int D, int KVT, int LPT, int MR>
static cudaError_t launch_one(const CUtensorMap& tmap, const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    using S = FmaShape<D, KVT, LPT, MR, kFmaNbuf>;
    auto kern = decode_fma_kernel<D, KVT, LPT, MR, kFmaNbuf>;
    static PerDevice state;
    cudaError_t e = kernel_setup(state, kern, kNW * 32, S::SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, kNW * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}

#define PKD_FMA_VARIANTS(X)                                                   \
    X(128, 0, 8, 2) X(128, 0, 8, 4) X(128, 0, 16, 8)                          \
    X(128, 1, 8, 2) X(128, 1, 8, 4) X(128, 1, 16, 8)                          \
    X(128, 2, 8, 2) X(128, 2, 8, 4) X(128, 2, 16, 8)                          \
    X(64, 0, 8, 2) X(64, 0, 8, 4) X(64, 0, 16, 8)                             \
    X(64, 1, 8, 2) X(64, 1, 8, 4) X(64, 1, 16, 8)

cudaError_t launch_decode_fma(int D, int kvt, int LPT, int MR, const CUtensorMap& tmap,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream) {
#define PKD_FMA_CASE(d, k, l, m) \
    if (D == d && kvt == k && LPT == l && MR == m) return launch_one<d, k, l, m>(tmap, p, grid, stream);
    PKD_FMA_VARIANTS(PKD_FMA_CASE)
#undef PKD_FMA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkd
