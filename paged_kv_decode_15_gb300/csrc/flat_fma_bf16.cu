// Flat-partition decode, CUDA-core warps, bf16 caches.
#include "flat_launch.cuh"

namespace pkd {

cudaError_t launch_flat_fma_bf16(int D, int LPT, int MR, const CUtensorMap& tmap, const DecodeParams& p, int max_ctas,
                                 cudaStream_t stream) {
#define PKD_CASE(d, l, m) \
    if (D == d && LPT == l && MR == m) \
        return launch_flat_one<FmaWarp<d, 0, l, m>, d, KvType<0>::ELT>(tmap, p, max_ctas, stream);
    PKD_CASE(128, 8, 2) PKD_CASE(128, 8, 4) PKD_CASE(128, 16, 8)
    PKD_CASE(64, 8, 2) PKD_CASE(64, 8, 4) PKD_CASE(64, 16, 8)
#undef PKD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkd
