// Flat-partition decode, tensor-core warps, fp8-e4m3 caches (widened to fp16 in shared memory).
#include "flat_launch.cuh"

namespace pkd {

cudaError_t launch_flat_mma_fp8(int D, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p, int max_ctas,
                                cudaStream_t stream) {
#define PKD_CASE(mt, nt) \
    if (D == 128 && MT == mt && NT == nt) return launch_flat_one<Fp8MmaWarp<mt, nt>, 128, 1>(tmap, p, max_ctas, stream);
    PKD_CASE(1, 1) PKD_CASE(1, 2)
    // 17..32 rows: two warps per unit, 16 rows each
    if (D == 128 && MT == 2) return launch_flat_one<Fp8MmaWarp<1, 2>, 128, 1, 2>(tmap, p, max_ctas, stream);
#undef PKD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkd
