// Flat-partition decode, tensor-core warps, bf16 caches.
#include "flat_launch.cuh"

namespace pkd {

cudaError_t launch_flat_mma_bf16(int D, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p, int max_ctas,
                                cudaStream_t stream) {
#define PKD_CASE(d, mt, nt) \
    if (D == d && MT == mt && NT == nt) return launch_flat_one<MmaWarp<d, true, mt, nt>, d, 2>(tmap, p, max_ctas, stream);
    PKD_CASE(128, 1, 1) PKD_CASE(128, 1, 2) PKD_CASE(64, 1, 1) PKD_CASE(64, 1, 2)
    // 17..32 rows: two warps per unit, 16 rows each
    if (MT == 2 && D == 128) return launch_flat_one<MmaWarp<128, true, 1, 2>, 128, 2, 2>(tmap, p, max_ctas, stream);
    if (MT == 2 && D == 64) return launch_flat_one<MmaWarp<64, true, 1, 2>, 64, 2, 2>(tmap, p, max_ctas, stream);
#undef PKD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkd
