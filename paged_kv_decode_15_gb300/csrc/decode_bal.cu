// Instantiations of the persistent per-CTA-partition decode kernel.
#include "decode_bal.cuh"
#include "launch.h"

namespace pkd {

template <class Body, int D>
static cudaError_t launch_bal_one(const CUtensorMap& tmap, const DecodeParams& p, cudaStream_t stream) {
    using S = typename Body::S;
    auto kern = decode_bal_kernel<Body, D>;
    static PerDevice state;
    int per_sm = 1, grid = 1;
    cudaError_t e = kernel_setup(state, kern, kNW * 32, S::SMEM, &per_sm);
    if (e != cudaSuccess) return e;
    e = persistent_grid(per_sm, kBalMaxCtas, grid);
    if (e != cudaSuccess) return e;
    kern<<<grid, kNW * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}

cudaError_t launch_decode_bal(int D, bool bf16, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p,
                              cudaStream_t stream) {
#define PKD_BAL_CASE(d, nt)                                                                     \
    if (D == d && MT == 1 && NT == nt)                                                          \
        return bf16 ? launch_bal_one<WarpsBody<d, true, nt>, d>(tmap, p, stream)                \
                    : launch_bal_one<WarpsBody<d, false, nt>, d>(tmap, p, stream);
    PKD_BAL_CASE(128, 1) PKD_BAL_CASE(128, 2) PKD_BAL_CASE(64, 1) PKD_BAL_CASE(64, 2)
#undef PKD_BAL_CASE
    if (MT == 2 && D == 128) return bf16 ? launch_bal_one<PairBody<128, true>, 128>(tmap, p, stream)
                                         : launch_bal_one<PairBody<128, false>, 128>(tmap, p, stream);
    if (MT == 2 && D == 64) return bf16 ? launch_bal_one<PairBody<64, true>, 64>(tmap, p, stream)
                                        : launch_bal_one<PairBody<64, false>, 64>(tmap, p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkd
