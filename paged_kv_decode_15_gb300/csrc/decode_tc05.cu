// Launch of the tcgen05 query-block decode kernel: one persistent CTA per SM.
#include "decode_tc05.cuh"
#include "launch.h"

namespace pkd {

template <bool kBF16, bool kCausal>
static cudaError_t launch_tc(const CUtensorMap& kvmap, const CUtensorMap& qmap, const DecodeParams& p,
                             cudaStream_t stream) {
    auto kern = decode_tc05_kernel<kBF16, kCausal>;
    static PerDevice state;
    int per_sm = 1, grid = 1;
    cudaError_t e = kernel_setup(state, kern, kTcThreads, TcShape::SMEM, &per_sm);
    if (e != cudaSuccess) return e;
    e = persistent_grid(1, 1 << 20, grid);
    if (e != cudaSuccess) return e;
    kern<<<grid, kTcThreads, TcShape::SMEM, stream>>>(kvmap, qmap, p);
    return cudaGetLastError();
}

cudaError_t launch_decode_tc05(bool bf16, const CUtensorMap& kvmap, const CUtensorMap& qmap, const DecodeParams& p,
                               cudaStream_t stream) {
    if (p.causal)
        return bf16 ? launch_tc<true, true>(kvmap, qmap, p, stream) : launch_tc<false, true>(kvmap, qmap, p, stream);
    return bf16 ? launch_tc<true, false>(kvmap, qmap, p, stream) : launch_tc<false, false>(kvmap, qmap, p, stream);
}

}  // namespace pkd
