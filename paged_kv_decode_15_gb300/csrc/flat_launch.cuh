// Launch helper for the persistent flat-partition decode kernel; included by
// the per-dtype translation units so that they compile in parallel.
#pragma once

#include "decode_flat.cuh"
#include "launch.h"

namespace pkd {

template <class W, int D, int ELT, int RT = 1>
cudaError_t launch_flat_one(const CUtensorMap& tmap, const DecodeParams& p, int max_ctas, cudaStream_t stream) {
    using S = FlatShape<D, ELT, W::kNbuf, W::kScratchBytes>;
    auto kern = decode_flat_kernel<W, D, ELT, W::kNbuf, RT>;
    static PerDevice state;
    int per_sm = 1, grid = 1;
    cudaError_t e = kernel_setup(state, kern, kNW * 32, S::SMEM, &per_sm);
    if (e != cudaSuccess) return e;
    e = persistent_grid(per_sm, max_ctas, grid);
    if (e != cudaSuccess) return e;
    kern<<<grid, kNW * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}

}  // namespace pkd
