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
    static int per_sm = 0;  // benign race: every thread computes the same value
    if (per_sm == 0) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kNW * 32, S::SMEM);
        if (e != cudaSuccess) return e;
        per_sm = n > 0 ? n : 1;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int grid = sms * per_sm;
    if (grid > max_ctas) grid = max_ctas;
    kern<<<grid, kNW * 32, S::SMEM, stream>>>(tmap, p);
    return cudaGetLastError();
}

}  // namespace pkd
