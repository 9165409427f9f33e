// Host-side entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pkd.h"

namespace pkd {

struct DecodeParams;

// Dynamic shared memory of a decode kernel variant (bytes), or -1 if the
// variant is not built.
int decode_mma_smem(int D, int MT, int NT);
int decode_fma_smem(int D, int kvt, int LPT, int MR);

// Launch one decode kernel variant on `stream`; grid = (max_splits, Hkv, B).
cudaError_t launch_decode_mma(int D, bool bf16, int MT, int NT, const CUtensorMap& tmap,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream);
cudaError_t launch_decode_fma(int D, int kvt, int LPT, int MR, const CUtensorMap& tmap,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream);

// Record `fmt` as this thread's last error message and return `st`.
int report_status(int st, const char* fmt, ...);
template <class... A>
inline pkd_status report(pkd_status st, const char* fmt, A... a) {
    return static_cast<pkd_status>(report_status(static_cast<int>(st), fmt, a...));
}

struct SegmentParams;
struct MergeParams;
cudaError_t launch_segmented(const SegmentParams& p, cudaStream_t stream);
cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream);

}  // namespace pkd
