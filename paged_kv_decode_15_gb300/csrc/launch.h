// Host-side entry points of the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pkd.h"
#include "device_state.h"

namespace pkd {

// Set the dynamic shared-memory limit of `kern` on the current device, once
// per device, and report how many CTAs of `threads` threads fit one SM there.
template <class K>
cudaError_t kernel_setup(PerDevice& state, K kern, int threads, int smem, int* per_sm = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaError_t err = cudaSuccess;
    const int n = state.get(
        dev,
        [&]() -> int {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (err != cudaSuccess) return -1;
            int b = 0;
            err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, threads, smem);
            if (err != cudaSuccess) return -1;
            return b > 0 ? b : 1;  // a kernel that fits nowhere fails at launch
        },
        -2);
    if (n == -2) return cudaErrorInvalidDevice;
    if (n <= 0) return err;
    if (per_sm) *per_sm = n;
    return cudaSuccess;
}

// Resident CTAs of a persistent grid on the current device: SMs x per_sm.
inline cudaError_t persistent_grid(int per_sm, int max_ctas, int& grid) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    grid = sms * per_sm;
    if (grid > max_ctas) grid = max_ctas;
    if (grid < 1) grid = 1;
    return cudaSuccess;
}

struct DecodeParams;

// Launch one decode kernel variant on `stream`; grid = (max_splits, Hkv, B).
cudaError_t launch_decode_mma(int D, bool bf16, int MT, int NT, const CUtensorMap& tmap,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream);
// Query blocks of 17-32 rows (16-bit caches, head_dim 128, no causal mask) on
// tcgen05 tensor cores: persistent CTAs, one per SM, taking work items from a
// queue.  kvmap: the stage map with boxes of 8 rows and every 128-byte chunk;
// qmap: q as {dims, heads, tokens} with boxes {64, G, sq}.
cudaError_t launch_decode_tc05(bool bf16, const CUtensorMap& kvmap, const CUtensorMap& qmap, const DecodeParams& p,
                               cudaStream_t stream);
// e4m3 caches on tensor cores in the chunked grid (M <= 16)
cudaError_t launch_decode_mma_fp8(int D, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p, dim3 grid,
                                  cudaStream_t stream);
cudaError_t launch_decode_fma(int D, int kvt, int LPT, int MR, const CUtensorMap& tmap,
                              const DecodeParams& p, dim3 grid, cudaStream_t stream);

// Persistent per-CTA partition, tensor cores, 16-bit caches: the grid fills
// the GPU once (at most 512 CTAs, two partial slots each in the workspace).
cudaError_t launch_decode_bal(int D, bool bf16, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p,
                              cudaStream_t stream);

// Persistent flat-partition decode: the grid fills the GPU once (at most
// max_ctas CTAs, one partial slot pair per warp in the workspace).
cudaError_t launch_flat_mma_bf16(int D, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p,
                                 int max_ctas, cudaStream_t stream);
cudaError_t launch_flat_mma_fp16(int D, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p,
                                 int max_ctas, cudaStream_t stream);
cudaError_t launch_flat_mma_fp8(int D, int MT, int NT, const CUtensorMap& tmap, const DecodeParams& p,
                                int max_ctas, cudaStream_t stream);
cudaError_t launch_flat_fma_bf16(int D, int LPT, int MR, const CUtensorMap& tmap, const DecodeParams& p,
                                 int max_ctas, cudaStream_t stream);
cudaError_t launch_flat_fma_fp16(int D, int LPT, int MR, const CUtensorMap& tmap, const DecodeParams& p,
                                 int max_ctas, cudaStream_t stream);
cudaError_t launch_flat_fma_fp8(int D, int LPT, int MR, const CUtensorMap& tmap, const DecodeParams& p,
                                int max_ctas, cudaStream_t stream);

// Record `fmt` as this thread's last error message and return `st`.
int report_status(int st, const char* fmt, ...);
template <class... A>
inline pkd_status report(pkd_status st, const char* fmt, A... a) {
    return static_cast<pkd_status>(report_status(static_cast<int>(st), fmt, a...));
}

cudaError_t launch_cache_write(const void* key, const void* value, int in_dtype, const int64_t* slots,
                               long long T, long long key_stride, long long value_stride, int Hkv, int D, int P,
                               long long num_pages, void* cache, int kv_dtype, float k_scale, float v_scale,
                               cudaStream_t stream);

struct SegmentParams;
struct MergeParams;
cudaError_t launch_segmented(const SegmentParams& p, cudaStream_t stream);
cudaError_t launch_lse_merge(const MergeParams& p, cudaStream_t stream);

}  // namespace pkd
