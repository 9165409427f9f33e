// Paged decode with a library-owned, statically allocated scratch area.
//
// pkd_paged_decode needs a workspace for its Split-KV partial results, and
// asks the caller to provide it.  Some callers cannot allocate device memory
// when they need to run decode: plug-ins hosted by a runtime that owns all
// device memory and hands none out, serving loops that must not allocate once
// their memory budget is fixed, or C callers that link only this library and
// have no allocator of their own.  pkd_paged_decode_static serves them: it uses the
// fixed scratch array below, which is part of the library image, so the call
// itself allocates nothing.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "../../include/pkd.h"
#include "launch.h"

namespace {

// Every GPU that loads the library reserves this much device memory until
// the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

using pkd::kMaxDevices;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per
// device.  In host code the name g_scratch is only a host-side stand-in, so
// the address must come from the runtime.  The address is kept for the life
// of the process: a device reset (cudaDeviceReset) reloads the module and may
// move the array, so the static call must not be used across one.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" pkd_status pkd_paged_decode_static(const void* q, pkd_dtype q_dtype, const void* kv_cache,
                                              pkd_dtype kv_dtype, int64_t num_pages, const int32_t* block_table,
                                              int64_t block_table_stride, const int32_t* seq_lens, int batch,
                                              int sq, int num_heads, int num_kv_heads, int head_dim, int page_size,
                                              int max_kv_len, float scale, float q_scale, float k_scale,
                                              float v_scale, int window, void* out, pkd_dtype out_dtype,
                                              float* lse, int chunk_tokens, unsigned flags, void* stream) {
    const size_t need = pkd_paged_decode_workspace_size(batch, sq, num_heads, num_kv_heads, head_dim, page_size,
                                                        max_kv_len, kv_dtype, window, chunk_tokens, flags);
    if (need == 0) return PKD_EINVAL;  // the plan was rejected; pkd_last_error says why
    if (need > kStaticScratchBytes) {
        const char* kern = pkd_paged_decode_kernel_name(batch, sq, num_heads, num_kv_heads, head_dim, page_size,
                                                        max_kv_len, kv_dtype, window, chunk_tokens, flags);
        const bool chunked = kern && std::strncmp(kern, "chunked grid", 12) == 0;
        return pkd::report(PKD_EUNSUPPORTED, "the plan (%s) needs %zu bytes of scratch, above the static %zu; use "
                           "pkd_paged_decode with a caller workspace%s", kern ? kern : "?", need,
                           kStaticScratchBytes, chunked ? ", or a larger chunk_tokens" : "");
    }
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return pkd::report(PKD_ECUDA, "static scratch address: %s", cudaGetErrorString(e));
    // the last call's counters and status word may be left over: start from zero
    pkd_status st = pkd_workspace_init(scratch, need, stream);
    if (st != PKD_OK) return st;
    return pkd_paged_decode(q, q_dtype, kv_cache, kv_dtype, num_pages, block_table, block_table_stride, seq_lens,
                            batch, sq, num_heads, num_kv_heads, head_dim, page_size, max_kv_len, scale, q_scale,
                            k_scale, v_scale, window, out, out_dtype, lse, scratch, kStaticScratchBytes,
                            chunk_tokens, flags, stream);
}

extern "C" pkd_status pkd_paged_decode_static_check(void* stream) {
    void* scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return pkd::report(PKD_ECUDA, "static scratch address: %s", cudaGetErrorString(e));
    // the status word sits at the start of the scratch, as in a caller workspace
    return pkd_workspace_check(scratch, kStaticScratchBytes, stream);
}
