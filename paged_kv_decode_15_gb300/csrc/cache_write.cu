// KV-cache write: new key/value rows into their slots of the paged cache,
// quantised to e4m3 for an fp8 cache.
//
// Each warp moves kItemsPerWarp (token, kv head) rows; lanes 0-15 move key
// rows, lanes 16-31 value rows, 16 input bytes each, all loads issued first.  A 16-bit cache receives the input bits; an
// fp8 cache receives e4m3(x / scale) rounded to nearest even with saturation
// (cvt.rn.satfinite), the quotient an IEEE fp32 division (a multiply by the
// exact reciprocal when the scale is a power of two: the same rounded value).
#include "launch.h"
#include "ptx.cuh"

namespace pkd {

struct CacheWriteParams {
    const uint8_t* key;     // [T, Hkv, D] rows, token stride key_stride elements
    const uint8_t* value;
    const int64_t* slots;   // [T]
    uint8_t* cache;         // [num_pages, Hkv, P, 2D]
    long long T, key_stride, value_stride, num_pages;
    int Hkv, D, P, in_elt, kv_elt, in_bf16;
    float k_scale, v_scale;
    float k_inv, v_inv;  // 1/scale when that scale is a power of two (then x*inv == x/scale exactly), else 0
};

// x / scale rounded to nearest: a multiply when the reciprocal is exact
__device__ __forceinline__ float scaled(float x, float scale, float inv) {
    return inv != 0.f ? x * inv : __fdiv_rn(x, scale);
}

__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

constexpr int kItemsPerWarp = 4;  // (token, kv head) rows per warp, loaded before any is stored

__global__ void __launch_bounds__(128) cache_write_kernel(const CacheWriteParams p) {
    const long long w0 = (static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5)) * kItemsPerWarp;
    const int lane = threadIdx.x & 31;
    const int part = lane >> 4, c = lane & 15;  // part 0: key, 1: value; 16-byte input chunk c
    const int chunks = p.D * p.in_elt / 16;
    const long long total = p.T * p.Hkv;
    uint4 v[kItemsPerWarp];
    long long slot[kItemsPerWarp];
    uint8_t* dst[kItemsPerWarp];
    // every load first (rows and slots are independent), then the stores
#pragma unroll
    for (int it = 0; it < kItemsPerWarp; ++it) {
        const long long wid = w0 + it;
        slot[it] = -1;
        if (wid >= total || c >= chunks) continue;
        const long long t = wid / p.Hkv;  // consecutive rows: the kv heads of one token, then the next token
        const int h = static_cast<int>(wid % p.Hkv);
        const uint8_t* src = (part ? p.value + (t * p.value_stride + static_cast<long long>(h) * p.D) * p.in_elt
                                   : p.key + (t * p.key_stride + static_cast<long long>(h) * p.D) * p.in_elt) +
                             c * 16;
        v[it] = __ldg(reinterpret_cast<const uint4*>(src));
        slot[it] = __ldg(p.slots + t);
    }
#pragma unroll
    for (int it = 0; it < kItemsPerWarp; ++it) {
        dst[it] = nullptr;
        const long long s = slot[it];
        if (s < 0 || s / p.P >= p.num_pages) continue;
        const long long wid = w0 + it;
        const int h = static_cast<int>(wid % p.Hkv);
        const long long page = s / p.P, off = s % p.P;
        dst[it] = p.cache + (((page * p.Hkv + h) * p.P + off) * 2 * p.D + part * p.D) * p.kv_elt;
    }
    const float scale = part ? p.v_scale : p.k_scale;
    const float inv = part ? p.v_inv : p.k_inv;
#pragma unroll
    for (int it = 0; it < kItemsPerWarp; ++it) {
        if (!dst[it]) continue;
        if (p.kv_elt == 2) {
            *reinterpret_cast<uint4*>(dst[it] + c * 16) = v[it];
            continue;
        }
        const uint32_t w[4] = {v[it].x, v[it].y, v[it].z, v[it].w};
        uint32_t out[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float f[4];
            if (p.in_bf16) {
                bf16x2_to_f32(w[2 * i], f[0], f[1]);
                bf16x2_to_f32(w[2 * i + 1], f[2], f[3]);
            } else {
                f16x2_to_f32(w[2 * i], f[0], f[1]);
                f16x2_to_f32(w[2 * i + 1], f[2], f[3]);
            }
            out[i] = f32x2_to_e4m3x2(scaled(f[0], scale, inv), scaled(f[1], scale, inv)) |
                     (f32x2_to_e4m3x2(scaled(f[2], scale, inv), scaled(f[3], scale, inv)) << 16);
        }
        *reinterpret_cast<uint2*>(dst[it] + c * 8) = make_uint2(out[0], out[1]);
    }
}

cudaError_t launch_cache_write(const void* key, const void* value, int in_dtype, const int64_t* slots,
                               long long T, long long key_stride, long long value_stride, int Hkv, int D, int P,
                               long long num_pages, void* cache, int kv_dtype, float k_scale, float v_scale,
                               cudaStream_t stream) {
    CacheWriteParams p;
    p.key = static_cast<const uint8_t*>(key);
    p.value = static_cast<const uint8_t*>(value);
    p.slots = slots;
    p.cache = static_cast<uint8_t*>(cache);
    p.T = T;
    p.key_stride = key_stride;
    p.value_stride = value_stride;
    p.num_pages = num_pages;
    p.Hkv = Hkv;
    p.D = D;
    p.P = P;
    p.in_elt = 2;
    p.kv_elt = kv_dtype == 2 ? 1 : 2;
    p.in_bf16 = in_dtype == 0;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    // a power-of-two scale has an exact reciprocal (within the normal range)
    auto exact_inv = [](float s) {
        int e;
        const float m = frexpf(s, &e);
        return (m == 0.5f && e > -120 && e < 120) ? 1.0f / s : 0.0f;
    };
    p.k_inv = exact_inv(k_scale);
    p.v_inv = exact_inv(v_scale);
    const long long warps = (T * Hkv + kItemsPerWarp - 1) / kItemsPerWarp;
    if (warps == 0) return cudaSuccess;
    cache_write_kernel<<<static_cast<unsigned>((warps + 3) / 4), 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkd
