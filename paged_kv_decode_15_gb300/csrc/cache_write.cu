// KV-cache write: new key/value rows into their slots of the paged cache,
// quantised to e4m3 for an fp8 cache.
//
// One warp per token.  The token's slot (page, offset) is resolved once; the
// token's key rows of every kv head (Hkv * D contiguous elements) and its
// value rows are then moved as 16-byte input chunks, 32 lanes side by side,
// every load issued before any store.  Chunk c < Hkv*D/8 is key chunk c, the
// rest value chunks; chunk j of a part lies in head j / (D/8) at element
// 8 * (j % (D/8)).  A 16-bit cache receives the input bits; an fp8 cache
// receives e4m3(x / scale) rounded to nearest even with saturation
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
    long long T, key_stride, value_stride, num_slots;  // num_slots = num_pages * P
    int Hkv, D, P, kv_elt, in_bf16;
    float k_scale, v_scale;
    float k_inv, v_inv;     // 1/scale when that scale is a power of two (then x*inv == x/scale exactly), else 0
};

__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

constexpr int kChunksPerLane = 8;  // loads in flight per lane (a token of 8 heads x 128: all of it)

// D, the cache type, the input type and the division mode are template
// parameters so that the per-chunk work has no runtime branches.
template <int D, bool kFp8, bool kBF16In, bool kExactInv>
__global__ void __launch_bounds__(128) cache_write_kernel(const CacheWriteParams p) {
    constexpr int kDShift = D == 128 ? 4 : 3;  // log2 of the 16-byte input chunks per head row
    constexpr int kEltOut = kFp8 ? 1 : 2;
    const long long t = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= p.T) return;
    const long long s = __ldg(p.slots + t);
    if (s < 0 || s >= p.num_slots) return;  // padding (negative) or outside the cache: nothing written
    const int page = static_cast<int>(s / p.P), off = static_cast<int>(s % p.P);
    const int per_part = p.Hkv << kDShift;  // 16-byte input chunks of the key rows (and of the value rows)
    const int total = 2 * per_part;
    constexpr int dmask = (1 << kDShift) - 1;
    const uint8_t* krow = p.key + t * p.key_stride * 2;
    const uint8_t* vrow = p.value + t * p.value_stride * 2;
    // cache row of (page, head 0, off): heads are P rows apart
    uint8_t* dst0 = p.cache + ((static_cast<long long>(page) * p.Hkv * p.P + off) * 2 * D) * kEltOut;
    const long long head_stride = static_cast<long long>(p.P) * 2 * D * kEltOut;

    for (int base = 0; base < total; base += 32 * kChunksPerLane) {
        uint4 v[kChunksPerLane];
#pragma unroll
        for (int i = 0; i < kChunksPerLane; ++i) {
            const int c = base + i * 32 + lane;
            if (c < total) {
                const int part = c >= per_part, j = c - part * per_part;
                v[i] = __ldg(reinterpret_cast<const uint4*>((part ? vrow : krow) + j * 16));
            }
        }
#pragma unroll
        for (int i = 0; i < kChunksPerLane; ++i) {
            const int c = base + i * 32 + lane;
            if (c >= total) continue;
            const int part = c >= per_part, j = c - part * per_part;
            const int h = j >> kDShift, e = (j & dmask) * 8;  // head, first element of the chunk
            uint8_t* dst = dst0 + h * head_stride + (part * D + e) * kEltOut;
            if constexpr (!kFp8) {
                *reinterpret_cast<uint4*>(dst) = v[i];
            } else {
                const float scale = part ? p.v_scale : p.k_scale;
                const float inv = part ? p.v_inv : p.k_inv;
                auto q8 = [&](float x) { return kExactInv ? x * inv : __fdiv_rn(x, scale); };
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t out[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float f[4];
                    if constexpr (kBF16In) {
                        bf16x2_to_f32(w[2 * q], f[0], f[1]);
                        bf16x2_to_f32(w[2 * q + 1], f[2], f[3]);
                    } else {
                        f16x2_to_f32(w[2 * q], f[0], f[1]);
                        f16x2_to_f32(w[2 * q + 1], f[2], f[3]);
                    }
                    out[q] = f32x2_to_e4m3x2(q8(f[0]), q8(f[1])) | (f32x2_to_e4m3x2(q8(f[2]), q8(f[3])) << 16);
                }
                *reinterpret_cast<uint2*>(dst) = make_uint2(out[0], out[1]);
            }
        }
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
    p.num_slots = num_pages * P;
    p.Hkv = Hkv;
    p.D = D;
    p.P = P;
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
    if (T == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((T + 3) / 4));
    const bool fp8 = p.kv_elt == 1, exact = p.k_inv != 0.f && p.v_inv != 0.f;
#define PKD_CW(d, f8, bf, ex) \
    if (D == d && fp8 == f8 && (f8 ? (p.in_bf16 != 0) == bf && exact == ex : !bf && !ex)) \
        cache_write_kernel<d, f8, bf, ex><<<grid, 128, 0, stream>>>(p);
    PKD_CW(128, false, false, false) PKD_CW(64, false, false, false)
    PKD_CW(128, true, true, true) PKD_CW(128, true, true, false) PKD_CW(128, true, false, true) PKD_CW(128, true, false, false)
    PKD_CW(64, true, true, true) PKD_CW(64, true, true, false) PKD_CW(64, true, false, true) PKD_CW(64, true, false, false)
#undef PKD_CW
    return cudaGetLastError();
}

}  // namespace pkd
