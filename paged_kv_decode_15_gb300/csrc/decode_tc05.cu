// Launch of the tcgen05 query-block decode kernel (one persistent CTA per SM)
// and, when requests may be split into several chunks, of the merge kernel.
#include "decode_tc05.cuh"
#include "launch.h"

namespace pkd {

// LSE merge of the chunk partials of split (request, kv head) units.  One
// warp per (unit, query row), eight rows per CTA: lane j reads chunk j's LSE
// (blocks of 32 chunks), shuffles give the maximum, the weights and their
// sum, and each lane sums dims 4*lane .. +3 over the chunks with every load
// of a block issued before the first is used.  Units with one chunk were
// written by the main kernel and are skipped.
constexpr int kTcMergeRows = 8;

__global__ void __launch_bounds__(kTcMergeRows * 32)
tc_merge_kernel(const DecodeParams p) {
    const int unit = blockIdx.x / (kTcRows / kTcMergeRows), b = unit / p.Hkv, hk = unit - b * p.Hkv;
    const int r = (blockIdx.x % (kTcRows / kTcMergeRows)) * kTcMergeRows + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= p.M) return;
    // launched as a programmatic dependent of the main kernel: wait for it to
    // complete (and its partials to be visible) before reading them
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int L = clamp_len(p, b, false), vis = L - visible_lo(p, L);
    const int nch = (vis + p.chunk - 1) / p.chunk;
    if (nch <= 1) return;
    const float* pl = p.part_lse + static_cast<long long>(unit) * p.max_splits * kTcRows + r;
    const float* pob = p.part_out + (static_cast<long long>(unit) * p.max_splits * kTcRows + r) * 128 + 4 * lane;
    float mx = -INFINITY;
    for (int cc = lane; cc < nch; cc += 32) mx = fmaxf(mx, __ldcg(pl + cc * kTcRows));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    float ws = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cb = 0; cb < nch; cb += 32) {
        const int cc = cb + lane, n = min(32, nch - cb);
        const float lc = cc < nch ? __ldcg(pl + cc * kTcRows) : -INFINITY;
        const float wl = lc == -INFINITY ? 0.f : fast_exp2(lc - mx);
        ws += wl;
        float4 v[8];
        for (int j0 = 0; j0 < n; j0 += 8) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = j0 + j < n ? __ldcg(reinterpret_cast<const float4*>(pob + static_cast<long long>(cb + j0 + j) * kTcRows * 128))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float w = __shfl_sync(kFull, wl, (j0 + j) & 31);
                if (j0 + j < n && w > 0.f)
                    acc = make_float4(fmaf(w, v[j].x, acc.x), fmaf(w, v[j].y, acc.y), fmaf(w, v[j].z, acc.z),
                                      fmaf(w, v[j].w, acc.w));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(kFull, ws, o);
    const float sc = ws > 0.f ? p.v_scale / ws : 0.f;
    const long long orow = static_cast<long long>(b) * p.sq * p.Hq + hk * p.G + static_cast<long long>(r / p.G) * p.Hq + r % p.G;
    const long long o0 = orow * 128 + 4 * lane;
    store_out(p.out, o0 + 0, acc.x * sc, p.out_dtype);
    store_out(p.out, o0 + 1, acc.y * sc, p.out_dtype);
    store_out(p.out, o0 + 2, acc.z * sc, p.out_dtype);
    store_out(p.out, o0 + 3, acc.w * sc, p.out_dtype);
    if (lane == 0 && p.lse) p.lse[orow] = ws > 0.f ? (mx + __log2f(ws)) * kLn2 : -INFINITY;
}

template <bool kBF16>
static cudaError_t launch_tc(const CUtensorMap& kvmap, const CUtensorMap& qmap, const DecodeParams& p,
                             cudaStream_t stream) {
    auto kern = decode_tc05_kernel<kBF16>;
    static PerDevice state;
    int per_sm = 1, grid = 1;
    cudaError_t e = kernel_setup(state, kern, kTcThreads, TcShape::SMEM, &per_sm);
    if (e != cudaSuccess) return e;
    e = persistent_grid(1, 1 << 20, grid);
    if (e != cudaSuccess) return e;
    kern<<<grid, kTcThreads, TcShape::SMEM, stream>>>(kvmap, qmap, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the chunk partials of split units, merged by LSE; a programmatic
    // dependent launch, so that its CTAs are resident when the main kernel ends
    if (p.max_splits > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(p.B * p.Hkv * (kTcRows / kTcMergeRows));
        cfg.blockDim = dim3(kTcMergeRows * 32);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, tc_merge_kernel, p);
    }
    return e;
}

cudaError_t launch_decode_tc05(bool bf16, const CUtensorMap& kvmap, const CUtensorMap& qmap, const DecodeParams& p,
                               cudaStream_t stream) {
    return bf16 ? launch_tc<true>(kvmap, qmap, p, stream) : launch_tc<false>(kvmap, qmap, p, stream);
}

}  // namespace pkd
