// Shared pieces of the paged-decode kernels: launch parameters, the per-CTA
// work decomposition (visible keys, Split-KV chunk), the swizzled stage
// layout that the TMA loads produce, and the CTA epilogue that merges the
// warps' partial softmax states and then, across CTAs, the Split-KV chunks.
#pragma once

#include "page_math.h"
#include "ptx.cuh"

namespace pkd {

constexpr int kNW = 4;          // consumer warps per CTA (one warp group)
constexpr int kStageTok = 16;   // keys per pipeline stage (one TMA box height)
constexpr int kMaxCtaPages = 256;
constexpr int kFlatMaxBatch = 1024;    // the flat kernel keeps per-request tables in shared memory
constexpr int kFlatMaxWorkers = 2048;  // and two partial slots per warp in the workspace
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct DecodeParams {
    const void* q;               // [B, sq, Hq, D]
    const int32_t* block_table;  // [B, bt_stride]
    const int32_t* seq_lens;     // [B]
    void* out;                   // [B, sq, Hq, D]
    float* lse;                  // [B, sq, Hq] or null
    int32_t* status;             // workspace status word
    int32_t* counters;           // [B * Hkv] Split-KV arrival counters
    float* part_lse;             // [B * Hkv, max_splits, M] (log2 domain)
    float* part_out;             // [B * Hkv, max_splits, M, D]
    long long bt_stride;
    long long num_pages;
    int B, sq, Hq, Hkv, G, M, P;
    int max_kv_len, chunk, max_splits, window, causal;
    int chunk_share;             // tcgen05 kernel: chunk when CTAs take tile shares
    int out_dtype;               // 0 bf16, 1 fp16, 3 fp32
    uint32_t pmagic;             // tok / P == (tok * pmagic) >> pmshift for 0 <= tok < 2^31
    int pmshift;
    float scale_log2;            // scale * q_scale * k_scale * log2(e)
    float v_scale;
    uint64_t wait_ns;            // limit of a wait on a stage's copy (0: test once)
};

struct CtaWork {
    int b, hk, split, nsplit;
    int L;        // sequence length (clamped to [0, max_kv_len])
    int t0, t1;   // this CTA's keys [t0, t1)
};

__device__ __forceinline__ void raise_status(const DecodeParams& p, int bits) {
    atomicOr(p.status, bits);
}

// Byte offset of (row, byte) inside a region of 16-row TMA boxes, each box
// 128 bytes wide and written with the 128-byte swizzle: the 16-byte chunk
// index is XOR-ed with (row % 8).  Consecutive boxes of a row are 2 KiB apart.
__device__ __forceinline__ uint32_t swz(int row, int byte) {
    const int box = byte >> 7;
    const int chunk = (byte >> 4) & 7;
    return static_cast<uint32_t>(box * 2048 + row * 128 + (((chunk ^ (row & 7)) << 4) | (byte & 15)));
}

__device__ __forceinline__ void store_out(void* out, long long idx, float v, int dt) {
    if (dt == 0)
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else if (dt == 1)
        reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
    else
        reinterpret_cast<float*>(out)[idx] = v;
}

// Output element index of (row r = i*G + g, dim d) of (b, hk).
__device__ __forceinline__ long long out_index(const DecodeParams& p, int b, int hk, int r, int d, int D) {
    const int i = r / p.G, g = r - (r / p.G) * p.G;
    return ((static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g) * D + d;
}

// Sequence length of request b, clamped to [0, max_kv_len]; an out-of-range
// length raises the status word when `report` is set.
__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b, bool report) {
    int L = p.seq_lens[b];
    if (L < 0 || L > p.max_kv_len) {
        if (report) raise_status(p, kErrBounds);
        L = L < 0 ? 0 : p.max_kv_len;
    }
    return L;
}

// First visible key of a request of length L: 0, or with a window the
// page-aligned start shared by the query block (dense), or the earliest key
// any row of the block can see, page-aligned (causal).
__device__ __forceinline__ int visible_lo(const DecodeParams& p, int L) {
    if (p.window <= 0) return 0;
    const int first = p.causal ? L - p.sq - p.window + 1 : L - (p.window + p.sq - 1);
    return first > 0 ? (first / p.P) * p.P : 0;
}

// out = 0, lse = -inf for every row of request b (it has no visible key).
template <int D>
__device__ __forceinline__ void write_empty_request(const DecodeParams& p, int b) {
    for (int e = threadIdx.x; e < p.Hkv * p.M * D; e += blockDim.x) {
        const int hk = e / (p.M * D), r = (e / D) % p.M, d = e % D;
        store_out(p.out, out_index(p, b, hk, r, d, D), 0.f, p.out_dtype);
        if (d == 0 && p.lse) {
            const int i = r / p.G, g = r % p.G;
            p.lse[(static_cast<long long>(b) * p.sq + i) * p.Hq + hk * p.G + g] = -INFINITY;
        }
    }
}

// Visible-key range and Split-KV chunk of this CTA.  Returns false when the
// CTA has nothing to do (it has then written what it owed).
template <int D>
__device__ bool cta_setup(const DecodeParams& p, CtaWork& w) {
    w.split = blockIdx.x;
    w.hk = blockIdx.y;
    w.b = blockIdx.z;
    int L = p.seq_lens[w.b];
    if (L < 0 || L > p.max_kv_len) {
        if (threadIdx.x == 0) raise_status(p, kErrBounds);
        L = L < 0 ? 0 : p.max_kv_len;
    }
    w.L = L;
    int lo = 0;
    if (p.window > 0) {
        // dense: the page-aligned suffix shared by the whole query block;
        // causal: the earliest key any row of the block can see, page-aligned.
        const int first = p.causal ? L - p.sq - p.window + 1 : L - (p.window + p.sq - 1);
        lo = first > 0 ? (first / p.P) * p.P : 0;
    }
    const int nvis = L - lo;
    w.nsplit = nvis > 0 ? (nvis + p.chunk - 1) / p.chunk : 0;
    if (w.nsplit > p.max_splits) {
        if (threadIdx.x == 0) raise_status(p, kErrBounds);
        w.nsplit = p.max_splits;
    }
    if (w.nsplit == 0) {
        // no visible key: out = 0, lse = -inf, written by the first chunk's CTA
        if (w.split == 0) {
            for (int e = threadIdx.x; e < p.M * D; e += blockDim.x)
                store_out(p.out, out_index(p, w.b, w.hk, e / D, e % D, D), 0.f, p.out_dtype);
            if (p.lse)
                for (int r = threadIdx.x; r < p.M; r += blockDim.x) {
                    const int i = r / p.G, g = r % p.G;
                    p.lse[(static_cast<long long>(w.b) * p.sq + i) * p.Hq + w.hk * p.G + g] = -INFINITY;
                }
        }
        return false;
    }
    if (w.split >= w.nsplit) return false;
    w.t0 = lo + w.split * p.chunk;
    w.t1 = min(w.t0 + p.chunk, L);
    return true;
}

// Is key `tok` visible to query row `row` (row < M)?  Keys are already known
// to lie in this CTA's [t0, t1) and hence in the block's visible range.
__device__ __forceinline__ bool row_sees(const DecodeParams& p, int L, int row, int tok) {
    if (row >= p.M) return false;
    if (!p.causal) return true;
    const int pos = L - p.sq + row / p.G;
    if (tok > pos) return false;
    return p.window <= 0 || tok >= pos - (p.window - 1);
}

// Table column and slot of key `tok` without a division: a 32x32->64-bit
// multiply by a magic number and a shift (division by an invariant integer,
// Granlund and Montgomery, exact for every dividend below 2^31).
__device__ __forceinline__ int page_col(const DecodeParams& p, int tok) {
    return page_div(tok, p.pmagic, p.pmshift);
}
__device__ __forceinline__ int page_slot(const DecodeParams& p, int tok) { return tok - page_col(p, tok) * p.P; }

// Load the page indices of this CTA's keys [t0, t1) into shared memory
// (pages[i] holds table column t0/P + i; t0 need not be page-aligned); a page
// outside [0, num_pages) becomes -1 (its keys are skipped) and raises the
// status word.
__device__ __forceinline__ void load_cta_pages(const DecodeParams& p, const CtaWork& w, int* pages) {
    const int npages = w.t1 > w.t0 ? (w.t1 - 1) / p.P - w.t0 / p.P + 1 : 0;
    const long long base = static_cast<long long>(w.b) * p.bt_stride + w.t0 / p.P;
    for (int i = threadIdx.x; i < npages; i += blockDim.x) {
        int pg = p.block_table[base + i];
        if (pg < 0 || pg >= p.num_pages) {
            raise_status(p, kErrBounds);
            pg = -1;
        }
        pages[i] = pg;
    }
}

// Page of key `tok` (in [t0, t1)) from the list load_cta_pages made.
__device__ __forceinline__ int page_of(const DecodeParams& p, const CtaWork& w, const int* pages, int tok) {
    return pages[page_col(p, tok) - page_col(p, w.t0)];
}

// Issue the TMA load of one 16-key stage.  The stage map views the cache as
// {128-byte chunk, key row, chunk index}: one copy brings 16 key rows and lands
// them chunk-major -- K boxes, then V boxes, 2 KiB each, 128-byte swizzled --
// completing on `bar`.  A skipped page only arrives on the barrier.
template <int D, int ELT>
__device__ __forceinline__ void issue_stage(const CUtensorMap* tmap, const DecodeParams& p,
                                            const CtaWork& w, const int* pages, int stage,
                                            uint32_t buf, uint32_t bar, uint64_t policy) {
    constexpr int ROWB = D * ELT;     // bytes of the K (or V) half of a key row
    constexpr int KBOX = ROWB / 128;  // 128-byte boxes per half
    constexpr int HALF = KBOX * 2048;
    const int tok = w.t0 + stage * kStageTok;
    const int pg = page_of(p, w, pages, tok);
    if (pg < 0) {
        mbar_arrive(bar);
        return;
    }
    const int row = (pg * p.Hkv + w.hk) * p.P + page_slot(p, tok);
    mbar_arrive_expect_tx(bar, 2 * HALF);
    tma_load_3d(buf, tmap, 0, row, 0, bar, policy);  // the whole 16-key stage in one copy
}

// Zero the V rows [nvalid, 16) of a stage so that masked keys (past the
// sequence end, or of a skipped page) cannot bring NaN into p*V.
template <int D, int ELT>
__device__ __forceinline__ void zero_tail_v(uint8_t* stage_gen, int nvalid, int lane) {
    constexpr int ROWB = D * ELT;
    constexpr int KBOX = ROWB / 128;
    constexpr int HALF = KBOX * 2048;
    const int nchunks = (kStageTok - nvalid) * KBOX * 8;  // 16-byte chunks
    for (int c = lane; c < nchunks; c += 32) {
        const int row = nvalid + c / (KBOX * 8);
        const int rem = c % (KBOX * 8);
        const int box = rem / 8, chunk = rem % 8;
        *reinterpret_cast<uint4*>(stage_gen + HALF + box * 2048 + row * 128 + chunk * 16) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();
    __syncwarp();
}

// CTA epilogue.  Each warp left, per query row r < M, its running max m (log2
// domain), its sum l and its unnormalised output O[w][r][0..D) in shared
// memory.  Merge the warps; then either write the result (one chunk) or
// publish the chunk's (normalised output, LSE) and let the last chunk's CTA
// merge all chunks by LSE.
// NS: number of per-warp (or per-warp-pair) states to merge, state k at
// rows k*mrows of wm, wl and O.
// part_of(j) is the workspace slot of split j of the unit (this CTA's split
// is w.split): [M] LSEs at part_lse + slot*M, [M, D] outputs at part_out +
// slot*M*D.
template <int D, int OSTRIDE, int NS, class PartOf>
__device__ void cta_finish_parts(const DecodeParams& p, const CtaWork& w, const float* O, const float* wm,
                                 const float* wl, int mrows, int* flag, PartOf part_of) {
    const int M = p.M;
    const int unit = w.b * p.Hkv + w.hk;
    const bool single = w.nsplit == 1;
    float* pout = p.part_out + static_cast<long long>(part_of(w.split)) * M * D;
    float* plse = p.part_lse + static_cast<long long>(part_of(w.split)) * M;

    for (int e = threadIdx.x; e < M * D; e += blockDim.x) {
        const int r = e / D, d = e % D;
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < NS; ++k) mx = fmaxf(mx, wm[k * mrows + r]);
        float lsum = 0.f, o = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
                const float s = fast_exp2(wm[k * mrows + r] - mx);
                lsum += wl[k * mrows + r] * s;
                o += O[(k * mrows + r) * OSTRIDE + d] * s;
            }
        }
        const float on = lsum > 0.f ? o / lsum : 0.f;
        const float l2 = lsum > 0.f ? mx + __log2f(lsum) : -INFINITY;
        if (single) {
            store_out(p.out, out_index(p, w.b, w.hk, r, d, D), on * p.v_scale, p.out_dtype);
            if (d == 0 && p.lse) {
                const int i = r / p.G, g = r % p.G;
                p.lse[(static_cast<long long>(w.b) * p.sq + i) * p.Hq + w.hk * p.G + g] = l2 * kLn2;
            }
        } else {
            __stcg(pout + e, on);
            if (d == 0) __stcg(plse + r, l2);
        }
    }
    if (single) return;

    // Split-KV: the last CTA of (b, hk) to arrive merges every chunk.  The
    // CTA barrier orders every thread's partial stores before one arrival with
    // acquire-release semantics at GPU scope (release covers them; the acquire,
    // passed on by the next barrier, covers the other chunks' partials).
    __syncthreads();
    if (threadIdx.x == 0) {
        const int prev = atom_add_acq_rel_gpu(p.counters + unit);
        const int last = prev == w.nsplit - 1;
        if (last) atomicExch(p.counters + unit, 0);  // ready for the next call
        *flag = last;
    }
    __syncthreads();
    if (!*flag) return;
    for (int e = threadIdx.x; e < M * D; e += blockDim.x) {
        const int r = e / D, d = e % D;
        float mx = -INFINITY;
        for (int c = 0; c < w.nsplit; ++c) mx = fmaxf(mx, __ldcg(p.part_lse + static_cast<long long>(part_of(c)) * M + r));
        float wsum = 0.f, o = 0.f;
        if (mx != -INFINITY) {
            for (int c = 0; c < w.nsplit; ++c) {
                const long long slot = part_of(c);
                const float lc = __ldcg(p.part_lse + slot * M + r);
                if (lc == -INFINITY) continue;  // an empty chunk is never read
                const float s = fast_exp2(lc - mx);
                wsum += s;
                o += s * __ldcg(p.part_out + (slot * M + r) * D + d);
            }
        }
        const float on = wsum > 0.f ? o / wsum : 0.f;
        store_out(p.out, out_index(p, w.b, w.hk, r, d, D), on * p.v_scale, p.out_dtype);
        if (d == 0 && p.lse) {
            const int i = r / p.G, g = r % p.G;
            p.lse[(static_cast<long long>(w.b) * p.sq + i) * p.Hq + w.hk * p.G + g] =
                wsum > 0.f ? (mx + __log2f(wsum)) * kLn2 : -INFINITY;
        }
    }
}

// The chunked grid: split j of unit u has slot u * max_splits + j.
template <int D, int OSTRIDE, int NS = kNW>
__device__ void cta_finish(const DecodeParams& p, const CtaWork& w, const float* O, const float* wm,
                           const float* wl, int mrows, int* flag) {
    const long long unit = static_cast<long long>(w.b) * p.Hkv + w.hk;
    cta_finish_parts<D, OSTRIDE, NS>(p, w, O, wm, wl, mrows, flag,
                                     [&](int j) { return unit * p.max_splits + j; });
}

}  // namespace pkd
