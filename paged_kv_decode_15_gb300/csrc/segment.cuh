// Parameters of the DASH segmented-attention and LSE-merge kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace pkd {

struct SegmentParams {
    CUtensorMap kmap, vmap;   // 3-D maps over k, v: {head_dim, Hkv, rows}; paged: kmap is the
                              // cache's stage map {128-byte chunk, pages*Hkv*P rows, chunks}
                              // and vmap is unused
    const int32_t* block_table;  // paged: [n, bt_stride]
    const int32_t* seg_start;    // paged: [n, topk+1] first key position of each segment
    const void* k;               // k rows [rows, Hkv, D] (paged: the cache), for row-exact copies
    const void* v;               // v rows [rows, Hkv, D] (paged: unused)
    long long bt_stride, num_pages;
    int P, max_kv_len, paged;
    uint32_t pmagic;          // paged: tok / P == (tok * pmagic) >> pmshift for 0 <= tok < 2^31
    int pmshift;
    const void* q;            // [n, Hq, D]
    const int32_t* used;      // [n, topk+1]
    const float* bias;        // [n, topk]
    void* out;                // [n, Hq, D] (q dtype)
    float* seg_out;           // [n, topk+1, Hq, D] or null
    float* seg_lse;           // [n, topk+1, Hq] or null
    int n, Hq, Hkv, G, D, topk, bs, local;
    int bf16;
    float scale_log2;         // D^-0.5 * log2(e)
};

struct MergeParams {
    const float* part_out;    // [n, parts, heads, D]
    const float* part_lse;    // [n, parts, heads], natural log
    const float* prior;       // [n, prior_cols] or null; parts >= prior_cols get prior 0
    const int32_t* live;      // [n, parts] or null
    int n, parts, heads, D;
    int prior_cols;
    void* out;                // [n, heads, D]
    int out_dtype;
    float* lse_out;           // [n, heads] or null
};

}  // namespace pkd
