/*
 * pkd -- attention over a paged KV cache on GB300 (sm_103a).
 *
 * C ABI.  Every pointer named "device" is a CUDA device address owned by the
 * caller; the library never allocates, frees or synchronises on its own (the
 * one exception is pkd_workspace_check, which reads a status word back).
 * Calls are asynchronous on the stream passed as `stream` (a cudaStream_t;
 * NULL is the legacy default stream).  All functions are thread-safe; the
 * message of the last failure is kept per host thread (pkd_last_error).
 * A process may call the library on several GPUs: each kernel's launch
 * set-up is made once per device, with that device current.
 *
 * Sources of the operations (vLLM API pages, by title and section):
 *   [TS]   vllm.v1.attention.backends.flashinfer_ts -- module docstring
 *          ("Layout", "Sliding window"), FlashInferTSImpl.forward,
 *          FlashInferTSImpl._kv_views, FlashInferTSMetadataBuilder.build,
 *          ._restrict_to_window, ._get_plan, _kv_kernel_dtype.
 *   [DASH] vllm.v1.attention.ops.dash_attention -- flash_dash_attention.
 *   [FA]   vllm.v1.attention.backends.fa_utils --
 *          FlashAttentionCuTeDSLCompileSpec (Split-KV, return_softmax_lse).
 */
#ifndef PKD_H_
#define PKD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKD_OK = 0,
    PKD_EINVAL = 1,          /* bad pointer, size, stride or alignment */
    PKD_EUNSUPPORTED = 2,    /* valid request outside what the kernels implement */
    PKD_ECUDA = 3,           /* a CUDA runtime/driver call failed (message has the CUDA error) */
    PKD_EDEVICE_BOUNDS = 4,  /* a kernel met an out-of-range page or length (see pkd_workspace_check) */
    PKD_ETIMEOUT = 5         /* a kernel gave up waiting on one of its own copies */
} pkd_status;

typedef enum {
    PKD_BF16 = 0,
    PKD_FP16 = 1,
    PKD_FP8_E4M3 = 2,        /* e4m3 "fn": uint8 storage, no infinities [TS _kv_kernel_dtype] */
    PKD_FP32 = 3
} pkd_dtype;

/* Flags for pkd_paged_decode. */
#define PKD_FLAG_CAUSAL 1u      /* causal mask inside the query block, exact per-token window */
#define PKD_FLAG_MMA_SMALL_M 2u /* tensor cores for sq*Hq/Hkv < 16 (already the default; kept for callers) */
#define PKD_FLAG_FMA 4u         /* CUDA cores instead (only when sq*Hq/Hkv <= 8) */
#define PKD_FLAG_GRID 8u        /* the chunked grid: one CTA per Split-KV chunk */
#define PKD_FLAG_FLAT 16u       /* the persistent flat partition whatever the shapes (batch <= 1024) */
#define PKD_FLAG_BALANCED 32u   /* the persistent per-CTA partition (16-bit caches, tensor cores) */
/* q, block_table, seq_lens, out and lse are pinned host memory (cudaHostAlloc,
 * cudaMallocHost or cudaHostRegister), which under unified addressing has the
 * same address on the device: the kernels read and write it in place over the
 * host link, with no copy before or after the launch.  kv_cache and the
 * workspace stay device memory.  Each of those five pointers is checked with
 * cudaPointerGetAttributes (host memory mapped at the same address, else
 * PKD_EINVAL).  The tcgen05 kernel, whose q goes through a tensor-map copy,
 * is not used with it: its shapes run on the chunked grid instead (the
 * workspace size and kernel name follow the flag). */
#define PKD_FLAG_HOST_IO 128u
/* Diagnostic: every wait on a stage's copy tests its barrier once instead of
 * waiting up to 200 ms, so a call reports PKD_ETIMEOUT whenever a copy has not
 * landed by its first test.  The kernels still let every issued copy land
 * before they leave.  It exists to exercise the timeout path; zero the
 * workspace again (pkd_workspace_init) after such a call. */
#define PKD_FLAG_TEST_TIMEOUT 64u

/* Library version, major*10000 + minor*100 + patch. */
int pkd_version(void);

/* Message of the last non-OK status returned on this host thread ("" if none). */
const char* pkd_last_error(void);

/*
 * Bytes of workspace pkd_paged_decode needs for a plan.  The plan is fixed by
 * the shapes and by max_kv_len, an upper bound on every seq_lens entry (the
 * constant K/V capacity of [TS FlashInferTSMetadataBuilder._max_kv_len]), so
 * one workspace serves every call with the same shapes, e.g. every replay of
 * a captured CUDA graph.  chunk_tokens is the Split-KV chunk (0 = automatic;
 * otherwise a multiple of page_size).  flags as for pkd_paged_decode.
 * Returns 0 for an invalid request (the reason is in pkd_last_error).
 */
size_t pkd_paged_decode_workspace_size(int batch, int sq, int num_heads, int num_kv_heads,
                                       int head_dim, int page_size, int max_kv_len,
                                       pkd_dtype kv_dtype, int window, int chunk_tokens,
                                       unsigned flags);

/*
 * Which kernel pkd_paged_decode launches for a plan (same arguments as
 * pkd_paged_decode_workspace_size): a static string such as
 * "chunked grid, tensor cores".  Host-only, no CUDA call.  Returns NULL for
 * an invalid request (the reason is in pkd_last_error).  The pages have no
 * counterpart of this call; it makes the library's choice of kernel visible
 * to callers and benchmarks.
 */
const char* pkd_paged_decode_kernel_name(int batch, int sq, int num_heads, int num_kv_heads, int head_dim,
                                         int page_size, int max_kv_len, pkd_dtype kv_dtype, int window,
                                         int chunk_tokens, unsigned flags);

/*
 * Zero a workspace (asynchronously on `stream`).  Needed once, before its
 * first use: every later call leaves the workspace ready for the next one.
 */
pkd_status pkd_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronise `stream`, read the workspace's status word and clear it.
 * Returns PKD_OK, PKD_EDEVICE_BOUNDS (a seq_lens entry above max_kv_len or
 * below 0, or a block-table entry outside [0, num_pages): the kernel skipped
 * those keys) or PKD_ETIMEOUT.  The kernels never trap.
 */
pkd_status pkd_workspace_check(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Paged decode: attention of a uniform query block per request over that
 * request's keys in a paged cache [TS FlashInferTSImpl.forward].
 *
 *   q            device, [batch, sq, num_heads, head_dim] contiguous, q_dtype
 *   kv_cache     device, [num_pages, num_kv_heads, page_size, 2*head_dim]
 *                contiguous, kv_dtype.  K = [..., :head_dim], V = [..., head_dim:]
 *                (token stride 2*head_dim [TS _kv_views, "Layout"]); 16-byte aligned.
 *   block_table  device int32 [batch, block_table_stride]: token t of request b
 *                lives in page block_table[b, t / page_size], slot t % page_size.
 *                Columns past a request's last page are never read.
 *   seq_lens     device int32 [batch], each in [0, max_kv_len].
 *   out          device, [batch, sq, num_heads, head_dim], out_dtype (bf16, fp16, fp32)
 *   lse          device fp32 [batch, sq, num_heads] natural-log LSE, or NULL
 *   workspace    device, >= pkd_paged_decode_workspace_size(...) bytes,
 *                zeroed once by pkd_workspace_init; 256-byte aligned.
 * With PKD_FLAG_HOST_IO, q, block_table, seq_lens, out and lse are pinned
 * host memory instead, read and written by the kernels in place.
 *
 * Query head h reads KV head h / (num_heads / num_kv_heads).  Logits are
 * (scale * q_scale * k_scale) * q.k and the output is scaled by v_scale
 * (bmm1 / bmm2 of [TS forward]); for fp8 caches q is already fp8 with
 * scale q_scale (q_dtype must equal kv_dtype).
 *
 * Masks.  Without PKD_FLAG_CAUSAL every query token of the block sees every
 * visible key ("dense", [TS module docstring]).  window > 0 restricts the
 * visible keys to the page-aligned suffix of [TS _restrict_to_window]:
 *   start_page = max(0, floor((L - (window + sq - 1)) / page_size)),
 * keys [start_page * page_size, L), one start for the whole block.  With
 * PKD_FLAG_CAUSAL query token i (position L - sq + i) sees keys up to its
 * position and, when window > 0, from position - (window - 1) on
 * ([TS _get_plan] mask_type "causal", window_left = window - 1).
 * A query row with no visible key gets out = 0 and lse = -inf.
 *
 * Split-KV [FA num_splits]: the keys of a (request, kv head) may be shared
 * between several workers whose partial results are merged by LSE inside
 * the same launch.  By default a chunked grid runs one CTA per chunk of
 * chunk_tokens keys (0: chosen by the library: about 2048 CTAs, chunks of at
 * most 4096 keys -- 32 chunks for 64 (request, kv head) units of 131,072
 * keys).  16-bit query blocks of M = sq * num_heads / num_kv_heads = 17-32
 * rows with head_dim 128 and batch <= 512 (dense or causal) run instead on a
 * persistent kernel with one CTA per SM on the tcgen05 tensor cores: chunks
 * of at most chunk_tokens keys (0: a quarter of the longest visible range in
 * whole 128-key tiles, between 1024 and 2048 keys; 2048 at most), equal
 * within a request; with more chunks than SMs every CTA takes an equal
 * share of all 128-key tiles (consecutive chunks of a (request, kv head)
 * accumulate together), and only units cut by a share boundary leave
 * partial results, merged by LSE by the CTA that completes the unit's last
 * piece -- one launch.  Other 16-bit blocks of 17-32 rows run the
 * chunked grid with two warps sharing each chunk's stages, 16 rows each
 * (as few chunks of at most 4096 keys as possible).  fp8
 * caches with M > 16 run, for batch <= 1024, on a persistent grid that gives
 * every warp an equal slice of all requests' keys laid end to end.  PKD_FLAG_GRID, PKD_FLAG_FLAT and PKD_FLAG_BALANCED
 * (a persistent grid with an equal slice per CTA) force a kernel;
 * pkd_paged_decode_kernel_name says which one a call launches.
 *
 * Limits: head_dim 64 or 128; page_size a multiple of 16; num_heads a
 * multiple of num_kv_heads; M <= 32 on tensor cores, <= 8 on CUDA cores
 * (PKD_FLAG_FMA); fp8 caches need head_dim 128, and M > 16 with fp8 needs the
 * per-warp persistent grid.  Anything else: PKD_EUNSUPPORTED.  After a
 * PKD_ETIMEOUT, zero the workspace again before reusing it.
 */
pkd_status pkd_paged_decode(const void* q, pkd_dtype q_dtype,
                            const void* kv_cache, pkd_dtype kv_dtype, int64_t num_pages,
                            const int32_t* block_table, int64_t block_table_stride,
                            const int32_t* seq_lens,
                            int batch, int sq, int num_heads, int num_kv_heads, int head_dim,
                            int page_size, int max_kv_len,
                            float scale, float q_scale, float k_scale, float v_scale, int window,
                            void* out, pkd_dtype out_dtype, float* lse,
                            void* workspace, size_t workspace_bytes, int chunk_tokens,
                            unsigned flags, void* stream);

/*
 * pkd_paged_decode without a caller workspace.  The pages have no counterpart
 * of this call: it exists for callers that cannot allocate device memory at
 * the point where they run decode -- plug-ins whose host runtime owns all
 * device memory and hands none out, serving loops that must not allocate once
 * their memory budget is fixed, or C callers with no device allocator of
 * their own.
 *
 * It takes the same arguments as pkd_paged_decode minus the workspace and
 * uses instead a scratch array compiled into the library: 32 MiB of device
 * memory that every GPU loading the library holds until the process exits.
 * A plan whose workspace (pkd_paged_decode_workspace_size) exceeds 32 MiB is
 * rejected with PKD_EUNSUPPORTED.  fp8 caches with more than 16 query rows
 * per kv head always are: their persistent per-warp kernel keeps two partial
 * slots per worker warp whatever the batch (64 MiB at 32 rows).  The call
 * allocates nothing; it clears the part of the scratch it uses
 * (cudaMemsetAsync on `stream`) and launches the decode kernel.  The first
 * call on each device looks up the scratch address on that device (make it
 * before any stream capture); the address is kept for the process, so the
 * call must not be used across a cudaDeviceReset.  All calls share the one
 * scratch array: calls that may overlap on the GPU (different streams, or
 * different host threads on one device) race and must be serialised by the
 * caller.  The device-side status word (out-of-range lengths or pages, a
 * wait that timed out) is cleared by the next call: read it with
 * pkd_paged_decode_static_check before then.
 */
pkd_status pkd_paged_decode_static(const void* q, pkd_dtype q_dtype,
                                   const void* kv_cache, pkd_dtype kv_dtype, int64_t num_pages,
                                   const int32_t* block_table, int64_t block_table_stride,
                                   const int32_t* seq_lens,
                                   int batch, int sq, int num_heads, int num_kv_heads, int head_dim,
                                   int page_size, int max_kv_len,
                                   float scale, float q_scale, float k_scale, float v_scale, int window,
                                   void* out, pkd_dtype out_dtype, float* lse,
                                   int chunk_tokens, unsigned flags, void* stream);

/*
 * The device-side status word of the last pkd_paged_decode_static call on
 * the current device, like pkd_workspace_check on a caller workspace: waits
 * for `stream`, returns PKD_OK, PKD_EDEVICE_BOUNDS (a seq_lens entry outside
 * [0, max_kv_len] or a block-table entry outside [0, num_pages): those keys
 * were skipped) or PKD_ETIMEOUT (a kernel gave up waiting on its own copies),
 * and clears the word.  No counterpart in the pages (see
 * pkd_paged_decode_static).  Allocates nothing.
 */
pkd_status pkd_paged_decode_static_check(void* stream);

/*
 * KV-cache write [TS FlashInferTSImpl.do_kv_cache_update, reshape_and_cache_flash]:
 * the key and value rows of num_tokens new tokens go to their slots.
 *
 *   key, value    device [num_tokens, num_kv_heads, head_dim], in_dtype (bf16 or
 *                 fp16); rows of one token contiguous, key_stride / value_stride
 *                 elements between tokens (multiples of 8); 16-byte aligned
 *   slot_mapping  device int64 [num_tokens]: slot s is page s / page_size,
 *                 offset s % page_size; s < 0 (padding) and slots past the
 *                 cache write nothing
 *   kv_cache      device [num_pages, num_kv_heads, page_size, 2*head_dim]
 *                 kv_dtype: key into [..., :head_dim], value into [..., head_dim:]
 *
 * kv_dtype == in_dtype stores the input bits.  PKD_FP8_E4M3 stores
 * e4m3(x / k_scale) for keys and e4m3(x / v_scale) for values: the quotient is
 * an IEEE fp32 division, rounded to nearest even and saturated to +-448.
 */
pkd_status pkd_cache_write(const void* key, const void* value, pkd_dtype in_dtype, int64_t key_stride,
                           int64_t value_stride, const int64_t* slot_mapping, int64_t num_tokens,
                           int num_kv_heads, int head_dim, int page_size, int64_t num_pages,
                           void* kv_cache, pkd_dtype kv_dtype, float k_scale, float v_scale, void* stream);

/*
 * DASH segmented attention with its combine [DASH flash_dash_attention].
 *
 *   q        device [n, num_heads, head_dim], dtype (bf16 or fp16)
 *   k, v     device [n * (topk*bs + local), num_kv_heads, head_dim], dtype, contiguous
 *   used     device int32 [n * (topk + 1)]: valid prefix length of each segment;
 *            query i's segment g < topk starts at row i*(topk*bs+local) + g*bs
 *            (capacity bs), its local segment at i*(topk*bs+local) + topk*bs
 *            (capacity local).  Values are clamped to [0, capacity].
 *   bias     device fp32 [n, topk] prior of each gathered segment (the local
 *            segment's prior is 0); may be NULL when topk == 0.
 *   out      device [n, num_heads, head_dim], dtype
 *   seg_out  device fp32 [n, topk+1, num_heads, head_dim] per-segment outputs, or NULL
 *   seg_lse  device fp32 [n, topk+1, num_heads] per-segment natural-log LSE, or NULL
 *
 * Each (query, segment, head) is softmax attention over the segment's used
 * rows with scale head_dim^-0.5, giving (o_g, lse_g); an empty segment gives
 * (0, -inf).  out = sum_g w_g o_g with w = softmax over live segments
 * (used > 0) of lse_g + prior_g; a query with no live segment gets 0.
 * Limits: head_dim 64 or 128, bs and local multiples of 8, num_heads a
 * multiple of num_kv_heads with num_heads / num_kv_heads <= 16.
 */
pkd_status pkd_segmented_attention(const void* q, const void* k, const void* v, pkd_dtype dtype,
                                   const int32_t* used, const float* bias,
                                   int n, int num_heads, int num_kv_heads, int head_dim,
                                   int topk, int bs, int local,
                                   void* out, float* seg_out, float* seg_lse, void* stream);

/*
 * DASH segmented attention read straight from the paged cache: the segments
 * are key ranges of the query's own request, gathered through the block
 * table instead of being copied into contiguous k/v first (the copy that
 * feeds [DASH flash_dash_attention]).
 *
 *   q            device [n, num_heads, head_dim], dtype (bf16 or fp16)
 *   kv_cache     device [num_pages, num_kv_heads, page_size, 2*head_dim], dtype
 *   block_table  device int32 [n, block_table_stride]: row i is query i's request
 *   seg_start    device int32 [n, topk+1]: position of the first key of each
 *                segment in that request ([topk gathered, local] order)
 *   used         device int32 [n, topk+1]: keys in each segment, clamped to
 *                [0, bs] (gathered) or [0, local] (local segment) and to max_kv_len
 *   bias, out, seg_out, seg_lse as for pkd_segmented_attention
 *
 * Segment g of query i holds keys [seg_start, seg_start + used) of request i;
 * everything else (scale, per-segment (o, lse), the combine) is as in
 * pkd_segmented_attention.  page_size must be a multiple of 16; pages outside
 * [0, num_pages) are skipped.
 */
pkd_status pkd_segmented_attention_paged(const void* q, pkd_dtype dtype, const void* kv_cache,
                                         int64_t num_pages, const int32_t* block_table,
                                         int64_t block_table_stride, const int32_t* seg_start,
                                         const int32_t* used, const float* bias, int n, int num_heads,
                                         int num_kv_heads, int head_dim, int page_size, int topk, int bs,
                                         int local, int max_kv_len, void* out, float* seg_out,
                                         float* seg_lse, void* stream);

/*
 * LSE merge of partial attention results: the Split-KV merge [FA] and, with a
 * prior and a live mask, the segment combine [DASH flash_dash_attention].
 *
 *   part_out  device fp32 [n, parts, heads, head_dim]
 *   part_lse  device fp32 [n, parts, heads] natural-log LSE of each part
 *   prior     device fp32 [n, parts] added to each part's LSE, or NULL
 *   live      device int32 [n, parts]; part p of row n is dead when <= 0, or NULL
 *   out       device [n, heads, head_dim], out_dtype (bf16, fp16, fp32)
 *   lse_out   device fp32 [n, heads] = ln sum_{live p} exp(lse_p + prior_p), or NULL
 *
 * out = sum over live parts of exp(lse_p + prior_p - lse_out) * part_out_p;
 * a dead part (or one with lse -inf) is never read; a row with no live part
 * gets out = 0 and lse_out = -inf.  Limits: head_dim <= 256, parts <= 1024.
 */
pkd_status pkd_lse_merge(const float* part_out, const float* part_lse, const float* prior,
                         const int32_t* live, int n, int parts, int heads, int head_dim,
                         void* out, pkd_dtype out_dtype, float* lse_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKD_H_ */
