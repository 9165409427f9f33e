// C ABI of the library: argument validation, the Split-KV plan, workspace
// layout, TMA descriptor construction and kernel launches.  No allocation,
// no synchronisation (except pkd_workspace_check), no CPU compute path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/pkd.h"
#include "decode_common.cuh"
#include "decode_tc05.cuh"
#include "launch.h"
#include "page_math.h"
#include "segment.cuh"

namespace {

thread_local std::string g_last_error;

pkd_status fail(pkd_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

pkd_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PKD_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elt_bytes(pkd_dtype dt) { return dt == PKD_FP8_E4M3 ? 1 : dt == PKD_FP32 ? 4 : 2; }

// ---------------------------------------------------------------- plan
// Split-KV aims for about this many CTAs with one-tile kernels: measured on
// gqa_decode_b64 (M = 4) 2048 (1024-key chunks) beats 512- to 2048-key chunks.
constexpr int kTargetCtas = 2048;
constexpr int kMaxChunk = 4096;    // and never puts more keys than this in one chunk
constexpr size_t kHeader = 256;    // workspace status word lives in the first bytes
// Chunks of the tcgen05 kernel: automatic chunks of at least this many keys.
constexpr int kTcChunkMin = 1024;

struct Plan {
    bool mma;
    bool flat;     // persistent per-warp partition
    bool bal;      // persistent per-CTA partition
    bool tc;       // persistent tcgen05 kernel (query blocks of 17-32 rows)
    int M, G;
    int mt, nt;    // tensor-core tiles
    int lpt, mr;   // CUDA-core lanes per key, padded rows
    int max_vis, chunk, max_splits;
    size_t off_counters, off_lse, off_out, bytes;
};

pkd_status make_plan(int B, int sq, int Hq, int Hkv, int D, int P, int max_kv_len, pkd_dtype kv,
                     int window, int chunk_tokens, unsigned flags, Plan& pl) {
    if (B < 0 || sq < 1 || Hq < 1 || Hkv < 1 || P < 1 || max_kv_len < 0)
        return fail(PKD_EINVAL, "invalid shape: batch=%d sq=%d num_heads=%d num_kv_heads=%d page_size=%d max_kv_len=%d",
                    B, sq, Hq, Hkv, P, max_kv_len);
    if (Hq % Hkv != 0)
        return fail(PKD_EUNSUPPORTED, "num_heads (%d) must be a multiple of num_kv_heads (%d)", Hq, Hkv);
    if (D != 64 && D != 128) return fail(PKD_EUNSUPPORTED, "head_dim %d not supported (64 or 128)", D);
    if (P % 16 != 0) return fail(PKD_EUNSUPPORTED, "page_size %d must be a multiple of 16", P);
    if (kv != PKD_BF16 && kv != PKD_FP16 && kv != PKD_FP8_E4M3)
        return fail(PKD_EUNSUPPORTED, "kv dtype %d not supported (bf16, fp16, fp8-e4m3)", (int)kv);
    if (kv == PKD_FP8_E4M3 && D != 128) return fail(PKD_EUNSUPPORTED, "fp8 caches need head_dim 128");
    pl.G = Hq / Hkv;
    pl.M = sq * pl.G;
    const int M = pl.M;
    // Kernel choice (measured): the chunked grid, whose hardware CTA
    // scheduling keeps every SM busy to the end (gqa_decode_b64: 101 us
    // against 124 us per-warp and 115 us per-CTA partitions; fp8_long_b8: 408
    // against 476 us; query_block_sq8 with warp pairs: 193 against 214 us;
    // tiny problems: 8.5 against 36.5 us).  fp8 caches with M > 16 have no
    // warp-pair kernel and take the persistent per-warp partition.
    // PKD_FLAG_GRID, PKD_FLAG_FLAT and PKD_FLAG_BALANCED force a kernel.
    const bool flat_default = kv == PKD_FP8_E4M3 && (long long)sq * (Hq / Hkv) > 16;
    if (((flags & PKD_FLAG_GRID) != 0) + ((flags & PKD_FLAG_FLAT) != 0) + ((flags & PKD_FLAG_BALANCED) != 0) > 1)
        return fail(PKD_EINVAL, "PKD_FLAG_GRID, PKD_FLAG_FLAT and PKD_FLAG_BALANCED exclude each other");
    pl.bal = false;
    if (flags & PKD_FLAG_BALANCED) {
        if (kv == PKD_FP8_E4M3 || (flags & PKD_FLAG_FMA))
            return fail(PKD_EUNSUPPORTED, "the per-CTA partition runs 16-bit caches on tensor cores only");
        pl.bal = true;
    }
    pl.flat = !pl.bal && B <= pkd::kFlatMaxBatch && !(flags & PKD_FLAG_GRID) &&
              ((flags & PKD_FLAG_FLAT) || flat_default);
    // 16-bit query blocks of 17-32 rows, dense or causal: the tcgen05 kernel
    // (query_block_sq8: see the kernel-choice table of the design notes)
    pl.tc = !pl.bal && !pl.flat && (kv == PKD_BF16 || kv == PKD_FP16) && D == 128 && sq * (Hq / Hkv) > 16 &&
            sq * (Hq / Hkv) <= 32 && B <= pkd::kTcMaxBatch &&
            !(flags & (PKD_FLAG_GRID | PKD_FLAG_FMA | PKD_FLAG_HOST_IO)) &&
            (chunk_tokens <= 0 || chunk_tokens <= pkd::kTcMaxChunk);
    if (kv == PKD_FP8_E4M3 && (flags & PKD_FLAG_FMA)) {
        if (M > 8) return fail(PKD_EUNSUPPORTED, "fp8 on CUDA cores supports sq*num_heads/num_kv_heads <= 8 (got %d)", M);
        pl.mma = false;
    } else if (kv == PKD_FP8_E4M3 && !pl.flat && M > 16) {
        return fail(PKD_EUNSUPPORTED,
                    "fp8 caches with more than 16 query rows per kv head (got %d) run on the flat partition only "
                    "(batch <= %d, no PKD_FLAG_GRID)", M, pkd::kFlatMaxBatch);
    } else if (flags & PKD_FLAG_FMA) {
        if (M > 8) return fail(PKD_EUNSUPPORTED, "the CUDA-core kernel supports sq*num_heads/num_kv_heads <= 8 (got %d)", M);
        pl.mma = false;
    } else {
        // 16-bit caches use the tensor-core kernel at every M (measured faster
        // than CUDA cores also for M < 16); PKD_FLAG_FMA selects CUDA cores.
        pl.mma = true;
    }
    if (pl.mma) {
        if (M > 32) return fail(PKD_EUNSUPPORTED, "sq*num_heads/num_kv_heads = %d > 32", M);
        pl.mt = (M + 15) / 16;
        pl.nt = (M + 7) / 8;
        if (pl.mt == 1 && pl.nt > 2) pl.nt = 2;
    } else {
        pl.lpt = M <= 4 ? 8 : 16;
        pl.mr = M <= 2 ? 2 : M <= 4 ? 4 : 8;
    }
    const long long span = window > 0 ? (long long)window + sq - 1 + P - 1 : (long long)max_kv_len;
    pl.max_vis = (int)(span < max_kv_len ? span : max_kv_len);
    const int units = B * Hkv > 0 ? B * Hkv : 1;
    if (pl.tc) {
        // chunks of at most `chunk` keys (equal within a request, whole 128-key
        // tiles where the chunk allows); a (request, kv head) unit of n chunks
        // is one piece per chunk (one chunk per CTA) or per CTA share it meets
        // (shares at least a chunk long): at most n + 1 partial slots of 32
        // rows, and an arrival counter
        if (chunk_tokens > 0 && chunk_tokens % P != 0)
            return fail(PKD_EINVAL, "chunk_tokens %d must be a multiple of page_size %d", chunk_tokens, P);
        // automatic: a quarter of the longest visible range in whole tiles,
        // 1024-2048 keys, when every chunk has a CTA of its own; when CTAs
        // take tile shares, chunks of the largest size (fewer items per run;
        // at most as many pieces per unit as the plan's chunks + 1)
        int auto_chunk = (pl.max_vis / 4 + pkd::kTcTile - 1) / pkd::kTcTile * pkd::kTcTile;
        if (auto_chunk < kTcChunkMin) auto_chunk = kTcChunkMin;
        if (auto_chunk > pkd::kTcMaxChunk) auto_chunk = pkd::kTcMaxChunk;
        pl.chunk = chunk_tokens > 0 ? chunk_tokens : auto_chunk;
        pl.max_splits = (pl.max_vis > 0 ? (pl.max_vis + pl.chunk - 1) / pl.chunk : 1) + 1;
        const size_t parts = (size_t)units * pl.max_splits;
        pl.off_counters = kHeader;
        pl.off_lse = pl.off_counters + round_up((size_t)units * 4, 256);
        pl.off_out = pl.off_lse + round_up(parts * pkd::kTcRows * 4, 256);
        pl.bytes = pl.off_out + round_up(parts * pkd::kTcRows * 128 * 4, 256);
        return PKD_OK;
    }
    if (chunk_tokens > 0) {
        if (chunk_tokens % P != 0)
            return fail(PKD_EINVAL, "chunk_tokens %d must be a multiple of page_size %d", chunk_tokens, P);
        if (chunk_tokens / P > pkd::kMaxCtaPages)
            return fail(PKD_EINVAL, "chunk_tokens %d spans more than %d pages", chunk_tokens, pkd::kMaxCtaPages);
        pl.chunk = chunk_tokens;
    } else {
        // one-tile kernels: about kTargetCtas CTAs; warp pairs (M > 16): as few
        // chunks as the chunk limit allows, since each partial is M x D floats
        // (query_block_sq8: 4096-key chunks 193 us, 2048 216 us, 1024 246 us)
        // (the e4m3 grid too: fp8_long_b8, 64 units of 131,072 keys, takes 32
        // chunks of 4096, 364 us, against 373-392 us for chunks of 2048-3840
        // and 378-400 us for 4416-8192)
        const bool pair = pl.mma && pl.mt == 2 && !pl.flat && !pl.bal;
        int splits = pair ? 1 : (kTargetCtas + units - 1) / units;
        const int by_len = (pl.max_vis + kMaxChunk - 1) / kMaxChunk;
        if (by_len > splits) splits = by_len;
        if (splits < 1) splits = 1;
        int chunk = (pl.max_vis + splits - 1) / splits;
        const int floor_chunk = P > 256 ? P : 256;
        if (chunk < floor_chunk) chunk = floor_chunk;
        chunk = (int)round_up((size_t)chunk, (size_t)P);
        if (chunk / P > pkd::kMaxCtaPages) chunk = pkd::kMaxCtaPages * P;
        pl.chunk = chunk;
    }
    pl.max_splits = pl.max_vis > 0 ? (pl.max_vis + pl.chunk - 1) / pl.chunk : 1;
    pl.off_counters = kHeader;
    pl.off_lse = pl.off_counters + round_up((size_t)units * 4, 256);
    // partial results: per (unit, chunk) for the chunked grid, per (warp, side)
    // for the flat partition
    const size_t parts = pl.flat  ? (size_t)pkd::kFlatMaxWorkers * 2
                         : pl.bal ? (size_t)pkd::kFlatMaxWorkers / pkd::kNW * 2  // two per CTA, <= 512 CTAs
                                  : (size_t)units * pl.max_splits;
    pl.off_out = pl.off_lse + round_up(parts * M * 4, 256);
    pl.bytes = pl.off_out + round_up(parts * M * D * 4, 256);
    return PKD_OK;
}

using pkd::page_magic;

// ---------------------------------------------------------- TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct MapKey {
    const void* base;
    uint64_t d0, d1, d2, s1, s2;
    int rank, dtype;
    bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof *this) == 0; }
};

struct MapCache {
    static constexpr int N = 64;
    MapKey key[N];
    CUtensorMap map[N];
    int used = 0, next = 0;
    std::mutex mu;
};

MapCache& map_cache() {
    static MapCache c;
    return c;
}

// A 2-D (rank 2) or 3-D (rank 3) tiled map, 128-byte swizzle, boxes of 128
// bytes by `box_rows` rows (one element of the middle dimension for rank 3).
pkd_status get_map(CUtensorMap& out, const void* base, int rank, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t s1, uint64_t s2, pkd_dtype dt, int box_rows) {
    MapKey k;
    std::memset(&k, 0, sizeof k);
    k.base = base; k.d0 = d0; k.d1 = d1; k.d2 = d2; k.s1 = s1; k.s2 = s2; k.rank = rank; k.dtype = dt;
    MapCache& c = map_cache();
    {
        std::lock_guard<std::mutex> g(c.mu);
        for (int i = 0; i < c.used; ++i)
            if (c.key[i] == k) {
                out = c.map[i];
                return PKD_OK;
            }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PKD_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int elt = elt_bytes(dt);
    const CUtensorMapDataType t = dt == PKD_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : dt == PKD_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elt), rank == 2 ? (cuuint32_t)box_rows : 1u, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap m;
    CUresult r = enc(&m, t, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKD_ECUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    {
        std::lock_guard<std::mutex> g(c.mu);
        const int slot = c.used < MapCache::N ? c.used++ : (c.next++ % MapCache::N);
        c.key[slot] = k;
        c.map[slot] = m;
    }
    out = m;
    return PKD_OK;
}

// The "stage map" of a paged cache: {128-byte chunk, key row, chunk of the
// row}, strides {row bytes, 128 B}, box {one chunk, 16 rows, every chunk},
// so one TMA copy loads a 16-key stage (K and V) chunk-major.
// Boxes of the stage map: a whole 16-key stage (every chunk), or the tcgen05
// kernel's stage: a 4-D view {chunk elements, 8 rows, chunk, 8-row group}
// whose box {all, 8, all, 2} lands a 16-key stage as two 8-row groups, each
// holding every chunk of its rows.
enum StageBox { kStageFull = 0, kStageTcGroup = 2 };

pkd_status get_stage_map(CUtensorMap& out, const void* cache, uint64_t rows, int row_bytes, pkd_dtype dt,
                         StageBox mode = kStageFull) {
    const int elt = elt_bytes(dt);
    MapKey k;
    std::memset(&k, 0, sizeof k);
    k.base = cache; k.d0 = 128 / elt; k.d1 = rows; k.d2 = row_bytes / 128; k.s1 = row_bytes; k.s2 = 128;
    k.rank = mode == kStageTcGroup ? 140 : 103; k.dtype = dt;
    MapCache& c = map_cache();
    {
        std::lock_guard<std::mutex> g(c.mu);
        for (int i = 0; i < c.used; ++i)
            if (c.key[i] == k) {
                out = c.map[i];
                return PKD_OK;
            }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PKD_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const CUtensorMapDataType t = dt == PKD_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : dt == PKD_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUtensorMap m;
    CUresult r;
    if (mode == kStageTcGroup) {
        // rows is a multiple of 16 (page_size is)
        cuuint64_t dims[4] = {k.d0, 8, k.d2, k.d1 / 8};
        cuuint64_t strides[3] = {k.s1, k.s2, 8 * k.s1};
        cuuint32_t box[4] = {(cuuint32_t)(128 / elt), 8, (cuuint32_t)(row_bytes / 128), 2};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = enc(&m, t, 4, const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[3] = {k.d0, k.d1, k.d2};
        cuuint64_t strides[2] = {k.s1, k.s2};
        cuuint32_t box[3] = {(cuuint32_t)(128 / elt), (cuuint32_t)pkd::kStageTok, (cuuint32_t)(row_bytes / 128)};
        cuuint32_t estr[3] = {1, 1, 1};
        r = enc(&m, t, 3, const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return fail(PKD_ECUDA, "cuTensorMapEncodeTiled (stage map) failed (CUresult %d)", (int)r);
    {
        std::lock_guard<std::mutex> g(c.mu);
        const int slot = c.used < MapCache::N ? c.used++ : (c.next++ % MapCache::N);
        c.key[slot] = k;
        c.map[slot] = m;
    }
    out = m;
    return PKD_OK;
}

// The q rows of one (request, kv head) as a TMA box: q [tokens, Hq, D] viewed
// as {D, Hq, tokens}, box {64 dims, G heads, sq tokens}, 128-byte swizzle, so
// that one copy lands 64 dims of rows r = i*G + g at 128 bytes per row.
pkd_status get_q_map(CUtensorMap& out, const void* q, int D, int Hq, uint64_t tokens, int G, int sq, pkd_dtype dt) {
    MapKey k;
    std::memset(&k, 0, sizeof k);
    k.base = q; k.d0 = (uint64_t)D; k.d1 = (uint64_t)Hq; k.d2 = tokens; k.s1 = (uint64_t)D * 2;
    k.s2 = (uint64_t)Hq * D * 2; k.rank = 1000 + G * 64 + sq; k.dtype = dt;
    MapCache& c = map_cache();
    {
        std::lock_guard<std::mutex> g(c.mu);
        for (int i = 0; i < c.used; ++i)
            if (c.key[i] == k) {
                out = c.map[i];
                return PKD_OK;
            }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PKD_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const CUtensorMapDataType t = dt == PKD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[3] = {k.d0, k.d1, k.d2};
    cuuint64_t strides[2] = {k.s1, k.s2};
    cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)sq};
    cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap m;
    CUresult r = enc(&m, t, 3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKD_ECUDA, "cuTensorMapEncodeTiled (q map) failed (CUresult %d)", (int)r);
    {
        std::lock_guard<std::mutex> g(c.mu);
        const int slot = c.used < MapCache::N ? c.used++ : (c.next++ % MapCache::N);
        c.key[slot] = k;
        c.map[slot] = m;
    }
    out = m;
    return PKD_OK;
}

}  // namespace

int pkd::report_status(int st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

extern "C" {

int pkd_version(void) { return 10000; }

const char* pkd_last_error(void) { return g_last_error.c_str(); }

size_t pkd_paged_decode_workspace_size(int batch, int sq, int num_heads, int num_kv_heads, int head_dim,
                                       int page_size, int max_kv_len, pkd_dtype kv_dtype, int window,
                                       int chunk_tokens, unsigned flags) {
    Plan pl;
    if (make_plan(batch, sq, num_heads, num_kv_heads, head_dim, page_size, max_kv_len, kv_dtype, window,
                  chunk_tokens, flags, pl) != PKD_OK)
        return 0;
    return pl.bytes;
}

const char* pkd_paged_decode_kernel_name(int batch, int sq, int num_heads, int num_kv_heads, int head_dim,
                                         int page_size, int max_kv_len, pkd_dtype kv_dtype, int window,
                                         int chunk_tokens, unsigned flags) {
    Plan pl;
    if (make_plan(batch, sq, num_heads, num_kv_heads, head_dim, page_size, max_kv_len, kv_dtype, window,
                  chunk_tokens, flags, pl) != PKD_OK)
        return nullptr;
    if (pl.tc) return "persistent tcgen05 kernel, TMEM accumulators";
    if (pl.bal) return "persistent per-CTA partition, tensor cores";
    if (pl.flat) return pl.mma ? "persistent flat partition, tensor cores" : "persistent flat partition, CUDA cores";
    return pl.mma ? "chunked grid, tensor cores" : "chunked grid, CUDA cores";
}

pkd_status pkd_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kHeader) return fail(PKD_EINVAL, "workspace is null or too small");
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream);
    return e == cudaSuccess ? PKD_OK : cuda_fail(e, "pkd_workspace_init");
}

pkd_status pkd_workspace_check(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kHeader) return fail(PKD_EINVAL, "workspace is null or too small");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "pkd_workspace_check: stream");
    int32_t word = 0;
    e = cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "pkd_workspace_check: read");
    if (word == 0) return PKD_OK;
    e = cudaMemset(workspace, 0, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "pkd_workspace_check: clear");
    if (word & pkd::kErrTimeout) return fail(PKD_ETIMEOUT, "a kernel gave up waiting on its own copies");
    return fail(PKD_EDEVICE_BOUNDS, "a kernel met a seq_lens entry outside [0, max_kv_len] or a block-table "
                                    "entry outside [0, num_pages); those keys were skipped");
}

// Host memory registered with CUDA (pinned) whose device address, under
// unified addressing, is the host address itself.
static bool mapped_host(const void* ptr) {
    cudaPointerAttributes a;
    std::memset(&a, 0, sizeof a);
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost && a.devicePointer == ptr;
}

pkd_status pkd_paged_decode(const void* q, pkd_dtype q_dtype, const void* kv_cache, pkd_dtype kv_dtype,
                            int64_t num_pages, const int32_t* block_table, int64_t block_table_stride,
                            const int32_t* seq_lens, int batch, int sq, int num_heads, int num_kv_heads,
                            int head_dim, int page_size, int max_kv_len, float scale, float q_scale,
                            float k_scale, float v_scale, int window, void* out, pkd_dtype out_dtype, float* lse,
                            void* workspace, size_t workspace_bytes, int chunk_tokens, unsigned flags,
                            void* stream) {
    Plan pl;
    pkd_status st = make_plan(batch, sq, num_heads, num_kv_heads, head_dim, page_size, max_kv_len, kv_dtype, window,
                              chunk_tokens, flags, pl);
    if (st != PKD_OK) return st;
    if (q_dtype != kv_dtype)
        return fail(PKD_EUNSUPPORTED, "q dtype (%d) must equal the cache dtype (%d)", (int)q_dtype, (int)kv_dtype);
    if (out_dtype != PKD_BF16 && out_dtype != PKD_FP16 && out_dtype != PKD_FP32)
        return fail(PKD_EUNSUPPORTED, "out dtype %d not supported (bf16, fp16, fp32)", (int)out_dtype);
    if (batch == 0) return PKD_OK;
    if (!q || !kv_cache || !block_table || !seq_lens || !out || !workspace)
        return fail(PKD_EINVAL, "null pointer argument");
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(workspace, 256) ||
        (lse && !aligned(lse, 4)) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return fail(PKD_EINVAL, "misaligned pointer (q, kv_cache, out: 16 B; workspace: 256 B)");
    if (flags & PKD_FLAG_HOST_IO) {
        const void* io[5] = {q, block_table, seq_lens, out, lse};
        static const char* const names[5] = {"q", "block_table", "seq_lens", "out", "lse"};
        for (int i = 0; i < 5; ++i)
            if (io[i] && !mapped_host(io[i]))
                return fail(PKD_EINVAL, "PKD_FLAG_HOST_IO: %s is not pinned host memory mapped at its own address",
                            names[i]);
    }
    if (num_pages < 1) return fail(PKD_EINVAL, "num_pages must be >= 1");
    if ((int64_t)num_pages * num_kv_heads * page_size >= (int64_t)1 << 31)
        return fail(PKD_EUNSUPPORTED, "cache too large: num_pages*num_kv_heads*page_size must be < 2^31");
    const int64_t need_cols = ((int64_t)max_kv_len + page_size - 1) / page_size;
    if (block_table_stride < need_cols)
        return fail(PKD_EINVAL, "block_table_stride %lld < ceil(max_kv_len/page_size) = %lld",
                    (long long)block_table_stride, (long long)need_cols);
    if (workspace_bytes < pl.bytes)
        return fail(PKD_EINVAL, "workspace too small: %zu < %zu bytes", workspace_bytes, pl.bytes);
    if (!(scale == scale) || !(q_scale == q_scale) || !(k_scale == k_scale) || !(v_scale == v_scale))
        return fail(PKD_EINVAL, "NaN scale");

    CUtensorMap tmap;
    const int elt = elt_bytes(kv_dtype);
    const uint64_t rows = (uint64_t)num_pages * num_kv_heads * page_size;
    st = get_stage_map(tmap, kv_cache, rows, 2 * head_dim * elt, kv_dtype);
    if (st != PKD_OK) return st;

    pkd::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.q = q;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out = out;
    p.lse = lse;
    p.status = reinterpret_cast<int32_t*>(ws);
    p.counters = reinterpret_cast<int32_t*>(ws + pl.off_counters);
    p.part_lse = reinterpret_cast<float*>(ws + pl.off_lse);
    p.part_out = reinterpret_cast<float*>(ws + pl.off_out);
    p.bt_stride = block_table_stride;
    p.num_pages = num_pages;
    p.B = batch;
    p.sq = sq;
    p.Hq = num_heads;
    p.Hkv = num_kv_heads;
    p.G = pl.G;
    p.M = pl.M;
    p.P = page_size;
    p.max_kv_len = max_kv_len;
    p.chunk = pl.chunk;
    p.chunk_share = chunk_tokens > 0 ? chunk_tokens : pkd::kTcMaxChunk;
    p.max_splits = pl.max_splits;
    p.window = window > 0 ? window : 0;
    p.causal = (flags & PKD_FLAG_CAUSAL) ? 1 : 0;
    p.out_dtype = (int)out_dtype;
    page_magic(page_size, p.pmagic, p.pmshift);
    p.scale_log2 = scale * q_scale * k_scale * pkd::kLog2e;
    p.v_scale = v_scale;
    p.wait_ns = (flags & PKD_FLAG_TEST_TIMEOUT) ? 0 : pkd::kWaitNs;

    cudaError_t e;
    cudaStream_t s = (cudaStream_t)stream;
    const int max_ctas = pkd::kFlatMaxWorkers / pkd::kNW;
    if (pl.tc) {
        CUtensorMap kvmap, qmap;
        st = get_stage_map(kvmap, kv_cache, rows, 2 * head_dim * elt, kv_dtype, kStageTcGroup);
        if (st != PKD_OK) return st;
        st = get_q_map(qmap, q, head_dim, num_heads, (uint64_t)batch * sq, pl.G, sq, kv_dtype);
        if (st != PKD_OK) return st;
        e = pkd::launch_decode_tc05(kv_dtype == PKD_BF16, kvmap, qmap, p, s);
    } else if (pl.bal)
        e = pkd::launch_decode_bal(head_dim, kv_dtype == PKD_BF16, pl.mt, pl.nt, tmap, p, s);
    else if (pl.flat && pl.mma)
        e = kv_dtype == PKD_BF16   ? pkd::launch_flat_mma_bf16(head_dim, pl.mt, pl.nt, tmap, p, max_ctas, s)
            : kv_dtype == PKD_FP16 ? pkd::launch_flat_mma_fp16(head_dim, pl.mt, pl.nt, tmap, p, max_ctas, s)
                                   : pkd::launch_flat_mma_fp8(head_dim, pl.mt, pl.nt, tmap, p, max_ctas, s);
    else if (pl.flat)
        e = kv_dtype == PKD_BF16   ? pkd::launch_flat_fma_bf16(head_dim, pl.lpt, pl.mr, tmap, p, max_ctas, s)
            : kv_dtype == PKD_FP16 ? pkd::launch_flat_fma_fp16(head_dim, pl.lpt, pl.mr, tmap, p, max_ctas, s)
                                   : pkd::launch_flat_fma_fp8(head_dim, pl.lpt, pl.mr, tmap, p, max_ctas, s);
    else if (pl.mma && kv_dtype == PKD_FP8_E4M3)
        e = pkd::launch_decode_mma_fp8(head_dim, pl.mt, pl.nt, tmap, p, dim3(pl.max_splits, num_kv_heads, batch), s);
    else if (pl.mma)
        e = pkd::launch_decode_mma(head_dim, kv_dtype == PKD_BF16, pl.mt, pl.nt, tmap, p,
                                   dim3(pl.max_splits, num_kv_heads, batch), s);
    else
        e = pkd::launch_decode_fma(head_dim, (int)kv_dtype, pl.lpt, pl.mr, tmap, p,
                                   dim3(pl.max_splits, num_kv_heads, batch), s);
    if (e != cudaSuccess) return cuda_fail(e, "pkd_paged_decode launch");
    return PKD_OK;
}

pkd_status pkd_cache_write(const void* key, const void* value, pkd_dtype in_dtype, int64_t key_stride,
                           int64_t value_stride, const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                           int head_dim, int page_size, int64_t num_pages, void* kv_cache, pkd_dtype kv_dtype,
                           float k_scale, float v_scale, void* stream) {
    if (num_tokens < 0 || num_kv_heads < 1 || page_size < 1 || num_pages < 1)
        return fail(PKD_EINVAL, "invalid shape: num_tokens=%lld num_kv_heads=%d page_size=%d num_pages=%lld",
                    (long long)num_tokens, num_kv_heads, page_size, (long long)num_pages);
    if (head_dim != 64 && head_dim != 128) return fail(PKD_EUNSUPPORTED, "head_dim %d not supported", head_dim);
    if (in_dtype != PKD_BF16 && in_dtype != PKD_FP16)
        return fail(PKD_EUNSUPPORTED, "key/value dtype %d not supported (bf16, fp16)", (int)in_dtype);
    if (kv_dtype != in_dtype && kv_dtype != PKD_FP8_E4M3)
        return fail(PKD_EUNSUPPORTED, "cache dtype %d must equal the input dtype or be fp8-e4m3", (int)kv_dtype);
    if (key_stride < (int64_t)num_kv_heads * head_dim || value_stride < (int64_t)num_kv_heads * head_dim ||
        key_stride % 8 || value_stride % 8)
        return fail(PKD_EINVAL, "token strides must be >= num_kv_heads*head_dim and multiples of 8 elements");
    if (kv_dtype == PKD_FP8_E4M3 && (!(k_scale > 0.f) || !(v_scale > 0.f)))
        return fail(PKD_EINVAL, "fp8 scales must be positive");
    if (num_tokens == 0) return PKD_OK;
    if (!key || !value || !slot_mapping || !kv_cache) return fail(PKD_EINVAL, "null pointer argument");
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(kv_cache, 16) || !aligned(slot_mapping, 8))
        return fail(PKD_EINVAL, "key, value and kv_cache must be 16-byte aligned");
    cudaError_t e = pkd::launch_cache_write(key, value, (int)in_dtype, slot_mapping, num_tokens, key_stride,
                                            value_stride, num_kv_heads, head_dim, page_size, num_pages, kv_cache,
                                            (int)kv_dtype, k_scale, v_scale, (cudaStream_t)stream);
    return e == cudaSuccess ? PKD_OK : cuda_fail(e, "pkd_cache_write launch");
}

pkd_status pkd_segmented_attention(const void* q, const void* k, const void* v, pkd_dtype dtype, const int32_t* used,
                                   const float* bias, int n, int num_heads, int num_kv_heads, int head_dim, int topk,
                                   int bs, int local, void* out, float* seg_out, float* seg_lse, void* stream) {
    if (n < 0 || num_heads < 1 || num_kv_heads < 1 || topk < 0 || bs < 0 || local < 0)
        return fail(PKD_EINVAL, "invalid shape: n=%d num_heads=%d num_kv_heads=%d topk=%d bs=%d local=%d", n,
                    num_heads, num_kv_heads, topk, bs, local);
    if (dtype != PKD_BF16 && dtype != PKD_FP16)
        return fail(PKD_EUNSUPPORTED, "segmented attention needs fp16 or bf16 (got dtype %d)", (int)dtype);
    if (bs % 8 || local % 8) return fail(PKD_EUNSUPPORTED, "bs (%d) and local (%d) must be multiples of 8", bs, local);
    if (head_dim != 64 && head_dim != 128) return fail(PKD_EUNSUPPORTED, "head_dim %d not supported", head_dim);
    if (num_heads % num_kv_heads) return fail(PKD_EUNSUPPORTED, "num_heads must be a multiple of num_kv_heads");
    const int G = num_heads / num_kv_heads;
    if (G > 16) return fail(PKD_EUNSUPPORTED, "num_heads/num_kv_heads = %d > 16", G);
    if ((seg_out == nullptr) != (seg_lse == nullptr))
        return fail(PKD_EINVAL, "seg_out and seg_lse must be given together");
    if (n == 0) return PKD_OK;
    const long long rows = (long long)n * ((long long)topk * bs + local);
    if (rows == 0 || topk + 1 > 64) return fail(PKD_EUNSUPPORTED, "need 1 <= rows and topk < 64");
    if (!q || !k || !v || !used || !out || (topk > 0 && !bias)) return fail(PKD_EINVAL, "null pointer argument");
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return fail(PKD_EINVAL, "q, k, v and out must be 16-byte aligned");
    if (rows * num_kv_heads >= (long long)1 << 31) return fail(PKD_EUNSUPPORTED, "k/v too large");

    CUtensorMap kmap, vmap;
    const uint64_t d0 = head_dim, d1 = num_kv_heads, d2 = (uint64_t)rows;
    const uint64_t s1 = (uint64_t)head_dim * 2, s2 = (uint64_t)num_kv_heads * head_dim * 2;
    pkd_status st = get_map(kmap, k, 3, d0, d1, d2, s1, s2, dtype, pkd::kStageTok);
    if (st != PKD_OK) return st;
    st = get_map(vmap, v, 3, d0, d1, d2, s1, s2, dtype, pkd::kStageTok);
    if (st != PKD_OK) return st;

    pkd::SegmentParams p;
    std::memset(&p, 0, sizeof p);
    p.kmap = kmap;
    p.vmap = vmap;
    p.k = k;
    p.v = v;
    p.q = q;
    p.used = used;
    p.bias = bias;
    p.out = out;
    p.seg_out = seg_out;
    p.seg_lse = seg_lse;
    p.n = n;
    p.Hq = num_heads;
    p.Hkv = num_kv_heads;
    p.G = G;
    p.D = head_dim;
    p.topk = topk;
    p.bs = bs;
    p.local = local;
    p.bf16 = dtype == PKD_BF16;
    p.scale_log2 = pkd::kLog2e / sqrtf((float)head_dim);
    cudaError_t e = pkd::launch_segmented(p, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "pkd_segmented_attention launch");
    return PKD_OK;
}

pkd_status pkd_segmented_attention_paged(const void* q, pkd_dtype dtype, const void* kv_cache, int64_t num_pages,
                                         const int32_t* block_table, int64_t block_table_stride,
                                         const int32_t* seg_start, const int32_t* used, const float* bias, int n,
                                         int num_heads, int num_kv_heads, int head_dim, int page_size, int topk,
                                         int bs, int local, int max_kv_len, void* out, float* seg_out,
                                         float* seg_lse, void* stream) {
    if (n < 0 || num_heads < 1 || num_kv_heads < 1 || topk < 0 || bs < 0 || local < 0 || max_kv_len < 0 ||
        num_pages < 1 || page_size < 1)
        return fail(PKD_EINVAL, "invalid shape: n=%d num_heads=%d num_kv_heads=%d topk=%d bs=%d local=%d", n,
                    num_heads, num_kv_heads, topk, bs, local);
    if (dtype != PKD_BF16 && dtype != PKD_FP16)
        return fail(PKD_EUNSUPPORTED, "segmented attention needs fp16 or bf16 (got dtype %d)", (int)dtype);
    if (head_dim != 64 && head_dim != 128) return fail(PKD_EUNSUPPORTED, "head_dim %d not supported", head_dim);
    if (page_size % 16) return fail(PKD_EUNSUPPORTED, "page_size %d must be a multiple of 16", page_size);
    if (num_heads % num_kv_heads) return fail(PKD_EUNSUPPORTED, "num_heads must be a multiple of num_kv_heads");
    const int G = num_heads / num_kv_heads;
    if (G > 16) return fail(PKD_EUNSUPPORTED, "num_heads/num_kv_heads = %d > 16", G);
    if (topk + 1 > 64) return fail(PKD_EUNSUPPORTED, "topk must be < 64");
    const long long stages = (long long)topk * ((bs + 15) / 16 + 1) + (local + 15) / 16 + 1;
    if (stages > 512) return fail(PKD_EUNSUPPORTED, "segments span more than 512 16-key stages per query");
    if ((seg_out == nullptr) != (seg_lse == nullptr))
        return fail(PKD_EINVAL, "seg_out and seg_lse must be given together");
    if (block_table_stride < ((int64_t)max_kv_len + page_size - 1) / page_size)
        return fail(PKD_EINVAL, "block_table_stride < ceil(max_kv_len/page_size)");
    if ((int64_t)num_pages * num_kv_heads * page_size >= (int64_t)1 << 31)
        return fail(PKD_EUNSUPPORTED, "cache too large");
    if (n == 0) return PKD_OK;
    if (!q || !kv_cache || !block_table || !seg_start || !used || !out || (topk > 0 && !bias))
        return fail(PKD_EINVAL, "null pointer argument");
    if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16))
        return fail(PKD_EINVAL, "q, kv_cache and out must be 16-byte aligned");

    pkd::SegmentParams p;
    std::memset(&p, 0, sizeof p);
    const uint64_t rows = (uint64_t)num_pages * num_kv_heads * page_size;
    pkd_status st = get_stage_map(p.kmap, kv_cache, rows, 4 * head_dim, dtype);
    if (st != PKD_OK) return st;
    p.vmap = p.kmap;  // unused: a stage's K and V rows come in one copy
    p.k = kv_cache;
    p.paged = 1;
    page_magic(page_size, p.pmagic, p.pmshift);
    p.block_table = block_table;
    p.bt_stride = block_table_stride;
    p.seg_start = seg_start;
    p.num_pages = num_pages;
    p.P = page_size;
    p.max_kv_len = max_kv_len;
    p.q = q;
    p.used = used;
    p.bias = bias;
    p.out = out;
    p.seg_out = seg_out;
    p.seg_lse = seg_lse;
    p.n = n;
    p.Hq = num_heads;
    p.Hkv = num_kv_heads;
    p.G = G;
    p.D = head_dim;
    p.topk = topk;
    p.bs = bs;
    p.local = local;
    p.bf16 = dtype == PKD_BF16;
    p.scale_log2 = pkd::kLog2e / sqrtf((float)head_dim);
    cudaError_t e = pkd::launch_segmented(p, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "pkd_segmented_attention_paged launch");
    return PKD_OK;
}

pkd_status pkd_lse_merge(const float* part_out, const float* part_lse, const float* prior, const int32_t* live, int n,
                         int parts, int heads, int head_dim, void* out, pkd_dtype out_dtype, float* lse_out,
                         void* stream) {
    if (n < 0 || parts < 0 || heads < 1 || head_dim < 1)
        return fail(PKD_EINVAL, "invalid shape: n=%d parts=%d heads=%d head_dim=%d", n, parts, heads, head_dim);
    if (head_dim > 256 || parts > 1024)
        return fail(PKD_EUNSUPPORTED, "lse_merge supports head_dim <= 256 and parts <= 1024");
    if (out_dtype != PKD_BF16 && out_dtype != PKD_FP16 && out_dtype != PKD_FP32)
        return fail(PKD_EUNSUPPORTED, "out dtype %d not supported", (int)out_dtype);
    if (n == 0) return PKD_OK;
    if ((parts > 0 && (!part_out || !part_lse)) || !out) return fail(PKD_EINVAL, "null pointer argument");
    pkd::MergeParams p;
    std::memset(&p, 0, sizeof p);
    p.part_out = part_out;
    p.part_lse = part_lse;
    p.prior = prior;
    p.live = live;
    p.n = n;
    p.parts = parts;
    p.prior_cols = parts;
    p.heads = heads;
    p.D = head_dim;
    p.out = out;
    p.out_dtype = (int)out_dtype;
    p.lse_out = lse_out;
    cudaError_t e = pkd::launch_lse_merge(p, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "pkd_lse_merge launch");
    return PKD_OK;
}

}  // extern "C"
