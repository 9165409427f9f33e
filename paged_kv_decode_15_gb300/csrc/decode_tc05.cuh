// Paged decode of query blocks with 17-32 rows per kv head (M = sq * Hq/Hkv)
// on the 5th-generation tensor cores, accumulators in tensor memory (TMEM);
// dense or causal (each query token sees the keys up to its own position,
// within the window).
//
// One persistent CTA per SM.  A request's visible keys are cut into chunks
// of at most `chunk` keys (whole 128-key tiles where the chunk allows).
// With no more (request, kv head, chunk) items than CTAs each CTA takes one
// chunk.  Otherwise the launch's work is the sequence of all tiles in the
// order (request, kv head, chunk, tile) and each CTA takes an equal share --
// a contiguous range at least one chunk long -- so that every CTA streams
// the same number of bytes and none waits for a straggler at the end.  A CTA
// walks its range as work items of at most one chunk (the block-table entries
// of an item fit in shared memory); consecutive items of one (request, kv
// head) unit form a run that keeps accumulating in TMEM, so a unit is split
// -- partial result per run, merged by LSE -- only where a share boundary
// cuts it.  Per 128-key tile of an item:
//   S^T = K Q^T      tcgen05.mma, M = 128 keys, N = 32 query rows, K = 128
//                    dims: A = the K tile as TMA lands it (K-major, 128-byte
//                    swizzle), B = the run's q rows (K-major); S^T in TMEM.
//   softmax          one key per thread of a warp group (TMEM lane = key):
//                    tcgen05.ld of its group's 16 scores, online softmax per query
//                    row in fp32 whose reference maximum moves only when a
//                    row's maximum grows by more than 2^8 (then O and l are
//                    rescaled), P written in the operand type over the
//                    tile's K in shared memory (dead once S is computed), so
//                    that each slot carries its own P.
//   O^T += V^T P^T   M = 128 dims, N = 32 rows, K = 128 keys: A = the V tile
//                    read MN-major, B = P (K-major); O^T accumulates in TMEM
//                    over the run's tiles.
// A tile lands as sixteen 4 KB groups of 8 keys, every group holding the
// four 128-byte chunks of its rows (K dims 0-63, K 64-127, V 0-63, V 64-127;
// 1 KB each, 128-byte swizzle), so that both products see rows at a uniform
// 4 KB stride; a 16-key stage (two groups, contiguous in the page) is one
// TMA copy of a 4-D view of the cache.
// Warp roles: warps 0-7 run the softmax in two groups of four, each group
// taking 16 of the 32 query rows, warps 8-11 the epilogue (read O^T,
// normalise, write out and LSE -- or, for a unit split into several runs,
// write the run's partial result), warp 12 loads (the item's block-table
// entries, q per run, the K/V tiles), warp 13 issues S^T = K Q^T and warp 14
// O^T += V^T P^T (one thread each, so that a tile's K/V slot is released as
// soon as its P is written).  A split unit's runs count their arrivals in
// the workspace; the epilogue of the CTA that completes the last one merges
// the partials by LSE (at most a few units per CTA, the shares being at
// least a chunk long).
// Every wait is bounded; a failure raises the status word and every role
// leaves after letting its own copies and products complete.
#pragma once

#include "decode_common.cuh"
#include "tc05.cuh"

namespace pkd {

constexpr int kTcTile = 128;      // keys per tile: the M of S^T = K Q^T
constexpr int kTcRows = 32;       // query rows per unit, padded: the N of both products
constexpr int kTcNS = 3;          // K/V tile ring
constexpr int kTcNI = 4;          // work-item ring
constexpr int kTcMaxChunk = 2048; // keys per chunk at most
constexpr int kTcItemPages = kTcMaxChunk / kStageTok + 8;
constexpr int kTcMaxBatch = 512;  // requests whose lengths and work prefix the CTA keeps in shared memory
constexpr int kTcPageRegs = (kTcItemPages + 31) / 32;  // block-table entries of an item per producer lane
constexpr int kTcThreads = 480;   // two softmax groups and the epilogue (four warps each), loads, S MMAs, O MMAs
constexpr int kTcGroupRows = 16;  // query rows of a softmax group
constexpr float kTcRescale = 8.f; // log2 units: P stays below 2^8 between rescales

// cont: the item continues the previous item's run (same unit, same
// accumulators); last: the run ends with it (the epilogue follows); slot: the
// run's partial slot in its unit; pieces: the unit's runs (1: this run is
// the whole unit); L: the request's length (for the causal mask).
struct TcItem {
    int b, hk, slot, pieces, cont, last, t0, t1, ntiles, bad, end, L, pad[4];
    int pages[kTcItemPages];      // table columns t0/P ..; -1: outside the pool (keys skipped)
};

// The chunks of a visible range of `vis` keys for chunks of at most C keys:
// n chunks of `len` keys (whole 128-key tiles unless C is smaller or not a
// multiple of 128), the last one shorter; all non-empty.
struct TcChunks {
    int n, len, tiles_full, tiles_last, tiles;  // tiles: of one kv head, all chunks
};
__host__ __device__ __forceinline__ TcChunks tc_chunks(int vis, int C) {
    TcChunks ch{0, C, 0, 0, 0};
    if (vis <= 0) return ch;
    const int n0 = (vis + C - 1) / C, even = (vis + n0 - 1) / n0;
    const int whole = (even + kTcTile - 1) / kTcTile * kTcTile;
    ch.len = whole < C ? whole : C;
    ch.n = (vis + ch.len - 1) / ch.len;
    ch.tiles_full = (ch.len + kTcTile - 1) / kTcTile;
    ch.tiles_last = (vis - (ch.n - 1) * ch.len + kTcTile - 1) / kTcTile;
    ch.tiles = (ch.n - 1) * ch.tiles_full + ch.tiles_last;
    return ch;
}

// Shared memory.  Operand regions are 1024-byte aligned (128-byte swizzle atoms).
struct TcShape {
    static constexpr int GROUP = 4096;                 // 8 keys: K 0-63 | K 64-127 | V 0-63 | V 64-127
    static constexpr int TILE = (kTcTile / 8) * GROUP; // 64 KB
    static constexpr int QB = kTcRows * 256;           // q rows: two regions of 32 x 128 bytes
    // P of a tile goes where its K was (dead once S is computed): 8-row group
    // g of key half h in the first 1 KB of the slot's 4 KB group 4h + g
    static constexpr int OFF_KV = 0;
    static constexpr int OFF_Q = OFF_KV + kTcNS * TILE;
    static constexpr int OFF_ITEM = OFF_Q + 2 * QB;
    static constexpr int OFF_STAT = OFF_ITEM + kTcNI * static_cast<int>(sizeof(TcItem));  // [2][4 warps + m][32]
    static constexpr int OFF_RED = OFF_STAT + 2 * 5 * kTcRows * 4;  // float [2][32 rows][4 warps]
    static constexpr int OFF_VOTE = OFF_RED + 2 * kTcRows * 4 * 4;  // int votes [2][4] per group; [24]: arrivals
    static constexpr int OFF_PREF = OFF_VOTE + 128;                 // int [kTcMaxBatch + 1]: work prefix
    static constexpr int OFF_LENS = OFF_PREF + (kTcMaxBatch + 1) * 4;  // int [kTcMaxBatch]: clamped lengths
    static constexpr int OFF_BAR = (OFF_LENS + kTcMaxBatch * 4 + 7) & ~7;
    // barriers: K/V full/empty (the empty one also says P.V is done), q
    // full/empty, S full/empty, P full (per slot), O full/free, stats
    // full/free, item full/empty, final drain
    static constexpr int B_TF = 0, B_TE = B_TF + kTcNS, B_QF = B_TE + kTcNS, B_QE = B_QF + 2;
    static constexpr int B_SF = B_QE + 2, B_SE = B_SF + 2, B_PF = B_SE + 2;
    static constexpr int B_OF = B_PF + kTcNS, B_OE = B_OF + 2, B_XF = B_OE + 2, B_XE = B_XF + 2;
    static constexpr int B_IF = B_XE + 2, B_IE = B_IF + kTcNI, B_DR = B_IE + kTcNI, NBAR = B_DR + 2;
    static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_TMEM + 16 + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    static_assert(SMEM > 114 * 1024, "one CTA per SM: its 128 TMEM columns are always free");
};

// Row reduction of a warp's 32 keys: each lane holds v[r] for its key and
// rows r = 0..31; returns, in lane r, op over the warp's keys of row r.
// (At each step the lane keeps the half of its rows whose index bit matches
// its own lane bit and receives its partner's values for them.)
template <class Op>
__device__ __forceinline__ float tc_row_reduce(const float (&v)[32], int lane, Op op) {
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const bool up = lane & 16;
        a[i] = op(up ? v[i + 16] : v[i], __shfl_xor_sync(kFull, up ? v[i] : v[i + 16], 16));
    }
    float b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = lane & 8;
        b[i] = op(up ? a[i + 8] : a[i], __shfl_xor_sync(kFull, up ? a[i] : a[i + 8], 8));
    }
    float c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = lane & 4;
        c[i] = op(up ? b[i + 4] : b[i], __shfl_xor_sync(kFull, up ? b[i] : b[i + 4], 4));
    }
    float d[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = lane & 2;
        d[i] = op(up ? c[i + 2] : c[i], __shfl_xor_sync(kFull, up ? c[i] : c[i + 2], 2));
    }
    const bool up = lane & 1;
    return op(up ? d[1] : d[0], __shfl_xor_sync(kFull, up ? d[0] : d[1], 1));
}

// The same for 16 rows: lanes 2r and 2r + 1 both return the reduction of row r.
template <class Op>
__device__ __forceinline__ float tc_row_reduce16(const float (&v)[16], int lane, Op op) {
    float b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = lane & 16;
        b[i] = op(up ? v[i + 8] : v[i], __shfl_xor_sync(kFull, up ? v[i] : v[i + 8], 16));
    }
    float c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = lane & 8;
        c[i] = op(up ? b[i + 4] : b[i], __shfl_xor_sync(kFull, up ? b[i] : b[i + 4], 8));
    }
    float d[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = lane & 4;
        d[i] = op(up ? c[i + 2] : c[i], __shfl_xor_sync(kFull, up ? c[i] : c[i + 2], 4));
    }
    const bool up = lane & 2;
    const float e = op(up ? d[1] : d[0], __shfl_xor_sync(kFull, up ? d[0] : d[1], 2));
    return op(e, __shfl_xor_sync(kFull, e, 1));
}

// A four-warp group's own barrier: named barrier `id`, 128 threads.
__device__ __forceinline__ void tc_group_sync(int id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// A vote of a four-warp group: OR of `bits` over the group.  Votes alternate
// between two buffers: a warp writes buffer v only after the barrier of vote
// v - 1, which every warp passes after reading vote v - 2.
__device__ __forceinline__ int tc_vote(int* votes, int id, int& nvote, int q4, int lane, int bits) {
    bits = __reduce_or_sync(kFull, bits);
    int* v = votes + (nvote & 1) * 4;
    ++nvote;
    if (lane == 0) v[q4] = bits;
    tc_group_sync(id);
    return v[0] | v[1] | v[2] | v[3];
}

// A wait every lane of the warp takes, with a warp-uniform result.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, const DecodeParams& p, uint64_t limit) {
    return __all_sync(kFull, mbar_wait(bar, parity, p.status, limit));
}

__device__ __forceinline__ float tc_pick16(const float (&v)[16], int r) {
    float x = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) x = i == r ? v[i] : x;
    return x;
}

// Element r of a register array, r not known at compile time (no local memory).
__device__ __forceinline__ float tc_pick(const float (&v)[32], int r) {
    float x = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) x = i == r ? v[i] : x;
    return x;
}

// LSE merge of the `np` pieces (partial results) of a split unit, run by the
// epilogue warps of the CTA that completed its last piece.  Warp q4 takes
// query rows q4, q4 + 4, ... (four at a time); lane j reads piece j's LSE
// (blocks of 32 pieces) and sums dims 4j .. 4j+3 over the pieces, all loads
// of a block issued before the first is used.  Pieces were written by other
// CTAs: L2 loads only.
__device__ __forceinline__ void tc_merge_unit(const DecodeParams& p, long long unit, long long row0, int np, int q4,
                                              int lane) {
    constexpr int R = 4;
    const float* pl = p.part_lse + unit * p.max_splits * kTcRows;
    const float* po = p.part_out + unit * p.max_splits * kTcRows * 128 + 4 * lane;
#pragma unroll 1
    for (int r0 = q4; r0 < p.M; r0 += 4 * R) {
        float lc0[R], mx[R], ws[R];
        float4 acc[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = r0 + 4 * i;
            lc0[i] = (lane < np && r < p.M) ? __ldcg(pl + lane * kTcRows + r) : -INFINITY;
            mx[i] = lc0[i];
            ws[i] = 0.f;
            acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int s = 32 + lane; s - lane < np; s += 32)
#pragma unroll
            for (int i = 0; i < R; ++i)
                if (s < np && r0 + 4 * i < p.M) mx[i] = fmaxf(mx[i], __ldcg(pl + s * kTcRows + r0 + 4 * i));
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx[i] = fmaxf(mx[i], __shfl_xor_sync(kFull, mx[i], o));
        for (int s0 = 0; s0 < np; s0 += 32) {
            const int n = min(32, np - s0);
            float wl[R];
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int r = r0 + 4 * i;
                const float lc = s0 == 0 ? lc0[i]
                                         : (s0 + lane < np && r < p.M ? __ldcg(pl + (s0 + lane) * kTcRows + r) : -INFINITY);
                wl[i] = lc == -INFINITY ? 0.f : fast_exp2(lc - mx[i]);
                ws[i] += wl[i];
            }
            for (int j = 0; j < n; ++j) {
                float4 v[R];
#pragma unroll
                for (int i = 0; i < R; ++i)
                    v[i] = r0 + 4 * i < p.M
                               ? __ldcg(reinterpret_cast<const float4*>(po + ((s0 + j) * kTcRows + r0 + 4 * i) * 128))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    const float w = __shfl_sync(kFull, wl[i], j);
                    acc[i] = make_float4(fmaf(w, v[i].x, acc[i].x), fmaf(w, v[i].y, acc[i].y),
                                         fmaf(w, v[i].z, acc[i].z), fmaf(w, v[i].w, acc[i].w));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int r = r0 + 4 * i;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ws[i] += __shfl_xor_sync(kFull, ws[i], o);
            if (r >= p.M) continue;
            const float sc = ws[i] > 0.f ? p.v_scale / ws[i] : 0.f;
            const long long orow = row0 + static_cast<long long>(r / p.G) * p.Hq + r % p.G;
            const long long o0 = orow * 128 + 4 * lane;
            store_out(p.out, o0 + 0, acc[i].x * sc, p.out_dtype);
            store_out(p.out, o0 + 1, acc[i].y * sc, p.out_dtype);
            store_out(p.out, o0 + 2, acc[i].z * sc, p.out_dtype);
            store_out(p.out, o0 + 3, acc[i].w * sc, p.out_dtype);
            if (lane == 0 && p.lse) p.lse[orow] = ws[i] > 0.f ? (mx[i] + __log2f(ws[i])) * kLn2 : -INFINITY;
        }
    }
}

template <bool kBF16, bool kCausal>
__global__ void __launch_bounds__(kTcThreads, 1)
decode_tc05_kernel(const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap qmap,
                   const DecodeParams p) {
    using S = TcShape;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb0 = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
    TcItem* items = reinterpret_cast<TcItem*>(smem + S::OFF_ITEM);
    float* stats = reinterpret_cast<float*>(smem + S::OFF_STAT);
    float* red = reinterpret_cast<float*>(smem + S::OFF_RED);
    int* votes = reinterpret_cast<int*>(smem + S::OFF_VOTE);
    int* pref = reinterpret_cast<int*>(smem + S::OFF_PREF);
    int* lens = reinterpret_cast<int*>(smem + S::OFF_LENS);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TMEM);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.Hkv, M = p.M;
    int C = p.chunk;  // warp 12: the chunk of the launch's mode
    auto bar = [&](int i) { return smem_u32(bars + i); };

    // ------------------------------------------------------------ set-up
    if (tid == 0) {
        for (int i = 0; i < kTcNS; ++i) {
            mbar_init(bar(S::B_TF + i), 1);
            mbar_init(bar(S::B_TE + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(S::B_QF + i), 1);
            mbar_init(bar(S::B_QE + i), 1);
            mbar_init(bar(S::B_SF + i), 1);
            mbar_init(bar(S::B_SE + i), 256);
            mbar_init(bar(S::B_OF + i), 1);
            mbar_init(bar(S::B_OE + i), 128);
            mbar_init(bar(S::B_XF + i), 256);
            mbar_init(bar(S::B_XE + i), 128);
        }
        for (int i = 0; i < kTcNS; ++i) mbar_init(bar(S::B_PF + i), 256);
        for (int i = 0; i < kTcNI; ++i) {
            mbar_init(bar(S::B_IF + i), 32);
            mbar_init(bar(S::B_IE + i), 2 + 256 + 128);  // both MMA threads, softmax and epilogue groups
        }
        mbar_init(bar(S::B_DR), 1);
        mbar_init(bar(S::B_DR + 1), 1);
        fence_barrier_init();
    }
    if (warp == 13) {
        tc05::alloc(smem_u32(tslot), 128);  // S^T: columns 0-63 (two buffers), O^T: 64-127 (two)
        tc05::relinquish_alloc_permit();
    }
    // warp 12: the launch's work -- chunks (item mode, no more than CTAs) or
    // tiles of the share mode's chunks -- and its prefix per request in pref
    bool by_item = true;
    int total = 0;
    if (warp == 12) {
        int n_items = 0, n_tiles = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            int ni = 0, nt = 0;
            if (b < p.B) {
                const int L = clamp_len(p, b, true), vis = L - visible_lo(p, L);
                ni = tc_chunks(vis, p.chunk).n * Hkv;
                nt = tc_chunks(vis, p.chunk_share).tiles * Hkv;
                lens[b] = L;
            }
            n_items += __reduce_add_sync(kFull, ni);
            n_tiles += __reduce_add_sync(kFull, nt);
        }
        by_item = n_items <= static_cast<int>(gridDim.x);
        total = by_item ? n_items : n_tiles;
        C = by_item ? p.chunk : p.chunk_share;
        int run = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            int n = 0;
            if (b < p.B) {
                const int L = lens[b];
                const TcChunks ch = tc_chunks(L - visible_lo(p, L), C);
                n = (by_item ? ch.n : ch.tiles) * Hkv;
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, n, o);
                if (lane >= o) n += y;
            }
            if (b < p.B) pref[b + 1] = run + n;
            run += __shfl_sync(kFull, n, 31);
        }
        if (lane == 0) pref[0] = 0;
    }
    if (warp < 4 && M < kTcRows) {
        // q rows M..31 of both buffers stay zero (the copies fill rows < M)
        for (int e = tid; e < 2 * 2 * (kTcRows - M) * 8; e += 128) {
            const int chunk = e & 7, row = M + (e >> 3) % (kTcRows - M), reg = (e >> 3) / (kTcRows - M);
            *reinterpret_cast<uint4*>(smem + S::OFF_Q + reg * 4096 + row * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
    }
    if (warp >= 8 && warp < 12) {
        // requests without a visible key: out = 0, lse = -inf
        const int et = tid - 256;
        for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
            const int L = clamp_len(p, b, false);
            if (L - visible_lo(p, L) > 0) continue;
            for (int e = et; e < Hkv * M * 128; e += 128) {
                const int hk = e / (M * 128), r = (e / 128) % M, d = e % 128;
                store_out(p.out, out_index(p, b, hk, r, d, 128), 0.f, p.out_dtype);
                if (d == 0 && p.lse)
                    p.lse[(static_cast<long long>(b) * p.sq + r / p.G) * p.Hq + hk * p.G + r % p.G] = -INFINITY;
            }
        }
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tmem = *tslot;
    constexpr uint32_t kIdS = tc05::idesc_f16(kBF16, kTcTile, kTcRows, false, false);  // S^T = K Q^T
    constexpr uint32_t kIdO = tc05::idesc_f16(kBF16, kTcTile, kTcRows, true, false);   // O^T += V^T P^T

    if (warp == 12) {
        // ---------------------------------------------------------- loads
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            prefetch_tmap(&kvmap);
            prefetch_tmap(&qmap);
        }
        int t = 0, tiss = 0, qiss = 0;
        bool ok = true;
        // This CTA's work, [cur, stop) of the launch's sequence: item
        // blockIdx.x in item mode; in share mode an equal share of the tiles,
        // at least one chunk long (so that a unit of n chunks has at most n + 1
        // pieces).  It is walked item by item, one ahead: the next item is
        // decoded while this one streams (to know where a run ends), and its
        // block-table entries are loaded into registers (lane j holds entries
        // j, j + 32, ...) so that they have landed when it is published.
        const int G = static_cast<int>(gridDim.x), me = static_cast<int>(blockIdx.x);
        const int share = max((total + G - 1) / G, (C + kTcTile - 1) / kTcTile);
        int cur = by_item ? me : static_cast<int>(min(static_cast<long long>(total), static_cast<long long>(me) * share));
        const int stop = by_item ? min(total, me + 1) : min(total, cur + share);
        struct Work {
            int b, hk, unit, slot, pieces, t0, t1, ntiles, col0, npg, L;
            bool valid, cont;
        };
        int prev_unit = -1;
        auto next_work = [&](Work& x) {
            x.valid = cur < stop;
            if (!x.valid) return;
            int lo_b = 0, hi_b = p.B;  // pref[lo_b] <= cur < pref[hi_b]
            while (hi_b - lo_b > 1) {
                const int mid = (lo_b + hi_b) >> 1;
                if (pref[mid] <= cur) lo_b = mid; else hi_b = mid;
            }
            const int L = lens[lo_b], lo = visible_lo(p, L);
            const TcChunks ch = tc_chunks(L - lo, C);
            const int r = cur - pref[lo_b];
            int hk, c, k0, k1;
            if (by_item) {
                hk = r / ch.n;
                c = r - hk * ch.n;
                k0 = 0;
                k1 = c < ch.n - 1 ? ch.tiles_full : ch.tiles_last;
                x.slot = c;
                x.pieces = ch.n;
            } else {
                // tile rr of the unit: chunk c, its tile k0
                hk = r / ch.tiles;
                const int rr = r - hk * ch.tiles, ustart = cur - rr;
                c = min(rr / ch.tiles_full, ch.n - 1);
                k0 = rr - c * ch.tiles_full;
                k1 = min(c < ch.n - 1 ? ch.tiles_full : ch.tiles_last, k0 + (stop - cur));
                // the unit's pieces: one per share it meets
                x.slot = me - ustart / share;
                x.pieces = (ustart + ch.tiles - 1) / share - ustart / share + 1;
            }
            const int cs = lo + c * ch.len, ce = min(cs + ch.len, L);
            x.b = lo_b;
            x.hk = hk;
            x.L = L;
            x.unit = lo_b * Hkv + hk;
            x.t0 = cs + k0 * kTcTile;
            x.t1 = min(cs + k1 * kTcTile, ce);
            x.ntiles = k1 - k0;
            x.cont = x.unit == prev_unit;
            x.col0 = page_div(x.t0, p.pmagic, p.pmshift);
            x.npg = page_div(x.t1 - 1, p.pmagic, p.pmshift) - x.col0 + 1;
            prev_unit = x.unit;
            cur += by_item ? 1 : k1 - k0;
        };
        int pg_next[kTcPageRegs];
        auto load_pages = [&](const Work& x) {
#pragma unroll
            for (int k = 0; k < kTcPageRegs; ++k) {
                const int j = lane + 32 * k;
                pg_next[k] = (x.valid && j < x.npg)
                                 ? p.block_table[static_cast<long long>(x.b) * p.bt_stride + x.col0 + j] : -1;
            }
        };
        Work w, wn;
        next_work(w);
        load_pages(w);
        next_work(wn);
        int ru = 0;  // runs started
        for (int it = 0;; ++it) {
            const int slot = it % kTcNI;
            if (it >= kTcNI && !tc_wait(bar(S::B_IE + slot), ((it / kTcNI) - 1) & 1, p, kWaitNs)) { ok = false; break; }
            TcItem& I = items[slot];
            if (!w.valid) {
                if (lane == 0) I.end = 1;
                __syncwarp();
                mbar_arrive(bar(S::B_IF + slot));
                break;
            }
            const int b = w.b, hk = w.hk, t0 = w.t0, t1 = w.t1, ntiles = w.ntiles, col0 = w.col0;
            int bad = 0;
#pragma unroll
            for (int k = 0; k < kTcPageRegs; ++k) {
                const int j = lane + 32 * k;
                if (j < w.npg) {
                    int pg = pg_next[k];
                    if (pg < 0 || pg >= p.num_pages) {
                        raise_status(p, kErrBounds);
                        pg = -1;
                        bad = 1;
                    }
                    I.pages[j] = pg;
                }
            }
            bad = __any_sync(kFull, bad);
            if (lane == 0) {
                I.b = b; I.hk = hk; I.slot = w.slot; I.pieces = w.pieces; I.L = w.L;
                I.cont = w.cont; I.last = !wn.valid || wn.unit != w.unit;
                I.t0 = t0; I.t1 = t1; I.ntiles = ntiles; I.bad = bad; I.end = 0;
            }
            __syncwarp();
            mbar_arrive(bar(S::B_IF + slot));
            const bool new_run = !w.cont;
            // the next item's table entries, requested while this one streams
            load_pages(wn);
            // a run's q rows (two 64-dim halves)
            if (new_run) {
                const int qb = ru & 1;
                if (ru >= 2 && !tc_wait(bar(S::B_QE + qb), ((ru >> 1) - 1) & 1, p, kWaitNs)) { ok = false; break; }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar(S::B_QF + qb), M * 256);
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(sb0 + S::OFF_Q + qb * S::QB + h * 4096, &qmap, 64 * h, hk * p.G, b * p.sq,
                                    bar(S::B_QF + qb), pol);
                }
                ++qiss;
                ++ru;
            }
            // K/V tiles: lane s < 8 loads stage s (16 keys: two 4 KB groups, one copy)
            for (int k = 0; k < ntiles; ++k, ++t) {
                const int tok0 = t0 + k * kTcTile, ts = t % kTcNS;
                if (t >= kTcNS && !tc_wait(bar(S::B_TE + ts), ((t / kTcNS) - 1) & 1, p, kWaitNs)) { ok = false; break; }
                const int tok = tok0 + lane * kStageTok;
                const int col = page_div(tok, p.pmagic, p.pmshift);
                const int pg = (lane < kTcTile / kStageTok && tok < t1) ? I.pages[col - col0] : -1;
                const unsigned loaded = __ballot_sync(kFull, pg >= 0);
                if (lane == 0) mbar_arrive_expect_tx(bar(S::B_TF + ts), __popc(loaded) * 2 * S::GROUP);
                __syncwarp();
                if (pg >= 0) {
                    const int row = (pg * Hkv + hk) * p.P + (tok - col * p.P);  // a multiple of 16
                    const uint32_t dst = sb0 + S::OFF_KV + ts * S::TILE + 2 * lane * S::GROUP;
                    tma_load_4d(dst, &kvmap, 0, 0, 0, row >> 3, bar(S::B_TF + ts), pol);
                }
                ++tiss;
            }
            if (!ok) break;
            w = wn;
            next_work(wn);
        }
        if (!ok) {
            // let every issued copy land before the CTA leaves
            if (lane == 0) raise_status(p, kErrTimeout);
            for (int j = max(0, tiss - kTcNS); j < tiss; ++j) mbar_wait(bar(S::B_TF + j % kTcNS), (j / kTcNS) & 1);
            for (int j = max(0, qiss - 2); j < qiss; ++j) mbar_wait(bar(S::B_QF + (j & 1)), (j >> 1) & 1);
        }
    } else if (warp == 13) {
        // ----------------------------------------------------- S^T = K Q^T
        if (lane == 0) {
            bool ok = true;
            int t = 0, ru = 0;
            for (int it = 0; ok; ++it) {
                const int slot = it % kTcNI;
                if (!mbar_wait(bar(S::B_IF + slot), (it / kTcNI) & 1, p.status)) { ok = false; break; }
                const TcItem& I = items[slot];
                if (I.end) break;
                const int ntiles = I.ntiles, last = I.last;
                if (!I.cont) ++ru;
                const int qb = (ru - 1) & 1;
                mbar_arrive(bar(S::B_IE + slot));
                if (!I.cont && !mbar_wait(bar(S::B_QF + qb), ((ru - 1) >> 1) & 1, p.status, p.wait_ns)) { ok = false; break; }
                for (int k = 0; k < ntiles; ++k, ++t) {
                    const int ts = t % kTcNS, sbuf = t & 1;
                    if (!mbar_wait(bar(S::B_TF + ts), (t / kTcNS) & 1, p.status, p.wait_ns)) { ok = false; break; }
                    if (t >= 2 && !mbar_wait(bar(S::B_SE + sbuf), ((t >> 1) - 1) & 1, p.status)) { ok = false; break; }
                    tc05::fence_after_sync();
                    const uint32_t tile = sb0 + S::OFF_KV + ts * S::TILE, qt = sb0 + S::OFF_Q + qb * S::QB;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc05::mma_f16(tmem + 32 * sbuf,
                                      tc05::smem_desc(tile + (kk >> 2) * 1024 + (kk & 3) * 32, 16, S::GROUP),
                                      tc05::smem_desc(qt + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024), kIdS, kk > 0);
                    tc05::commit(bar(S::B_SF + sbuf));
                    if (last && k == ntiles - 1) tc05::commit(bar(S::B_QE + qb));
                }
            }
            if (!ok) raise_status(p, kErrTimeout);
            // every product issued has completed before TMEM is freed
            tc05::commit(bar(S::B_DR));
            mbar_wait(bar(S::B_DR), 0);
        }
        __syncwarp();
    } else if (warp == 14) {
        // ------------------------------------------------- O^T += V^T P^T
        // issued as soon as the softmax has written P, so that the tile's
        // K/V slot is released without waiting for the next tile's keys
        if (lane == 0) {
            bool ok = true;
            int t = 0, ru = 0;
            for (int it = 0; ok; ++it) {
                const int slot = it % kTcNI;
                if (!mbar_wait(bar(S::B_IF + slot), (it / kTcNI) & 1, p.status)) { ok = false; break; }
                const TcItem& I = items[slot];
                if (I.end) break;
                const int ntiles = I.ntiles, last = I.last, cont = I.cont;
                if (!cont) ++ru;
                const int ob = (ru - 1) & 1;
                mbar_arrive(bar(S::B_IE + slot));
                for (int k = 0; k < ntiles; ++k, ++t) {
                    const int ts = t % kTcNS;
                    const bool run_start = !cont && k == 0;
                    if (!mbar_wait(bar(S::B_PF + ts), (t / kTcNS) & 1, p.status)) { ok = false; break; }
                    if (run_start && ru >= 3 && !mbar_wait(bar(S::B_OE + ob), (((ru - 1) >> 1) - 1) & 1, p.status)) { ok = false; break; }
                    tc05::fence_after_sync();
                    const uint32_t tile = sb0 + S::OFF_KV + ts * S::TILE;
#pragma unroll
                    for (int j = 0; j < kTcTile / 16; ++j)
                        tc05::mma_f16(tmem + 64 + 32 * ob,
                                      tc05::smem_desc(tile + 2 * j * S::GROUP + 2048, 1024, S::GROUP),
                                      tc05::smem_desc(tile + (j >> 2) * 4 * S::GROUP + (j & 3) * 32, 16, S::GROUP),
                                      kIdO, !(run_start && j == 0));
                    tc05::commit(bar(S::B_TE + ts));
                    if (last && k == ntiles - 1) tc05::commit(bar(S::B_OF + ob));
                }
            }
            if (!ok) raise_status(p, kErrTimeout);
            tc05::commit(bar(S::B_DR + 1));
            mbar_wait(bar(S::B_DR + 1), 0);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------- softmax
        // two groups of four warps: group g takes query rows 16g .. 16g+15
        // (columns of S^T and O^T), with votes and reductions of its own
        constexpr int RG = kTcGroupRows;
        const int grp = warp >> 2, q4 = warp & 3, rbase = RG * grp, key = 32 * q4 + lane;  // key: TMEM lane of S^T
        const int gid = 1 + 2 * grp;  // the group's named barrier
        int* gvotes = votes + 8 * grp;
        float* gred = red + grp * 2 * RG * 4;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q4) << 16;
        const float scale2 = p.scale_log2;
        int nvote = 0, t = 0, ru = 0;
        float m_used[RG], lp[RG];
        for (int it = 0;; ++it) {
            const int slot = it % kTcNI;
            const int fail = !tc_wait(bar(S::B_IF + slot), (it / kTcNI) & 1, p, kWaitNs);
            const TcItem& I = items[slot];
            const int end = fail ? 1 : I.end;
            if (tc_vote(gvotes, gid, nvote, q4, lane, (fail ? 2 : 0) | (end ? 1 : 0))) {
                if (fail) raise_status(p, kErrTimeout);
                break;
            }
            const int t0 = I.t0, t1 = I.t1, ntiles = I.ntiles, bad = I.bad, cont = I.cont, last = I.last;
            // causal: query token i = row / G sits at L - sq + i and sees keys up
            // to it (and, with a window, from window - 1 before it on)
            const int first_pos = I.L - p.sq;
            const int col0 = page_div(t0, p.pmagic, p.pmshift);
            if (!cont) {
                // a new run: fresh statistics
                ++ru;
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    m_used[r] = -INFINITY;
                    lp[r] = 0.f;
                }
            }
            const int ob = (ru - 1) & 1;
            bool abort = false;
            for (int k = 0; k < ntiles; ++k, ++t) {
                const int sbuf = t & 1, ts = t % kTcNS;
                const int tok0 = t0 + k * kTcTile;
                const int nvalid = min(kTcTile, t1 - tok0);
                bool valid = key < nvalid;
                // causal: this key is visible to the rows [rmin, rmax) of the group
                int rmin = 0, rmax = RG;
                if constexpr (kCausal) {
                    const int d = tok0 + key - first_pos;  // first token that sees the key
                    rmin = d * p.G - rbase;
                    if (p.window > 0) rmax = (d + p.window) * p.G - rbase;
                }
                if (bad && valid) valid = I.pages[page_div(tok0 + key, p.pmagic, p.pmshift) - col0] >= 0;
                float x[RG];
                const bool got = tc_wait(bar(S::B_SF + sbuf), (t >> 1) & 1, p, kWaitNs);
                if (got) {
                    tc05::fence_after_sync();
                    uint32_t sr[RG];
                    tc05::ld_32x32b_x16(tmem + lane_addr + 32 * sbuf + rbase, sr);
                    tc05::wait_ld();
                    tc05::fence_before_sync();
                    mbar_arrive(bar(S::B_SE + sbuf));
#pragma unroll
                    for (int r = 0; r < RG; ++r)
                        x[r] = (valid && rbase + r < M && (!kCausal || (r >= rmin && r < rmax)))
                                   ? __uint_as_float(sr[r]) * scale2
                                   : -INFINITY;
                } else {
#pragma unroll
                    for (int r = 0; r < RG; ++r) x[r] = -INFINITY;
                }
                int need = 0;
#pragma unroll
                for (int r = 0; r < RG; ++r) need |= x[r] > m_used[r] + kTcRescale;
                const int v = tc_vote(gvotes, gid, nvote, q4, lane, (got ? 0 : 2) | need);
                if (v & 2) {
                    raise_status(p, kErrTimeout);
                    abort = true;
                    break;
                }
                if (v & 1) {
                    // a row's maximum grew past the reference: new references from
                    // the tile's row maxima (lanes 2r and 2r+1 reduce row r), and O
                    // and l rescaled to them
                    float* rb = gred + (nvote & 1) * RG * 4;
                    const float y = tc_row_reduce16(x, lane, [](float a, float b2) { return fmaxf(a, b2); });
                    if ((lane & 1) == 0) rb[(lane >> 1) * 4 + q4] = y;
                    tc_group_sync(gid);
                    const int rl = lane & (RG - 1);
                    const float4 w = *reinterpret_cast<const float4*>(rb + rl * 4);
                    const float m_old = tc_pick16(m_used, rl);
                    const float m_new = fmaxf(m_old, fmaxf(fmaxf(w.x, w.y), fmaxf(w.z, w.w)));
                    const float a_lane = m_new == m_old ? 1.f : fast_exp2(m_old - m_new);
                    const bool grew = __any_sync(kFull, m_new > m_old);
#pragma unroll
                    for (int r = 0; r < RG; ++r) {
                        m_used[r] = __shfl_sync(kFull, m_new, r);
                        lp[r] *= __shfl_sync(kFull, a_lane, r);
                    }
                    if (grew && (cont || k > 0)) {
                        // O holds the run's earlier tiles: rescale once their P.V has
                        // completed (the previous tile's slot released)
                        if (tc_wait(bar(S::B_TE + (t - 1) % kTcNS), ((t - 1) / kTcNS) & 1, p, kWaitNs)) {
                            tc05::fence_after_sync();
                            uint32_t o[RG];
                            tc05::ld_32x32b_x16(tmem + lane_addr + 64 + 32 * ob + rbase, o);
                            tc05::wait_ld();
#pragma unroll
                            for (int r = 0; r < RG; ++r)
                                o[r] = __float_as_uint(__uint_as_float(o[r]) * __shfl_sync(kFull, a_lane, r));
                            tc05::st_32x32b_x16(tmem + lane_addr + 64 + 32 * ob + rbase, o);
                            tc05::wait_st();
                        } else {
                            abort = true;  // reported at the next vote
                        }
                    }
                }
                // P (rows past M and keys outside the chunk are 0), over the tile's K
                float pr[RG];
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    pr[r] = m_used[r] == -INFINITY ? 0.f : fast_exp2(x[r] - m_used[r]);
                    lp[r] += pr[r];
                }
                uint8_t* ptile = smem + S::OFF_KV + ts * S::TILE + (key >> 6) * 4 * S::GROUP;
                const int kc = (key & 63) >> 3, kb2 = (key & 7) * 2;
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    const int row = rbase + r;
                    const uint32_t h = pack2<kBF16>(pr[r], 0.f);
                    *reinterpret_cast<uint16_t*>(ptile + (row >> 3) * S::GROUP + (row & 7) * 128 +
                                                 (((kc ^ (row & 7)) << 4) | kb2)) = static_cast<uint16_t>(h & 0xffffu);
                }
                if (grp == 0 && __any_sync(kFull, !valid)) {
                    // keys outside the chunk (or on a skipped page) get P = 0; their V
                    // rows, stale or never loaded, are zeroed so that 0 * NaN cannot
                    // occur (each lane starts at its own chunk: no bank conflicts)
                    if (!tc_wait(bar(S::B_TF + ts), (t / kTcNS) & 1, p, kWaitNs)) abort = true;
                    if (!valid) {
                        uint8_t* vrow = smem + S::OFF_KV + ts * S::TILE + (key >> 3) * S::GROUP + 2048 + (key & 7) * 128;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int c = ((j + lane) & 7) * 16;
                            *reinterpret_cast<uint4*>(vrow + c) = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4*>(vrow + 1024 + c) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async();      // P and zeroed rows are read by the tensor cores
                tc05::fence_before_sync();
                mbar_arrive(bar(S::B_PF + ts));
            }
            if (tc_vote(gvotes, gid, nvote, q4, lane, abort ? 2 : 0) & 2) {
                raise_status(p, kErrTimeout);
                break;
            }
            bool free_ok = true;
            if (last) {
                // row statistics of the run for the epilogue: this warp's share of l, and m
                const float lw = tc_row_reduce16(lp, lane, [](float a, float b2) { return a + b2; });
                free_ok = ru < 3 || tc_wait(bar(S::B_XE + ob), (((ru - 1) >> 1) - 1) & 1, p, kWaitNs);
                float* st = stats + ob * 5 * kTcRows;
                if ((lane & 1) == 0) st[q4 * kTcRows + rbase + (lane >> 1)] = lw;
                if (q4 == 0 && lane < RG) st[4 * kTcRows + rbase + lane] = tc_pick16(m_used, lane);
                mbar_arrive(bar(S::B_XF + ob));
            }
            mbar_arrive(bar(S::B_IE + slot));
            if (!free_ok) {
                raise_status(p, kErrTimeout);  // the next vote stops the group
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        const int q4 = warp & 3, d = 32 * q4 + lane;  // TMEM lane of O^T: the head dim
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q4) << 16;
        int* evotes = votes + 16;
        int nvote = 0, er = 0;  // er: runs written
        for (int it = 0;; ++it) {
            const int slot = it % kTcNI, ob = er & 1;
            int fail = !tc_wait(bar(S::B_IF + slot), (it / kTcNI) & 1, p, kWaitNs);
            const TcItem& I = items[slot];
            const int end = fail ? 1 : I.end, last = end ? 0 : I.last;
            if (last) {
                fail |= !tc_wait(bar(S::B_XF + ob), (er >> 1) & 1, p, kWaitNs);
                fail |= !tc_wait(bar(S::B_OF + ob), (er >> 1) & 1, p, kWaitNs);
            }
            if (tc_vote(evotes, 2, nvote, q4, lane, (fail ? 2 : 0) | (end ? 1 : 0))) {
                if (fail) raise_status(p, kErrTimeout);
                break;
            }
            if (!last) {
                // the run goes on in the next item
                mbar_arrive(bar(S::B_IE + slot));
                continue;
            }
            ++er;
            const int b = I.b, hk = I.hk, pslot = I.slot, np = I.pieces;
            // O^T of the item (this thread's head dim, 32 rows); l and m per row
            // are read from the softmax's statistics as they are needed
            tc05::fence_after_sync();
            uint32_t o[32];
            tc05::ld_32x32b_x32(tmem + lane_addr + 64 + 32 * ob, o);
            tc05::wait_ld();
            tc05::fence_before_sync();
            mbar_arrive(bar(S::B_OE + ob));
            const float* st = stats + ob * 5 * kTcRows;
            auto lrow = [&](int r) { return (st[r] + st[kTcRows + r]) + (st[2 * kTcRows + r] + st[3 * kTcRows + r]); };
            const long long unit = static_cast<long long>(b) * Hkv + hk;
            const long long row0 = static_cast<long long>(b) * p.sq * p.Hq + hk * p.G;  // output row of query row 0
            auto out_row = [&](int r) { return row0 + static_cast<long long>(r / p.G) * p.Hq + r % p.G; };
            if (np == 1) {
                int i = 0, g = 0;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    if (r >= M) break;
                    const float l = lrow(r);
                    store_out(p.out, (row0 + static_cast<long long>(i) * p.Hq + g) * 128 + d,
                              l > 0.f ? __uint_as_float(o[r]) / l * p.v_scale : 0.f, p.out_dtype);
                    if (++g == p.G) {
                        g = 0;
                        ++i;
                    }
                }
                if (p.lse && d < M) {
                    const float l = lrow(d);
                    p.lse[out_row(d)] = l > 0.f ? (st[4 * kTcRows + d] + __log2f(l)) * kLn2 : -INFINITY;
                }
                mbar_arrive(bar(S::B_XE + ob));
            } else {
                // this run's partial (normalised O, LSE in log2 units); the CTA
                // that completes the unit's last piece merges them
                const long long slot2 = unit * p.max_splits + pslot;
                float* po = p.part_out + slot2 * kTcRows * 128;
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    if (r >= M) break;
                    const float l = lrow(r);
                    __stcg(po + r * 128 + d, l > 0.f ? __uint_as_float(o[r]) / l : 0.f);
                }
                if (d < M) {
                    const float l = lrow(d);
                    __stcg(p.part_lse + slot2 * kTcRows + d, l > 0.f ? st[4 * kTcRows + d] + __log2f(l) : -INFINITY);
                }
                mbar_arrive(bar(S::B_XE + ob));
                // publish the piece: the group's barrier, then one arrival with
                // release semantics at GPU scope (cumulative over the stores the
                // barrier ordered before it); the arrival that completes the unit
                // acquires the other pieces' partials for the whole group
                tc_group_sync(2);
                if (q4 == 0 && lane == 0) votes[24] = atom_add_acq_rel_gpu(p.counters + unit);
                tc_group_sync(2);
                if (votes[24] == np - 1) {
                    tc_merge_unit(p, unit, row0, np, q4, lane);
                    if (q4 == 0 && lane == 0) p.counters[unit] = 0;  // every piece has arrived: ready for the next call
                }
            }
            mbar_arrive(bar(S::B_IE + slot));
        }
    }

    // ---------------------------------------------------------- tear-down
    tc05::fence_before_sync();
    __syncthreads();
    if (warp == 13) {
        tc05::fence_after_sync();
        tc05::dealloc(tmem, 128);
    }
}

}  // namespace pkd
