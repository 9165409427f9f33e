// Page column of a key index without a division.
//
// Every stage the kernels stream needs tok / P and tok % P for a page size P
// known only at run time.  An integer division there cost 2-10 % of the
// decode time, so the host computes, once per call, a magic number m and a
// shift s with tok / P == (tok * m) >> s for every 0 <= tok < 2^31
// (division by an invariant integer, Granlund and Montgomery): with
// l = ceil(log2 P), m = floor(2^(31+l) / P) + 1 (2^31 when P is a power of
// two) and s = 31 + l.  The product fits 64 bits since m < 2^32.
// Plain C++ so that host tests can check it exhaustively without a GPU.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define PKD_HOST_DEVICE __host__ __device__ __forceinline__
#else
#define PKD_HOST_DEVICE inline
#endif

namespace pkd {

// Magic number and shift for division by P (1 <= P < 2^31).
inline void page_magic(int P, uint32_t& magic, int& shift) {
    int l = 0;
    while ((1LL << l) < P) ++l;
    const bool pow2 = (P & (P - 1)) == 0;
    magic = pow2 ? 0x80000000u : (uint32_t)(((uint64_t)1 << (31 + l)) / (uint64_t)P + 1);
    shift = 31 + l;
}

// tok / P for 0 <= tok < 2^31, from page_magic's (magic, shift).
PKD_HOST_DEVICE int page_div(int tok, uint32_t magic, int shift) {
    return (int)(((uint64_t)(uint32_t)tok * magic) >> shift);
}

}  // namespace pkd
