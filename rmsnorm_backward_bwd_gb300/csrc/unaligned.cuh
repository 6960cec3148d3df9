// Helpers of the engines for rows that are not 16-byte multiples (the
// realigning engine, the vector generic kernels and the vector forward).
#pragma once

#include "common.cuh"

namespace rn {

// Bytes [sh, sh + 16) of the 32 bytes lo|hi (byte 0 = lowest byte of lo.x),
// sh in [0, 16). Callers pass an sh that is uniform across the CTA (a row's
// alignment phase): the switch does not diverge and every word index is a
// constant.
__device__ __forceinline__ uint4 shift_bytes(const uint4 &lo, const uint4 &hi, int sh) {
    const int b = (sh & 3) * 8;
    uint32_t a0, a1, a2, a3, a4;
    switch (sh >> 2) {
    case 0: a0 = lo.x; a1 = lo.y; a2 = lo.z; a3 = lo.w; a4 = hi.x; break;
    case 1: a0 = lo.y; a1 = lo.z; a2 = lo.w; a3 = hi.x; a4 = hi.y; break;
    case 2: a0 = lo.z; a1 = lo.w; a2 = hi.x; a3 = hi.y; a4 = hi.z; break;
    default: a0 = lo.w; a1 = hi.x; a2 = hi.y; a3 = hi.z; a4 = hi.w; break;
    }
    return make_uint4(__funnelshift_r(a0, a1, b), __funnelshift_r(a1, a2, b),
                      __funnelshift_r(a2, a3, b), __funnelshift_r(a3, a4, b));
}

// The 16 bytes of elements p[0 .. 16/sizeof(T)), loaded one element at a time
// (p need only be element-aligned), packed as one 16-byte chunk.
template <typename T>
__device__ __forceinline__ uint4 gather_chunk(const T *p) {
    union {
        T e[16 / sizeof(T)];
        uint4 v;
    } u;
#pragma unroll
    for (int k = 0; k < (int)(16 / sizeof(T)); ++k) u.e[k] = p[k];
    return u.v;
}

// The generic engines' per-column shared arrays are padded by one word per
// 32 columns: a warp's lanes touch columns 16/s apart, which without the pad
// share banks. vpad is column c's padded index; vec_words is the padded
// length of one array (a multiple of 4 words, so arrays stay 16-byte aligned).
__device__ __forceinline__ int vpad(int c) { return c + (c >> 5); }
inline size_t vec_words(int N) { return ((size_t)N + (size_t)(N >> 5) + 4) & ~(size_t)3; }

}  // namespace rn
