// Packed-pair arithmetic of the LayerNorm backward (FlyDSL issue #769,
// LayerNorm backward plan: x_hat = (x - mean)*rstd, wdy = dy*gamma): chunks of
// the I/O dtype widened to fp32 pairs, dy*gamma as exact products of the
// packed 16-bit halves, x - mean by one mixed-precision FMA per element, and
// fp32 pairs rounded back to a chunk. Shared by the LayerNorm row engine and
// the LayerNorm staged phase-class kernel.
#pragma once

#include "common.cuh"

namespace rn {

// A 16-byte chunk as fp32 pairs.
template <typename T> __device__ __forceinline__ void chunk_pairs(const uint4 &u, f32x2 *p);
template <> __device__ __forceinline__ void chunk_pairs<float>(const uint4 &u, f32x2 *p) {
    p[0] = f2_make(__uint_as_float(u.x), __uint_as_float(u.y));
    p[1] = f2_make(__uint_as_float(u.z), __uint_as_float(u.w));
}
template <> __device__ __forceinline__ void chunk_pairs<__nv_bfloat16>(const uint4 &u, f32x2 *p) {
    p[0] = widen_bf16x2(u.x);
    p[1] = widen_bf16x2(u.y);
    p[2] = widen_bf16x2(u.z);
    p[3] = widen_bf16x2(u.w);
}
template <> __device__ __forceinline__ void chunk_pairs<__half>(const uint4 &u, f32x2 *p) {
    p[0] = widen_f16x2(u.x);
    p[1] = widen_f16x2(u.y);
    p[2] = widen_f16x2(u.z);
    p[3] = widen_f16x2(u.w);
}

// dy*gamma for a chunk, as fp32 pairs: for 16-bit types the exact products of
// the packed halves (one mixed-precision FMA per element, no unpacking).
template <typename T>
__device__ __forceinline__ void mul_chunk_pairs(const uint4 &d, const uint4 &g, f32x2 *p);
template <>
__device__ __forceinline__ void mul_chunk_pairs<__nv_bfloat16>(const uint4 &d, const uint4 &g,
                                                               f32x2 *p) {
    p[0] = mul_bf16x2(d.x, g.x);
    p[1] = mul_bf16x2(d.y, g.y);
    p[2] = mul_bf16x2(d.z, g.z);
    p[3] = mul_bf16x2(d.w, g.w);
}
template <>
__device__ __forceinline__ void mul_chunk_pairs<__half>(const uint4 &d, const uint4 &g, f32x2 *p) {
    p[0] = mul_f16x2(d.x, g.x);
    p[1] = mul_f16x2(d.y, g.y);
    p[2] = mul_f16x2(d.z, g.z);
    p[3] = mul_f16x2(d.w, g.w);
}

// x - mean for a chunk, as fp32 pairs: for 16-bit types one mixed-precision
// FMA per element, x*1 + (-mean), rounded once -- the same value as widening
// x and subtracting in fp32, without the unpacking.
template <typename T>
__device__ __forceinline__ void centre_chunk_pairs(const uint4 &x, f32x2 nmu2, float nmu, f32x2 *p);
template <>
__device__ __forceinline__ void centre_chunk_pairs<float>(const uint4 &x, f32x2 nmu2, float,
                                                          f32x2 *p) {
    chunk_pairs<float>(x, p);
    p[0] = f2_add(p[0], nmu2);
    p[1] = f2_add(p[1], nmu2);
}
__device__ __forceinline__ f32x2 centre_bf16x2(uint32_t w, float c) {
    f32x2 d;
    asm("{\n\t.reg .b16 xl, xh, one;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b32 {xl, xh}, %1;\n\tmov.b16 one, 0x3F80;\n\t"
        "fma.rn.f32.bf16 lo, xl, one, %2;\n\t"
        "fma.rn.f32.bf16 hi, xh, one, %2;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(d)
        : "r"(w), "f"(c));
    return d;
}
__device__ __forceinline__ f32x2 centre_f16x2(uint32_t w, float c) {
    f32x2 d;
    asm("{\n\t.reg .b16 xl, xh, one;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b32 {xl, xh}, %1;\n\tmov.b16 one, 0x3C00;\n\t"
        "fma.rn.f32.f16 lo, xl, one, %2;\n\t"
        "fma.rn.f32.f16 hi, xh, one, %2;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(d)
        : "r"(w), "f"(c));
    return d;
}
template <>
__device__ __forceinline__ void centre_chunk_pairs<__nv_bfloat16>(const uint4 &x, f32x2,
                                                                  float nmu, f32x2 *p) {
    p[0] = centre_bf16x2(x.x, nmu);
    p[1] = centre_bf16x2(x.y, nmu);
    p[2] = centre_bf16x2(x.z, nmu);
    p[3] = centre_bf16x2(x.w, nmu);
}
template <>
__device__ __forceinline__ void centre_chunk_pairs<__half>(const uint4 &x, f32x2, float nmu,
                                                           f32x2 *p) {
    p[0] = centre_f16x2(x.x, nmu);
    p[1] = centre_f16x2(x.y, nmu);
    p[2] = centre_f16x2(x.z, nmu);
    p[3] = centre_f16x2(x.w, nmu);
}

// fp32 pairs back to a 16-byte chunk of T (round to nearest even).
template <typename T> __device__ __forceinline__ uint4 pairs_chunk(const f32x2 *p);
template <> __device__ __forceinline__ uint4 pairs_chunk<float>(const f32x2 *p) {
    float a, b, c, d;
    f2_split(p[0], a, b);
    f2_split(p[1], c, d);
    return make_uint4(__float_as_uint(a), __float_as_uint(b), __float_as_uint(c),
                      __float_as_uint(d));
}
template <> __device__ __forceinline__ uint4 pairs_chunk<__nv_bfloat16>(const f32x2 *p) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float lo, hi;
        f2_split(p[q], lo, hi);
        w[q] = pack_bf16x2(lo, hi);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
template <> __device__ __forceinline__ uint4 pairs_chunk<__half>(const f32x2 *p) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float lo, hi;
        f2_split(p[q], lo, hi);
        w[q] = pack_f16x2(lo, hi);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace rn
