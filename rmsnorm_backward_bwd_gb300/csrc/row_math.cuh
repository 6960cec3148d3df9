// Per-chunk arithmetic of the RMSNorm backward's two passes (FlyDSL issue
// #769, "Math": pass 1 sums x*dy*gamma over the row; pass 2 forms
// dx = (wdy - x_hat*c1)*rstd = wdy*rstd + x*b with b = -rstd^2*c1, adds
// dresidual_out for the fused-add variant of PR #800, and accumulates
// dy*x_hat for the weight gradient). Shared by the row engine and the
// cluster engine.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace rn {

// Per-chunk arithmetic of the two passes, by I/O dtype, on packed fp32
// pairs (one f32x2 instruction per two elements). For bf16/f16 the products
// x*dy and dy*gamma come exact from mixed-precision FMAs on the packed
// 16-bit halves, so the inputs are never unpacked for them.
template <typename T> struct RowMath;

template <> struct RowMath<float> {
    static constexpr int kPairs = 2;
    static constexpr bool kNeedsGammaF = true;  // the fp32 path always reads gamma as fp32
    // part2 + (x*dy)*g, pairwise
    static __device__ __forceinline__ f32x2 pass1(const uint4 &x, const uint4 &dy, const uint4 &,
                                                  const f32x2 *g2, f32x2 part2) {
        const f32x2 x0 = f2_make(__uint_as_float(x.x), __uint_as_float(x.y));
        const f32x2 x1 = f2_make(__uint_as_float(x.z), __uint_as_float(x.w));
        const f32x2 d0 = f2_make(__uint_as_float(dy.x), __uint_as_float(dy.y));
        const f32x2 d1 = f2_make(__uint_as_float(dy.z), __uint_as_float(dy.w));
        part2 = f2_fma(f2_mul(x0, d0), g2[0], part2);
        return f2_fma(f2_mul(x1, d1), g2[1], part2);
    }
    // dx = wdy*rs + x*b (rounded to the dtype); acc += (x*dy)*rs
    template <bool HAS_DRES>
    static __device__ __forceinline__ uint4 pass2(const uint4 &x, const uint4 &dy, const uint4 &r,
                                                  const uint4 &, const f32x2 *g2, f32x2 rs2,
                                                  f32x2 b2, f32x2 *acc2) {
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, dw[4] = {dy.x, dy.y, dy.z, dy.w};
        const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const f32x2 x2 = f2_make(__uint_as_float(xw[2 * q]), __uint_as_float(xw[2 * q + 1]));
            const f32x2 d2 = f2_make(__uint_as_float(dw[2 * q]), __uint_as_float(dw[2 * q + 1]));
            acc2[q] = f2_fma(f2_mul(x2, d2), rs2, acc2[q]);
            f32x2 v = f2_fma(x2, b2, f2_mul(f2_mul(d2, g2[q]), rs2));
            if (HAS_DRES)
                v = f2_add(v, f2_make(__uint_as_float(rw[2 * q]), __uint_as_float(rw[2 * q + 1])));
            float lo, hi;
            f2_split(v, lo, hi);
            o[2 * q] = __float_as_uint(lo);
            o[2 * q + 1] = __float_as_uint(hi);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};

template <typename T> struct RowMath16 {
    static constexpr int kPairs = 4;
    static constexpr bool kNeedsGammaF = false;
    static constexpr bool kBF = std::is_same<T, __nv_bfloat16>::value;
    static __device__ __forceinline__ f32x2 mul(uint32_t a, uint32_t b) {
        return kBF ? mul_bf16x2(a, b) : mul_f16x2(a, b);
    }
    static __device__ __forceinline__ f32x2 widen(uint32_t a) {
        return kBF ? widen_bf16x2(a) : widen_f16x2(a);
    }
    static __device__ __forceinline__ uint32_t pack(f32x2 v) {
        float lo, hi;
        f2_split(v, lo, hi);
        return kBF ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
    }
    // part2 + (x*dy)*g pairwise; without fp32 gamma (g2 == nullptr): x*(dy*gamma)
    static __device__ __forceinline__ f32x2 pass1(const uint4 &x, const uint4 &dy,
                                                  const uint4 &gp, const f32x2 *g2, f32x2 part2) {
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, dw[4] = {dy.x, dy.y, dy.z, dy.w};
        const uint32_t gw[4] = {gp.x, gp.y, gp.z, gp.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (g2) part2 = f2_fma(mul(xw[q], dw[q]), g2[q], part2);
            else part2 = f2_fma(widen(xw[q]), mul(dw[q], gw[q]), part2);
        }
        return part2;
    }
    template <bool HAS_DRES>
    static __device__ __forceinline__ uint4 pass2(const uint4 &x, const uint4 &dy, const uint4 &r,
                                                  const uint4 &gp, const f32x2 *, f32x2 rs2,
                                                  f32x2 b2, f32x2 *acc2) {
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, dw[4] = {dy.x, dy.y, dy.z, dy.w};
        const uint32_t gw[4] = {gp.x, gp.y, gp.z, gp.w}, rw[4] = {r.x, r.y, r.z, r.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            acc2[q] = f2_fma(mul(xw[q], dw[q]), rs2, acc2[q]);                 // += dy*x_hat
            f32x2 v = f2_fma(widen(xw[q]), b2, f2_mul(mul(dw[q], gw[q]), rs2)); // wdy*rs + x*b
            if (HAS_DRES) v = f2_add(v, widen(rw[q]));
            o[q] = pack(v);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};
template <> struct RowMath<__nv_bfloat16> : RowMath16<__nv_bfloat16> {};
template <> struct RowMath<__half> : RowMath16<__half> {};

}  // namespace rn
