// Shared device helpers for the sm_103a RMSNorm kernels: I/O dtype traits,
// 16-byte chunk packing, warp reductions, and inline-PTX wrappers for async
// 16-byte copies, mixed-precision (bf16/f16 x bf16/f16 + fp32) arithmetic
// and programmatic dependent launch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rn {

// ---------------------------------------------------------------- dtypes
// A "chunk" is 16 bytes of one row: 4 f32 or 8 f16/bf16 elements, moved with
// one 128-bit load or store.
template <typename T> struct Traits;
template <> struct Traits<float> { static constexpr int kVec = 4; };
template <> struct Traits<__half> { static constexpr int kVec = 8; };
template <> struct Traits<__nv_bfloat16> { static constexpr int kVec = 8; };

template <typename T>
__device__ __forceinline__ void chunk_to_float(const uint4 &u, float *f);

template <>
__device__ __forceinline__ void chunk_to_float<float>(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}

__device__ __forceinline__ void bf16x2_to_float(uint32_t w, float &lo, float &hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}

template <>
__device__ __forceinline__ void chunk_to_float<__nv_bfloat16>(const uint4 &u, float *f) {
    bf16x2_to_float(u.x, f[0], f[1]);
    bf16x2_to_float(u.y, f[2], f[3]);
    bf16x2_to_float(u.z, f[4], f[5]);
    bf16x2_to_float(u.w, f[6], f[7]);
}

__device__ __forceinline__ void f16x2_to_float(uint32_t w, float &lo, float &hi) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    float2 v = __half22float2(h);
    lo = v.x;
    hi = v.y;
}

template <>
__device__ __forceinline__ void chunk_to_float<__half>(const uint4 &u, float *f) {
    f16x2_to_float(u.x, f[0], f[1]);
    f16x2_to_float(u.y, f[2], f[3]);
    f16x2_to_float(u.z, f[4], f[5]);
    f16x2_to_float(u.w, f[6], f[7]);
}

template <typename T>
__device__ __forceinline__ uint4 float_to_chunk(const float *f);

template <>
__device__ __forceinline__ uint4 float_to_chunk<float>(const float *f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t *>(&h);
}

template <>
__device__ __forceinline__ uint4 float_to_chunk<__nv_bfloat16>(const float *f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <>
__device__ __forceinline__ uint4 float_to_chunk<__half>(const float *f) {
    return make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                      pack_f16x2(f[6], f[7]));
}

// Scalar element access for the generic (unaligned) engine.
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Round an fp32 value to T and back (the value a T store would hold).
template <typename T> __device__ __forceinline__ float round_through(float v) {
    return to_f(from_f<T>(v));
}

// ------------------------------------------------------------ reductions
// xor butterfly: every lane ends with the same bits (fp add is commutative).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Named CTA barrier over `nthreads` threads (a multiple of 32). bar.sync is
// the aligned form: every thread of a warp must execute it together, and
// the PTX ISA leaves a diverged warp at an aligned barrier undefined. The
// compiler cannot see that this inline asm needs a converged warp: code
// such as `if (lane == 0) slot[w] = v;` just before it may be compiled as a
// branch and leave the warp diverged here. On GB300 that stops the kernel
// with "an illegal instruction was encountered". __syncwarp() is a
// convergence point the compiler honours, so the whole warp reaches the
// barrier together whatever the code before it compiled to.
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    __syncwarp();
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// -------------------------------------------------------------- 128-bit I/O
__device__ __forceinline__ uint4 ld_global_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Same, with an L2 eviction policy (createpolicy).
__device__ __forceinline__ uint4 ld_global_nc_v4_hint(const void *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ void st_global_v4(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------- async 16-byte copies
// One 16-byte asynchronous copy global -> shared through the load/store
// path (L1 bypassed), with an L2 eviction policy. Completion is tracked per
// thread with commit / wait groups: a thread that reads back only what it
// copied itself needs no other synchronisation.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
                 "l"(src), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Wait until at most `pending` of this thread's newest commit groups are
// still in flight (0 <= pending <= 7).
__device__ __forceinline__ void cp_async_wait_pending(int pending) {
    switch (pending) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------ mixed-precision arithmetic
// d_lo = a_lo*b_lo + c_lo and d_hi = a_hi*b_hi + c_hi on the two 16-bit
// halves of packed words, with an fp32 addend and result and one rounding
// (the product of two bf16 or two f16 values is exact in fp32).
__device__ __forceinline__ void fma2_bf16(uint32_t a, uint32_t b, float c0, float c1, float &d0,
                                          float &d1) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %4;\n\tfma.rn.f32.bf16 %1, ah, bh, %5;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(a), "r"(b), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void fma2_f16(uint32_t a, uint32_t b, float c0, float c1, float &d0,
                                         float &d1) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %4;\n\tfma.rn.f32.f16 %1, ah, bh, %5;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(a), "r"(b), "f"(c0), "f"(c1));
}

// d = a + c with a a 16-bit half of a packed word and c fp32 (one rounding).
__device__ __forceinline__ void add2_bf16(uint32_t a, float c0, float c1, float &d0, float &d1) {
    asm("{\n\t.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"
        "add.rn.f32.bf16 %0, al, %3;\n\tadd.rn.f32.bf16 %1, ah, %4;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(a), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void add2_f16(uint32_t a, float c0, float c1, float &d0, float &d1) {
    asm("{\n\t.reg .b16 al, ah;\n\tmov.b32 {al, ah}, %2;\n\t"
        "add.rn.f32.f16 %0, al, %3;\n\tadd.rn.f32.f16 %1, ah, %4;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(a), "f"(c0), "f"(c1));
}

// ------------------------------------------------------ packed fp32 pairs
// Two fp32 values in one 64-bit register pair; one f32x2 instruction does
// both lanes (each lane rounded exactly as the scalar fp32 operation).
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Exact products of the two 16-bit halves of packed words, as an fp32 pair
// (mixed-precision FMA with a zero addend; bf16*bf16 and f16*f16 products
// are exact in fp32).
__device__ __forceinline__ f32x2 mul_bf16x2(uint32_t a, uint32_t b) {
    f32x2 d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 lo, al, bl, 0f00000000;\n\t"
        "fma.rn.f32.bf16 hi, ah, bh, 0f00000000;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(d)
        : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ f32x2 mul_f16x2(uint32_t a, uint32_t b) {
    f32x2 d;
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 lo, hi;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 lo, al, bl, 0f00000000;\n\t"
        "fma.rn.f32.f16 hi, ah, bh, 0f00000000;\n\t"
        "mov.b64 %0, {lo, hi};\n\t}"
        : "=l"(d)
        : "r"(a), "r"(b));
    return d;
}
// The two 16-bit halves of a packed word, widened to an fp32 pair.
__device__ __forceinline__ f32x2 widen_bf16x2(uint32_t w) {
    return f2_make(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ f32x2 widen_f16x2(uint32_t w) {
    float lo, hi;
    f16x2_to_float(w, lo, hi);
    return f2_make(lo, hi);
}

// ------------------------------------------- programmatic dependent launch
// Block until every grid this one depends on programmatically has completed
// and its memory is visible (no-op when launched without such a dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the dependent grid (if any) to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Workspace: the partial rows start after a 256-byte header (kept free so
// that the partials stay 256-byte aligned).
constexpr size_t kWsHeaderBytes = 256;

}  // namespace rn
