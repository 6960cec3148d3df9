// Shared device helpers for the sm_103a RMSNorm kernels: I/O dtype traits,
// 16-byte chunk packing, warp reductions, and inline-PTX wrappers for
// mbarriers, bulk async copies (global -> shared) and programmatic dependent
// launch.
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

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
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

// ------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of an mbarrier to complete, giving up after
// `limit_cycles` SM clock cycles. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  long long limit_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit_cycles) return false;
    }
}

// One bulk asynchronous copy global -> this CTA's shared memory; completion
// is signalled as transaction bytes on `bar`. dst, src 16-byte aligned;
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------- programmatic dependent launch
// Block until every grid this one depends on programmatically has completed
// and its memory is visible (no-op when launched without such a dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the dependent grid (if any) to begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ~1 s at GB300 clocks: the limit on any device-side wait.
constexpr long long kWaitLimitCycles = 2000000000LL;

// Workspace header: status word at byte 0; partials start at byte 256.
constexpr size_t kWsHeaderBytes = 256;

}  // namespace rn
