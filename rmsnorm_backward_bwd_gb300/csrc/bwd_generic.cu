// Backward generic engine: any N, any element alignment (the rows that the
// bulk-copy row engine cannot take: N*elem_bytes not a multiple of 16, a base
// pointer not 16-byte aligned, or a row longer than its tile).
//
// Same math as the row engine (FlyDSL issue #769 "Math"; fused-add from
// PR #800 "What's included"). One CTA owns one row at a time (persistent,
// grid-stride over rows). Pass 1 reduces sum_j x_j*dy_j*gamma_j with scalar
// loads; pass 2 re-reads the row (now an L2 hit), writes dx and adds dy*x_hat
// into the CTA's weight-gradient partial. Column j always belongs to thread
// j % blockDim.x, so the partial needs no atomics: it lives in shared memory
// when N fp32 values fit there, otherwise in the CTA's workspace row.
#include "common.cuh"
#include "launch.h"

namespace rn {

size_t generic_smem_bytes(int N, bool smem_dw) {
    return 256 + (smem_dw ? (size_t)N * 4 : 0);
}

struct GenArgs {
    const void *x;
    const void *gamma;
    const void *dy;
    const float *rstd;
    const void *dres;
    void *dx;
    float *dw_out;   // scratch: partial rows [gridDim.x][N]; atomic: dweight_f32
    int64_t M;
    int N;
    float inv_n;
};

template <typename T, bool HAS_DRES, bool ATOMIC, bool SMEM_DW>
__global__ void __launch_bounds__(512) bwd_generic_kernel(const GenArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);          // 32 warp sums + total
    float *sdw = reinterpret_cast<float *>(smem + 256);    // N floats when SMEM_DW
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N;
    float *part = ATOMIC ? nullptr : a.dw_out + (size_t)blockIdx.x * N;
    float *dw = SMEM_DW ? sdw : part;  // !SMEM_DW implies scratch mode

    for (int j = tid; j < N; j += nthr) dw[j] = 0.f;

    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const float rs = __ldg(a.rstd + row);
        const T *xr = x + (size_t)row * N;
        const T *dyr = dy + (size_t)row * N;
        float s = 0.f;
        for (int j = tid; j < N; j += nthr) s = fmaf(to_f(xr[j]), to_f(dyr[j]) * to_f(g[j]), s);
        s = warp_sum(s);
        if (lane == 0) red[warp] = s;
        __syncthreads();
        float tot = 0.f;
        for (int w = 0; w < nwarps; ++w) tot += red[w];
        __syncthreads();  // red is rewritten by the next row
        const float c1 = rs * tot * a.inv_n;
        T *dxr = dx + (size_t)row * N;
        const T *rr = HAS_DRES ? dres + (size_t)row * N : nullptr;
        for (int j = tid; j < N; j += nthr) {
            const float xv = to_f(xr[j]), dv = to_f(dyr[j]);
            const float xh = xv * rs;
            float d = fmaf(-xh, c1, dv * to_f(g[j])) * rs;
            if (HAS_DRES) d += to_f(rr[j]);
            dxr[j] = from_f<T>(d);
            dw[j] = fmaf(dv, xh, dw[j]);
        }
    }
    pdl_launch_dependents();
    if (SMEM_DW || ATOMIC) {
        if (ATOMIC) {
            pdl_wait();
            for (int j = tid; j < N; j += nthr) atomicAdd(a.dw_out + j, dw[j]);
        } else {
            for (int j = tid; j < N; j += nthr) part[j] = dw[j];
        }
    }
}

template <typename T, bool HAS_DRES, bool ATOMIC, bool SMEM_DW>
static cudaError_t launch_gen_t(const GenArgs &args, const GenericPlan &plan, cudaStream_t s,
                                bool pdl) {
    auto kern = bwd_generic_kernel<T, HAS_DRES, ATOMIC, SMEM_DW>;
    cudaError_t e = ensure_smem_attr((const void *)kern, plan.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.threads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

template <typename T>
static cudaError_t launch_gen_dt(const GenArgs &args, const GenericPlan &plan, bool has_dres,
                                 cudaStream_t s, bool pdl) {
    if (plan.atomic) {
        // atomic mode always keeps the partial in shared memory
        return has_dres ? launch_gen_t<T, true, true, true>(args, plan, s, pdl)
                        : launch_gen_t<T, false, true, true>(args, plan, s, pdl);
    }
    if (plan.smem_dw)
        return has_dres ? launch_gen_t<T, true, false, true>(args, plan, s, pdl)
                        : launch_gen_t<T, false, false, true>(args, plan, s, pdl);
    return has_dres ? launch_gen_t<T, true, false, false>(args, plan, s, pdl)
                    : launch_gen_t<T, false, false, false>(args, plan, s, pdl);
}

cudaError_t launch_bwd_generic(const BwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                               bool pdl_after_zero) {
    GenArgs a;
    a.x = p.x;
    a.gamma = p.gamma;
    a.dy = p.dy;
    a.rstd = p.rstd;
    a.dres = p.dres;
    a.dx = p.dx;
    a.dw_out = plan.atomic ? p.dw_f32 : reinterpret_cast<float *>(p.ws + kWsHeaderBytes);
    a.M = p.M;
    a.N = p.N;
    a.inv_n = 1.0f / (float)p.N;
    const bool has_dres = p.dres != nullptr;
    switch (p.dtype) {
    case kF32: return launch_gen_dt<float>(a, plan, has_dres, s, pdl_after_zero);
    case kF16: return launch_gen_dt<__half>(a, plan, has_dres, s, pdl_after_zero);
    case kBF16: return launch_gen_dt<__nv_bfloat16>(a, plan, has_dres, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
