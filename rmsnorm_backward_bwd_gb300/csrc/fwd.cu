// Forward kernels: plain RMSNorm and fused-add (prenorm) RMSNorm, both
// storing the per-row fp32 rstd the backward consumes.
//
// rstd = 1/sqrt(mean_j x_j^2 + eps), y = x * rstd * gamma (FlyDSL issue #769,
// "Current state"; rstd is fp32 of shape (M,), PR #800 commit message
// "Makes RMSNorm training-capable"). Fused-add (PR #800, "What's included"):
// added = x + residual is rounded to the I/O dtype and stored as
// residual_out; the statistic and the output are taken from that rounded
// value, which is exactly the tensor the backward will read.
//
// This file holds the generic engine (unaligned rows, or rows longer than
// the row engine's tile): one CTA per row, scalar loads, two passes. Aligned
// rows take the forward row engine (fwd_row.cu).
#include "common.cuh"
#include "launch.h"

namespace rn {

struct FwdArgs {
    const uint8_t *x;
    const uint8_t *res;
    const uint8_t *gamma;
    uint8_t *y;
    uint8_t *res_out;
    float *rstd;
    int64_t M;
    int N;
    float inv_n;
    float eps;
};

template <typename T, bool FUSED>
__global__ void __launch_bounds__(256) fwd_generic_kernel(const FwdArgs a) {
    __shared__ float red[32];
    const T *x = reinterpret_cast<const T *>(a.x);
    const T *res = reinterpret_cast<const T *>(a.res);
    const T *g = reinterpret_cast<const T *>(a.gamma);
    T *y = reinterpret_cast<T *>(a.y);
    T *res_out = reinterpret_cast<T *>(a.res_out);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N;
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const size_t off = (size_t)row * N;
        float ss = 0.f;
        for (int j = tid; j < N; j += nthr) {
            float v = to_f(x[off + j]);
            if (FUSED) {
                v = round_through<T>(v + to_f(res[off + j]));
                res_out[off + j] = from_f<T>(v);
            }
            ss = fmaf(v, v, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int w = 0; w < nwarps; ++w) tot += red[w];
        __syncthreads();
        const float rs = rsqrtf(tot * a.inv_n + a.eps);
        if (tid == 0 && a.rstd) a.rstd[row] = rs;
        for (int j = tid; j < N; j += nthr) {
            // fused: read back this thread's own residual_out element
            const float v = FUSED ? to_f(res_out[off + j]) : to_f(x[off + j]);
            y[off + j] = from_f<T>(v * rs * to_f(g[j]));
        }
    }
}

template <typename T, bool FUSED>
static cudaError_t launch_fwd_t(const FwdArgs &a, int num_sms, cudaStream_t s) {
    int64_t grid = (int64_t)num_sms * 8;
    if (grid > a.M) grid = a.M;
    fwd_generic_kernel<T, FUSED><<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdProblem &p, int num_sms, cudaStream_t s) {
    FwdArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.res = static_cast<const uint8_t *>(p.residual);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.y = static_cast<uint8_t *>(p.y);
    a.res_out = static_cast<uint8_t *>(p.residual_out);
    a.rstd = p.rstd;
    a.M = p.M;
    a.N = p.N;
    a.inv_n = 1.0f / (float)p.N;
    a.eps = p.eps;
    const bool fused = p.residual != nullptr;
    switch (p.dtype) {
    case kF32:
        return fused ? launch_fwd_t<float, true>(a, num_sms, s)
                     : launch_fwd_t<float, false>(a, num_sms, s);
    case kF16:
        return fused ? launch_fwd_t<__half, true>(a, num_sms, s)
                     : launch_fwd_t<__half, false>(a, num_sms, s);
    case kBF16:
        return fused ? launch_fwd_t<__nv_bfloat16, true>(a, num_sms, s)
                     : launch_fwd_t<__nv_bfloat16, false>(a, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
