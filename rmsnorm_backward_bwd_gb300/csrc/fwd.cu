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
// Vector engine: a team of threads per row, 16-byte chunks, rows striding
// over a grid sized to fill the GPU; sum of squares reduced with warp
// shuffles and a named barrier across the team. Generic engine (unaligned
// rows): one CTA per row, scalar loads, two passes.
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
    int nchunks;
    int row_bytes;
    int team_threads;
    int teams;
    float inv_n;
    float eps;
};

template <typename T, int CPT, bool FUSED>
__global__ void __launch_bounds__(512) fwd_vec_kernel(const FwdArgs a) {
    constexpr int V = Traits<T>::kVec;
    __shared__ float red[2][32];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int team = tid / a.team_threads;
    const int tt = tid - team * a.team_threads;
    const int team_warps = a.team_threads >> 5;
    const int first_warp = team * team_warps;

    uint4 g[CPT];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        const int c = tt + kk * a.team_threads;
        g[kk] = c < a.nchunks ? ld_global_nc_v4(a.gamma + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
    }
    const int64_t stride = (int64_t)gridDim.x * a.teams;
    int parity = 0;
    for (int64_t row = (int64_t)blockIdx.x * a.teams + team; row < a.M; row += stride) {
        const size_t off = (size_t)row * a.row_bytes;
        float v[CPT][V];
        float ss = 0.f;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = tt + kk * a.team_threads;
            if (c < a.nchunks) {
                chunk_to_float<T>(ld_global_nc_v4(a.x + off + 16u * c), v[kk]);
                if (FUSED) {
                    float r[V];
                    chunk_to_float<T>(ld_global_nc_v4(a.res + off + 16u * c), r);
#pragma unroll
                    for (int e = 0; e < V; ++e) v[kk][e] = v[kk][e] + r[e];
                    const uint4 packed = float_to_chunk<T>(v[kk]);
                    st_global_v4(a.res_out + off + 16u * c, packed);
                    chunk_to_float<T>(packed, v[kk]);  // continue from the stored value
                }
#pragma unroll
                for (int e = 0; e < V; ++e) ss = fmaf(v[kk][e], v[kk][e], ss);
            }
        }
        ss = warp_sum(ss);
        if (team_warps > 1) {
            if (lane == 0) red[parity][warp] = ss;
            named_barrier_sync(1 + team, a.team_threads);
            float tot = 0.f;
            for (int w = 0; w < team_warps; ++w) tot += red[parity][first_warp + w];
            ss = tot;
            parity ^= 1;
        }
        const float rs = rsqrtf(ss * a.inv_n + a.eps);
        if (tt == 0 && a.rstd) a.rstd[row] = rs;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = tt + kk * a.team_threads;
            if (c < a.nchunks) {
                float gf[V], o[V];
                chunk_to_float<T>(g[kk], gf);
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = v[kk][e] * rs * gf[e];
                st_global_v4(a.y + off + 16u * c, float_to_chunk<T>(o));
            }
        }
    }
}

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
static cudaError_t launch_fwd_t(const FwdArgs &a0, bool vector_ok, int num_sms, cudaStream_t s) {
    FwdArgs a = a0;
    if (vector_ok) {
        // team shape: about 256 threads per row, up to 4 chunks per thread
        int team = (a.nchunks + 1) / 2;
        team = ((team + 31) / 32) * 32;
        if (team > 256) team = 256;
        int cpt = (a.nchunks + team - 1) / team;
        cpt = cpt <= 1 ? 1 : (cpt <= 2 ? 2 : 4);
        if (cpt == 4) team = (((a.nchunks + 3) / 4 + 31) / 32) * 32;
        if (team <= 512) {
            a.team_threads = team;
            a.teams = 512 / team;
            if (a.teams > 15) a.teams = 15;
            const void *fn = nullptr;
            if (cpt == 1) fn = (const void *)fwd_vec_kernel<T, 1, FUSED>;
            else if (cpt == 2) fn = (const void *)fwd_vec_kernel<T, 2, FUSED>;
            else fn = (const void *)fwd_vec_kernel<T, 4, FUSED>;
            int per_sm = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, fn, a.teams * a.team_threads, 0);
            if (e != cudaSuccess) return e;
            if (per_sm < 1) per_sm = 1;
            int64_t need = (a.M + a.teams - 1) / a.teams;
            int64_t grid = (int64_t)num_sms * per_sm;
            if (grid > need) grid = need;
            dim3 block(a.teams * a.team_threads);
            if (cpt == 1) fwd_vec_kernel<T, 1, FUSED><<<(unsigned)grid, block, 0, s>>>(a);
            else if (cpt == 2) fwd_vec_kernel<T, 2, FUSED><<<(unsigned)grid, block, 0, s>>>(a);
            else fwd_vec_kernel<T, 4, FUSED><<<(unsigned)grid, block, 0, s>>>(a);
            return cudaGetLastError();
        }
    }
    int64_t grid = (int64_t)num_sms * 8;
    if (grid > a.M) grid = a.M;
    fwd_generic_kernel<T, FUSED><<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdProblem &p, bool vector_ok, int num_sms, cudaStream_t s) {
    FwdArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.res = static_cast<const uint8_t *>(p.residual);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.y = static_cast<uint8_t *>(p.y);
    a.res_out = static_cast<uint8_t *>(p.residual_out);
    a.rstd = p.rstd;
    a.M = p.M;
    a.N = p.N;
    a.row_bytes = p.N * elem_bytes(p.dtype);
    a.nchunks = a.row_bytes / 16;
    a.team_threads = 0;
    a.teams = 0;
    a.inv_n = 1.0f / (float)p.N;
    a.eps = p.eps;
    const bool fused = p.residual != nullptr;
    switch (p.dtype) {
    case kF32:
        return fused ? launch_fwd_t<float, true>(a, vector_ok, num_sms, s)
                     : launch_fwd_t<float, false>(a, vector_ok, num_sms, s);
    case kF16:
        return fused ? launch_fwd_t<__half, true>(a, vector_ok, num_sms, s)
                     : launch_fwd_t<__half, false>(a, vector_ok, num_sms, s);
    case kBF16:
        return fused ? launch_fwd_t<__nv_bfloat16, true>(a, vector_ok, num_sms, s)
                     : launch_fwd_t<__nv_bfloat16, false>(a, vector_ok, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
