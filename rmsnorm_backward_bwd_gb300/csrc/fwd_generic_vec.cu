// Forwards for rows that are not 16-byte multiples (RMSNorm, fused-add
// RMSNorm, LayerNorm), when the row tensors (x, y; residual and
// residual_out) share one alignment phase and gamma (beta) start on a
// 16-byte boundary.
//
// What is computed is the forward row engine's (FlyDSL issue #769,
// "Current state"; PR #800 "What's included" for the fused-add variant, whose
// statistic and output are taken from the dtype-rounded residual_out; issue
// #769's LayerNorm plan, mean then centred variance). The data path differs:
// one CTA per row at a time (persistent, many CTAs per SM); each row splits
// into a head (the elements before its first 16-byte boundary), whole
// 16-byte chunks moved with 128-bit loads and stores, and a tail; later
// passes re-read the row through L1. A chunk's gamma (beta) columns start at
// the row's phase, so they come from two aligned 16-byte loads and a funnel
// shift (element by element for a window at the end of the vector).
#include "common.cuh"
#include "unaligned.cuh"
#include "launch.h"

namespace rn {

namespace {

struct FwdVecArgs {
    const uint8_t *x;
    const uint8_t *res;     // fused-add
    const uint8_t *gamma;
    const uint8_t *beta;    // LayerNorm, nullable
    uint8_t *y;
    uint8_t *res_out;       // fused-add
    float *mean;            // LayerNorm, nullable
    float *rstd;            // nullable
    int64_t M;
    int N;
    float inv_n;
    float eps;
};

// 16 read-only bytes through L1 (later passes re-read the row there).
__device__ __forceinline__ uint4 ld_ro_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The V values of a 1-D parameter vector (16-byte aligned, nbytes long) at
// byte offsets [start, start + 16), as floats.
template <typename T>
__device__ __forceinline__ void param_window(const uint8_t *p, int start, int nbytes, float *f) {
    constexpr int V = 16 / (int)sizeof(T);
    const int al = start & ~15, sh = start & 15;
    if (sh == 0) {
        chunk_to_float<T>(ld_ro_v4(p + al), f);
    } else if (al + 32 <= nbytes) {
        chunk_to_float<T>(shift_bytes(ld_ro_v4(p + al), ld_ro_v4(p + al + 16), sh), f);
    } else {
        // the window nearest the end: no read past the vector
        const T *e = reinterpret_cast<const T *>(p + start);
#pragma unroll
        for (int k = 0; k < V; ++k) f[k] = to_f(e[k]);
    }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(256) fwd_generic_vec_kernel(const FwdVecArgs a) {
    constexpr int S = sizeof(T), V = 16 / S;
    __shared__ float red[32];
    const T *x = reinterpret_cast<const T *>(a.x);
    const T *res = reinterpret_cast<const T *>(a.res);
    const T *g = reinterpret_cast<const T *>(a.gamma);
    const T *bt = reinterpret_cast<const T *>(a.beta);
    T *y = reinterpret_cast<T *>(a.y);
    T *ro = reinterpret_cast<T *>(a.res_out);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N, nbytes = N * S;
    auto block_sum = [&](float v) {
        v = warp_sum(v);
        if (lane == 0) red[warp] = v;
        __syncthreads();
        float t = 0.f;
        for (int w = 0; w < nwarps; ++w) t += red[w];
        __syncthreads();  // red is rewritten by the next sum
        return t;
    };
    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const size_t base = (size_t)row * N;
        const uintptr_t ad = reinterpret_cast<uintptr_t>(x + base);
        int h = (int)(((16u - (unsigned)(ad & 15u)) & 15u) / S);
        if (h > N) h = N;
        const int nv = (N - h) / V, nt = N - h - nv * V;
        // this thread's head or tail element (threads below h + nt)
        const bool has_e = tid < h + nt;
        const int je = tid < h ? tid : h + nv * V + (tid - h);

        // pass 1: sum (LayerNorm) or sum of squares; fused-add stores
        // residual_out = round(x + residual) first and sums its squares
        float s = 0.f;
        for (int i = tid; i < nv; i += nthr) {
            const size_t e0 = base + h + (size_t)i * V;
            float v[V];
            chunk_to_float<T>(ld_ro_v4(x + e0), v);
            if (MODE == kFwdFused) {
                float r[V];
                chunk_to_float<T>(ld_ro_v4(res + e0), r);
#pragma unroll
                for (int e = 0; e < V; ++e) v[e] += r[e];
                const uint4 o = float_to_chunk<T>(v);
                st_global_v4(ro + e0, o);
                chunk_to_float<T>(o, v);
            }
#pragma unroll
            for (int e = 0; e < V; ++e) s = MODE == kFwdLn ? s + v[e] : fmaf(v[e], v[e], s);
        }
        float xe = 0.f;
        if (has_e) {
            xe = to_f(x[base + je]);
            if (MODE == kFwdFused) {
                xe = round_through<T>(xe + to_f(res[base + je]));
                ro[base + je] = from_f<T>(xe);
            }
            s = MODE == kFwdLn ? s + xe : fmaf(xe, xe, s);
        }
        float mu = 0.f, rs;
        if (MODE == kFwdLn) {
            mu = block_sum(s) * a.inv_n;
            // pass 2: centred sum of squares (no cancellation)
            float q = 0.f;
            for (int i = tid; i < nv; i += nthr) {
                float v[V];
                chunk_to_float<T>(ld_ro_v4(x + base + h + (size_t)i * V), v);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float d = v[e] - mu;
                    q = fmaf(d, d, q);
                }
            }
            if (has_e) q = fmaf(xe - mu, xe - mu, q);
            rs = rsqrtf(block_sum(q) * a.inv_n + a.eps);
        } else {
            rs = rsqrtf(block_sum(s) * a.inv_n + a.eps);
        }
        if (tid == 0) {
            if (MODE == kFwdLn && a.mean) a.mean[row] = mu;
            if (a.rstd) a.rstd[row] = rs;
        }
        // output pass (fused-add re-reads its own residual_out stores)
        for (int i = tid; i < nv; i += nthr) {
            const size_t e0 = base + h + (size_t)i * V;
            float v[V], gf[V], o[V];
            if (MODE == kFwdFused) chunk_to_float<T>(*reinterpret_cast<const uint4 *>(ro + e0), v);
            else chunk_to_float<T>(ld_ro_v4(x + e0), v);
            const int cb = (h + i * V) * S;  // the chunk's first column, in bytes
            param_window<T>(a.gamma, cb, nbytes, gf);
            if (MODE == kFwdLn) {
                float bf[V];
                if (bt) param_window<T>(a.beta, cb, nbytes, bf);
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = fmaf((v[e] - mu) * rs, gf[e], bt ? bf[e] : 0.f);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = v[e] * rs * gf[e];
            }
            st_global_v4(y + e0, float_to_chunk<T>(o));
        }
        if (has_e) {
            const float ge = to_f(g[je]);
            y[base + je] = from_f<T>(MODE == kFwdLn ? fmaf((xe - mu) * rs, ge, bt ? to_f(bt[je]) : 0.f)
                                                    : xe * rs * ge);
        }
    }
}

template <typename T, int MODE>
cudaError_t launch_t(const FwdVecArgs &a, int num_sms, cudaStream_t s) {
    int64_t grid = (int64_t)num_sms * 8;
    if (grid > a.M) grid = a.M;
    fwd_generic_vec_kernel<T, MODE><<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const FwdVecArgs &a, int dtype, int num_sms, cudaStream_t s) {
    switch (dtype) {
    case kF32: return launch_t<float, MODE>(a, num_sms, s);
    case kF16: return launch_t<__half, MODE>(a, num_sms, s);
    case kBF16: return launch_t<__nv_bfloat16, MODE>(a, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool fwd_generic_vec_ok(const FwdRowProblem &p) {
    const uintptr_t S = (uintptr_t)elem_bytes(p.dtype);
    const uintptr_t ph = (uintptr_t)p.x & 15u;
    for (const void *q : {p.x, static_cast<const void *>(p.y), p.residual,
                          static_cast<const void *>(p.residual_out)}) {
        if (q == nullptr) continue;
        if (((uintptr_t)q & 15u) != ph || ((uintptr_t)q % S) != 0) return false;
    }
    return ((uintptr_t)p.gamma & 15u) == 0 && (p.beta == nullptr || ((uintptr_t)p.beta & 15u) == 0);
}

cudaError_t launch_fwd_generic_vec(const FwdRowProblem &p, int num_sms, cudaStream_t s) {
    FwdVecArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.res = static_cast<const uint8_t *>(p.residual);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.beta = static_cast<const uint8_t *>(p.beta);
    a.y = static_cast<uint8_t *>(p.y);
    a.res_out = static_cast<uint8_t *>(p.residual_out);
    a.mean = p.mean;
    a.rstd = p.rstd;
    a.M = p.M;
    a.N = p.N;
    a.inv_n = 1.0f / (float)p.N;
    a.eps = p.eps;
    switch (p.mode) {
    case kFwdRms: return launch_mode<kFwdRms>(a, p.dtype, num_sms, s);
    case kFwdFused: return launch_mode<kFwdFused>(a, p.dtype, num_sms, s);
    case kFwdLn: return launch_mode<kFwdLn>(a, p.dtype, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
