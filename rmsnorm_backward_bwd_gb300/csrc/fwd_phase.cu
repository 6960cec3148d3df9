// Forwards for rows that are not 16-byte multiples (RMSNorm, fused-add
// RMSNorm, LayerNorm), the row tensors (x, y; residual and residual_out) at
// one alignment phase, rows of at most 1024 whole 16-byte chunks.
//
// What is computed is the forward row engine's (FlyDSL issue #769, "Current
// state"; PR #800 "What's included": the fused-add statistic and output come
// from the dtype-rounded residual_out; issue #769's LayerNorm plan: mean,
// then the centred variance). The work split is the backward phase-class
// kernel's: row r starts r*N*s bytes past the base, so its alignment phase
// repeats with period P = 16 / gcd(16, N*s mod 16) rows; each CTA takes the
// rows of one residue class modulo P, where every row splits the same way
// into head elements, whole 16-byte chunks and tail elements. A thread so
// owns the same columns in every row: gamma (and beta) stay in registers as
// fp32 pairs, and the rows stay in registers between the passes (the
// LayerNorm variance is taken from them, not re-read). A CTA takes two rows
// of its class per iteration under one CTA barrier per row sum, and loads the
// next two while it computes these.
#include "common.cuh"
#include "launch.h"
#include "unaligned.cuh"

namespace rn {

namespace {

struct FwdPhaseArgs {
    const uint8_t *x;
    const uint8_t *res;     // fused-add
    const uint8_t *gamma;   // any element alignment
    const uint8_t *beta;    // LayerNorm, nullable
    uint8_t *y;
    uint8_t *res_out;       // fused-add
    float *mean;            // LayerNorm, nullable
    float *rstd;            // nullable
    int64_t M;
    int N;
    float inv_n;
    float eps;
    int period;             // P
};

// The chunk's V elements as fp32 pairs.
template <typename T, int V>
__device__ __forceinline__ void chunk_pairs2(const uint4 &u, f32x2 *p) {
    float f[V];
    chunk_to_float<T>(u, f);
#pragma unroll
    for (int q = 0; q < V / 2; ++q) p[q] = f2_make(f[2 * q], f[2 * q + 1]);
}

template <typename T, int V>
__device__ __forceinline__ uint4 pairs_to_chunk(const f32x2 *p) {
    float f[V];
#pragma unroll
    for (int q = 0; q < V / 2; ++q) f2_split(p[q], f[2 * q], f[2 * q + 1]);
    return float_to_chunk<T>(f);
}

template <typename T, int MODE, int J, int R>
__global__ void __launch_bounds__(512) fwd_phase_kernel(const FwdPhaseArgs a) {
    constexpr int S = sizeof(T), V = 16 / S, P2 = V / 2;
    constexpr bool kFused = MODE == kFwdFused, kLn = MODE == kFwdLn;
    __shared__ float red[2][R][16];  // warp sums of the R rows, alternating between sums
    const T *x = reinterpret_cast<const T *>(a.x);
    const T *res = reinterpret_cast<const T *>(a.res);
    const T *g = reinterpret_cast<const T *>(a.gamma);
    const T *bt = reinterpret_cast<const T *>(a.beta);
    T *y = reinterpret_cast<T *>(a.y);
    T *ro = reinterpret_cast<T *>(a.res_out);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N, P = a.period;
    const int cls = (int)(blockIdx.x % (unsigned)P);
    const int64_t rank = blockIdx.x / (unsigned)P;
    const int64_t nper = ((int64_t)gridDim.x - cls + P - 1) / P;  // CTAs of this class
    const int64_t rstride = nper * P;
    const int64_t row0 = cls + rank * P;

    // the class's split (address arithmetic on row cls; nothing is read there)
    const uintptr_t start = reinterpret_cast<uintptr_t>(a.x) + (uintptr_t)cls * (uintptr_t)N * S;
    int h = (int)(((16u - (unsigned)(start & 15u)) & 15u) / S);
    if (h > N) h = N;
    const int nv = (N - h) / V, tail = N - h - nv * V;

    bool own[J];
    int col[J];
    f32x2 g2[J][P2], b2[kLn ? J : 1][kLn ? P2 : 1];
#pragma unroll
    for (int k = 0; k < J; ++k) {
        const int i = tid + k * nthr;
        own[k] = i < nv;
        col[k] = h + i * V;
        chunk_pairs2<T, V>(own[k] ? gather_chunk<T>(g + col[k]) : make_uint4(0, 0, 0, 0), g2[k]);
        if (kLn)
            chunk_pairs2<T, V>(own[k] && bt ? gather_chunk<T>(bt + col[k]) : make_uint4(0, 0, 0, 0),
                               b2[kLn ? k : 0]);
    }
    const bool e_own = tid < h + tail;
    const int je = tid < h ? tid : h + nv * V + (tid - h);
    const float ge = e_own ? to_f(g[je]) : 0.f;
    const float be = (kLn && e_own && bt) ? to_f(bt[je]) : 0.f;

    // rv: J residual chunks (fused-add only)
    auto load = [&](int64_t row, uint4 (&xv)[J], uint4 *rv, float &xe, float &re) {
        const size_t base = (size_t)row * N;
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                xv[k] = ld_global_nc_v4(x + base + col[k]);
                if (kFused) rv[kFused ? k : 0] = ld_global_nc_v4(res + base + col[k]);
            }
        }
        if (e_own) {
            xe = to_f(x[base + je]);
            if (kFused) re = to_f(res[base + je]);
        }
    };
    // CTA-wide sums of the R rows' per-thread values (one barrier)
    int buf = 0;
    auto row_sums = [&](float (&v)[R]) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float w = warp_sum(v[r]);
            if (lane == 0) red[buf][r][warp] = w;
        }
        __syncthreads();  // also orders the reads of red[buf] two sums back before these writes
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float t = 0.f;
            for (int w = 0; w < nwarps; ++w) t += red[buf][r][w];
            v[r] = t;
        }
        buf ^= 1;
    };

    constexpr int JR = kFused ? J : 1;
    uint4 xc[R][J], rc[R][JR], xn[R][J], rn_[R][JR];
    float xec[R], rec[R], xen[R], ren[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int k = 0; k < J; ++k) xc[r][k] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int k = 0; k < JR; ++k) rc[r][k] = make_uint4(0, 0, 0, 0);
        xec[r] = rec[r] = 0.f;
        const int64_t row = row0 + r * rstride;
        if (row < a.M) load(row, xc[r], rc[r], xec[r], rec[r]);
    }
    for (int64_t rb = row0; rb < a.M; rb += R * rstride) {
        // the next iteration's rows, in flight while these are computed
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int k = 0; k < J; ++k) xn[r][k] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < JR; ++k) rn_[r][k] = make_uint4(0, 0, 0, 0);
            xen[r] = ren[r] = 0.f;
            const int64_t nrow = rb + (R + r) * rstride;
            if (nrow < a.M) load(nrow, xn[r], rn_[r], xen[r], ren[r]);
        }

        // fused-add: residual_out = round(x + residual), kept (packed) as the row
        if (kFused) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int64_t row = rb + r * rstride;
                if (row >= a.M) break;  // uniform across the CTA
                const size_t base = (size_t)row * N;
#pragma unroll
                for (int k = 0; k < J; ++k) {
                    if (own[k]) {
                        f32x2 v[P2], w[P2];
                        chunk_pairs2<T, V>(xc[r][k], v);
                        chunk_pairs2<T, V>(rc[r][kFused ? k : 0], w);
#pragma unroll
                        for (int q = 0; q < P2; ++q) v[q] = f2_add(v[q], w[q]);
                        xc[r][k] = pairs_to_chunk<T, V>(v);
                        st_global_v4(ro + base + col[k], xc[r][k]);
                    }
                }
                if (e_own) {
                    xec[r] = round_through<T>(xec[r] + rec[r]);
                    ro[base + je] = from_f<T>(xec[r]);
                }
            }
        }

        // pass 1: sum of squares (LayerNorm: sum) of each row (a row past M sums zeros)
        float s[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            f32x2 s2 = f2_make(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < J; ++k) {
                if (own[k]) {
                    f32x2 v[P2];
                    chunk_pairs2<T, V>(xc[r][k], v);
#pragma unroll
                    for (int q = 0; q < P2; ++q) s2 = kLn ? f2_add(v[q], s2) : f2_fma(v[q], v[q], s2);
                }
            }
            float lo, hi;
            f2_split(s2, lo, hi);
            s[r] = lo + hi;
            if (e_own) s[r] = kLn ? s[r] + xec[r] : fmaf(xec[r], xec[r], s[r]);
        }
        row_sums(s);
        float mu[R], rs[R];
        if (kLn) {
            // pass 2: the centred sum of squares, from the registers (no cancellation)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                mu[r] = s[r] * a.inv_n;
                const f32x2 m2 = f2_make(-mu[r], -mu[r]);
                f32x2 q2 = f2_make(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < J; ++k) {
                    if (own[k]) {
                        f32x2 v[P2];
                        chunk_pairs2<T, V>(xc[r][k], v);
#pragma unroll
                        for (int q = 0; q < P2; ++q) {
                            const f32x2 d = f2_add(v[q], m2);
                            q2 = f2_fma(d, d, q2);
                        }
                    }
                }
                float lo, hi;
                f2_split(q2, lo, hi);
                s[r] = lo + hi;
                if (e_own) s[r] = fmaf(xec[r] - mu[r], xec[r] - mu[r], s[r]);
            }
            row_sums(s);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (!kLn) mu[r] = 0.f;
            rs[r] = rsqrtf(s[r] * a.inv_n + a.eps);
        }

        // output pass: y = x*rs*gamma (LayerNorm: (x - mean)*rs*gamma + beta)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = rb + r * rstride;
            if (row >= a.M) break;  // uniform across the CTA
            const size_t base = (size_t)row * N;
            if (tid == 0) {
                if (kLn && a.mean) a.mean[row] = mu[r];
                if (a.rstd) a.rstd[row] = rs[r];
            }
            const f32x2 rs2 = f2_make(rs[r], rs[r]), m2 = f2_make(-mu[r], -mu[r]);
#pragma unroll
            for (int k = 0; k < J; ++k) {
                if (own[k]) {
                    f32x2 v[P2];
                    chunk_pairs2<T, V>(xc[r][k], v);
#pragma unroll
                    for (int q = 0; q < P2; ++q) {
                        if (kLn)
                            v[q] = f2_fma(f2_mul(f2_add(v[q], m2), rs2), g2[k][q],
                                          b2[kLn ? k : 0][kLn ? q : 0]);
                        else
                            v[q] = f2_mul(f2_mul(v[q], rs2), g2[k][q]);
                    }
                    st_global_v4(y + base + col[k], pairs_to_chunk<T, V>(v));
                }
            }
            if (e_own)
                y[base + je] = from_f<T>(kLn ? fmaf((xec[r] - mu[r]) * rs[r], ge, be)
                                              : xec[r] * rs[r] * ge);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int k = 0; k < J; ++k) xc[r][k] = xn[r][k];
#pragma unroll
            for (int k = 0; k < JR; ++k) rc[r][k] = rn_[r][k];
            xec[r] = xen[r];
            rec[r] = ren[r];
        }
    }
}

template <typename T, int MODE, int J>
cudaError_t launch_t(const FwdPhaseArgs &a, int grid, int threads, cudaStream_t s) {
    fwd_phase_kernel<T, MODE, J, 2><<<grid, threads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int MODE>
cudaError_t launch_j(const FwdPhaseArgs &a, int cpt, int grid, int threads, cudaStream_t s) {
    return cpt == 2 ? launch_t<T, MODE, 2>(a, grid, threads, s)
                    : launch_t<T, MODE, 1>(a, grid, threads, s);
}

template <int MODE>
cudaError_t launch_mode(const FwdPhaseArgs &a, int dtype, int cpt, int grid, int threads,
                        cudaStream_t s) {
    switch (dtype) {
    case kF32: return launch_j<float, MODE>(a, cpt, grid, threads, s);
    case kF16: return launch_j<__half, MODE>(a, cpt, grid, threads, s);
    case kBF16: return launch_j<__nv_bfloat16, MODE>(a, cpt, grid, threads, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool fwd_phase_ok(const FwdRowProblem &p) {
    const uintptr_t S = (uintptr_t)elem_bytes(p.dtype);
    const uintptr_t ph = (uintptr_t)p.x & 15u;
    for (const void *q : {p.x, static_cast<const void *>(p.y), p.residual,
                          static_cast<const void *>(p.residual_out)}) {
        if (q == nullptr) continue;
        if (((uintptr_t)q & 15u) != ph || ((uintptr_t)q % S) != 0) return false;
    }
    return (int64_t)p.N * elem_bytes(p.dtype) / 16 <= 1024;
}

cudaError_t launch_fwd_phase(const FwdRowProblem &p, int cpt, int grid, int threads,
                             cudaStream_t s) {
    FwdPhaseArgs a;
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
    a.period = phase_period(p.N, p.dtype);
    // a residue class without a CTA would leave its rows unwritten
    if (p.M > 0 && grid < (p.M < a.period ? p.M : a.period)) return cudaErrorInvalidValue;
    if ((cpt != 1 && cpt != 2) || threads < 32 || threads > 512 || (threads & 31))
        return cudaErrorInvalidValue;
    switch (p.mode) {
    case kFwdRms: return launch_mode<kFwdRms>(a, p.dtype, cpt, grid, threads, s);
    case kFwdFused: return launch_mode<kFwdFused>(a, p.dtype, cpt, grid, threads, s);
    case kFwdLn: return launch_mode<kFwdLn>(a, p.dtype, cpt, grid, threads, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
