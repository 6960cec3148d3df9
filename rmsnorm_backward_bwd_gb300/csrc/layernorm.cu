// LayerNorm forward (saving mean and rstd) and backward (dx, dgamma, dbeta).
//
// The FlyDSL pages plan the LayerNorm backward as the RMSNorm backward with
// mean handling and a bias gradient added, over a forward that saves the
// per-row mean and rstd (issue #769, plan item 6 and "PR 5 -- LayerNorm
// backward"). The formulas are the textbook ones:
//   forward:  mean = (1/N) sum_j x_j,  var = (1/N) sum_j (x_j - mean)^2,
//             rstd = 1/sqrt(var + eps),  y = (x - mean) * rstd * gamma + beta
//   backward: x_hat = (x - mean) * rstd,  wdy = dy * gamma,
//             c1 = mean_j(x_hat * wdy),  c2 = mean_j(wdy),
//             dx = (wdy - c2 - x_hat * c1) * rstd,
//             dgamma = sum_rows dy * x_hat,  dbeta = sum_rows dy   (fp32)
//
// The engines mirror the RMSNorm ones:
//   * forward: aligned rows take the forward row engine (fwd_row.cu); here is
//     the one-CTA-per-row version for the others, in three sweeps (sum,
//     centred sum of squares, output).
//   * backward, aligned rows: the persistent row engine -- per-thread
//     cp.async ring of x and dy rows in shared memory, pass 1 reduces the two
//     row sums (x - mean)*wdy and wdy together, pass 2 stores dx and adds dy*x_hat
//     and dy into fp32 register partials; at the end the CTA's teams combine
//     their partials in a fixed order in shared memory and the CTA adds them
//     with fp32 vector atomics (atomic mode) or stores one partial row of
//     [dgamma | dbeta] to the workspace for the finalize kernel (scratch mode).
//   * backward, aligned rows longer than one CTA's tile: the cluster engine
//     of the RMSNorm backward (a row split across a thread-block cluster, the
//     two row sums exchanged through distributed shared memory behind one
//     cluster barrier per row), with the LayerNorm arithmetic.
//   * backward, unaligned rows: one CTA per row, scalar, two passes; the
//     partials live in shared memory when 2N floats fit, else in the CTA's
//     workspace row.
#include "cluster.cuh"
#include "common.cuh"
#include "ln_math.cuh"
#include "unaligned.cuh"
#include "launch.h"

namespace rn {

// ------------------------------------------------------------------ forward
struct LnFwdArgs {
    const uint8_t *x;
    const uint8_t *gamma;
    const uint8_t *beta;  // nullable
    uint8_t *y;
    float *mean;          // nullable
    float *rstd;          // nullable
    int64_t M;
    int N;
    float inv_n;
    float eps;
};

template <typename T>
__global__ void __launch_bounds__(256) ln_fwd_generic_kernel(const LnFwdArgs a) {
    __shared__ float red[32];
    const T *x = reinterpret_cast<const T *>(a.x);
    const T *g = reinterpret_cast<const T *>(a.gamma);
    const T *bt = reinterpret_cast<const T *>(a.beta);
    T *y = reinterpret_cast<T *>(a.y);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N;
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
        const T *xr = x + (size_t)row * N;
        float s = 0.f;
        for (int j = tid; j < N; j += nthr) s += to_f(xr[j]);
        const float mu = block_sum(s) * a.inv_n;
        float q = 0.f;
        for (int j = tid; j < N; j += nthr) {
            const float d = to_f(xr[j]) - mu;
            q = fmaf(d, d, q);
        }
        const float rs = rsqrtf(block_sum(q) * a.inv_n + a.eps);
        if (tid == 0) {
            if (a.mean) a.mean[row] = mu;
            if (a.rstd) a.rstd[row] = rs;
        }
        T *yr = y + (size_t)row * N;
        for (int j = tid; j < N; j += nthr) {
            const float bv = bt ? to_f(bt[j]) : 0.f;
            yr[j] = from_f<T>(fmaf((to_f(xr[j]) - mu) * rs, to_f(g[j]), bv));
        }
    }
}

template <typename T>
static cudaError_t launch_ln_fwd_t(const LnFwdArgs &a, int num_sms, cudaStream_t s) {
    int64_t grid = (int64_t)num_sms * 8;
    if (grid > a.M) grid = a.M;
    ln_fwd_generic_kernel<T><<<(unsigned)grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ln_fwd(const LnFwdProblem &p, int num_sms, cudaStream_t s) {
    LnFwdArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.beta = static_cast<const uint8_t *>(p.beta);
    a.y = static_cast<uint8_t *>(p.y);
    a.mean = p.mean;
    a.rstd = p.rstd;
    a.M = p.M;
    a.N = p.N;
    a.inv_n = 1.0f / (float)p.N;
    a.eps = p.eps;
    switch (p.dtype) {
    case kF32: return launch_ln_fwd_t<float>(a, num_sms, s);
    case kF16: return launch_ln_fwd_t<__half>(a, num_sms, s);
    case kBF16: return launch_ln_fwd_t<__nv_bfloat16>(a, num_sms, s);
    default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------- backward, row engine
// Two fp32 accumulators per element pair (dgamma, dbeta) need up to 128
// registers a thread: at most 512 threads a CTA for every tile.
int ln_row_max_threads(int) { return 512; }
constexpr int kLnMaxThreads = 512;

// [2 parities][2 sums][32 warps] fp32 partial sums, then the ring
constexpr int kLnRingOffset = 512;

size_t ln_row_smem_bytes(int teams, int stages, int team_chunks) {
    return (size_t)kLnRingOffset + (size_t)teams * stages * 2 * (size_t)team_chunks * 16;
}

struct LnRowArgs {
    const uint8_t *x;
    const uint8_t *gamma;
    const uint8_t *dy;
    const float *mean;
    const float *rstd;
    uint8_t *dx;
    // atomic: dgamma_f32 / dbeta_f32 (dbeta nullable);
    // scratch: the workspace's partial rows [gridDim.x][2N], dgamma then dbeta
    float *dg_out;
    float *db_out;
    int64_t M;
    int N;
    int nchunks;
    int row_bytes;
    int team_threads;
    int teams;
    int stages;
    float inv_n;
};

// Two team-wide sums at once; every thread of the team gets the same bits.
__device__ __forceinline__ void ln_team_sum2(float &u, float &v, float *red, int parity, int warp,
                                             int lane, int team, int team_warps, int first_warp,
                                             int team_threads) {
    u = warp_sum(u);
    v = warp_sum(v);
    if (team_warps == 1) return;
    float *slot = red + parity * 64;
    if (lane == 0) {
        slot[warp] = u;
        slot[32 + warp] = v;
    }
    named_barrier_sync(1 + team, team_threads);
    const float a = lane < team_warps ? slot[first_warp + lane] : 0.f;
    const float b = lane < team_warps ? slot[32 + first_warp + lane] : 0.f;
    u = warp_sum(a);
    v = warp_sum(b);
}

// The CTA's partials of dgamma and dbeta (each team's registers; with several
// teams, combined in a fixed team order through shared memory, float4 q of
// chunk c at q*tc + c, the dbeta copy after the dgamma one): added atomically
// into dg / db (atomic mode) or stored there as the CTA's partial rows
// (scratch). db may be NULL (no bias gradient). `scratch` must hold 2N floats
// and be free of other use; the caller synchronises the CTA before.
template <int CPT, int P, bool ATOMIC>
__device__ __forceinline__ void ln_cta_out(const f32x2 (&accg)[CPT][P],
                                           const f32x2 (&accb)[CPT][P], float *dg, float *db,
                                           const LnRowArgs &a, uint8_t *scratch, int team,
                                           int tt) {
    constexpr int Q = P / 2;  // float4 per chunk
    auto put = [](float *dst4, const float4 &v) {
        if (ATOMIC) atomicAdd(reinterpret_cast<float4 *>(dst4), v);
        else *reinterpret_cast<float4 *>(dst4) = v;
    };
    if (a.teams == 1) {
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = tt + kk * a.team_threads;
            if (c < a.nchunks) {
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const size_t off = (size_t)c * (2 * P) + 4 * q;
                    float4 v;
                    f2_split(accg[kk][2 * q], v.x, v.y);
                    f2_split(accg[kk][2 * q + 1], v.z, v.w);
                    put(dg + off, v);
                    if (db) {
                        f2_split(accb[kk][2 * q], v.x, v.y);
                        f2_split(accb[kk][2 * q + 1], v.z, v.w);
                        put(db + off, v);
                    }
                }
            }
        }
        return;
    }
    const int tc = CPT * a.team_threads;
    float4 *sg = reinterpret_cast<float4 *>(scratch);
    float4 *sb = sg + (size_t)Q * tc;
    auto acc4 = [](float4 *p, float4 v, bool add) {
        if (add) {
            const float4 o = *p;
            v.x += o.x;
            v.y += o.y;
            v.z += o.z;
            v.w += o.w;
        }
        *p = v;
    };
    for (int t = 0; t < a.teams; ++t) {
        if (team == t) {
#pragma unroll
            for (int kk = 0; kk < CPT; ++kk) {
                const int c = tt + kk * a.team_threads;
                if (c < a.nchunks) {
#pragma unroll
                    for (int q = 0; q < Q; ++q) {
                        const size_t i = (size_t)q * tc + c;
                        float4 v;
                        f2_split(accg[kk][2 * q], v.x, v.y);
                        f2_split(accg[kk][2 * q + 1], v.z, v.w);
                        acc4(sg + i, v, t > 0);
                        f2_split(accb[kk][2 * q], v.x, v.y);
                        f2_split(accb[kk][2 * q + 1], v.z, v.w);
                        acc4(sb + i, v, t > 0);
                    }
                }
            }
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < a.N / 4; i += blockDim.x) {
        const int c = i / Q, q = i - c * Q;
        const size_t j = (size_t)q * tc + c;
        put(dg + 4 * (size_t)i, sg[j]);
        if (db) put(db + 4 * (size_t)i, sb[j]);
    }
}

template <typename T, int CPT, bool ATOMIC>
__global__ void __launch_bounds__(kLnMaxThreads, 1) ln_bwd_row_kernel(const LnRowArgs a) {
    constexpr int V = Traits<T>::kVec;
    constexpr int P = V / 2;  // fp32 pairs per chunk
    // fp32 gamma is kept as pairs; 16-bit gamma stays packed (see mul_chunk_pairs)
    constexpr bool kF32 = sizeof(T) == 4;
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    uint8_t *ring = smem + kLnRingOffset;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int team = tid / a.team_threads;
    const int tt = tid - team * a.team_threads;
    const int team_warps = a.team_threads >> 5;
    const int first_warp = team * team_warps;
    const int S = a.stages;

    // This thread's ring: chunk kk of tensor t (0 = x, 1 = dy) in slot s at
    // my0 + s*slot_bytes + t*tensor_bytes + kk*kk_bytes.
    const int tc = CPT * a.team_threads;
    const uint32_t kk_bytes = 16u * a.team_threads;
    const uint32_t tensor_bytes = 16u * tc;
    const uint32_t slot_bytes = 2 * tensor_bytes;
    const uint32_t my0 = smem_addr(ring) + (uint32_t)team * S * slot_bytes + 16u * tt;

    const int64_t team_stride = (int64_t)gridDim.x * a.teams;
    const int64_t row0 = (int64_t)blockIdx.x * a.teams + team;
    const int64_t nrows = row0 < a.M ? (a.M - 1 - row0) / team_stride + 1 : 0;
    const uint64_t policy = l2_policy_evict_first();

    uint32_t coff[CPT];
    bool cok[CPT];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        const int c = tt + kk * a.team_threads;
        coff[kk] = 16u * c;
        cok[kk] = c < a.nchunks;
    }

    auto issue = [&](int64_t row, int s) {
        const size_t off = (size_t)row * a.row_bytes;
        const uint8_t *xr = a.x + off, *dr = a.dy + off;
        const uint32_t d = my0 + (uint32_t)s * slot_bytes;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                cp_async16(d + kk * kk_bytes, xr + coff[kk], policy);
                cp_async16(d + tensor_bytes + kk * kk_bytes, dr + coff[kk], policy);
            }
        }
    };
    for (int j = 0; j < S - 1; ++j) {
        if (j < nrows) issue(row0 + j * team_stride, j);
        cp_async_commit();
    }

    uint4 gp[CPT];
    f32x2 g2[kF32 ? CPT : 1][kF32 ? P : 1];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        gp[kk] = cok[kk] ? ld_global_nc_v4(a.gamma + coff[kk]) : make_uint4(0, 0, 0, 0);
        if (kF32) chunk_pairs<T>(gp[kk], g2[kF32 ? kk : 0]);
    }
    // wdy = dy*gamma of chunk kk as fp32 pairs (d2: dy as pairs, fp32 only)
    auto wdy = [&](int kk, const uint4 &dv, const f32x2 *d2, f32x2 *w) {
        if constexpr (kF32) {
#pragma unroll
            for (int q = 0; q < P; ++q) w[q] = f2_mul(d2[q], g2[kF32 ? kk : 0][kF32 ? q : 0]);
        } else {
            mul_chunk_pairs<T>(dv, gp[kk], w);
        }
    };
    f32x2 accg[CPT][P], accb[CPT][P];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk)
#pragma unroll
        for (int q = 0; q < P; ++q) accg[kk][q] = accb[kk][q] = f2_make(0.f, 0.f);

    const int64_t ahead = (int64_t)(S - 1) * team_stride;
    float mu_next = nrows > 0 ? __ldg(a.mean + row0) : 0.f;
    float rs_next = nrows > 0 ? __ldg(a.rstd + row0) : 0.f;
    int slot = 0, fill = S - 1;
    int64_t row = row0;
    for (int64_t k = 0; k < nrows; ++k, row += team_stride) {
        if (k + S - 1 < nrows) issue(row + ahead, fill);
        cp_async_commit();
        const float mu = mu_next, rs = rs_next;
        if (k + 1 < nrows) {
            mu_next = __ldg(a.mean + row + team_stride);
            rs_next = __ldg(a.rstd + row + team_stride);
        }
        cp_async_wait_pending(S - 1);
        const uint32_t sb = my0 + (uint32_t)slot * slot_bytes;
        const f32x2 nmu2 = f2_make(-mu, -mu);

        // pass 1: sum (x - mean)*wdy and sum wdy over the row
        f32x2 s1 = f2_make(0.f, 0.f), s2 = f2_make(0.f, 0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                f32x2 xc[P], d2[P], w[P];
                const uint4 dv = ld_shared_v4(sb + tensor_bytes + kk * kk_bytes);
                centre_chunk_pairs<T>(ld_shared_v4(sb + kk * kk_bytes), nmu2, -mu, xc);
                if (kF32) chunk_pairs<T>(dv, d2);
                wdy(kk, dv, d2, w);
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    s1 = f2_fma(xc[q], w[q], s1);
                    s2 = f2_add(w[q], s2);
                }
            }
        }
        float u, v, uh, vh;
        f2_split(s1, u, uh);
        f2_split(s2, v, vh);
        u += uh;
        v += vh;
        ln_team_sum2(u, v, red, (int)(k & 1), warp, lane, team, team_warps, first_warp,
                     a.team_threads);

        // dx = (wdy - c2 - x_hat*c1)*rstd = wdy*rstd + (x - mean)*B + A with
        // c1 = rstd*u/N, c2 = v/N, B = -rstd^2*c1, A = -c2*rstd
        const float c1 = rs * u * a.inv_n;
        const float c2 = v * a.inv_n;
        const float B = -rs * rs * c1, A = -c2 * rs;
        const f32x2 rs2 = f2_make(rs, rs), B2 = f2_make(B, B), A2 = f2_make(A, A);
        uint8_t *dxrow = a.dx + (size_t)row * a.row_bytes;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                f32x2 xc[P], d2[P], w[P], o2[P];
                const uint4 dv = ld_shared_v4(sb + tensor_bytes + kk * kk_bytes);
                centre_chunk_pairs<T>(ld_shared_v4(sb + kk * kk_bytes), nmu2, -mu, xc);
                chunk_pairs<T>(dv, d2);
                wdy(kk, dv, d2, w);
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    o2[q] = f2_fma(w[q], rs2, f2_fma(xc[q], B2, A2));
                    accg[kk][q] = f2_fma(d2[q], f2_mul(xc[q], rs2), accg[kk][q]);
                    accb[kk][q] = f2_add(d2[q], accb[kk][q]);
                }
                st_global_v4(dxrow + coff[kk], pairs_chunk<T>(o2));
            }
        }
        if (++slot == S) slot = 0;
        if (++fill == S) fill = 0;
    }

    pdl_launch_dependents();
    __syncthreads();  // every team is done with its ring (all real copies waited for)
    if (ATOMIC) pdl_wait();  // the zeroing kernel ahead of this one has finished
    float *dg = ATOMIC ? a.dg_out : a.dg_out + (size_t)blockIdx.x * 2 * a.N;
    float *db = ATOMIC ? a.db_out : dg + a.N;
    ln_cta_out<CPT, P, ATOMIC>(accg, accb, dg, db, a, ring, team, tt);
}

template <typename T, int CPT, bool ATOMIC>
static cudaError_t launch_ln_row_t(const LnRowArgs &args, const RowPlan &plan, cudaStream_t s,
                                   bool pdl) {
    auto kern = ln_bwd_row_kernel<T, CPT, ATOMIC>;
    cudaError_t e = ensure_smem_attr((const void *)kern, plan.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(plan.teams * plan.team_threads);
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
static cudaError_t launch_ln_row_dt(const LnRowArgs &args, const RowPlan &plan, cudaStream_t s,
                                    bool pdl) {
    switch (plan.cpt) {
    case 1:
        return plan.atomic ? launch_ln_row_t<T, 1, true>(args, plan, s, pdl)
                           : launch_ln_row_t<T, 1, false>(args, plan, s, pdl);
    case 2:
        return plan.atomic ? launch_ln_row_t<T, 2, true>(args, plan, s, pdl)
                           : launch_ln_row_t<T, 2, false>(args, plan, s, pdl);
    case 4:
        return plan.atomic ? launch_ln_row_t<T, 4, true>(args, plan, s, pdl)
                           : launch_ln_row_t<T, 4, false>(args, plan, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_ln_bwd_row(const LnBwdProblem &p, const RowPlan &plan, cudaStream_t s,
                              bool pdl_after_zero) {
    LnRowArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.dy = static_cast<const uint8_t *>(p.dy);
    a.mean = p.mean;
    a.rstd = p.rstd;
    a.dx = static_cast<uint8_t *>(p.dx);
    if (plan.atomic) {
        a.dg_out = p.dg_f32;
        a.db_out = p.db_f32;
    } else {
        a.dg_out = reinterpret_cast<float *>(p.ws + kWsHeaderBytes);
        a.db_out = nullptr;  // the kernel derives the dbeta half of each partial row
    }
    a.M = p.M;
    a.N = p.N;
    a.row_bytes = p.N * elem_bytes(p.dtype);
    a.nchunks = a.row_bytes / 16;
    a.team_threads = plan.team_threads;
    a.teams = plan.teams;
    a.stages = plan.stages;
    a.inv_n = 1.0f / (float)p.N;
    switch (p.dtype) {
    case kF32: return launch_ln_row_dt<float>(a, plan, s, pdl_after_zero);
    case kF16: return launch_ln_row_dt<__half>(a, plan, s, pdl_after_zero);
    case kBF16: return launch_ln_row_dt<__nv_bfloat16>(a, plan, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

// -------------------------------------------------- backward, cluster engine
// [2 parities][2 sums][16 warps] fp32 warp sums, then the ring
constexpr int kLnClusterRingOffset = 512;

size_t ln_cluster_smem_bytes(int stages, int cpt, int threads) {
    return (size_t)kLnClusterRingOffset + (size_t)stages * 2 * cpt * threads * 16;
}

struct LnClusterArgs {
    const uint8_t *x;
    const uint8_t *gamma;
    const uint8_t *dy;
    const float *mean;
    const float *rstd;
    uint8_t *dx;
    // atomic: dgamma_f32 / dbeta_f32 (dbeta nullable);
    // scratch: partial rows [clusters][2N], dgamma then dbeta
    float *dg_out;
    float *db_out;
    int64_t M;
    int N;
    int nchunks;
    int row_bytes;
    int slice;  // chunks per CTA slice
    int stages;
    float inv_n;
};

template <typename T, int CPT, bool ATOMIC>
__global__ void __launch_bounds__(512, 1) ln_bwd_cluster_kernel(const LnClusterArgs a) {
    constexpr int V = Traits<T>::kVec;
    constexpr int P = V / 2;
    constexpr int Q = P / 2;  // float4 per chunk
    constexpr bool kF32 = sizeof(T) == 4;
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    uint8_t *ring = smem + kLnClusterRingOffset;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const uint32_t crank = cluster_rank();
    const int csize = (int)cluster_size_x();
    const int64_t cid = cluster_index_x();
    const int64_t ncl = cluster_count_x();
    const int S = a.stages;

    const int c0 = (int)crank * a.slice;
    int c1 = c0 + a.slice;
    if (c1 > a.nchunks) c1 = a.nchunks;

    const uint32_t kk_bytes = 16u * nthr;
    const uint32_t tensor_bytes = kk_bytes * CPT;
    const uint32_t slot_bytes = 2 * tensor_bytes;
    const uint32_t my0 = smem_addr(ring) + 16u * tid;
    const uint32_t red_addr = smem_addr(red);

    const int64_t nrows = cid < a.M ? (a.M - 1 - cid) / ncl + 1 : 0;
    const uint64_t policy = l2_policy_evict_first();

    uint32_t coff[CPT];
    bool cok[CPT];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        const int c = c0 + tid + kk * nthr;
        coff[kk] = 16u * c;
        cok[kk] = c < c1;
    }

    auto issue = [&](int64_t row, int s) {
        const size_t off = (size_t)row * a.row_bytes;
        const uint8_t *xr = a.x + off, *dr = a.dy + off;
        const uint32_t d = my0 + (uint32_t)s * slot_bytes;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                cp_async16(d + kk * kk_bytes, xr + coff[kk], policy);
                cp_async16(d + tensor_bytes + kk * kk_bytes, dr + coff[kk], policy);
            }
        }
    };
    for (int j = 0; j < S - 1; ++j) {
        if (j < nrows) issue(cid + j * ncl, j);
        cp_async_commit();
    }

    uint4 gp[CPT];
    f32x2 g2[kF32 ? CPT : 1][kF32 ? P : 1];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        gp[kk] = cok[kk] ? ld_global_nc_v4(a.gamma + coff[kk]) : make_uint4(0, 0, 0, 0);
        if (kF32) chunk_pairs<T>(gp[kk], g2[kF32 ? kk : 0]);
    }
    auto wdy = [&](int kk, const uint4 &dv, const f32x2 *d2, f32x2 *w) {
        if constexpr (kF32) {
#pragma unroll
            for (int q = 0; q < P; ++q) w[q] = f2_mul(d2[q], g2[kF32 ? kk : 0][kF32 ? q : 0]);
        } else {
            mul_chunk_pairs<T>(dv, gp[kk], w);
        }
    };
    f32x2 accg[CPT][P], accb[CPT][P];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk)
#pragma unroll
        for (int q = 0; q < P; ++q) accg[kk][q] = accb[kk][q] = f2_make(0.f, 0.f);

    const int64_t ahead = (int64_t)(S - 1) * ncl;
    const int nparts = csize * nwarps;  // <= 16 x 16
    float mu_next = nrows > 0 ? __ldg(a.mean + cid) : 0.f;
    float rs_next = nrows > 0 ? __ldg(a.rstd + cid) : 0.f;
    int slot = 0, fill = S - 1;
    int64_t row = cid;
    for (int64_t k = 0; k < nrows; ++k, row += ncl) {
        if (k + S - 1 < nrows) issue(row + ahead, fill);
        cp_async_commit();
        const float mu = mu_next, rs = rs_next;
        if (k + 1 < nrows) {
            mu_next = __ldg(a.mean + row + ncl);
            rs_next = __ldg(a.rstd + row + ncl);
        }
        cp_async_wait_pending(S - 1);
        const uint32_t sb = my0 + (uint32_t)slot * slot_bytes;
        const f32x2 nmu2 = f2_make(-mu, -mu);

        // pass 1: this thread's share of sum (x - mean)*wdy and sum wdy
        f32x2 s1 = f2_make(0.f, 0.f), s2 = f2_make(0.f, 0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                f32x2 xc[P], d2[P], w[P];
                const uint4 dv = ld_shared_v4(sb + tensor_bytes + kk * kk_bytes);
                centre_chunk_pairs<T>(ld_shared_v4(sb + kk * kk_bytes), nmu2, -mu, xc);
                if (kF32) chunk_pairs<T>(dv, d2);
                wdy(kk, dv, d2, w);
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    s1 = f2_fma(xc[q], w[q], s1);
                    s2 = f2_add(w[q], s2);
                }
            }
        }
        float u, v, uh, vh;
        f2_split(s1, u, uh);
        f2_split(s2, v, vh);
        u = warp_sum(u + uh);
        v = warp_sum(v + vh);
        const int par = (int)(k & 1) * 32;
        if (lane == 0) {
            red[par + warp] = u;
            red[par + 16 + warp] = v;
        }
        cluster_sync_all();
        // lane l reads partial l of the cluster's C x warps partials
        float tu = 0.f, tv = 0.f;
        for (int i = lane; i < nparts; i += 32) {
            const int r = i / nwarps, w = i - r * nwarps;
            tu += ld_peer_f32(red_addr + 4u * (par + w), (uint32_t)r);
            tv += ld_peer_f32(red_addr + 4u * (par + 16 + w), (uint32_t)r);
        }
        u = warp_sum(tu);
        v = warp_sum(tv);

        const float c1v = rs * u * a.inv_n;
        const float c2 = v * a.inv_n;
        const float B = -rs * rs * c1v, A = -c2 * rs;
        const f32x2 rs2 = f2_make(rs, rs), B2 = f2_make(B, B), A2 = f2_make(A, A);
        uint8_t *dxrow = a.dx + (size_t)row * a.row_bytes;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                f32x2 xc[P], d2[P], w[P], o2[P];
                const uint4 dv = ld_shared_v4(sb + tensor_bytes + kk * kk_bytes);
                centre_chunk_pairs<T>(ld_shared_v4(sb + kk * kk_bytes), nmu2, -mu, xc);
                chunk_pairs<T>(dv, d2);
                wdy(kk, dv, d2, w);
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    o2[q] = f2_fma(w[q], rs2, f2_fma(xc[q], B2, A2));
                    accg[kk][q] = f2_fma(d2[q], f2_mul(xc[q], rs2), accg[kk][q]);
                    accb[kk][q] = f2_add(d2[q], accb[kk][q]);
                }
                st_global_v4(dxrow + coff[kk], pairs_chunk<T>(o2));
            }
        }
        if (++slot == S) slot = 0;
        if (++fill == S) fill = 0;
    }
    // peers may still read this CTA's partial slots of the last row
    cluster_sync_all();

    pdl_launch_dependents();
    if (ATOMIC) pdl_wait();  // the zeroing kernel ahead of this one has finished
    float *dg = ATOMIC ? a.dg_out : a.dg_out + (size_t)cid * 2 * a.N;
    float *db = ATOMIC ? a.db_out : dg + a.N;
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        if (cok[kk]) {
            const int c = c0 + tid + kk * nthr;
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const size_t off = (size_t)c * V + 4 * q;
                float4 vg, vb;
                f2_split(accg[kk][2 * q], vg.x, vg.y);
                f2_split(accg[kk][2 * q + 1], vg.z, vg.w);
                f2_split(accb[kk][2 * q], vb.x, vb.y);
                f2_split(accb[kk][2 * q + 1], vb.z, vb.w);
                if (ATOMIC) {
                    atomicAdd(reinterpret_cast<float4 *>(dg + off), vg);
                    if (db) atomicAdd(reinterpret_cast<float4 *>(db + off), vb);
                } else {
                    *reinterpret_cast<float4 *>(dg + off) = vg;
                    *reinterpret_cast<float4 *>(db + off) = vb;
                }
            }
        }
    }
}

template <typename T, int CPT, bool ATOMIC>
static const void *ln_cluster_ptr() {
    return (const void *)ln_bwd_cluster_kernel<T, CPT, ATOMIC>;
}

template <typename T>
static const void *ln_cluster_kernel_for(int cpt, bool atomic) {
    if (cpt == 1) return atomic ? ln_cluster_ptr<T, 1, true>() : ln_cluster_ptr<T, 1, false>();
    if (cpt == 2) return atomic ? ln_cluster_ptr<T, 2, true>() : ln_cluster_ptr<T, 2, false>();
    return atomic ? ln_cluster_ptr<T, 4, true>() : ln_cluster_ptr<T, 4, false>();
}

static const void *ln_cluster_kernel_dt(int dtype, int cpt, bool atomic) {
    switch (dtype) {
    case kF32: return ln_cluster_kernel_for<float>(cpt, atomic);
    case kF16: return ln_cluster_kernel_for<__half>(cpt, atomic);
    case kBF16: return ln_cluster_kernel_for<__nv_bfloat16>(cpt, atomic);
    default: return nullptr;
    }
}

static cudaError_t ln_cluster_prepare(const void *kern, const ClusterPlan &plan) {
    cudaError_t e = ensure_smem_attr(kern, plan.smem);
    if (e != cudaSuccess) return e;
    if (plan.csize > 8)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

cudaError_t ln_cluster_max_active(const LnBwdProblem &p, const ClusterPlan &plan, int *clusters) {
    const void *kern = ln_cluster_kernel_dt(p.dtype, plan.cpt, plan.atomic);
    if (!kern) return cudaErrorInvalidValue;
    cudaError_t e = ln_cluster_prepare(kern, plan);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.csize);
    cfg.blockDim = dim3(plan.threads);
    cfg.dynamicSmemBytes = plan.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = plan.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, kern, &cfg);
}

template <typename T, int CPT, bool ATOMIC>
static cudaError_t launch_ln_cluster_t(const LnClusterArgs &args, const ClusterPlan &plan,
                                       cudaStream_t s, bool pdl) {
    auto kern = ln_bwd_cluster_kernel<T, CPT, ATOMIC>;
    cudaError_t e = ln_cluster_prepare((const void *)kern, plan);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.clusters * plan.csize);
    cfg.blockDim = dim3(plan.threads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = plan.csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

template <typename T>
static cudaError_t launch_ln_cluster_dt(const LnClusterArgs &args, const ClusterPlan &plan,
                                        cudaStream_t s, bool pdl) {
    switch (plan.cpt) {
    case 1:
        return plan.atomic ? launch_ln_cluster_t<T, 1, true>(args, plan, s, pdl)
                           : launch_ln_cluster_t<T, 1, false>(args, plan, s, pdl);
    case 2:
        return plan.atomic ? launch_ln_cluster_t<T, 2, true>(args, plan, s, pdl)
                           : launch_ln_cluster_t<T, 2, false>(args, plan, s, pdl);
    case 4:
        return plan.atomic ? launch_ln_cluster_t<T, 4, true>(args, plan, s, pdl)
                           : launch_ln_cluster_t<T, 4, false>(args, plan, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_ln_bwd_cluster(const LnBwdProblem &p, const ClusterPlan &plan, cudaStream_t s,
                                  bool pdl_after_zero) {
    LnClusterArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.dy = static_cast<const uint8_t *>(p.dy);
    a.mean = p.mean;
    a.rstd = p.rstd;
    a.dx = static_cast<uint8_t *>(p.dx);
    if (plan.atomic) {
        a.dg_out = p.dg_f32;
        a.db_out = p.db_f32;
    } else {
        a.dg_out = reinterpret_cast<float *>(p.ws + kWsHeaderBytes);
        a.db_out = nullptr;  // the kernel derives the dbeta half of each partial row
    }
    a.M = p.M;
    a.N = p.N;
    a.row_bytes = p.N * elem_bytes(p.dtype);
    a.nchunks = a.row_bytes / 16;
    a.slice = plan.slice;
    a.stages = plan.stages;
    a.inv_n = 1.0f / (float)p.N;
    switch (p.dtype) {
    case kF32: return launch_ln_cluster_dt<float>(a, plan, s, pdl_after_zero);
    case kF16: return launch_ln_cluster_dt<__half>(a, plan, s, pdl_after_zero);
    case kBF16: return launch_ln_cluster_dt<__nv_bfloat16>(a, plan, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

// -------------------------------------------------- backward, generic engine
size_t ln_generic_smem_bytes(int N, bool smem_dw) {
    return 512 + (smem_dw ? (size_t)N * 8 : 0);
}

struct LnGenArgs {
    const void *x;
    const void *gamma;
    const void *dy;
    const float *mean;
    const float *rstd;
    void *dx;
    // scratch: partial rows [gridDim.x][2N] (dgamma | dbeta); atomic: the outputs
    float *dg_out;
    float *db_out;  // atomic mode only; nullable
    int64_t M;
    int N;
    float inv_n;
    int words;  // vector variant: padded length of each shared array
};

template <typename T, bool ATOMIC, bool SMEM_DW>
__global__ void __launch_bounds__(512) ln_bwd_generic_kernel(const LnGenArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);        // [2 sums][32 warps]
    float *sdw = reinterpret_cast<float *>(smem + 512);  // 2N floats when SMEM_DW
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N;
    float *part = ATOMIC ? nullptr : a.dg_out + (size_t)blockIdx.x * 2 * N;
    float *dw = SMEM_DW ? sdw : part;  // [dgamma | dbeta]; !SMEM_DW implies scratch mode

    for (int j = tid; j < 2 * N; j += nthr) dw[j] = 0.f;

    for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x) {
        const float mu = __ldg(a.mean + row), rs = __ldg(a.rstd + row);
        const T *xr = x + (size_t)row * N;
        const T *dyr = dy + (size_t)row * N;
        float s1 = 0.f, s2 = 0.f;
        for (int j = tid; j < N; j += nthr) {
            const float w = to_f(dyr[j]) * to_f(g[j]);
            s1 = fmaf(to_f(xr[j]) - mu, w, s1);
            s2 += w;
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        if (lane == 0) {
            red[warp] = s1;
            red[32 + warp] = s2;
        }
        __syncthreads();
        float t1 = 0.f, t2 = 0.f;
        for (int w = 0; w < nwarps; ++w) {
            t1 += red[w];
            t2 += red[32 + w];
        }
        __syncthreads();  // red is rewritten by the next row
        const float c1 = rs * t1 * a.inv_n, c2 = t2 * a.inv_n;
        T *dxr = dx + (size_t)row * N;
        for (int j = tid; j < N; j += nthr) {
            const float dv = to_f(dyr[j]);
            const float xh = (to_f(xr[j]) - mu) * rs;
            const float w = dv * to_f(g[j]);
            dxr[j] = from_f<T>((w - c2 - xh * c1) * rs);
            dw[j] = fmaf(dv, xh, dw[j]);
            dw[N + j] += dv;
        }
    }
    pdl_launch_dependents();
    if (SMEM_DW || ATOMIC) {
        if (ATOMIC) {
            pdl_wait();
            for (int j = tid; j < N; j += nthr) {
                atomicAdd(a.dg_out + j, dw[j]);
                if (a.db_out) atomicAdd(a.db_out + j, dw[N + j]);
            }
        } else {
            for (int j = tid; j < 2 * N; j += nthr) part[j] = dw[j];
        }
    }
}

// Vector variant of the generic engine (rows that are not 16-byte multiples,
// x, dy and dx at one alignment phase), the LayerNorm counterpart of the
// RMSNorm one: each row splits into a head, whole 16-byte chunks (128-bit
// loads and stores) and a tail; R rows per CTA iteration, their two sums
// reduced together; gamma as fp32 and the dgamma / dbeta partials in padded
// shared memory (a column's owner thread changes with the row's phase, so
// the partials take shared atomic adds).
size_t ln_generic_vec_smem_bytes(int N) { return 1024 + 3 * 4 * vec_words(N); }

template <typename T, bool ATOMIC, int R>
__global__ void __launch_bounds__(512, 2) ln_bwd_generic_vec_kernel(const LnGenArgs a) {
    constexpr int S = sizeof(T), V = 16 / S;
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);            // [R][2 sums][32 warps]
    float *sg = reinterpret_cast<float *>(smem + 1024);      // gamma, fp32, padded columns
    float *sdg = sg + a.words;                               // dgamma partial, padded
    float *sdb = sdg + a.words;                              // dbeta partial, padded
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N;

    for (int j = tid; j < N; j += nthr) {
        sdg[vpad(j)] = 0.f;
        sdb[vpad(j)] = 0.f;
        sg[vpad(j)] = to_f(g[j]);
    }
    __syncthreads();

    for (int64_t row0 = (int64_t)blockIdx.x * R; row0 < a.M; row0 += (int64_t)gridDim.x * R) {
        int h[R], nv[R], nt[R];
        float mu[R], rs[R], s1[R], s2[R];
        int nvmax = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = row0 + r;
            h[r] = nv[r] = nt[r] = 0;
            mu[r] = rs[r] = s1[r] = s2[r] = 0.f;
            if (row < a.M) {
                const uintptr_t ad = reinterpret_cast<uintptr_t>(x + (size_t)row * N);
                int hh = (int)(((16u - (unsigned)(ad & 15u)) & 15u) / S);
                if (hh > N) hh = N;
                h[r] = hh;
                nv[r] = (N - hh) / V;
                nt[r] = N - hh - nv[r] * V;
                mu[r] = __ldg(a.mean + row);
                rs[r] = __ldg(a.rstd + row);
            }
            if (nv[r] > nvmax) nvmax = nv[r];
        }
        // pass 1: sum (x - mean)*wdy and sum wdy of each row
        for (int i = tid; i < nvmax; i += nthr) {
            uint4 xv[R], dv[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (i < nv[r]) {
                    const size_t e0 = (size_t)(row0 + r) * N + h[r] + (size_t)i * V;
                    xv[r] = ld_global_nc_v4(x + e0);
                    dv[r] = ld_global_nc_v4(dy + e0);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (i < nv[r]) {
                    float xf[V], df[V];
                    chunk_to_float<T>(xv[r], xf);
                    chunk_to_float<T>(dv[r], df);
                    const int c0 = h[r] + i * V;
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float w = df[e] * sg[vpad(c0 + e)];
                        s1[r] = fmaf(xf[e] - mu[r], w, s1[r]);
                        s2[r] += w;
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            // head and tail (fewer than V elements each)
            if (tid < h[r] + nt[r]) {
                const size_t base = (size_t)(row0 + r) * N;
                const int j = tid < h[r] ? tid : h[r] + nv[r] * V + (tid - h[r]);
                const float w = to_f(dy[base + j]) * sg[vpad(j)];
                s1[r] = fmaf(to_f(x[base + j]) - mu[r], w, s1[r]);
                s2[r] += w;
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float w1 = warp_sum(s1[r]), w2 = warp_sum(s2[r]);
            if (lane == 0) {
                red[r * 64 + warp] = w1;
                red[r * 64 + 32 + warp] = w2;
            }
        }
        __syncthreads();
        float B[R], A[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float t1 = 0.f, t2 = 0.f;
            for (int w = 0; w < nwarps; ++w) {
                t1 += red[r * 64 + w];
                t2 += red[r * 64 + 32 + w];
            }
            // dx = (wdy - c2 - x_hat*c1)*rstd = wdy*rstd + (x - mean)*B + A
            const float c1 = rs[r] * t1 * a.inv_n, c2 = t2 * a.inv_n;
            B[r] = -rs[r] * rs[r] * c1;
            A[r] = -c2 * rs[r];
        }
        __syncthreads();  // red is rewritten by the next rows
        // pass 2: dx; dgamma / dbeta partials += dy*x_hat, dy
        for (int i = tid; i < nvmax; i += nthr) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (i < nv[r]) {
                    const int c0 = h[r] + i * V;
                    const size_t e0 = (size_t)(row0 + r) * N + c0;
                    float xf[V], df[V], o[V];
                    chunk_to_float<T>(ld_global_nc_v4(x + e0), xf);
                    chunk_to_float<T>(ld_global_nc_v4(dy + e0), df);
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float xc = xf[e] - mu[r];
                        const float w = df[e] * sg[vpad(c0 + e)];
                        o[e] = fmaf(w, rs[r], fmaf(xc, B[r], A[r]));
                        atomicAdd(sdg + vpad(c0 + e), df[e] * (xc * rs[r]));
                        atomicAdd(sdb + vpad(c0 + e), df[e]);
                    }
                    st_global_v4(dx + e0, float_to_chunk<T>(o));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (tid < h[r] + nt[r]) {
                const size_t base = (size_t)(row0 + r) * N;
                const int j = tid < h[r] ? tid : h[r] + nv[r] * V + (tid - h[r]);
                const float xc = to_f(x[base + j]) - mu[r], dv = to_f(dy[base + j]);
                const float w = dv * sg[vpad(j)];
                dx[base + j] = from_f<T>(fmaf(w, rs[r], fmaf(xc, B[r], A[r])));
                atomicAdd(sdg + vpad(j), dv * (xc * rs[r]));
                atomicAdd(sdb + vpad(j), dv);
            }
        }
    }
    pdl_launch_dependents();
    __syncthreads();  // every shared add of the partials is done
    if (ATOMIC) {
        pdl_wait();
        for (int j = tid; j < N; j += nthr) {
            atomicAdd(a.dg_out + j, sdg[vpad(j)]);
            if (a.db_out) atomicAdd(a.db_out + j, sdb[vpad(j)]);
        }
    } else {
        float *part = a.dg_out + (size_t)blockIdx.x * 2 * N;  // [dgamma | dbeta]
        for (int j = tid; j < N; j += nthr) {
            part[j] = sdg[vpad(j)];
            part[N + j] = sdb[vpad(j)];
        }
    }
}

template <typename T, bool ATOMIC, int R>
static cudaError_t launch_ln_gen_vec_t(const LnGenArgs &args, const GenericPlan &plan,
                                       cudaStream_t s, bool pdl) {
    auto kern = ln_bwd_generic_vec_kernel<T, ATOMIC, R>;
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

template <typename T, bool ATOMIC, bool SMEM_DW>
static cudaError_t launch_ln_gen_t(const LnGenArgs &args, const GenericPlan &plan,
                                   cudaStream_t s, bool pdl) {
    auto kern = ln_bwd_generic_kernel<T, ATOMIC, SMEM_DW>;
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
static cudaError_t launch_ln_gen_dt(const LnGenArgs &args, const GenericPlan &plan,
                                    cudaStream_t s, bool pdl) {
    if (plan.rows) {
        if (plan.atomic)
            return plan.rows == 4 ? launch_ln_gen_vec_t<T, true, 4>(args, plan, s, pdl)
                                  : launch_ln_gen_vec_t<T, true, 2>(args, plan, s, pdl);
        return plan.rows == 4 ? launch_ln_gen_vec_t<T, false, 4>(args, plan, s, pdl)
                              : launch_ln_gen_vec_t<T, false, 2>(args, plan, s, pdl);
    }
    if (plan.atomic) return launch_ln_gen_t<T, true, true>(args, plan, s, pdl);
    if (plan.smem_dw) return launch_ln_gen_t<T, false, true>(args, plan, s, pdl);
    return launch_ln_gen_t<T, false, false>(args, plan, s, pdl);
}

cudaError_t launch_ln_bwd_generic(const LnBwdProblem &p, const GenericPlan &plan,
                                  cudaStream_t s, bool pdl_after_zero) {
    LnGenArgs a;
    a.x = p.x;
    a.gamma = p.gamma;
    a.dy = p.dy;
    a.mean = p.mean;
    a.rstd = p.rstd;
    a.dx = p.dx;
    a.dg_out = plan.atomic ? p.dg_f32 : reinterpret_cast<float *>(p.ws + kWsHeaderBytes);
    a.db_out = plan.atomic ? p.db_f32 : nullptr;
    a.M = p.M;
    a.N = p.N;
    a.inv_n = 1.0f / (float)p.N;
    a.words = (int)vec_words(p.N);
    switch (p.dtype) {
    case kF32: return launch_ln_gen_dt<float>(a, plan, s, pdl_after_zero);
    case kF16: return launch_ln_gen_dt<__half>(a, plan, s, pdl_after_zero);
    case kBF16: return launch_ln_gen_dt<__nv_bfloat16>(a, plan, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
