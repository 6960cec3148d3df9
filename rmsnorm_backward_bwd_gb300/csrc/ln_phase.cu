// LayerNorm backward phase-class kernel: rows that are not 16-byte multiples
// (or whose base is off a 16-byte boundary), x, dy and dx at one alignment
// phase, rows of at most 1024 16-byte chunks.
//
// Same math as the LayerNorm row engine (FlyDSL issue #769, LayerNorm
// backward plan: dx = (wdy - c2 - x_hat*c1)*rstd with c1 = mean(x_hat*wdy),
// c2 = mean(wdy); dgamma += dy*x_hat, dbeta += dy). The work split is the
// RMSNorm phase-class kernel's: row r's alignment phase repeats with period
// P = 16 / gcd(16, N*s mod 16) rows, each CTA takes the rows of one residue
// class modulo P, so a thread owns the same columns in every row it touches.
// Gamma (packed), the row and the two partials stay in registers; the class's
// next row is loaded while the current one is computed; in atomic mode the
// partials go out through shared memory as 16-byte atomic adds.
#include "common.cuh"
#include "unaligned.cuh"
#include "launch.h"

namespace rn {

struct LnPhaseArgs {
    const void *x;
    const void *gamma;
    const void *dy;
    const float *mean;
    const float *rstd;
    void *dx;
    // scratch: partial rows [gridDim.x][2N] (dgamma | dbeta); atomic: the
    // outputs (16-byte aligned)
    float *dg_out;
    float *db_out;  // atomic mode only; nullable
    int64_t M;
    int N;
    float inv_n;
    int period;     // P
    int prefetch;   // 1: L2 prefetch of the row after the next one
};

// Padded length of the atomic mode's first staged partial: the second one
// starts 16-byte aligned.
__host__ __device__ __forceinline__ int ln_phase_stride(int N) { return (N + 3) & ~3; }

size_t ln_phase_smem_bytes(int N, bool atomic) {
    return atomic ? (size_t)2 * ln_phase_stride(N) * 4 : 0;
}

template <typename T, bool ATOMIC, int J>
__global__ void __launch_bounds__(512) ln_bwd_phase_kernel(const LnPhaseArgs a) {
    constexpr int S = sizeof(T), V = 16 / S;
    __shared__ float red[2][2][16];  // [row parity][sum][warp]
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N, P = a.period;
    const int cls = (int)(blockIdx.x % (unsigned)P);
    const int64_t rank = blockIdx.x / (unsigned)P;
    const int64_t nper = ((int64_t)gridDim.x - cls + P - 1) / P;  // CTAs of this class

    // the class's split (address arithmetic on row cls; nothing is read there)
    const uintptr_t start = reinterpret_cast<uintptr_t>(a.x) + (uintptr_t)cls * (uintptr_t)N * S;
    int h = (int)(((16u - (unsigned)(start & 15u)) & 15u) / S);
    if (h > N) h = N;
    const int nv = (N - h) / V, tail = N - h - nv * V;

    bool own[J];
    int col[J];
    uint4 gv[J];
    float dgp[J][V], dbp[J][V];
#pragma unroll
    for (int k = 0; k < J; ++k) {
        const int i = tid + k * nthr;
        own[k] = i < nv;
        col[k] = h + i * V;
        gv[k] = own[k] ? gather_chunk<T>(g + col[k]) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < V; ++e) dgp[k][e] = dbp[k][e] = 0.f;
    }
    const bool e_own = tid < h + tail;
    const int je = tid < h ? tid : h + nv * V + (tid - h);
    const float ge = e_own ? to_f(g[je]) : 0.f;
    float dge = 0.f, dbe = 0.f;

    auto load = [&](int64_t row, uint4 (&xv)[J], uint4 (&dv)[J], float &xe, float &de) {
        const size_t base = (size_t)row * N;
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                xv[k] = ld_global_nc_v4(x + base + col[k]);
                dv[k] = ld_global_nc_v4(dy + base + col[k]);
            }
        }
        if (e_own) {
            xe = to_f(x[base + je]);
            de = to_f(dy[base + je]);
        }
    };

    uint4 xc[J], dc[J];
#pragma unroll
    for (int k = 0; k < J; ++k) xc[k] = dc[k] = make_uint4(0, 0, 0, 0);
    float xec = 0.f, dec = 0.f;
    int64_t row = cls + rank * P;
    if (row < a.M) load(row, xc, dc, xec, dec);
    int buf = 0;
    while (row < a.M) {
        const int64_t nrow = row + nper * P;
        uint4 xn[J], dn[J];
#pragma unroll
        for (int k = 0; k < J; ++k) xn[k] = dn[k] = make_uint4(0, 0, 0, 0);
        float xen = 0.f, den = 0.f;
        if (nrow < a.M) load(nrow, xn, dn, xen, den);
        // the row after that into L2 (when the planner asks): its loads next iteration then
        // wait on L2, not DRAM
        const int64_t prow = nrow + nper * P;
        if (a.prefetch && prow < a.M) {
            const size_t pbase = (size_t)prow * N;
#pragma unroll
            for (int k = 0; k < J; ++k) {
                if (own[k]) {
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(x + pbase + col[k]));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(dy + pbase + col[k]));
                }
            }
        }
        const size_t base = (size_t)row * N;
        const float mu = __ldg(a.mean + row), rs = __ldg(a.rstd + row);

        // pass 1: sum (x - mean)*wdy and sum wdy
        float s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                float xf[V], df[V], gf[V];
                chunk_to_float<T>(xc[k], xf);
                chunk_to_float<T>(dc[k], df);
                chunk_to_float<T>(gv[k], gf);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float w = df[e] * gf[e];
                    s1 = fmaf(xf[e] - mu, w, s1);
                    s2 += w;
                }
            }
        }
        if (e_own) {
            const float w = dec * ge;
            s1 = fmaf(xec - mu, w, s1);
            s2 += w;
        }
        s1 = warp_sum(s1);
        s2 = warp_sum(s2);
        if (lane == 0) {
            red[buf][0][warp] = s1;
            red[buf][1][warp] = s2;
        }
        __syncthreads();  // also orders the reads of red[buf] two rows back before these writes
        float t1 = 0.f, t2 = 0.f;
        for (int w = 0; w < nwarps; ++w) {
            t1 += red[buf][0][w];
            t2 += red[buf][1][w];
        }
        buf ^= 1;
        // dx = (wdy - c2 - x_hat*c1)*rstd = wdy*rstd + (x - mean)*B + A
        const float c1 = rs * t1 * a.inv_n, c2 = t2 * a.inv_n;
        const float B = -rs * rs * c1, A = -c2 * rs;

        // pass 2: dx; dgamma / dbeta partials += dy*x_hat, dy
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                float xf[V], df[V], gf[V], o[V];
                chunk_to_float<T>(xc[k], xf);
                chunk_to_float<T>(dc[k], df);
                chunk_to_float<T>(gv[k], gf);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float xcen = xf[e] - mu;
                    o[e] = fmaf(df[e] * gf[e], rs, fmaf(xcen, B, A));
                    dgp[k][e] = fmaf(df[e], xcen * rs, dgp[k][e]);
                    dbp[k][e] += df[e];
                }
                st_global_v4(dx + base + col[k], float_to_chunk<T>(o));
            }
        }
        if (e_own) {
            const float xcen = xec - mu;
            dx[base + je] = from_f<T>(fmaf(dec * ge, rs, fmaf(xcen, B, A)));
            dge = fmaf(dec, xcen * rs, dge);
            dbe += dec;
        }
#pragma unroll
        for (int k = 0; k < J; ++k) {
            xc[k] = xn[k];
            dc[k] = dn[k];
        }
        xec = xen;
        dec = den;
        row = nrow;
    }
    pdl_launch_dependents();
    if (ATOMIC) {
        extern __shared__ __align__(16) float sdw[];  // dgamma | dbeta, each ln_phase_stride(N)
        float *sdg = sdw, *sdb = sdw + ln_phase_stride(N);
#pragma unroll
        for (int k = 0; k < J; ++k)
            if (own[k])
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    sdg[col[k] + e] = dgp[k][e];
                    sdb[col[k] + e] = dbp[k][e];
                }
        if (e_own) {
            sdg[je] = dge;
            sdb[je] = dbe;
        }
        __syncthreads();
        pdl_wait();
        const int n4 = N >> 2;
        for (int q = tid; q < n4; q += nthr) {
            atomicAdd(reinterpret_cast<float4 *>(a.dg_out) + q, reinterpret_cast<const float4 *>(sdg)[q]);
            if (a.db_out)
                atomicAdd(reinterpret_cast<float4 *>(a.db_out) + q, reinterpret_cast<const float4 *>(sdb)[q]);
        }
        for (int j = (n4 << 2) + tid; j < N; j += nthr) {
            atomicAdd(a.dg_out + j, sdg[j]);
            if (a.db_out) atomicAdd(a.db_out + j, sdb[j]);
        }
    } else {
        float *part = a.dg_out + (size_t)blockIdx.x * 2 * N;  // [dgamma | dbeta]
#pragma unroll
        for (int k = 0; k < J; ++k)
            if (own[k])
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    part[col[k] + e] = dgp[k][e];
                    part[N + col[k] + e] = dbp[k][e];
                }
        if (e_own) {
            part[je] = dge;
            part[N + je] = dbe;
        }
    }
}

template <typename T>
static const void *ln_phase_kernel_ptr(bool atomic, int cpt) {
    if (cpt == 2)
        return atomic ? (const void *)ln_bwd_phase_kernel<T, true, 2>
                      : (const void *)ln_bwd_phase_kernel<T, false, 2>;
    return atomic ? (const void *)ln_bwd_phase_kernel<T, true, 1>
                  : (const void *)ln_bwd_phase_kernel<T, false, 1>;
}

static const void *ln_phase_kernel_for(int dtype, bool atomic, int cpt) {
    return dtype == kF32 ? ln_phase_kernel_ptr<float>(atomic, cpt)
         : dtype == kF16 ? ln_phase_kernel_ptr<__half>(atomic, cpt)
                         : ln_phase_kernel_ptr<__nv_bfloat16>(atomic, cpt);
}

// Resident CTAs per SM of one instance at a CTA size (a multiple of 32 up to
// 512) with its dynamic shared memory; cached per instance, size and
// shared-memory bytes in 4 KB steps.
int ln_phase_blocks_per_sm(int dtype, bool atomic, int cpt, int threads, size_t smem) {
    static int cache[3][2][2][17][17];
    if (dtype < 0 || dtype > 2 || threads < 32 || threads > 512 || (threads & 31)) return 1;
    const size_t step = (smem + 4095) / 4096;
    if (step > 16) return 1;
    int &c = cache[dtype][atomic][cpt == 2][threads >> 5][step];
    if (c > 0) return c;
    const void *k = ln_phase_kernel_for(dtype, atomic, cpt);
    const size_t query = step * 4096;
    int n = 0;
    if (ensure_smem_attr(k, query) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, query) != cudaSuccess ||
        n < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    c = n;
    return n;
}

template <typename T, bool ATOMIC, int J>
static cudaError_t launch_ln_phase_t(const LnPhaseArgs &args, const GenericPlan &plan,
                                     cudaStream_t s, bool pdl) {
    auto kern = ln_bwd_phase_kernel<T, ATOMIC, J>;
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
static cudaError_t launch_ln_phase_dt(const LnPhaseArgs &args, const GenericPlan &plan,
                                      cudaStream_t s, bool pdl) {
    if (plan.atomic)
        return plan.phase == 2 ? launch_ln_phase_t<T, true, 2>(args, plan, s, pdl)
                               : launch_ln_phase_t<T, true, 1>(args, plan, s, pdl);
    return plan.phase == 2 ? launch_ln_phase_t<T, false, 2>(args, plan, s, pdl)
                           : launch_ln_phase_t<T, false, 1>(args, plan, s, pdl);
}

cudaError_t launch_ln_bwd_phase(const LnBwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                                bool pdl_after_zero) {
    LnPhaseArgs a;
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
    a.period = phase_period(p.N, p.dtype);
    a.prefetch = plan.prefetch ? 1 : 0;
    // a residue class without a CTA would leave its rows unwritten
    if (p.M > 0 && plan.grid < (p.M < a.period ? p.M : a.period)) return cudaErrorInvalidValue;
    if (plan.atomic && plan.smem < ln_phase_smem_bytes(p.N, true)) return cudaErrorInvalidValue;
    switch (p.dtype) {
    case kF32: return launch_ln_phase_dt<float>(a, plan, s, pdl_after_zero);
    case kF16: return launch_ln_phase_dt<__half>(a, plan, s, pdl_after_zero);
    case kBF16: return launch_ln_phase_dt<__nv_bfloat16>(a, plan, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
