// Backward phase-class kernel: rows that are not 16-byte multiples (or whose
// base is off a 16-byte boundary), x, dy, dx and dresidual_out at one
// alignment phase, rows of at most 2048 whole 16-byte chunks.
//
// Same math as the row engine (FlyDSL issue #769 "Math"; fused-add from
// PR #800 "What's included"). Row r starts at byte r*N*s past the base, so its
// alignment phase repeats with period P = 16 / gcd(16, N*s mod 16) rows (P = 1
// when only the base is off a boundary). Each CTA takes the rows of one
// residue class modulo P. Within a class every row splits the same way into
// head elements, whole 16-byte chunks and tail elements, so a thread owns the
// same columns in every row it touches. Its gamma chunks (packed, as loaded)
// and its weight-gradient partial stay in registers, as in the row engine
// (with four 16-bit chunks a thread the gamma chunks move to shared memory).
// The rows stay in registers between the two passes: a CTA takes R rows of
// its class per iteration (2, or 1 with four chunks a thread) under one CTA
// barrier, and the class's next R rows are loaded while the current ones are
// computed. The chunk arithmetic is the row engine's packed-pair RowMath. The
// generic vector kernel, by
// contrast, lets any CTA take any row, so a column's owner changes with the
// row's phase and gamma and the partial live in shared memory.
#include "common.cuh"
#include "launch.h"
#include "row_math.cuh"
#include "unaligned.cuh"

namespace rn {

// Ask L2 to fetch the line holding p (no register result, no completion to
// wait for; p must be a valid global address).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

struct PhaseArgs {
    const void *x;
    const void *gamma;
    const void *dy;
    const float *rstd;
    const void *dres;
    void *dx;
    float *dw_out;   // scratch: partial rows [gridDim.x][N]; atomic: dweight_f32 (16-byte aligned)
    int64_t M;
    int N;
    float inv_n;
    int period;      // P
    int prefetch;    // 1: L2 prefetch of the rows two iterations ahead
};

int phase_period(int N, int dtype) {
    const int d = (int)(((int64_t)N * elem_bytes(dtype)) & 15);
    if (d == 0) return 1;
    int g = 16, b = d;  // gcd(16, d)
    while (b) {
        const int t = g % b;
        g = b;
        b = t;
    }
    return 16 / g;
}

template <typename T, bool HAS_DRES, bool ATOMIC, int J, int R>
__global__ void __launch_bounds__(512) bwd_phase_kernel(const PhaseArgs a) {
    constexpr int S = sizeof(T), V = 16 / S;
    constexpr int P2 = RowMath<T>::kPairs;  // fp32 pairs per chunk
    // gamma also as fp32 pairs when the math needs it or when that fits
    constexpr bool kGammaF = RowMath<T>::kNeedsGammaF || J * V <= 8;
    __shared__ float red[2][R][16];  // warp sums of the R rows, alternating between iterations
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N, P = a.period;
    const int cls = (int)(blockIdx.x % (unsigned)P);
    const int64_t rank = blockIdx.x / (unsigned)P;
    const int64_t nper = ((int64_t)gridDim.x - cls + P - 1) / P;  // CTAs of this class
    // this CTA's rows: row0, row0 + rstride, ...; R of them per iteration
    const int64_t rstride = nper * P;
    const int64_t row0 = cls + rank * P;

    // the class's split (address arithmetic on row cls; nothing is read there)
    const uintptr_t start = reinterpret_cast<uintptr_t>(a.x) + (uintptr_t)cls * (uintptr_t)N * S;
    int h = (int)(((16u - (unsigned)(start & 15u)) & 15u) / S);
    if (h > N) h = N;
    const int nv = (N - h) / V, tail = N - h - nv * V;

    // this thread's chunks (i = tid + k*nthr) and its head or tail element. With four 16-bit
    // chunks a thread the packed gamma chunks wait in dynamic shared memory (at i), not in
    // registers: there are not enough.
    constexpr bool kGammaSmem = J == 4 && !kGammaF;
    extern __shared__ __align__(16) uint4 dyn[];
    bool own[J];
    int col[J];
    uint4 gv[kGammaSmem ? 1 : J];
    f32x2 g2[kGammaF ? J : 1][kGammaF ? P2 : 1];
    f32x2 acc2[J][P2];
#pragma unroll
    for (int k = 0; k < J; ++k) {
        const int i = tid + k * nthr;
        own[k] = i < nv;
        col[k] = h + i * V;
        const uint4 gk = own[k] ? gather_chunk<T>(g + col[k]) : make_uint4(0, 0, 0, 0);
        if (kGammaSmem) dyn[i] = gk;
        else gv[kGammaSmem ? 0 : k] = gk;
        if (kGammaF) {
            float gf[V];
            chunk_to_float<T>(gk, gf);
#pragma unroll
            for (int q = 0; q < P2; ++q)
                g2[kGammaF ? k : 0][kGammaF ? q : 0] = f2_make(gf[2 * q], gf[2 * q + 1]);
        }
#pragma unroll
        for (int q = 0; q < P2; ++q) acc2[k][q] = f2_make(0.f, 0.f);
    }
    const bool e_own = tid < h + tail;
    const int je = tid < h ? tid : h + nv * V + (tid - h);
    const float ge = e_own ? to_f(g[je]) : 0.f;
    float dwe = 0.f;

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

    uint4 xc[R][J], dc[R][J];
    float xec[R], dec[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int k = 0; k < J; ++k) xc[r][k] = dc[r][k] = make_uint4(0, 0, 0, 0);
        xec[r] = dec[r] = 0.f;
        const int64_t row = row0 + r * rstride;
        if (row < a.M) load(row, xc[r], dc[r], xec[r], dec[r]);
    }
    int buf = 0;
    for (int64_t rb = row0; rb < a.M; rb += R * rstride) {
        // the next iteration's rows, in flight while these are computed
        uint4 xn[R][J], dn[R][J];
        float xen[R], den[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int k = 0; k < J; ++k) xn[r][k] = dn[r][k] = make_uint4(0, 0, 0, 0);
            xen[r] = den[r] = 0.f;
            const int64_t nrow = rb + (R + r) * rstride;
            if (nrow < a.M) load(nrow, xn[r], dn[r], xen[r], den[r]);
        }
        // the rows after those into L2 (when the planner asks): their loads next iteration
        // then wait on L2, not DRAM (the rows in flight in registers are all the registers
        // allow)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t prow = rb + (2 * R + r) * rstride;
            if (a.prefetch && prow < a.M) {
                const size_t base = (size_t)prow * N;
#pragma unroll
                for (int k = 0; k < J; ++k) {
                    if (own[k]) {
                        prefetch_l2(x + base + col[k]);
                        prefetch_l2(dy + base + col[k]);
                        if (HAS_DRES) prefetch_l2(dres + base + col[k]);
                    }
                }
            }
        }

        // dresidual_out (a plain load: dx may overwrite it) and rstd of these rows; with four
        // chunks a thread dresidual_out is loaded in pass 2 (registers)
        constexpr bool kEarlyDres = HAS_DRES && J <= 2;
        uint4 rv[kEarlyDres ? R : 1][J];
        float re[R], rs[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = rb + r * rstride;
            const bool live = row < a.M;
            const size_t base = (size_t)row * N;
            re[r] = 0.f;
            if (kEarlyDres) {
#pragma unroll
                for (int k = 0; k < J; ++k)
                    rv[kEarlyDres ? r : 0][k] =
                        own[k] && live ? *reinterpret_cast<const uint4 *>(dres + base + col[k])
                                       : make_uint4(0, 0, 0, 0);
            }
            if (HAS_DRES && e_own && live) re[r] = to_f(dres[base + je]);
            rs[r] = live ? __ldg(a.rstd + row) : 0.f;
        }

        // pass 1: sum_j x_j*dy_j*gamma_j of each row (a row past M sums zeros)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            f32x2 part2 = f2_make(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < J; ++k)
                if (own[k])
                    part2 = RowMath<T>::pass1(xc[r][k], dc[r][k],
                                              kGammaSmem ? dyn[tid + k * nthr] : gv[kGammaSmem ? 0 : k],
                                              kGammaF ? g2[kGammaF ? k : 0] : nullptr, part2);
            float lo, hi;
            f2_split(part2, lo, hi);
            float s = lo + hi;
            if (e_own) s = fmaf(xec[r] * dec[r], ge, s);
            s = warp_sum(s);
            if (lane == 0) red[buf][r][warp] = s;
        }
        __syncthreads();  // also orders the reads of red[buf] two iterations back before these writes

        // pass 2: dx = wdy*rstd + x*b with b = -rstd^2*c1 (+ dres); partial += dy*x_hat
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = rb + r * rstride;
            if (row >= a.M) break;  // uniform across the CTA
            float tot = 0.f;
            for (int w = 0; w < nwarps; ++w) tot += red[buf][r][w];
            const float c1 = rs[r] * tot * a.inv_n;
            const float b = -rs[r] * rs[r] * c1;
            const f32x2 rs2 = f2_make(rs[r], rs[r]), b2 = f2_make(b, b);
            const size_t base = (size_t)row * N;
#pragma unroll
            for (int k = 0; k < J; ++k) {
                if (own[k]) {
                    uint4 rk = make_uint4(0, 0, 0, 0);
                    if (kEarlyDres) rk = rv[kEarlyDres ? r : 0][k];
                    else if (HAS_DRES) rk = *reinterpret_cast<const uint4 *>(dres + base + col[k]);
                    const uint4 o = RowMath<T>::template pass2<HAS_DRES>(
                        xc[r][k], dc[r][k], rk,
                        kGammaSmem ? dyn[tid + k * nthr] : gv[kGammaSmem ? 0 : k],
                        kGammaF ? g2[kGammaF ? k : 0] : nullptr, rs2, b2, acc2[k]);
                    st_global_v4(dx + base + col[k], o);
                }
            }
            if (e_own) {
                float d = fmaf(xec[r], b, (dec[r] * ge) * rs[r]);
                if (HAS_DRES) d += re[r];
                dx[base + je] = from_f<T>(d);
                dwe = fmaf(xec[r] * dec[r], rs[r], dwe);
            }
        }
        buf ^= 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int k = 0; k < J; ++k) {
                xc[r][k] = xn[r][k];
                dc[r][k] = dn[r][k];
            }
            xec[r] = xen[r];
            dec[r] = den[r];
        }
    }
    pdl_launch_dependents();
    if (ATOMIC) {
        // The partial goes through shared memory so that every class adds it
        // with 16-byte atomics (dweight_f32 is 16-byte aligned; a class's own
        // columns start at any element). It takes the place of the gamma chunks.
        float *sdw = reinterpret_cast<float *>(dyn);  // N floats
        if (kGammaSmem) __syncthreads();  // every thread is done with the gamma chunks
#pragma unroll
        for (int k = 0; k < J; ++k)
            if (own[k])
#pragma unroll
                for (int q = 0; q < P2; ++q)
                    f2_split(acc2[k][q], sdw[col[k] + 2 * q], sdw[col[k] + 2 * q + 1]);
        if (e_own) sdw[je] = dwe;
        __syncthreads();
        pdl_wait();
        const int n4 = N >> 2;
        for (int q = tid; q < n4; q += nthr)
            atomicAdd(reinterpret_cast<float4 *>(a.dw_out) + q, reinterpret_cast<const float4 *>(sdw)[q]);
        for (int j = (n4 << 2) + tid; j < N; j += nthr) atomicAdd(a.dw_out + j, sdw[j]);
    } else {
        float *part = a.dw_out + (size_t)blockIdx.x * N;
#pragma unroll
        for (int k = 0; k < J; ++k)
            if (own[k])
#pragma unroll
                for (int q = 0; q < P2; ++q)
                    f2_split(acc2[k][q], part[col[k] + 2 * q], part[col[k] + 2 * q + 1]);
        if (e_own) part[je] = dwe;
    }
}

template <typename T, bool HAS_DRES, bool ATOMIC, int J, int R>
static cudaError_t launch_phase_t(const PhaseArgs &args, const GenericPlan &plan, cudaStream_t s,
                                  bool pdl) {
    auto kern = bwd_phase_kernel<T, HAS_DRES, ATOMIC, J, R>;
    // the atomic mode stages N floats in dynamic shared memory: raise the
    // kernel's cap when a plan asks for more than the default 48 KB
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

template <typename T, bool HAS_DRES, bool ATOMIC>
static cudaError_t launch_phase_j(const PhaseArgs &args, const GenericPlan &plan, cudaStream_t s,
                                  bool pdl) {
    // four chunks a thread: one row per iteration (two would not fit the registers)
    if (plan.phase == 4) return launch_phase_t<T, HAS_DRES, ATOMIC, 4, 1>(args, plan, s, pdl);
    if (plan.phase_rows == 2)
        return plan.phase == 2 ? launch_phase_t<T, HAS_DRES, ATOMIC, 2, 2>(args, plan, s, pdl)
                               : launch_phase_t<T, HAS_DRES, ATOMIC, 1, 2>(args, plan, s, pdl);
    return plan.phase == 2 ? launch_phase_t<T, HAS_DRES, ATOMIC, 2, 1>(args, plan, s, pdl)
                           : launch_phase_t<T, HAS_DRES, ATOMIC, 1, 1>(args, plan, s, pdl);
}

template <typename T>
static cudaError_t launch_phase_dt(const PhaseArgs &args, const GenericPlan &plan, bool has_dres,
                                   cudaStream_t s, bool pdl) {
    if (plan.atomic)
        return has_dres ? launch_phase_j<T, true, true>(args, plan, s, pdl)
                        : launch_phase_j<T, false, true>(args, plan, s, pdl);
    return has_dres ? launch_phase_j<T, true, false>(args, plan, s, pdl)
                    : launch_phase_j<T, false, false>(args, plan, s, pdl);
}

template <typename T, int R>
static const void *phase_kernel_ptr_r(bool dres, bool atomic, int cpt) {
    if (cpt == 4)
        return dres ? (atomic ? (const void *)bwd_phase_kernel<T, true, true, 4, 1>
                              : (const void *)bwd_phase_kernel<T, true, false, 4, 1>)
                    : (atomic ? (const void *)bwd_phase_kernel<T, false, true, 4, 1>
                              : (const void *)bwd_phase_kernel<T, false, false, 4, 1>);
    if (cpt == 2)
        return dres ? (atomic ? (const void *)bwd_phase_kernel<T, true, true, 2, R>
                              : (const void *)bwd_phase_kernel<T, true, false, 2, R>)
                    : (atomic ? (const void *)bwd_phase_kernel<T, false, true, 2, R>
                              : (const void *)bwd_phase_kernel<T, false, false, 2, R>);
    return dres ? (atomic ? (const void *)bwd_phase_kernel<T, true, true, 1, R>
                          : (const void *)bwd_phase_kernel<T, true, false, 1, R>)
                : (atomic ? (const void *)bwd_phase_kernel<T, false, true, 1, R>
                          : (const void *)bwd_phase_kernel<T, false, false, 1, R>);
}

template <typename T>
static const void *phase_kernel_ptr(bool dres, bool atomic, int cpt, int rows) {
    return rows == 2 ? phase_kernel_ptr_r<T, 2>(dres, atomic, cpt)
                     : phase_kernel_ptr_r<T, 1>(dres, atomic, cpt);
}

// Resident CTAs per SM of one instance at a CTA size (a multiple of 32 up to
// 512), from the occupancy calculator without dynamic shared memory (the
// atomic mode's N floats, at most 33 KB, leave room for the 2 CTAs per SM the
// planner takes at most); cached per instance and size.
int phase_blocks_per_sm(int dtype, bool dres, bool atomic, int cpt, int rows, int threads) {
    static int cache[3][2][2][3][2][17];
    if (dtype < 0 || dtype > 2 || threads < 32 || threads > 512 || (threads & 31)) return 1;
    int &c = cache[dtype][dres][atomic][cpt == 4 ? 2 : cpt == 2][rows == 2][threads >> 5];
    if (c > 0) return c;
    const void *k = dtype == kF32 ? phase_kernel_ptr<float>(dres, atomic, cpt, rows)
                  : dtype == kF16 ? phase_kernel_ptr<__half>(dres, atomic, cpt, rows)
                                  : phase_kernel_ptr<__nv_bfloat16>(dres, atomic, cpt, rows);
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, 0) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    c = n;
    return n;
}

cudaError_t launch_bwd_phase(const BwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                             bool pdl_after_zero) {
    PhaseArgs a;
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
    a.period = phase_period(p.N, p.dtype);
    a.prefetch = plan.prefetch ? 1 : 0;
    // a residue class without a CTA would leave its rows unwritten
    if (p.M > 0 && plan.grid < (p.M < a.period ? p.M : a.period)) return cudaErrorInvalidValue;
    if (plan.atomic && plan.smem < (size_t)p.N * 4) return cudaErrorInvalidValue;
    if (plan.phase == 4 && p.dtype != kF32 && plan.smem < (size_t)plan.threads * 4 * 16)
        return cudaErrorInvalidValue;
    if (plan.phase_rows != 1 && plan.phase_rows != 2) return cudaErrorInvalidValue;
    const bool has_dres = p.dres != nullptr;
    switch (p.dtype) {
    case kF32: return launch_phase_dt<float>(a, plan, has_dres, s, pdl_after_zero);
    case kF16: return launch_phase_dt<__half>(a, plan, has_dres, s, pdl_after_zero);
    case kBF16: return launch_phase_dt<__nv_bfloat16>(a, plan, has_dres, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
