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
#include "unaligned.cuh"
#include "launch.h"

namespace rn {

size_t generic_smem_bytes(int N, bool smem_dw) {
    return 256 + (smem_dw ? (size_t)N * 4 : 0);
}

size_t generic_vec_smem_bytes(int N) { return 512 + 2 * 4 * vec_words(N); }

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
    int words;       // vector variant: padded length of each shared array
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

// Vector variant for rows whose start is not 16-byte aligned (N*s not a
// multiple of 16) when x, dy, dx and dresidual_out share one alignment phase
// (their base addresses agree modulo 16, as for tensors from one allocator).
// Each row splits into a head (the elements before its first 16-byte
// boundary), whole 16-byte chunks, and a tail; chunks move with 128-bit loads
// and stores, head and tail one element at a time. R rows are in flight per
// CTA iteration (their chunk loads issued together), and their sums are
// reduced together. A column's owner thread changes from row to row, so the
// CTA's weight-gradient partial (shared memory) takes shared-memory atomic
// adds. gamma is staged in shared memory as fp32. Both shared arrays are
// padded by one word per 32 columns: a warp's lanes touch columns 16/s apart,
// which without the pad share banks.
struct RowGeom {
    int h;     // head elements
    int nv;    // whole 16-byte chunks after the head
    int tail;  // elements after the chunks
};

template <typename T>
__device__ __forceinline__ RowGeom row_geom(const void *base, int64_t row, int N) {
    constexpr int S = sizeof(T), V = 16 / S;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(base) + (uintptr_t)row * N * S;
    int h = (int)(((16u - (unsigned)(addr & 15u)) & 15u) / S);
    if (h > N) h = N;
    RowGeom g;
    g.h = h;
    g.nv = (N - h) / V;
    g.tail = N - h - g.nv * V;
    return g;
}

// 4 rows in flight run with 256 threads (short rows), 2 rows with up to 512.
template <int R> struct GenVecBounds {
    static constexpr int kMaxThreads = R == 4 ? 256 : 512;
};

template <typename T, bool HAS_DRES, bool ATOMIC, int R>
__global__ void __launch_bounds__(GenVecBounds<R>::kMaxThreads, 2)
    bwd_generic_vec_kernel(const GenArgs a) {
    constexpr int V = 16 / (int)sizeof(T);
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);          // [R][32] warp sums
    float *sg = reinterpret_cast<float *>(smem + 512);     // gamma, fp32, padded columns
    float *sdw = sg + a.words;                             // weight-gradient partial, padded
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N;

    for (int j = tid; j < N; j += nthr) {
        sdw[vpad(j)] = 0.f;
        sg[vpad(j)] = to_f(g[j]);
    }
    __syncthreads();

    for (int64_t row0 = (int64_t)blockIdx.x * R; row0 < a.M; row0 += (int64_t)gridDim.x * R) {
        RowGeom geo[R];
        float sum[R], rs[R];
        int nvmax = 0;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = row0 + r;
            const bool ok = row < a.M;
            geo[r] = ok ? row_geom<T>(a.x, row, N) : RowGeom{0, 0, 0};
            rs[r] = ok ? __ldg(a.rstd + row) : 0.f;
            sum[r] = 0.f;
            if (geo[r].nv > nvmax) nvmax = geo[r].nv;
        }
        // pass 1: sum_j x_j*dy_j*gamma_j of each row
        for (int i = tid; i < nvmax; i += nthr) {
            uint4 xv[R], dv[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (i < geo[r].nv) {
                    const size_t e0 = (size_t)(row0 + r) * N + geo[r].h + (size_t)i * V;
                    xv[r] = ld_global_nc_v4(x + e0);
                    dv[r] = ld_global_nc_v4(dy + e0);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (i < geo[r].nv) {
                    float xf[V], df[V];
                    chunk_to_float<T>(xv[r], xf);
                    chunk_to_float<T>(dv[r], df);
                    const int c0 = geo[r].h + i * V;
#pragma unroll
                    for (int e = 0; e < V; ++e) sum[r] = fmaf(xf[e], df[e] * sg[vpad(c0 + e)], sum[r]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            // head and tail (fewer than V elements each)
            const size_t base = (size_t)(row0 + r) * N;
            const int j = tid < geo[r].h ? tid : geo[r].h + geo[r].nv * V + (tid - geo[r].h);
            if (tid < geo[r].h + geo[r].tail)
                sum[r] = fmaf(to_f(x[base + j]), to_f(dy[base + j]) * sg[vpad(j)], sum[r]);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float w = warp_sum(sum[r]);
            if (lane == 0) red[r * 32 + warp] = w;
        }
        __syncthreads();
        float c1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float tot = 0.f;
            for (int w = 0; w < nwarps; ++w) tot += red[r * 32 + w];
            c1[r] = rs[r] * tot * a.inv_n;
        }
        __syncthreads();  // red is rewritten by the next rows
        // pass 2: dx = (wdy - x_hat*c1)*rstd (+ dres); dweight partial += dy*x_hat
        for (int i = tid; i < nvmax; i += nthr) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (i < geo[r].nv) {
                    const int c0 = geo[r].h + i * V;
                    const size_t e0 = (size_t)(row0 + r) * N + c0;
                    float xf[V], df[V], o[V];
                    chunk_to_float<T>(ld_global_nc_v4(x + e0), xf);
                    chunk_to_float<T>(ld_global_nc_v4(dy + e0), df);
                    float rf[V];
                    if (HAS_DRES) chunk_to_float<T>(*reinterpret_cast<const uint4 *>(dres + e0), rf);
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float xh = xf[e] * rs[r];
                        o[e] = fmaf(-xh, c1[r], df[e] * sg[vpad(c0 + e)]) * rs[r];
                        if (HAS_DRES) o[e] += rf[e];
                        atomicAdd(sdw + vpad(c0 + e), df[e] * xh);
                    }
                    st_global_v4(dx + e0, float_to_chunk<T>(o));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const size_t base = (size_t)(row0 + r) * N;
            const int j = tid < geo[r].h ? tid : geo[r].h + geo[r].nv * V + (tid - geo[r].h);
            if (tid < geo[r].h + geo[r].tail) {
                const float xh = to_f(x[base + j]) * rs[r], dv = to_f(dy[base + j]);
                float d = fmaf(-xh, c1[r], dv * sg[vpad(j)]) * rs[r];
                if (HAS_DRES) d += to_f(dres[base + j]);
                dx[base + j] = from_f<T>(d);
                atomicAdd(sdw + vpad(j), dv * xh);
            }
        }
    }
    pdl_launch_dependents();
    __syncthreads();  // every shared add of the partial is done
    if (ATOMIC) {
        pdl_wait();
        for (int j = tid; j < N; j += nthr) atomicAdd(a.dw_out + j, sdw[vpad(j)]);
    } else {
        float *part = a.dw_out + (size_t)blockIdx.x * N;
        for (int j = tid; j < N; j += nthr) part[j] = sdw[vpad(j)];
    }
}

template <typename T, bool HAS_DRES, bool ATOMIC, int R>
static cudaError_t launch_gen_vec_t(const GenArgs &args, const GenericPlan &plan, cudaStream_t s,
                                    bool pdl) {
    auto kern = bwd_generic_vec_kernel<T, HAS_DRES, ATOMIC, R>;
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
static cudaError_t launch_gen_vec_r(const GenArgs &args, const GenericPlan &plan, cudaStream_t s,
                                    bool pdl) {
    return plan.rows == 4 ? launch_gen_vec_t<T, HAS_DRES, ATOMIC, 4>(args, plan, s, pdl)
                          : launch_gen_vec_t<T, HAS_DRES, ATOMIC, 2>(args, plan, s, pdl);
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
    if (plan.rows > 0) {
        if (plan.atomic)
            return has_dres ? launch_gen_vec_r<T, true, true>(args, plan, s, pdl)
                            : launch_gen_vec_r<T, false, true>(args, plan, s, pdl);
        return has_dres ? launch_gen_vec_r<T, true, false>(args, plan, s, pdl)
                        : launch_gen_vec_r<T, false, false>(args, plan, s, pdl);
    }
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
    a.words = (int)vec_words(p.N);
    const bool has_dres = p.dres != nullptr;
    switch (p.dtype) {
    case kF32: return launch_gen_dt<float>(a, plan, has_dres, s, pdl_after_zero);
    case kF16: return launch_gen_dt<__half>(a, plan, has_dres, s, pdl_after_zero);
    case kBF16: return launch_gen_dt<__nv_bfloat16>(a, plan, has_dres, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
