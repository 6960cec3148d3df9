// Backward row engine (aligned rows): RMSNorm and fused-add RMSNorm backward.
//
// Math per row (FlyDSL issue #769, section "Math"): with x_hat = x*rstd and
// wdy = dy*gamma, c1 = mean_j(x_hat*wdy) and dx = (wdy - x_hat*c1)*rstd; the
// weight gradient sums dy*x_hat over rows. Fused-add (PR #800, "What's
// included"): the same on the saved `added`, plus dresidual_out on dx.
//
// Design (sm_103a):
//   * Persistent grid, one CTA per SM. A CTA holds `teams` teams; a team of
//     team_threads threads owns one row at a time. Team t of CTA b walks rows
//     b*teams + t, then strides by gridDim.x*teams.
//   * Each team keeps a ring of `stages` shared-memory slots. Its leader
//     thread fills a slot with one bulk asynchronous copy per tensor row
//     (x|added, dy, [dresidual_out]) completing on the slot's mbarrier, so
//     several rows per team are in flight while the current row is reduced.
//     Every row is read from HBM exactly once.
//   * Thread tt of a team owns 16-byte chunks tt, tt+team_threads, ... of the
//     row (consecutive threads -> consecutive 16 B: conflict-free shared
//     reads, coalesced 128-bit dx stores). It keeps those chunks in registers
//     across the c1 reduction (warp shuffles, then one named barrier across
//     the team's warps), so dx needs no second read.
//   * The weight-gradient partial of the thread's columns lives in fp32
//     registers for every row the team handles; at the end the CTA's teams
//     add theirs in a fixed order in shared memory and the CTA either stores
//     one partial row to the workspace (deterministic; a finalize kernel sums
//     the rows and casts) or adds it with fp32 vector atomics into a zeroed
//     dweight_f32.
//   * Every mbarrier wait is bounded (~1 s); on timeout the whole team stops,
//     waits (bounded) for its copies in flight, and the CTA writes
//     RN_ERR_TIMEOUT into the workspace status word.
#include "common.cuh"
#include "launch.h"

namespace rn {

int row_max_threads(int cpt) { return cpt <= 1 ? 1024 : (cpt == 2 ? 768 : 512); }

template <int CPT> struct RowBounds {
    static constexpr int kMaxThreads = CPT <= 1 ? 1024 : (CPT == 2 ? 768 : 512);
};

constexpr int kBarBytes = 1024;      // up to 15 teams x 8 stages of 8-byte mbarriers
constexpr int kRedOffset = 1024;     // [2 parities][32 warps] fp32 partial sums
constexpr int kFlagOffset = 1280;    // [2 parities][32 warps] timeout flags
constexpr int kStageOffset = 2048;

static inline int round_up(int v, int a) { return (v + a - 1) / a * a; }

size_t row_smem_bytes(int teams, int stages, int ntensors, int row_bytes) {
    return (size_t)kStageOffset +
           (size_t)teams * stages * ntensors * (size_t)round_up(row_bytes, 128);
}

struct RowArgs {
    const uint8_t *x;
    const uint8_t *gamma;
    const uint8_t *dy;
    const float *rstd;
    const uint8_t *dres;
    uint8_t *dx;
    float *dw_out;   // scratch: partial rows [gridDim.x][N]; atomic: dweight_f32
    int *status;
    int64_t M;
    int N;
    int nchunks;
    int row_bytes;
    int row_pitch;
    int team_threads;
    int teams;
    int stages;
    float inv_n;
};

template <typename T, int CPT, bool HAS_DRES, bool ATOMIC>
__global__ void __launch_bounds__(RowBounds<CPT>::kMaxThreads, 1)
    bwd_row_kernel(const RowArgs a) {
    constexpr int V = Traits<T>::kVec;
    constexpr int NT = HAS_DRES ? 3 : 2;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + kRedOffset);
    int *redflag = reinterpret_cast<int *>(smem + kFlagOffset);
    uint8_t *stage_base = smem + kStageOffset;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int team = tid / a.team_threads;
    const int tt = tid - team * a.team_threads;
    const int team_warps = a.team_threads >> 5;
    const int first_warp = team * team_warps;
    const int S = a.stages;
    const int stage_bytes = NT * a.row_pitch;

    if (tid == 0) {
        for (int i = 0; i < a.teams * S; ++i) mbar_init(smem_addr(&bars[i]), 1);
        fence_mbarrier_init();
    }
    __syncthreads();

    const int64_t team_stride = (int64_t)gridDim.x * a.teams;
    const int64_t row0 = (int64_t)blockIdx.x * a.teams + team;
    const int64_t nrows = row0 < a.M ? (a.M - 1 - row0) / team_stride + 1 : 0;
    uint8_t *my_stages = stage_base + (size_t)team * S * stage_bytes;
    const uint32_t my_bars = smem_addr(&bars[team * S]);
    const uint32_t tx_bytes = (uint32_t)(NT * a.row_bytes);

    uint64_t policy = 0;
    if (tt == 0) policy = l2_policy_evict_first();

    // Leader only: load this team's k-th row into slot k % S.
    auto issue = [&](int64_t k) {
        const int s = (int)(k % S);
        const int64_t row = row0 + k * team_stride;
        const uint32_t bar = my_bars + 8u * s;
        const uint32_t dst = smem_addr(my_stages + (size_t)s * stage_bytes);
        const size_t off = (size_t)row * a.row_bytes;
        mbar_arrive_expect_tx(bar, tx_bytes);
        bulk_copy_g2s(dst, a.x + off, a.row_bytes, bar, policy);
        bulk_copy_g2s(dst + a.row_pitch, a.dy + off, a.row_bytes, bar, policy);
        if (HAS_DRES) bulk_copy_g2s(dst + 2 * a.row_pitch, a.dres + off, a.row_bytes, bar, policy);
    };

    if (tt == 0) {
        const int64_t n0 = nrows < S ? nrows : S;
        for (int64_t k = 0; k < n0; ++k) issue(k);
    }

    uint4 g[CPT];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        const int c = tt + kk * a.team_threads;
        g[kk] = c < a.nchunks ? ld_global_nc_v4(a.gamma + (size_t)c * 16) : make_uint4(0, 0, 0, 0);
    }
    float acc[CPT][V];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk)
#pragma unroll
        for (int e = 0; e < V; ++e) acc[kk][e] = 0.f;

    float rs_next = nrows > 0 ? __ldg(a.rstd + row0) : 0.f;
    int64_t k = 0;
    bool failed = false;
    for (; k < nrows; ++k) {
        const int s = (int)(k % S);
        const uint32_t parity = (uint32_t)((k / S) & 1);
        const int64_t row = row0 + k * team_stride;
        const float rs = rs_next;
        if (k + 1 < nrows) rs_next = __ldg(a.rstd + row + team_stride);

        const bool ok = mbar_wait_bounded(my_bars + 8u * s, parity, kWaitLimitCycles);
        const uint32_t sb = smem_addr(my_stages + (size_t)s * stage_bytes);

        uint4 xv[CPT], dv[CPT], rv[CPT];
        float part = 0.f;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = tt + kk * a.team_threads;
            if (c < a.nchunks) {
                xv[kk] = ld_shared_v4(sb + 16u * c);
                dv[kk] = ld_shared_v4(sb + a.row_pitch + 16u * c);
                if (HAS_DRES) rv[kk] = ld_shared_v4(sb + 2 * a.row_pitch + 16u * c);
                float xf[V], df[V], gf[V];
                chunk_to_float<T>(xv[kk], xf);
                chunk_to_float<T>(dv[kk], df);
                chunk_to_float<T>(g[kk], gf);
#pragma unroll
                for (int e = 0; e < V; ++e) part = fmaf(xf[e], df[e] * gf[e], part);
            }
        }
        // c1 reduction across the team; the same barrier also tells the
        // leader that every thread has finished reading slot s.
        part = warp_sum(part);
        int any_fail;
        if (team_warps > 1) {
            const int base = (int)(k & 1) * 32;
            if (lane == 0) {
                red[base + warp] = part;
                redflag[base + warp] = ok ? 0 : 1;
            }
            named_barrier_sync(1 + team, a.team_threads);
            float tot = 0.f;
            int fl = 0;
            for (int w = 0; w < team_warps; ++w) {
                tot += red[base + first_warp + w];
                fl |= redflag[base + first_warp + w];
            }
            part = tot;
            any_fail = fl;
        } else {
            any_fail = __any_sync(0xFFFFFFFFu, !ok);
            __syncwarp();
        }
        if (any_fail) {
            failed = true;
            break;
        }
        if (tt == 0 && k + S < nrows) {
            fence_proxy_async_shared();
            issue(k + S);
        }

        const float c1 = rs * part * a.inv_n;
        uint8_t *dxrow = a.dx + (size_t)row * a.row_bytes;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = tt + kk * a.team_threads;
            if (c < a.nchunks) {
                float xf[V], df[V], gf[V], rf[V], o[V];
                chunk_to_float<T>(xv[kk], xf);
                chunk_to_float<T>(dv[kk], df);
                chunk_to_float<T>(g[kk], gf);
                if (HAS_DRES) chunk_to_float<T>(rv[kk], rf);
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float xh = xf[e] * rs;
                    const float wdy = df[e] * gf[e];
                    float d = fmaf(-xh, c1, wdy) * rs;
                    if (HAS_DRES) d += rf[e];
                    o[e] = d;
                    acc[kk][e] = fmaf(df[e], xh, acc[kk][e]);
                }
                st_global_v4(dxrow + 16u * c, float_to_chunk<T>(o));
            }
        }
    }

    if (failed && tt == 0) {
        // Let the copies this team still has in flight land before exiting.
        for (int64_t j = k; j < nrows && j < k + S; ++j) {
            const int s = (int)(j % S);
            mbar_wait_bounded(my_bars + 8u * s, (uint32_t)((j / S) & 1), kWaitLimitCycles);
        }
        atomicExch(a.status, 5 /* RN_ERR_TIMEOUT */);
    }

    pdl_launch_dependents();

    // ---- weight-gradient partial of this CTA
    __syncthreads();  // all teams are done with their slots
    float *out_row = ATOMIC ? a.dw_out : a.dw_out + (size_t)blockIdx.x * a.N;
    if (ATOMIC) pdl_wait();  // the zeroing kernel ahead of this one has finished
    if (a.teams == 1) {
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = tt + kk * a.team_threads;
            if (c < a.nchunks) {
#pragma unroll
                for (int q = 0; q < V / 4; ++q) {
                    float4 v = make_float4(acc[kk][4 * q], acc[kk][4 * q + 1], acc[kk][4 * q + 2],
                                           acc[kk][4 * q + 3]);
                    float4 *dst = reinterpret_cast<float4 *>(out_row + (size_t)c * V + 4 * q);
                    if (ATOMIC) atomicAdd(dst, v);
                    else *dst = v;
                }
            }
        }
        return;
    }
    float *sdw = reinterpret_cast<float *>(stage_base);
    for (int t = 0; t < a.teams; ++t) {
        if (team == t) {
#pragma unroll
            for (int kk = 0; kk < CPT; ++kk) {
                const int c = tt + kk * a.team_threads;
                if (c < a.nchunks) {
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        float *p = sdw + (size_t)c * V + e;
                        *p = (t == 0) ? acc[kk][e] : *p + acc[kk][e];
                    }
                }
            }
        }
        __syncthreads();
    }
    for (int i = tid * 4; i < a.N; i += blockDim.x * 4) {
        float4 v = *reinterpret_cast<const float4 *>(sdw + i);
        float4 *dst = reinterpret_cast<float4 *>(out_row + i);
        if (ATOMIC) atomicAdd(dst, v);
        else *dst = v;
    }
}

template <typename T, int CPT, bool HAS_DRES, bool ATOMIC>
static cudaError_t launch_row_t(const RowArgs &args, const RowPlan &plan, cudaStream_t s,
                                bool pdl) {
    auto kern = bwd_row_kernel<T, CPT, HAS_DRES, ATOMIC>;
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

template <typename T, int CPT>
static cudaError_t launch_row_cpt(const RowArgs &args, const RowPlan &plan, bool has_dres,
                                  cudaStream_t s, bool pdl) {
    if (has_dres)
        return plan.atomic ? launch_row_t<T, CPT, true, true>(args, plan, s, pdl)
                           : launch_row_t<T, CPT, true, false>(args, plan, s, pdl);
    return plan.atomic ? launch_row_t<T, CPT, false, true>(args, plan, s, pdl)
                       : launch_row_t<T, CPT, false, false>(args, plan, s, pdl);
}

template <typename T>
static cudaError_t launch_row_dt(const RowArgs &args, const RowPlan &plan, bool has_dres,
                                 cudaStream_t s, bool pdl) {
    switch (plan.cpt) {
    case 1: return launch_row_cpt<T, 1>(args, plan, has_dres, s, pdl);
    case 2: return launch_row_cpt<T, 2>(args, plan, has_dres, s, pdl);
    case 4: return launch_row_cpt<T, 4>(args, plan, has_dres, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_row(const BwdProblem &p, const RowPlan &plan, cudaStream_t s,
                           bool pdl_after_zero) {
    RowArgs a;
    const int eb = elem_bytes(p.dtype);
    a.x = static_cast<const uint8_t *>(p.x);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.dy = static_cast<const uint8_t *>(p.dy);
    a.rstd = p.rstd;
    a.dres = static_cast<const uint8_t *>(p.dres);
    a.dx = static_cast<uint8_t *>(p.dx);
    a.dw_out = plan.atomic ? p.dw_f32 : reinterpret_cast<float *>(p.ws + kWsHeaderBytes);
    a.status = reinterpret_cast<int *>(p.ws);
    a.M = p.M;
    a.N = p.N;
    a.row_bytes = p.N * eb;
    a.nchunks = a.row_bytes / 16;
    a.row_pitch = round_up(a.row_bytes, 128);
    a.team_threads = plan.team_threads;
    a.teams = plan.teams;
    a.stages = plan.stages;
    a.inv_n = 1.0f / (float)p.N;
    const bool has_dres = p.dres != nullptr;
    switch (p.dtype) {
    case kF32: return launch_row_dt<float>(a, plan, has_dres, s, pdl_after_zero);
    case kF16: return launch_row_dt<__half>(a, plan, has_dres, s, pdl_after_zero);
    case kBF16: return launch_row_dt<__nv_bfloat16>(a, plan, has_dres, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
