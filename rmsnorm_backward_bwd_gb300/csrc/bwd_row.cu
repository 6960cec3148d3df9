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
//   * Thread tt of a team owns 16-byte chunks tt, tt+team_threads, ... of the
//     row (consecutive threads -> consecutive 16 B: coalesced loads and
//     128-bit dx stores, conflict-free shared accesses).
//   * Each thread streams its own chunks of the next `stages-1` rows into a
//     private ring of shared-memory slots with 16-byte asynchronous copies
//     (cp.async, L2 evict-first). A thread only ever reads back what it copied
//     itself, so the ring needs no barrier or mbarrier: per-thread commit
//     groups order everything, and no wait in this kernel can spin forever.
//     Every input byte is read from HBM exactly once.
//   * Pass 1 reduces sum_j x_j*dy_j*gamma_j (warp shuffles, then one named
//     barrier across the team's warps); pass 2 reads the slot again and
//     stores dx. The arithmetic runs on packed fp32 pairs (f32x2 FMA / MUL /
//     ADD: one instruction per two elements); for bf16/f16 the products
//     x*dy and dy*gamma come exact from mixed-precision FMAs on the packed
//     16-bit halves.
//   * The weight-gradient partial of the thread's columns lives in fp32
//     registers for every row the team handles; at the end the CTA's teams
//     add theirs in a fixed order in shared memory and the CTA either stores
//     one partial row to the workspace (deterministic; a finalize kernel sums
//     the rows and casts) or adds it with fp32 vector atomics into a zeroed
//     dweight_f32.
#include "common.cuh"
#include "launch.h"
#include "row_math.cuh"

namespace rn {

int row_max_threads(int cpt) { return cpt <= 2 ? 768 : 512; }

template <int CPT> struct RowBounds {
    static constexpr int kMaxThreads = CPT <= 2 ? 768 : 512;
};

constexpr int kRingOffset = 256;  // after [2 parities][32 warps] fp32 partial sums

size_t row_smem_bytes(int teams, int stages, int ntensors, int team_chunks) {
    return (size_t)kRingOffset + (size_t)teams * stages * ntensors * (size_t)team_chunks * 16;
}

struct RowArgs {
    const uint8_t *x;
    const uint8_t *gamma;
    const uint8_t *dy;
    const float *rstd;
    const uint8_t *dres;
    uint8_t *dx;
    float *dw_out;   // scratch: partial rows [gridDim.x][N]; atomic: dweight_f32
    int64_t M;
    int N;
    int nchunks;
    int row_bytes;
    int team_threads;
    int teams;
    int stages;
    float inv_n;
};

// The CTA's weight-gradient partial: teams add theirs in a fixed order in
// shared memory (deterministic), then the CTA stores one partial row to the
// workspace (scratch mode) or adds it with fp32 vector atomics into
// dweight_f32 (atomic mode, after the zeroing kernel ahead has finished).
// Layout in shared memory: the float4 `q` of chunk c sits at float4 index
// q*tc + c, so a warp's 16-byte accesses for one (kk, q) are consecutive (no
// bank conflicts). `scratch` must hold N floats and be free of other use.
template <typename T, int CPT, bool ATOMIC>
__device__ __forceinline__ void cta_partial_out(const f32x2 (&acc2)[CPT][RowMath<T>::kPairs],
                                                const RowArgs &a, uint8_t *scratch, int team,
                                                int tt) {
    constexpr int V = Traits<T>::kVec;
    float *out_row = ATOMIC ? a.dw_out : a.dw_out + (size_t)blockIdx.x * a.N;
    if (ATOMIC) pdl_wait();
    if (a.teams == 1) {
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            const int c = tt + kk * a.team_threads;
            if (c < a.nchunks) {
#pragma unroll
                for (int q = 0; q < V / 4; ++q) {
                    float4 v;
                    f2_split(acc2[kk][2 * q], v.x, v.y);
                    f2_split(acc2[kk][2 * q + 1], v.z, v.w);
                    float4 *dst = reinterpret_cast<float4 *>(out_row + (size_t)c * V + 4 * q);
                    if (ATOMIC) atomicAdd(dst, v);
                    else *dst = v;
                }
            }
        }
        return;
    }
    constexpr int Q = V / 4;
    const int tc = CPT * a.team_threads;
    float4 *sdw = reinterpret_cast<float4 *>(scratch);
    for (int t = 0; t < a.teams; ++t) {
        if (team == t) {
#pragma unroll
            for (int kk = 0; kk < CPT; ++kk) {
                const int c = tt + kk * a.team_threads;
                if (c < a.nchunks) {
#pragma unroll
                    for (int q = 0; q < Q; ++q) {
                        float4 *p = sdw + (size_t)q * tc + c;
                        float4 v;
                        f2_split(acc2[kk][2 * q], v.x, v.y);
                        f2_split(acc2[kk][2 * q + 1], v.z, v.w);
                        if (t > 0) {
                            const float4 o = *p;
                            v.x += o.x;
                            v.y += o.y;
                            v.z += o.z;
                            v.w += o.w;
                        }
                        *p = v;
                    }
                }
            }
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < a.N / 4; i += blockDim.x) {
        const int c = i / Q, q = i - c * Q;
        const float4 v = sdw[(size_t)q * tc + c];
        float4 *dst = reinterpret_cast<float4 *>(out_row) + i;
        if (ATOMIC) atomicAdd(dst, v);
        else *dst = v;
    }
}

// Sum of one value per thread over a team of team_warps warps: warp
// shuffles, then the warps' sums through shared memory (double-buffered by
// `parity`) and one named barrier, then a second shuffle; every thread of
// the team gets the same bits.
__device__ __forceinline__ float team_sum(float v, float *red, int parity, int team, int warp,
                                          int lane, int team_warps, int first_warp,
                                          int team_threads) {
    v = warp_sum(v);
    if (team_warps == 1) return v;
    float *slot = red + parity * 32;
    if (lane == 0) slot[warp] = v;
    named_barrier_sync(1 + team, team_threads);
    float w = lane < team_warps ? slot[first_warp + lane] : 0.f;
    return warp_sum(w);
}

template <typename T, int CPT, bool HAS_DRES, bool ATOMIC>
__global__ void __launch_bounds__(RowBounds<CPT>::kMaxThreads, 1)
    bwd_row_kernel(const RowArgs a) {
    constexpr int V = Traits<T>::kVec;
    constexpr int P = RowMath<T>::kPairs;  // fp32 pairs per chunk
    constexpr int NT = HAS_DRES ? 3 : 2;
    // gamma is also kept as fp32 pairs when the math needs it or when that
    // fits the register budget
    constexpr bool kGammaF = RowMath<T>::kNeedsGammaF || CPT * V <= 8;
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    uint8_t *ring = smem + kRingOffset;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int team = tid / a.team_threads;
    const int tt = tid - team * a.team_threads;
    const int team_warps = a.team_threads >> 5;
    const int first_warp = team * team_warps;
    const int S = a.stages;

    // This thread's ring: chunk kk of tensor t in slot s lives at
    // my0 + s*slot_bytes + t*tensor_bytes + kk*kk_bytes.
    const int tc = CPT * a.team_threads;
    const uint32_t kk_bytes = 16u * a.team_threads;
    const uint32_t tensor_bytes = 16u * tc;
    const uint32_t slot_bytes = NT * tensor_bytes;
    const uint32_t my0 = smem_addr(ring) + (uint32_t)team * S * slot_bytes + 16u * tt;

    const int64_t team_stride = (int64_t)gridDim.x * a.teams;
    const int64_t row0 = (int64_t)blockIdx.x * a.teams + team;
    const int64_t nrows = row0 < a.M ? (a.M - 1 - row0) / team_stride + 1 : 0;
    const uint64_t policy = l2_policy_evict_first();

    // byte offset of this thread's chunk kk within a row, and whether it exists
    uint32_t coff[CPT];
    bool cok[CPT];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        const int c = tt + kk * a.team_threads;
        coff[kk] = 16u * c;
        cok[kk] = c < a.nchunks;
    }

    // Copy this thread's chunks of row `row` into slot `s`.
    auto issue = [&](int64_t row, int s) {
        const size_t off = (size_t)row * a.row_bytes;
        const uint8_t *xr = a.x + off, *dr = a.dy + off, *rr = HAS_DRES ? a.dres + off : nullptr;
        const uint32_t d = my0 + (uint32_t)s * slot_bytes;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                cp_async16(d + kk * kk_bytes, xr + coff[kk], policy);
                cp_async16(d + tensor_bytes + kk * kk_bytes, dr + coff[kk], policy);
                if (HAS_DRES) cp_async16(d + 2 * tensor_bytes + kk * kk_bytes, rr + coff[kk], policy);
            }
        }
    };
    for (int j = 0; j < S - 1; ++j) {
        if (j < nrows) issue(row0 + j * team_stride, j);
        cp_async_commit();
    }

    uint4 gp[CPT];
    f32x2 g2[kGammaF ? CPT : 1][kGammaF ? P : 1];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        gp[kk] = cok[kk] ? ld_global_nc_v4(a.gamma + coff[kk]) : make_uint4(0, 0, 0, 0);
        if (kGammaF) {
            float gf[V];
            chunk_to_float<T>(gp[kk], gf);
#pragma unroll
            for (int q = 0; q < P; ++q)
                g2[kGammaF ? kk : 0][kGammaF ? q : 0] = f2_make(gf[2 * q], gf[2 * q + 1]);
        }
    }
    f32x2 acc2[CPT][P];
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk)
#pragma unroll
        for (int q = 0; q < P; ++q) acc2[kk][q] = f2_make(0.f, 0.f);

    const int64_t ahead = (int64_t)(S - 1) * team_stride;
    float rs_next = nrows > 0 ? __ldg(a.rstd + row0) : 0.f;
    int slot = 0, fill = S - 1;
    int64_t row = row0;
    for (int64_t k = 0; k < nrows; ++k, row += team_stride) {
        // Refill: row k+S-1 goes into the slot this thread finished with in
        // the previous iteration; then wait until row k's copies have landed.
        if (k + S - 1 < nrows) issue(row + ahead, fill);
        cp_async_commit();
        const float rs = rs_next;
        if (k + 1 < nrows) rs_next = __ldg(a.rstd + row + team_stride);
        cp_async_wait_pending(S - 1);
        const uint32_t sb = my0 + (uint32_t)slot * slot_bytes;

        f32x2 part2 = f2_make(0.f, 0.f);
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk])
                part2 = RowMath<T>::pass1(ld_shared_v4(sb + kk * kk_bytes),
                                          ld_shared_v4(sb + tensor_bytes + kk * kk_bytes), gp[kk],
                                          kGammaF ? g2[kGammaF ? kk : 0] : nullptr, part2);
        }
        float plo, phi;
        f2_split(part2, plo, phi);
        const float part = team_sum(plo + phi, red, (int)(k & 1), team, warp, lane, team_warps,
                                    first_warp, a.team_threads);

        // dx = (wdy - x_hat*c1)*rstd = wdy*rstd + x*b with b = -rstd^2*c1
        const float c1 = rs * part * a.inv_n;
        const float b = -rs * rs * c1;
        const f32x2 rs2 = f2_make(rs, rs), b2 = f2_make(b, b);
        uint8_t *dxrow = a.dx + (size_t)row * a.row_bytes;
#pragma unroll
        for (int kk = 0; kk < CPT; ++kk) {
            if (cok[kk]) {
                const uint4 r = HAS_DRES ? ld_shared_v4(sb + 2 * tensor_bytes + kk * kk_bytes)
                                         : make_uint4(0, 0, 0, 0);
                const uint4 o = RowMath<T>::template pass2<HAS_DRES>(
                    ld_shared_v4(sb + kk * kk_bytes), ld_shared_v4(sb + tensor_bytes + kk * kk_bytes),
                    r, gp[kk], kGammaF ? g2[kGammaF ? kk : 0] : nullptr, rs2, b2, acc2[kk]);
                st_global_v4(dxrow + coff[kk], o);
            }
        }
        if (++slot == S) slot = 0;
        if (++fill == S) fill = 0;
    }

    pdl_launch_dependents();
    __syncthreads();  // every team is done with its ring (all real copies waited for)
    cta_partial_out<T, CPT, ATOMIC>(acc2, a, ring, team, tt);
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
    a.M = p.M;
    a.N = p.N;
    a.row_bytes = p.N * eb;
    a.nchunks = a.row_bytes / 16;
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
