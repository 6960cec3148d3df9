// Forward staged phase-class kernel: RMSNorm, fused-add RMSNorm and LayerNorm
// forwards on rows that are not 16-byte multiples (or whose base is off a
// 16-byte boundary), every row tensor (x, y; residual, residual_out) at one
// alignment phase, at most 2048 whole 16-byte chunks per row.
//
// What is computed is the forward row engine's (FlyDSL issue #769, "Current
// state": rstd = 1/sqrt(mean(x^2) + eps), y = x*rstd*gamma; PR #800, "What's
// included": the fused-add statistic and output come from the dtype-rounded
// residual_out; issue #769's LayerNorm plan: the mean, then the centred
// variance, y = (x - mean)*rstd*gamma + beta).
//
// The work split and the staging are the backward staged kernel's:
//   * Row r starts r*N*s bytes past the base, so its alignment phase repeats
//     with period P = 16 / gcd(16, N*s mod 16) rows. CTA b takes the rows of
//     residue class b mod P, where every row splits the same way into h head
//     elements, nv whole 16-byte chunks and a few tail elements.
//   * Persistent grid; a CTA holds `teams` teams (named barriers 1..teams), a
//     team owns one row at a time. Warp w of a team owns the contiguous chunks
//     [w*32J, (w+1)*32J) of the row's whole-chunk middle; lane l takes chunks
//     w*32J + l + 32k.
//   * Each warp stages its own span of the team's next rows in shared memory
//     with bulk copies (one per streamed tensor and row, issued by lane 0,
//     completing on the warp's own mbarrier of the slot). At the top of row j
//     the warp refills the slot it finished with in row j-1, so no barrier
//     guards the ring. For 16-bit types the 16-byte blocks holding the head
//     and tail elements ride on the first and the last warp's copies (16
//     bytes early, 16 bytes late) where they lie inside the tensor; fp32
//     edges (and the blocks of the first and last rows) are loaded from
//     global memory.
//   * A lane reads its chunks from the slot once and keeps them in registers
//     for the whole row: fused-add rounds x + residual there and stores
//     residual_out; the sums (LayerNorm: the sum, then the centred sum of
//     squares) go through warp shuffles and the team's named barrier; y leaves
//     as 16-byte stores (the class's chunks are 16-byte aligned in every row
//     tensor). gamma (beta) may sit at any alignment: gathered once.
//   * Every mbarrier wait is bounded in time; a warp whose wait runs out tells
//     its team through the first row sum's exchange, the team stops, its
//     issuing lanes wait (bounded) for their copies still in flight, and the
//     kernel ORs 1 into its device status word (read by
//     rn_take_device_status()).
#include "common.cuh"
#include "launch.h"
#include "stage.cuh"
#include "unaligned.cuh"

namespace rn {

// Device status word of the forward staged kernel (bit 0: a bounded wait ran out).
__device__ unsigned int g_fwd_device_status;

namespace {

// Shared memory: [0,256) warp sums [2 parities][32 warps]; [256,512) wait outcomes, same
// layout; [512, 512 + 8*16*Sq) the warps' full barriers (warp w, slot u at w*Sq + u); the ring
// from fwd_stage_ring_offset(Sq): team t's slot u at (t*Sq + u)*stage_bytes, tensor k of a slot
// at k*tensor_bytes; within a tensor whole chunk i at kMid + 16i, the head block just before
// chunk 0 and the tail block just after the last whole chunk.
constexpr uint32_t kFwdBarOffset = 512;
constexpr uint32_t kFwdMid = 128;

uint32_t fwd_stage_ring_offset(int slots) {
    return (kFwdBarOffset + 8u * 16u * (uint32_t)slots + 127u) / 128u * 128u;
}

struct FwdStageArgs {
    const void *x;
    const void *res;       // fused-add
    const void *gamma;     // any element alignment
    const void *beta;      // LayerNorm, nullable
    void *y;
    void *res_out;         // fused-add
    float *mean;           // LayerNorm, nullable
    float *rstd;           // nullable
    int64_t M;
    int N;
    float inv_n;
    float eps;
    int period;            // P
    int teams;
    int team_threads;
    int slots;             // Sq
    uint32_t tensor_bytes;
    uint32_t stage_bytes;
    uint32_t ring_off;
    int64_t skip_row;      // test hook: CTA 0 team 0's local row whose copies its warp 0 never
                           // issues (its wait runs out); -1 = off
};

template <typename T, int MODE, int J>
__global__ void __launch_bounds__(512, 1) fwd_stage_kernel(const FwdStageArgs a) {
    constexpr int S = sizeof(T), V = 16 / S, P2 = V / 2;
    constexpr bool kFused = MODE == kFwdFused, kLn = MODE == kFwdLn;
    constexpr int NT = kFused ? 2 : 1;
    constexpr bool kFold = S == 2;
    extern __shared__ __align__(128) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    int *okf = reinterpret_cast<int *>(smem + 256);
    const T *x = static_cast<const T *>(a.x);
    const T *res = static_cast<const T *>(a.res);
    const T *g = static_cast<const T *>(a.gamma);
    const T *bt = static_cast<const T *>(a.beta);
    T *y = static_cast<T *>(a.y);
    T *ro = static_cast<T *>(a.res_out);
    const int tid = threadIdx.x;
    const int N = a.N, P = a.period, Sq = a.slots;

    // this CTA's rows: row0 + k*rstride (k < nrows), all of class cls
    const int cls = (int)(blockIdx.x % (unsigned)P);
    const int64_t nper = ((int64_t)gridDim.x - cls + P - 1) / P;  // CTAs of this class
    const int64_t rstride = nper * P;
    const int64_t row0 = cls + (int64_t)(blockIdx.x / (unsigned)P) * P;
    const int64_t nrows = row0 < a.M ? (a.M - 1 - row0) / rstride + 1 : 0;
    // the class's split (address arithmetic on row cls; nothing is read there)
    const uintptr_t start = reinterpret_cast<uintptr_t>(a.x) + (uintptr_t)cls * (uintptr_t)N * S;
    const int h_free = (int)(((16u - (unsigned)(start & 15u)) & 15u) / S);
    // a row that holds a 16-byte boundary has its head in the block that ends at the first
    // boundary and its tail in the block that starts at the last one
    const bool blocks = h_free <= N;
    const int h = blocks ? h_free : N;
    const int nv = (N - h) / V, tail = N - h - nv * V;
    const int64_t total = a.M * (int64_t)N;  // elements of a row tensor

    const int team_warps = a.team_threads >> 5;
    const int team = tid / a.team_threads;
    const int tt = tid - team * a.team_threads;
    const int warp = tid >> 5, lane = tid & 31;
    const int first_warp = team * team_warps;
    const int c0 = (warp - first_warp) * 32 * J;  // this warp's first chunk
    const int wn = nv - c0 < 0 ? 0 : (nv - c0 < 32 * J ? nv - c0 : 32 * J);
    // this team's rows: CTA rows team, team + teams, ...
    const int64_t tn = team < nrows ? (nrows - 1 - team) / a.teams + 1 : 0;
    const int64_t trow0 = row0 + (int64_t)team * rstride;
    const int64_t tstride = (int64_t)a.teams * rstride;  // rows between the team's rows
    const int64_t tstep = tstride * N;                    // elements between them
    const uint32_t wbar = smem_addr(smem + kFwdBarOffset) + 8u * (uint32_t)(warp * Sq);
    const uint32_t tring = smem_addr(smem + a.ring_off) + (uint32_t)(team * Sq) * a.stage_bytes;

    if (lane == 0) {
        for (int u = 0; u < Sq; ++u) mbar_init(wbar + 8u * u, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Lane 0: copies of this warp's span of the team's rows, in order (folded edge blocks on
    // the team's first warp and on the warp holding the last whole chunk).
    const uint64_t policy = l2_policy_evict_first();
    const uint32_t bytes = (uint32_t)wn * 16u;
    const int w_last = nv > 0 ? (nv - 1) / (32 * J) : 0;
    const bool w_head = warp == first_warp, w_tail = warp == first_warp + w_last;
    const bool skipper = a.skip_row >= 0 && blockIdx.x == 0 && tid == 0;
    int64_t issued = 0;                   // rows issued
    int64_t irow_e0 = trow0 * N + h;      // element of row `issued`'s first 16-byte boundary
    int iu = 0;                           // its slot
    auto issue = [&]() {
        const uint32_t bar = wbar + 8u * (uint32_t)iu;
        const int64_t e0 = irow_e0;
        const bool hb = kFold && w_head && blocks && h > 0 && e0 - V >= 0;
        const bool tb = kFold && w_tail && blocks && tail > 0 && e0 + (int64_t)(nv + 1) * V <= total;
        const uint32_t nbytes = bytes + (hb ? 16u : 0u) + (tb ? 16u : 0u);
        if (skipper && issued == a.skip_row) {
            // test hook: nothing arrives, so this slot's wait runs out
        } else if (nbytes == 0) {
            mbar_arrive(bar);
        } else {
            const size_t off = (size_t)(e0 + (int64_t)c0 * V - (hb ? V : 0));
            const uint32_t dst =
                tring + (uint32_t)iu * a.stage_bytes + kFwdMid + 16u * (uint32_t)c0 - (hb ? 16u : 0u);
            mbar_arrive_expect_tx(bar, NT * nbytes);
            bulk_copy_g2s(dst, x + off, nbytes, bar, policy);
            if (kFused) bulk_copy_g2s(dst + a.tensor_bytes, res + off, nbytes, bar, policy);
        }
        ++issued;
        irow_e0 += tstep;
        if (++iu == Sq) iu = 0;
    };
    if (lane == 0)
        while (issued < Sq - 1 && issued < tn) issue();

    // this thread's chunks (lane + 32k of the warp's span): gamma (beta) as fp32 pairs
    bool own[J];
    int col[J];
    f32x2 g2[J][P2], b2[kLn ? J : 1][kLn ? P2 : 1];
#pragma unroll
    for (int k = 0; k < J; ++k) {
        own[k] = lane + 32 * k < wn;
        col[k] = h + (c0 + lane + 32 * k) * V;
        float gf[V];
        chunk_to_float<T>(own[k] ? gather_chunk<T>(g + col[k]) : make_uint4(0, 0, 0, 0), gf);
#pragma unroll
        for (int q = 0; q < P2; ++q) g2[k][q] = f2_make(gf[2 * q], gf[2 * q + 1]);
        if (kLn) {
            chunk_to_float<T>(own[k] && bt ? gather_chunk<T>(bt + col[k]) : make_uint4(0, 0, 0, 0),
                              gf);
#pragma unroll
            for (int q = 0; q < P2; ++q) b2[kLn ? k : 0][kLn ? q : 0] = f2_make(gf[2 * q], gf[2 * q + 1]);
        }
    }
    // the head or tail element of this thread, its column and (folded) its byte offset in a
    // tensor's slot: head elements on the first lanes of the team's first warp, tail elements
    // on the last lanes of the warp copying the tail block; fp32: the first h + tail threads
    const bool e_head = kFold ? w_head && lane < h : tt < h;
    const bool e_tail = kFold ? w_tail && lane >= 32 - tail : tt >= h && tt < h + tail;
    const bool e_own = e_head || e_tail;
    const int je = e_head ? (kFold ? lane : tt)
                          : h + nv * V + (kFold ? lane - (32 - tail) : tt - h);
    const uint32_t e_soff = e_head ? kFwdMid - 16u + (uint32_t)(S * (V - h + lane))
                                   : kFwdMid + 16u * (uint32_t)nv + (uint32_t)(S * (lane - (32 - tail)));
    const float ge = e_own ? to_f(g[je]) : 0.f;
    const float be = (kLn && e_own && bt) ? to_f(bt[je]) : 0.f;
    // fp32: the team's next row's edge element, one row ahead in registers
    float xe_n = 0.f, re_n = 0.f;
    auto edge_next = [&](int64_t r) {
        if (!kFold && e_own) {
            const size_t e = (size_t)r * N + je;
            xe_n = to_f(x[e]);
            if (kFused) re_n = to_f(res[e]);
        }
    };
    if (tn > 0) edge_next(trow0);

    // team sum of v; with `ok`, also whether every warp's wait succeeded
    int par = 0;
    auto team_sum = [&](float v, bool ok, bool *all_ok) {
        const float wsum = warp_sum(v);
        const int wok = __all_sync(0xffffffffu, ok);
        if (lane == 0) {
            red[par * 32 + warp] = wsum;
            okf[par * 32 + warp] = wok;
        }
        named_barrier_sync(1 + team, a.team_threads);
        const float w = lane < team_warps ? red[par * 32 + first_warp + lane] : 0.f;
        const int o = lane < team_warps ? okf[par * 32 + first_warp + lane] : 1;
        *all_ok = __all_sync(0xffffffffu, o) != 0;
        par ^= 1;
        return warp_sum(w);
    };

    bool failed = false;
    int64_t j = 0;
    int u = 0;          // slot of row j
    uint32_t ph = 0;    // parity of its use
    int64_t row = trow0;
    size_t rbase = (size_t)trow0 * N;
    for (; j < tn; ++j) {
        // every lane of this warp is done with row j-1: its slot takes row j+Sq-1
        __syncwarp();
        if (lane == 0 && issued < tn) issue();
        float xe = xe_n, re = re_n;
        if (j + 1 < tn) edge_next(row + tstride);
        const bool ok = mbar_wait_bounded(wbar + 8u * (uint32_t)u, ph, kWaitLimitNs);
        const uint32_t sb = tring + (uint32_t)u * a.stage_bytes;
        const uint32_t sm = sb + kFwdMid;  // the row's whole chunks
        if (kFold && e_own) {
            const int64_t e0 = row * N + h;
            const bool e_smem = blocks && (e_head ? e0 - V >= 0 : e0 + (int64_t)(nv + 1) * V <= total);
            if (e_smem) {
                xe = lds_elem<T>(sb + e_soff);
                if (kFused) re = lds_elem<T>(sb + a.tensor_bytes + e_soff);
            } else {
                xe = to_f(x[rbase + je]);
                if (kFused) re = to_f(res[rbase + je]);
            }
        }
        // the row's chunks into registers; fused-add: round(x + residual), stored as residual_out
        uint4 xv[J];
#pragma unroll
        for (int k = 0; k < J; ++k) {
            const uint32_t c16 = 16u * (uint32_t)(c0 + lane + 32 * k);
            xv[k] = own[k] ? ld_shared_v4(sm + c16) : make_uint4(0, 0, 0, 0);
            if (kFused && own[k]) {
                float xf[V], rf[V];
                chunk_to_float<T>(xv[k], xf);
                chunk_to_float<T>(ld_shared_v4(sm + a.tensor_bytes + c16), rf);
#pragma unroll
                for (int q = 0; q < V; ++q) xf[q] += rf[q];
                xv[k] = float_to_chunk<T>(xf);
                st_global_v4(ro + rbase + col[k], xv[k]);
            }
        }
        if (kFused && e_own) {
            xe = round_through<T>(xe + re);
            ro[rbase + je] = from_f<T>(xe);
        }
        // pass 1: sum of squares (LayerNorm: sum)
        f32x2 s2 = f2_make(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                float f[V];
                chunk_to_float<T>(xv[k], f);
#pragma unroll
                for (int q = 0; q < P2; ++q) {
                    const f32x2 v = f2_make(f[2 * q], f[2 * q + 1]);
                    s2 = kLn ? f2_add(v, s2) : f2_fma(v, v, s2);
                }
            }
        }
        float lo, hi;
        f2_split(s2, lo, hi);
        float sv = lo + hi;
        if (e_own) sv = kLn ? sv + xe : fmaf(xe, xe, sv);
        bool all_ok;
        float tot = team_sum(sv, ok, &all_ok);
        if (!all_ok) {
            failed = true;
            break;
        }
        float mu = 0.f;
        if (kLn) {
            // the centred sum of squares, from the registers (no cancellation)
            mu = tot * a.inv_n;
            const f32x2 m2 = f2_make(-mu, -mu);
            f32x2 q2 = f2_make(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < J; ++k) {
                if (own[k]) {
                    float f[V];
                    chunk_to_float<T>(xv[k], f);
#pragma unroll
                    for (int q = 0; q < P2; ++q) {
                        const f32x2 d = f2_add(f2_make(f[2 * q], f[2 * q + 1]), m2);
                        q2 = f2_fma(d, d, q2);
                    }
                }
            }
            f2_split(q2, lo, hi);
            sv = lo + hi;
            if (e_own) sv = fmaf(xe - mu, xe - mu, sv);
            bool unused;
            tot = team_sum(sv, true, &unused);
        }
        const float rs = rsqrtf(tot * a.inv_n + a.eps);
        if (tt == 0) {
            if (kLn && a.mean) a.mean[row] = mu;
            if (a.rstd) a.rstd[row] = rs;
        }
        // y = x*rs*gamma (LayerNorm: (x - mean)*rs*gamma + beta)
        const f32x2 rs2 = f2_make(rs, rs), m2 = f2_make(-mu, -mu);
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                float f[V];
                chunk_to_float<T>(xv[k], f);
#pragma unroll
                for (int q = 0; q < P2; ++q) {
                    f32x2 v = f2_make(f[2 * q], f[2 * q + 1]);
                    if (kLn)
                        v = f2_fma(f2_mul(f2_add(v, m2), rs2), g2[k][q], b2[kLn ? k : 0][kLn ? q : 0]);
                    else
                        v = f2_mul(f2_mul(v, rs2), g2[k][q]);
                    f2_split(v, f[2 * q], f[2 * q + 1]);
                }
                st_global_v4(y + rbase + col[k], float_to_chunk<T>(f));
            }
        }
        if (e_own)
            y[rbase + je] = from_f<T>(kLn ? fmaf((xe - mu) * rs, ge, be) : xe * rs * ge);
        if (++u == Sq) {
            u = 0;
            ph ^= 1u;
        }
        row += tstride;
        rbase += (size_t)tstep;
    }
    if (failed) {
        // rows j .. issued-1 of this warp may still have copies in flight: wait for them
        // (bounded) before the CTA can exit
        if (lane == 0) {
            for (; j < issued; ++j) {
                (void)mbar_wait_bounded(wbar + 8u * (uint32_t)u, ph, kWaitLimitNs);
                if (++u == Sq) {
                    u = 0;
                    ph ^= 1u;
                }
            }
        }
        if (tt == 0) atomicOr(&g_fwd_device_status, 1u);
    }
}

template <typename T, int MODE, int J>
cudaError_t launch_t(const FwdStageArgs &a, int grid, int threads, size_t smem, cudaStream_t s) {
    auto k = fwd_stage_kernel<T, MODE, J>;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(k), smem);
    if (e != cudaSuccess) return e;
    k<<<grid, threads, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int MODE>
cudaError_t launch_j(const FwdStageArgs &a, int cpt, int grid, int threads, size_t smem,
                     cudaStream_t s) {
    switch (cpt) {
    case 1: return launch_t<T, MODE, 1>(a, grid, threads, smem, s);
    case 2: return launch_t<T, MODE, 2>(a, grid, threads, smem, s);
    case 4: return launch_t<T, MODE, 4>(a, grid, threads, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
const void *kernel_ptr(int mode, int cpt) {
#define RN_FWD_STAGE_K(M)                                                           \
    (cpt == 1 ? (const void *)fwd_stage_kernel<T, M, 1>                             \
              : cpt == 2 ? (const void *)fwd_stage_kernel<T, M, 2>                  \
                         : (const void *)fwd_stage_kernel<T, M, 4>)
    return mode == kFwdFused ? RN_FWD_STAGE_K(kFwdFused)
           : mode == kFwdLn  ? RN_FWD_STAGE_K(kFwdLn)
                             : RN_FWD_STAGE_K(kFwdRms);
#undef RN_FWD_STAGE_K
}

}  // namespace

size_t fwd_stage_smem_bytes(int N, int dtype, int mode, int teams, int slots) {
    const int V = 16 / elem_bytes(dtype);
    const int64_t maxnv = (int64_t)N / V;  // whole chunks of any class's row
    // a tensor's slot: the head block, the whole chunks, the tail block
    const size_t tb = (size_t)((kFwdMid + (maxnv + 1) * 16 + 127) / 128 * 128);
    return fwd_stage_ring_offset(slots) + (size_t)teams * slots * (mode == kFwdFused ? 2 : 1) * tb;
}

bool fwd_stage_ok(const FwdRowProblem &p) {
    const uintptr_t S = (uintptr_t)elem_bytes(p.dtype);
    const uintptr_t ph = (uintptr_t)p.x & 15u;
    for (const void *q : {p.x, static_cast<const void *>(p.y), p.residual,
                          static_cast<const void *>(p.residual_out)}) {
        if (q == nullptr) continue;
        if (((uintptr_t)q & 15u) != ph || ((uintptr_t)q % S) != 0) return false;
    }
    return (int64_t)p.N * elem_bytes(p.dtype) / 16 <= 2048;
}

int fwd_stage_blocks_per_sm(int dtype, int mode, int cpt, int threads, size_t smem) {
    const void *k = dtype == kF32 ? kernel_ptr<float>(mode, cpt)
                  : dtype == kF16 ? kernel_ptr<__half>(mode, cpt)
                                  : kernel_ptr<__nv_bfloat16>(mode, cpt);
    int n = 0;
    if (ensure_smem_attr(k, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess ||
        n < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    return n;
}

cudaError_t launch_fwd_stage(const FwdRowProblem &p, const StagePlan &plan, cudaStream_t s) {
    FwdStageArgs a;
    a.x = p.x;
    a.res = p.residual;
    a.gamma = p.gamma;
    a.beta = p.beta;
    a.y = p.y;
    a.res_out = p.residual_out;
    a.mean = p.mean;
    a.rstd = p.rstd;
    a.M = p.M;
    a.N = p.N;
    a.inv_n = 1.0f / (float)p.N;
    a.eps = p.eps;
    a.period = phase_period(p.N, p.dtype);
    a.teams = plan.teams;
    a.team_threads = plan.team_threads;
    a.slots = plan.slots;
    a.skip_row = plan.skip_row;
    const int V = 16 / elem_bytes(p.dtype);
    const int64_t maxnv = (int64_t)p.N / V;
    a.tensor_bytes = (uint32_t)((kFwdMid + (maxnv + 1) * 16 + 127) / 128 * 128);
    a.stage_bytes = (p.mode == kFwdFused ? 2 : 1) * a.tensor_bytes;
    a.ring_off = fwd_stage_ring_offset(plan.slots);
    const size_t need = fwd_stage_smem_bytes(p.N, p.dtype, p.mode, plan.teams, plan.slots);
    // the launch shape the kernel relies on: every chunk owned, named barrier IDs 1..15, at
    // most 16 warps (the barrier and sum areas), two or more slots, every residue class with a
    // CTA, the edge elements within the lanes of one warp, and the shared memory it indexes
    if (!fwd_stage_ok(p)) return cudaErrorInvalidValue;
    if (plan.cpt != 1 && plan.cpt != 2 && plan.cpt != 4) return cudaErrorInvalidValue;
    if (plan.team_threads < 32 || plan.team_threads % 32 || plan.teams < 1 || plan.teams > 15 ||
        plan.teams * plan.team_threads > 512)
        return cudaErrorInvalidValue;
    if ((int64_t)plan.cpt * plan.team_threads < maxnv) return cudaErrorInvalidValue;
    if (plan.slots < 2 || plan.slots > 4) return cudaErrorInvalidValue;
    if (plan.smem < need) return cudaErrorInvalidValue;
    if (p.M > 0 && plan.grid < (p.M < a.period ? p.M : a.period)) return cudaErrorInvalidValue;
    const int threads = plan.teams * plan.team_threads;
    switch (p.dtype) {
#define RN_FWD_STAGE_MODES(T)                                                                      \
    switch (p.mode) {                                                                              \
    case kFwdRms: return launch_j<T, kFwdRms>(a, plan.cpt, plan.grid, threads, plan.smem, s);     \
    case kFwdFused: return launch_j<T, kFwdFused>(a, plan.cpt, plan.grid, threads, plan.smem, s); \
    case kFwdLn: return launch_j<T, kFwdLn>(a, plan.cpt, plan.grid, threads, plan.smem, s);       \
    default: return cudaErrorInvalidValue;                                                         \
    }
    case kF32: RN_FWD_STAGE_MODES(float)
    case kF16: RN_FWD_STAGE_MODES(__half)
    case kBF16: RN_FWD_STAGE_MODES(__nv_bfloat16)
#undef RN_FWD_STAGE_MODES
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t take_fwd_device_status(unsigned int *status) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fwd_device_status, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_fwd_device_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
    *status = v;
    return cudaSuccess;
}

}  // namespace rn
