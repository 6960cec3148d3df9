// LayerNorm backward staged phase-class kernel: rows that are not 16-byte
// multiples (or whose base is off a 16-byte boundary), x, dy and dx at one
// alignment phase, at most 1024 whole 16-byte chunks per row.
//
// Math per row (FlyDSL issue #769, LayerNorm backward plan): x_hat =
// (x - mean)*rstd, wdy = dy*gamma, c1 = mean(x_hat*wdy), c2 = mean(wdy),
// dx = (wdy - c2 - x_hat*c1)*rstd = wdy*rstd + (x - mean)*B + A with
// B = -rstd^2*c1 and A = -c2*rstd; dgamma += dy*x_hat, dbeta += dy.
//
// Design: the RMSNorm staged kernel's (bwd_stage.cu) with the LayerNorm
// arithmetic of the row engine (ln_math.cuh):
//   * CTA b takes the rows of residue class b mod P (P = 16 / gcd(16,
//     N*s mod 16)); within a class every row splits into h head elements, nv
//     whole 16-byte chunks and a tail.
//   * Teams of warps own a row each; warp w of a team owns the contiguous
//     whole chunks [w*32J, (w+1)*32J) and stages its span of the team's next
//     rows in shared memory with one bulk copy per tensor (x, dy), completing
//     on its own mbarrier; it refills the slot it finished with at the top of
//     the next row. For 16-bit types the head and tail blocks ride on the
//     first and last warps' copies (where they lie inside the tensor); f32
//     loads the head and tail elements one row ahead into registers.
//   * Pass 1 sums (x - mean)*wdy and wdy over the row (warp shuffles, then
//     the team's named barrier, both sums at once); pass 2 stores dx and adds
//     dy*x_hat and dy into the thread's fp32 register partials.
//   * Waits are bounded (250 ms): a team whose wait runs out stops, drains
//     its copies (bounded again), and the CTA skips its partials and ORs 1
//     into this file's device status word (read with the library's one by
//     rn_take_device_status()).
//   * At the end each team stores its two partials in its own regions of the
//     drained ring by padded column; the CTA sums the teams' regions in team
//     order: fp32 vector atomics into dgamma / dbeta, or one partial row of
//     [dgamma | dbeta] of the workspace for the finalize kernel.
#include "common.cuh"
#include "launch.h"
#include "ln_math.cuh"
#include "stage.cuh"
#include "unaligned.cuh"

namespace rn {

// Device status word of the LayerNorm staged kernel (bit 0: a bounded wait ran out).
__device__ unsigned int g_ln_device_status;

namespace {

// Shared memory: [0,512) warp sums [2 parities][2 sums][32 warps]; [512,768)
// wait outcomes [2 parities][32 warps]; [768, 768 + 8*16*Sq) the warps' full
// barriers (warp w, slot u at w*Sq + u); the ring from ln_stage_ring_offset(Sq):
// team t's slot u at (t*Sq + u)*stage_bytes, x then dy in a slot; within a
// tensor whole chunk i at kLnMid + 16i, the head block just before chunk 0 and
// the tail block just after the last whole chunk.
constexpr uint32_t kLnStageOkOffset = 512;
constexpr uint32_t kLnStageBarOffset = 768;
constexpr uint32_t kLnMid = 128;

}  // namespace

uint32_t ln_stage_ring_offset(int slots) {
    return (kLnStageBarOffset + 8u * 16u * (uint32_t)slots + 127u) / 128u * 128u;
}

struct LnStageArgs {
    const void *x;
    const void *gamma;
    const void *dy;
    const float *mean;
    const float *rstd;
    void *dx;
    float *dg_out;  // atomic: dgamma_f32; scratch: partial rows [gridDim.x][2N] (dgamma | dbeta)
    float *db_out;  // atomic: dbeta_f32 (nullable); scratch: unused
    int64_t M;
    int N;
    float inv_n;
    int period;
    int teams;
    int team_threads;
    int slots;
    uint32_t tensor_bytes;
    uint32_t stage_bytes;
    uint32_t ring_off;
    uint32_t region_words;  // one padded partial region
    int64_t skip_row;       // test hook, as in the RMSNorm staged kernel; -1 = off
};

template <typename T, bool ATOMIC, int J>
__global__ void __launch_bounds__(512, 1) ln_bwd_stage_kernel(const LnStageArgs a) {
    constexpr int S = sizeof(T), V = 16 / S;
    constexpr int P2 = V / 2;  // fp32 pairs per chunk
    constexpr bool kF32 = S == 4;
    constexpr bool kFold = S == 2;  // f32 keeps the head and tail elements in registers
    extern __shared__ __align__(128) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    int *okf = reinterpret_cast<int *>(smem + kLnStageOkOffset);
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x;
    const int N = a.N, P = a.period, Sq = a.slots;

    // this CTA's rows: row0 + k*rstride (k < nrows), all of class cls
    const int cls = (int)(blockIdx.x % (unsigned)P);
    const int64_t nper = ((int64_t)gridDim.x - cls + P - 1) / P;
    const int64_t rstride = nper * P;
    const int64_t row0 = cls + (int64_t)(blockIdx.x / (unsigned)P) * P;
    const int64_t nrows = row0 < a.M ? (a.M - 1 - row0) / rstride + 1 : 0;
    // the class's split (address arithmetic on row cls; nothing is read there)
    const uintptr_t start = reinterpret_cast<uintptr_t>(a.x) + (uintptr_t)cls * (uintptr_t)N * S;
    const int h_free = (int)(((16u - (unsigned)(start & 15u)) & 15u) / S);
    const bool blocks = h_free <= N;  // the row holds a 16-byte boundary
    const int h = blocks ? h_free : N;
    const int nv = (N - h) / V, tail = N - h - nv * V;
    const int64_t total = a.M * (int64_t)N;

    const int team_warps = a.team_threads >> 5;
    const int team = tid / a.team_threads;
    const int tt = tid - team * a.team_threads;
    const int warp = tid >> 5, lane = tid & 31;
    const int first_warp = team * team_warps;
    const int c0 = (warp - first_warp) * 32 * J;
    const int wn = nv - c0 < 0 ? 0 : (nv - c0 < 32 * J ? nv - c0 : 32 * J);
    const int64_t tn = team < nrows ? (nrows - 1 - team) / a.teams + 1 : 0;
    const int64_t trow0 = row0 + (int64_t)team * rstride;
    const int64_t tstride = (int64_t)a.teams * rstride;
    const int64_t tstep = tstride * N;
    const uint32_t wbar = smem_addr(smem + kLnStageBarOffset) + 8u * (uint32_t)(warp * Sq);
    const uint32_t tring = smem_addr(smem + a.ring_off) + (uint32_t)(team * Sq) * a.stage_bytes;

    if (lane == 0) {
        for (int u = 0; u < Sq; ++u) mbar_init(wbar + 8u * u, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Lane 0: copies of this warp's span of the team's rows, in order (16-bit types: the first
    // warp's copy starts 16 bytes early with the head block, the last warp's ends 16 bytes late
    // with the tail block, where they lie inside the tensor).
    const uint64_t policy = l2_policy_evict_first();
    const uint32_t bytes = (uint32_t)wn * 16u;
    const int w_last = nv > 0 ? (nv - 1) / (32 * J) : 0;
    const bool w_head = warp == first_warp, w_tail = warp == first_warp + w_last;
    const bool skipper = a.skip_row >= 0 && blockIdx.x == 0 && tid == 0;
    int64_t issued = 0;
    int64_t irow_e0 = trow0 * N + h;  // element of row `issued`'s first 16-byte boundary
    int iu = 0;
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
                tring + (uint32_t)iu * a.stage_bytes + kLnMid + 16u * (uint32_t)c0 - (hb ? 16u : 0u);
            mbar_arrive_expect_tx(bar, 2u * nbytes);
            bulk_copy_g2s(dst, x + off, nbytes, bar, policy);
            bulk_copy_g2s(dst + a.tensor_bytes, dy + off, nbytes, bar, policy);
        }
        ++issued;
        irow_e0 += tstep;
        if (++iu == Sq) iu = 0;
    };
    if (lane == 0)
        while (issued < Sq - 1 && issued < tn) issue();

    // this thread's chunks, gamma (packed; fp32 pairs for f32) and partials
    bool own[J];
    int col[J];
    uint4 gp[J];
    f32x2 g2[kF32 ? J : 1][kF32 ? P2 : 1];
    f32x2 accg[J][P2], accb[J][P2];
#pragma unroll
    for (int k = 0; k < J; ++k) {
        own[k] = lane + 32 * k < wn;
        col[k] = h + (c0 + lane + 32 * k) * V;
        gp[k] = own[k] ? gather_chunk<T>(g + col[k]) : make_uint4(0, 0, 0, 0);
        if (kF32) chunk_pairs<T>(gp[k], g2[kF32 ? k : 0]);
#pragma unroll
        for (int q = 0; q < P2; ++q) accg[k][q] = accb[k][q] = f2_make(0.f, 0.f);
    }
    // wdy = dy*gamma of chunk k as fp32 pairs (d2: dy as pairs, f32 only)
    auto wdy = [&](int k, const uint4 &dv, const f32x2 *d2, f32x2 *w) {
        if constexpr (kF32) {
#pragma unroll
            for (int q = 0; q < P2; ++q) w[q] = f2_mul(d2[q], g2[kF32 ? k : 0][kF32 ? q : 0]);
        } else {
            mul_chunk_pairs<T>(dv, gp[k], w);
        }
    };
    // the head or tail element of this thread (as in the RMSNorm staged kernel)
    const bool e_head = kFold ? w_head && lane < h : tt < h;
    const bool e_tail = kFold ? w_tail && lane >= 32 - tail : tt >= h && tt < h + tail;
    const bool e_own = e_head || e_tail;
    const int je = e_head ? (kFold ? lane : tt)
                          : h + nv * V + (kFold ? lane - (32 - tail) : tt - h);
    const uint32_t e_soff = e_head ? kLnMid - 16u + (uint32_t)(S * (V - h + lane))
                                   : kLnMid + 16u * (uint32_t)nv + (uint32_t)(S * (lane - (32 - tail)));
    const float ge = e_own ? to_f(g[je]) : 0.f;
    float dge = 0.f, dbe = 0.f;
    float xe_n = 0.f, de_n = 0.f;
    auto edge_next = [&](int64_t r) {
        if (!kFold && e_own) {
            const size_t e = (size_t)r * N + je;
            xe_n = to_f(x[e]);
            de_n = to_f(dy[e]);
        }
    };
    if (tn > 0) edge_next(trow0);
    float mu_n = tn > 0 ? __ldg(a.mean + trow0) : 0.f;
    float rs_n = tn > 0 ? __ldg(a.rstd + trow0) : 0.f;

    bool failed = false;
    int64_t j = 0;
    int u = 0;
    uint32_t ph = 0;
    int64_t row = trow0;
    T *dxr = dx + (size_t)trow0 * N;
    for (; j < tn; ++j) {
        // every lane of this warp is done with row j-1: its slot takes row j+Sq-1
        __syncwarp();
        if (lane == 0 && issued < tn) issue();
        const float mu = mu_n, rs = rs_n;
        float xe = xe_n, de = de_n;
        if (j + 1 < tn) {
            mu_n = __ldg(a.mean + row + tstride);
            rs_n = __ldg(a.rstd + row + tstride);
            edge_next(row + tstride);
        }
        const bool ok = mbar_wait_bounded(wbar + 8u * (uint32_t)u, ph, kWaitLimitNs);
        const uint32_t sb = tring + (uint32_t)u * a.stage_bytes;
        const uint32_t sm = sb + kLnMid;
        if (kFold && e_own) {
            const int64_t e0 = row * N + h;
            if (blocks && (e_head ? e0 - V >= 0 : e0 + (int64_t)(nv + 1) * V <= total)) {
                xe = lds_elem<T>(sb + e_soff);
                de = lds_elem<T>(sb + a.tensor_bytes + e_soff);
            } else {
                const size_t e = (size_t)row * N + je;
                xe = to_f(x[e]);
                de = to_f(dy[e]);
            }
        }
        const f32x2 nmu2 = f2_make(-mu, -mu);

        // pass 1: sum (x - mean)*wdy and sum wdy over the row
        f32x2 s1 = f2_make(0.f, 0.f), s2 = f2_make(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                const uint32_t c16 = 16u * (uint32_t)(c0 + lane + 32 * k);
                f32x2 xc[P2], d2[P2], w[P2];
                const uint4 dv = ld_shared_v4(sm + a.tensor_bytes + c16);
                centre_chunk_pairs<T>(ld_shared_v4(sm + c16), nmu2, -mu, xc);
                if (kF32) chunk_pairs<T>(dv, d2);
                wdy(k, dv, d2, w);
#pragma unroll
                for (int q = 0; q < P2; ++q) {
                    s1 = f2_fma(xc[q], w[q], s1);
                    s2 = f2_add(w[q], s2);
                }
            }
        }
        float su, suh, sv, svh;
        f2_split(s1, su, suh);
        f2_split(s2, sv, svh);
        su += suh;
        sv += svh;
        if (e_own) {
            const float w = de * ge;
            su = fmaf(xe - mu, w, su);
            sv += w;
        }
        // the two sums over the team and the team's wait outcome (slots alternate between rows)
        su = warp_sum(su);
        sv = warp_sum(sv);
        const int wok = __all_sync(0xffffffffu, ok);
        const int par = (int)(j & 1);
        if (lane == 0) {
            red[par * 64 + warp] = su;
            red[par * 64 + 32 + warp] = sv;
            okf[par * 32 + warp] = wok;
        }
        named_barrier_sync(1 + team, a.team_threads);
        const bool in = lane < team_warps;
        const float tu = warp_sum(in ? red[par * 64 + first_warp + lane] : 0.f);
        const float tv = warp_sum(in ? red[par * 64 + 32 + first_warp + lane] : 0.f);
        const int o = in ? okf[par * 32 + first_warp + lane] : 1;
        if (!__all_sync(0xffffffffu, o)) {
            failed = true;
            break;
        }

        // dx = wdy*rstd + (x - mean)*B + A with c1 = rstd*tu/N, c2 = tv/N, B = -rstd^2*c1,
        // A = -c2*rstd; partials += dy*x_hat, dy
        const float c1 = rs * tu * a.inv_n, c2 = tv * a.inv_n;
        const float B = -rs * rs * c1, A = -c2 * rs;
        const f32x2 rs2 = f2_make(rs, rs), B2 = f2_make(B, B), A2 = f2_make(A, A);
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                const uint32_t c16 = 16u * (uint32_t)(c0 + lane + 32 * k);
                f32x2 xc[P2], d2[P2], w[P2], o2[P2];
                const uint4 dv = ld_shared_v4(sm + a.tensor_bytes + c16);
                centre_chunk_pairs<T>(ld_shared_v4(sm + c16), nmu2, -mu, xc);
                chunk_pairs<T>(dv, d2);
                wdy(k, dv, d2, w);
#pragma unroll
                for (int q = 0; q < P2; ++q) {
                    o2[q] = f2_fma(w[q], rs2, f2_fma(xc[q], B2, A2));
                    accg[k][q] = f2_fma(d2[q], f2_mul(xc[q], rs2), accg[k][q]);
                    accb[k][q] = f2_add(d2[q], accb[k][q]);
                }
                st_global_v4(dxr + col[k], pairs_chunk<T>(o2));
            }
        }
        if (e_own) {
            const float xcen = xe - mu;
            dxr[je] = from_f<T>(fmaf(de * ge, rs, fmaf(xcen, B, A)));
            dge = fmaf(de, xcen * rs, dge);
            dbe += de;
        }
        if (++u == Sq) {
            u = 0;
            ph ^= 1u;
        }
        row += tstride;
        dxr += tstep;
    }
    pdl_launch_dependents();

    __shared__ int cta_failed;
    if (tid == 0) cta_failed = 0;
    __syncthreads();
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
        if (tt == 0) {
            cta_failed = 1;
            atomicOr(&g_ln_device_status, 1u);
        }
    }
    __syncthreads();  // every copy has landed; the ring is free
    if (cta_failed) return;

    // team t's partials into regions t (dgamma) and teams + t (dbeta), by padded column
    float *reg = reinterpret_cast<float *>(smem + a.ring_off);
    const size_t rw = a.region_words;
    {
        float *rg = reg + (size_t)team * rw, *rb = reg + (size_t)(a.teams + team) * rw;
#pragma unroll
        for (int k = 0; k < J; ++k)
            if (own[k])
#pragma unroll
                for (int q = 0; q < P2; ++q) {
                    f2_split(accg[k][q], rg[vpad(col[k] + 2 * q)], rg[vpad(col[k] + 2 * q + 1)]);
                    f2_split(accb[k][q], rb[vpad(col[k] + 2 * q)], rb[vpad(col[k] + 2 * q + 1)]);
                }
        if (e_own) {
            rg[vpad(je)] = dge;
            rb[vpad(je)] = dbe;
        }
    }
    __syncthreads();
    const int nthr = a.teams * a.team_threads;
    const float *regb = reg + (size_t)a.teams * rw;
    auto colsum = [&](const float *r, int c) {
        float v = r[vpad(c)];
        for (int t = 1; t < a.teams; ++t) v += r[t * rw + vpad(c)];
        return v;
    };
    if (ATOMIC) {
        pdl_wait();  // the zeroing kernel is done with the outputs
        const int n4 = N >> 2;
        for (int i = tid; i < n4; i += nthr) {
            const int c = 4 * i;
            atomicAdd(reinterpret_cast<float4 *>(a.dg_out) + i,
                      make_float4(colsum(reg, c), colsum(reg, c + 1), colsum(reg, c + 2),
                                  colsum(reg, c + 3)));
            if (a.db_out)
                atomicAdd(reinterpret_cast<float4 *>(a.db_out) + i,
                          make_float4(colsum(regb, c), colsum(regb, c + 1), colsum(regb, c + 2),
                                      colsum(regb, c + 3)));
        }
        for (int c = (n4 << 2) + tid; c < N; c += nthr) {
            atomicAdd(a.dg_out + c, colsum(reg, c));
            if (a.db_out) atomicAdd(a.db_out + c, colsum(regb, c));
        }
    } else {
        float *out = a.dg_out + (size_t)blockIdx.x * 2 * N;  // [dgamma | dbeta]
        for (int c = tid; c < N; c += nthr) {
            out[c] = colsum(reg, c);
            out[N + c] = colsum(regb, c);
        }
    }
}

size_t ln_stage_smem_bytes(int N, int dtype, int teams, int slots, uint32_t *tensor_bytes,
                           uint32_t *region_words) {
    const int V = 16 / elem_bytes(dtype);
    const int64_t maxnv = (int64_t)N / V;  // whole chunks of any class's row
    const uint32_t tb = (uint32_t)((kLnMid + (maxnv + 1) * 16 + 127) / 128 * 128);
    const uint32_t rwords = (uint32_t)((vec_words(N) + 31) / 32 * 32);
    if (tensor_bytes) *tensor_bytes = tb;
    if (region_words) *region_words = rwords;
    const size_t ring = (size_t)teams * slots * 2 * tb;
    const size_t regions = (size_t)2 * teams * rwords * 4;
    return ln_stage_ring_offset(slots) + (ring > regions ? ring : regions);
}

template <typename T, bool ATOMIC, int J>
static cudaError_t launch_ln_stage_t(const LnStageArgs &args, const StagePlan &plan,
                                     cudaStream_t s, bool pdl) {
    auto kern = ln_bwd_stage_kernel<T, ATOMIC, J>;
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
static cudaError_t launch_ln_stage_dt(const LnStageArgs &args, const StagePlan &plan,
                                      cudaStream_t s, bool pdl) {
    if (plan.atomic)
        return plan.cpt == 4   ? launch_ln_stage_t<T, true, 4>(args, plan, s, pdl)
               : plan.cpt == 2 ? launch_ln_stage_t<T, true, 2>(args, plan, s, pdl)
                               : launch_ln_stage_t<T, true, 1>(args, plan, s, pdl);
    return plan.cpt == 4   ? launch_ln_stage_t<T, false, 4>(args, plan, s, pdl)
           : plan.cpt == 2 ? launch_ln_stage_t<T, false, 2>(args, plan, s, pdl)
                           : launch_ln_stage_t<T, false, 1>(args, plan, s, pdl);
}

template <typename T>
static const void *ln_stage_kernel_ptr(bool atomic, int cpt) {
    if (cpt == 4)
        return atomic ? (const void *)ln_bwd_stage_kernel<T, true, 4>
                      : (const void *)ln_bwd_stage_kernel<T, false, 4>;
    if (cpt == 2)
        return atomic ? (const void *)ln_bwd_stage_kernel<T, true, 2>
                      : (const void *)ln_bwd_stage_kernel<T, false, 2>;
    return atomic ? (const void *)ln_bwd_stage_kernel<T, true, 1>
                  : (const void *)ln_bwd_stage_kernel<T, false, 1>;
}

int ln_stage_blocks_per_sm(int dtype, bool atomic, int cpt, int threads, size_t smem) {
    const void *k = dtype == kF32 ? ln_stage_kernel_ptr<float>(atomic, cpt)
                  : dtype == kF16 ? ln_stage_kernel_ptr<__half>(atomic, cpt)
                                  : ln_stage_kernel_ptr<__nv_bfloat16>(atomic, cpt);
    int n = 0;
    if (ensure_smem_attr(k, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess ||
        n < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    return n;
}

cudaError_t launch_ln_bwd_stage(const LnBwdProblem &p, const StagePlan &plan, cudaStream_t s,
                                bool pdl_after_zero) {
    LnStageArgs a;
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
    a.teams = plan.teams;
    a.team_threads = plan.team_threads;
    a.slots = plan.slots;
    a.skip_row = plan.skip_row;
    const int V = 16 / elem_bytes(p.dtype);
    const size_t need = ln_stage_smem_bytes(p.N, p.dtype, plan.teams, plan.slots,
                                            &a.tensor_bytes, &a.region_words);
    a.stage_bytes = 2 * a.tensor_bytes;
    a.ring_off = ln_stage_ring_offset(plan.slots);
    // the launch shape the kernel relies on (as for the RMSNorm staged kernel)
    const int64_t maxnv = (int64_t)p.N / V;
    if (plan.cpt != 1 && plan.cpt != 2 && plan.cpt != 4) return cudaErrorInvalidValue;
    if (plan.team_threads < 32 || plan.team_threads % 32 || plan.teams < 1 || plan.teams > 15 ||
        plan.teams * plan.team_threads > 512)
        return cudaErrorInvalidValue;
    if ((int64_t)plan.cpt * plan.team_threads < maxnv) return cudaErrorInvalidValue;
    if (plan.slots < 2 || plan.slots > 4) return cudaErrorInvalidValue;
    if (plan.smem < need) return cudaErrorInvalidValue;
    if (p.M > 0 && plan.grid < (p.M < a.period ? p.M : a.period)) return cudaErrorInvalidValue;
    switch (p.dtype) {
    case kF32: return launch_ln_stage_dt<float>(a, plan, s, pdl_after_zero);
    case kF16: return launch_ln_stage_dt<__half>(a, plan, s, pdl_after_zero);
    case kBF16: return launch_ln_stage_dt<__nv_bfloat16>(a, plan, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t take_ln_device_status(unsigned int *status) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_ln_device_status, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_ln_device_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
    *status = v;
    return cudaSuccess;
}

}  // namespace rn
