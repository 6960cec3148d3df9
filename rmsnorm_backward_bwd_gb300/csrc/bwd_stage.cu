// Backward staged phase-class kernel: rows that are not 16-byte multiples (or
// whose base is off a 16-byte boundary), every row tensor at one alignment
// phase, at most 2048 whole 16-byte chunks per row. RMSNorm and fused-add
// RMSNorm backward.
//
// Math per row (FlyDSL issue #769, section "Math"): with x_hat = x*rstd and
// wdy = dy*gamma, c1 = mean_j(x_hat*wdy) and dx = (wdy - x_hat*c1)*rstd; the
// weight gradient sums dy*x_hat over rows. Fused-add (PR #800, "What's
// included"): the same on the saved `added`, plus dresidual_out on dx.
//
// Design (sm_103a):
//   * Row r starts at byte r*N*s past the base, so its alignment phase repeats
//     with period P = 16 / gcd(16, N*s mod 16) rows. CTA b takes the rows of
//     residue class b mod P. Within a class every row splits the same way
//     into h head elements, nv whole 16-byte chunks and a few tail elements.
//   * Persistent grid. A CTA holds `teams` teams (named barriers 1..teams);
//     a team owns one row at a time and walks the CTA's rows with stride
//     `teams`. Warp w of a team owns the contiguous chunks [w*32J, (w+1)*32J)
//     of the row's whole-chunk middle; lane l takes chunks w*32J + l + 32k.
//   * Each warp stages its own span of the team's next rows in shared memory
//     with bulk copies (cp.async.bulk, one per streamed tensor and row,
//     issued by lane 0, completing on the warp's own mbarrier of the slot).
//     A team has `Sq` slots; at the top of row j the warp refills the slot it
//     finished with in row j-1 with row j+Sq-1, so no barrier guards the
//     ring: only the warp itself reads what it copied. The 16-byte blocks
//     that hold the row's head and tail elements (fewer than 16 per row)
//     ride on the first warp's and the last warp's copies, which start 16
//     bytes early and end 16 bytes late; lanes of those warps own the
//     elements. A block that would reach outside the tensor (the first and
//     last rows) is not copied and its lanes read their elements from global
//     memory. rstd is loaded one row ahead.
//   * Pass 1 sums x*dy*gamma over the row (warp shuffles, then the team's
//     named barrier); pass 2 reads the slot again and stores dx with 16-byte
//     stores (the class's chunks are 16-byte aligned in every row tensor).
//     The chunk arithmetic is the row engine's packed-pair RowMath.
//   * Every wait on an mbarrier is bounded in time. A warp whose wait runs
//     out tells its team through the row sum's exchange; the team stops, its
//     issuing lanes wait (again bounded) for the copies they still have in
//     flight, the kernel ORs 1 into the library's device status word and the
//     CTA skips its weight-gradient output. The host reads the word with
//     rn_take_device_status().
//   * The weight-gradient partial of a thread's columns stays in fp32
//     registers. At the end each team stores its partial in its own region of
//     the drained ring, by column with one pad word per 32 columns (lanes 8
//     columns apart hit distinct banks), and the CTA sums the teams' regions
//     column by column in team order: fp32 vector atomics into dweight_f32, or
//     one partial row of the workspace for the finalize kernel.
#include "common.cuh"
#include "launch.h"
#include "row_math.cuh"
#include "stage.cuh"
#include "unaligned.cuh"

namespace rn {

// Device status word (bit 0: a bounded wait ran out); read and cleared by
// rn_take_device_status().
__device__ unsigned int g_device_status;

namespace {

// Shared memory: [0,256) warp sums [2 parities][32 warps]; [256,512) wait
// outcomes, same layout; [512, 512 + 8*16*Sq) the warps' full barriers
// (warp w, slot u at w*Sq + u); the ring from stage_ring_offset(Sq): team t's
// slot u at (t*Sq + u)*stage_bytes, tensor k of a slot at k*tensor_bytes;
// within a tensor whole chunk i at kMid + 16i, the head block just before
// chunk 0 and the tail block just after the last whole chunk.
constexpr uint32_t kStageBarOffset = 512;
// Within a tensor's slot: the whole chunks from byte kMid (128-byte aligned, as the bulk copies
// of the chunks land), the head block just before them, the tail block just after.
constexpr uint32_t kMid = 128;

}  // namespace

uint32_t stage_ring_offset(int slots) {
    return (kStageBarOffset + 8u * 16u * (uint32_t)slots + 127u) / 128u * 128u;
}

struct StageArgs {
    const void *x;
    const void *gamma;
    const void *dy;
    const float *rstd;
    const void *dres;
    void *dx;
    float *dw_out;        // scratch: partial rows [gridDim.x][N]; atomic: dweight_f32
    int64_t M;
    int N;
    float inv_n;
    int period;           // P
    int teams;
    int team_threads;
    int slots;            // Sq
    uint32_t tensor_bytes;
    uint32_t stage_bytes;
    uint32_t ring_off;
    uint32_t region_words;  // one team's padded weight-gradient region
    int64_t skip_row;     // test hook: CTA 0 team 0's local row whose copies its warp 0 never
                          // issues (its wait runs out); -1 = off
};

template <typename T, bool HAS_DRES, bool ATOMIC, int J>
__global__ void __launch_bounds__(512, 1) bwd_stage_kernel(const StageArgs a) {
    constexpr int S = sizeof(T), V = 16 / S;
    constexpr int P2 = RowMath<T>::kPairs;  // fp32 pairs per chunk
    constexpr int NT = HAS_DRES ? 3 : 2;
    // gamma also as fp32 pairs when the math needs it or when that fits
    constexpr bool kGammaF = RowMath<T>::kNeedsGammaF || J * V <= 8;
    // The head and tail elements come with the bulk copies (kFold) or are loaded one row ahead
    // into registers by lanes of the team's first warp. Measured on GB300 (us per call, registers
    // -> folded): bf16 4096 x 4095 27.6 -> 25.1, 4096 x 12290 66.6 -> 58.3, f16 16384 x 1001
    // 28.4 -> 27.2, f32 fused 4096 x 4095 +dres 43.3 -> 40.5; plain f32 loses (4096 x 4095
    // 31.9 -> 35.0, 8192 x 6001 94.1 -> 101.5, 4096 x 2047 21.5 -> 23.6), so it keeps registers.
    constexpr bool kFold = S == 2 || HAS_DRES;
    extern __shared__ __align__(128) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    int *okf = reinterpret_cast<int *>(smem + 256);
    const T *x = static_cast<const T *>(a.x);
    const T *g = static_cast<const T *>(a.gamma);
    const T *dy = static_cast<const T *>(a.dy);
    const T *dres = static_cast<const T *>(a.dres);
    T *dx = static_cast<T *>(a.dx);
    const int tid = threadIdx.x;
    const int N = a.N, P = a.period, Sq = a.slots;

    // this CTA's rows: row0 + k*rstride (k < nrows), all of class cls
    const int cls = (int)(blockIdx.x % (unsigned)P);
    const int64_t nper = ((int64_t)gridDim.x - cls + P - 1) / P;  // CTAs of this class
    const int64_t rstride = nper * P;
    const int64_t row0 = cls + (int64_t)(blockIdx.x / (unsigned)P) * P;
    const int64_t nrows = row0 < a.M ? (a.M - 1 - row0) / rstride + 1 : 0;
    // the class's split (address arithmetic on row cls; nothing is read there): h head
    // elements before the first 16-byte boundary, nv whole chunks, `tail` elements after
    const uintptr_t start = reinterpret_cast<uintptr_t>(a.x) + (uintptr_t)cls * (uintptr_t)N * S;
    const int h_free = (int)(((16u - (unsigned)(start & 15u)) & 15u) / S);
    // A row that holds a 16-byte boundary has its head in the 16-byte block that ends at the
    // first boundary and its tail in the block that starts at the last one; those blocks are
    // copied with the row wherever they lie inside the tensor.
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
    const uint32_t wbar = smem_addr(smem + kStageBarOffset) + 8u * (uint32_t)(warp * Sq);
    const uint32_t tring = smem_addr(smem + a.ring_off) + (uint32_t)(team * Sq) * a.stage_bytes;

    if (lane == 0) {
        for (int u = 0; u < Sq; ++u) mbar_init(wbar + 8u * u, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Lane 0: copies of this warp's span of the team's rows, in order. Folded edges: the team's
    // first warp also copies the head block (its copy starts 16 bytes early), the warp holding
    // the last whole chunk the tail block (its copy ends 16 bytes late), where they lie inside
    // the tensor.
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
                tring + (uint32_t)iu * a.stage_bytes + kMid + 16u * (uint32_t)c0 - (hb ? 16u : 0u);
            mbar_arrive_expect_tx(bar, NT * nbytes);
            bulk_copy_g2s(dst, x + off, nbytes, bar, policy);
            bulk_copy_g2s(dst + a.tensor_bytes, dy + off, nbytes, bar, policy);
            if (HAS_DRES) bulk_copy_g2s(dst + 2 * a.tensor_bytes, dres + off, nbytes, bar, policy);
        }
        ++issued;
        irow_e0 += tstep;
        if (++iu == Sq) iu = 0;
    };
    if (lane == 0)
        while (issued < Sq - 1 && issued < tn) issue();

    // this thread's chunks (lane + 32k of the warp's span) and its head or tail element
    bool own[J];
    int col[J];
    uint4 gp[J];
    f32x2 g2[kGammaF ? J : 1][kGammaF ? P2 : 1];
    f32x2 acc2[J][P2];
#pragma unroll
    for (int k = 0; k < J; ++k) {
        own[k] = lane + 32 * k < wn;
        col[k] = h + (c0 + lane + 32 * k) * V;
        gp[k] = own[k] ? gather_chunk<T>(g + col[k]) : make_uint4(0, 0, 0, 0);
        if (kGammaF) {
            float gf[V];
            chunk_to_float<T>(gp[k], gf);
#pragma unroll
            for (int q = 0; q < P2; ++q)
                g2[kGammaF ? k : 0][kGammaF ? q : 0] = f2_make(gf[2 * q], gf[2 * q + 1]);
        }
#pragma unroll
        for (int q = 0; q < P2; ++q) acc2[k][q] = f2_make(0.f, 0.f);
    }
    // the head or tail element of this thread and its column. Folded: head elements on the
    // first lanes of the team's first warp, tail elements on the last lanes of the warp that
    // copies the tail block (each reads only what its own warp copied), with the element's byte
    // offset in a tensor's slot. Otherwise: the first h + tail threads of the team.
    const bool e_head = kFold ? w_head && lane < h : tt < h;
    const bool e_tail = kFold ? w_tail && lane >= 32 - tail : tt >= h && tt < h + tail;
    const bool e_own = e_head || e_tail;
    const int je = e_head ? (kFold ? lane : tt)
                          : h + nv * V + (kFold ? lane - (32 - tail) : tt - h);
    const uint32_t e_soff = e_head ? kMid - 16u + (uint32_t)(S * (V - h + lane))
                                   : kMid + 16u * (uint32_t)nv + (uint32_t)(S * (lane - (32 - tail)));
    const float ge = e_own ? to_f(g[je]) : 0.f;
    float dwe = 0.f;
    // registers: the team's next row's head or tail element
    float xe_n = 0.f, de_n = 0.f, re_n = 0.f;
    auto edge_next = [&](int64_t r) {
        if (!kFold && e_own) {
            const size_t e = (size_t)r * N + je;
            xe_n = to_f(x[e]);
            de_n = to_f(dy[e]);
            if (HAS_DRES) re_n = to_f(dres[e]);
        }
    };
    if (tn > 0) edge_next(trow0);

    // rstd of the team's next row, one row ahead
    float rs_n = tn > 0 ? __ldg(a.rstd + trow0) : 0.f;

    bool failed = false;
    int64_t j = 0;
    int u = 0;          // slot of row j
    uint32_t ph = 0;    // parity of its use
    int64_t row = trow0;
    T *dxr = dx + (size_t)trow0 * N;
    for (; j < tn; ++j) {
        // every lane of this warp is done with row j-1: its slot takes row j+Sq-1
        __syncwarp();
        if (lane == 0 && issued < tn) issue();
        const float rs = rs_n;
        float xe = xe_n, de = de_n, re = re_n;
        if (j + 1 < tn) {
            rs_n = __ldg(a.rstd + row + tstride);
            edge_next(row + tstride);
        }
        const bool ok = mbar_wait_bounded(wbar + 8u * (uint32_t)u, ph, kWaitLimitNs);
        const uint32_t sb = tring + (uint32_t)u * a.stage_bytes;
        const uint32_t sm = sb + kMid;  // the row's whole chunks
        // folded: this row's head or tail element from its copied block, or (a block that would
        // reach outside the tensor: the first and last rows) from global memory
        bool e_smem = false;
        if (kFold && e_own) {
            const int64_t e0 = row * N + h;
            e_smem = blocks && (e_head ? e0 - V >= 0 : e0 + (int64_t)(nv + 1) * V <= total);
            if (e_smem) {
                xe = lds_elem<T>(sb + e_soff);
                de = lds_elem<T>(sb + a.tensor_bytes + e_soff);
                if (HAS_DRES) re = lds_elem<T>(sb + 2 * a.tensor_bytes + e_soff);
            } else {
                const size_t e = (size_t)row * N + je;
                xe = to_f(x[e]);
                de = to_f(dy[e]);
                if (HAS_DRES) re = to_f(dres[e]);
            }
        }
        f32x2 part2 = f2_make(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < J; ++k) {
            const uint32_t c16 = 16u * (uint32_t)(c0 + lane + 32 * k);
            if (own[k])
                part2 = RowMath<T>::pass1(ld_shared_v4(sm + c16), ld_shared_v4(sm + a.tensor_bytes + c16),
                                          gp[k], kGammaF ? g2[kGammaF ? k : 0] : nullptr, part2);
        }
        float plo, phi;
        f2_split(part2, plo, phi);
        float sv = plo + phi;
        if (e_own) sv = fmaf(xe * de, ge, sv);
        // team sum and the team's wait outcome (slots alternate between rows)
        const float wsum = warp_sum(sv);
        const int wok = __all_sync(0xffffffffu, ok);
        const int par = (int)(j & 1);
        if (lane == 0) {
            red[par * 32 + warp] = wsum;
            okf[par * 32 + warp] = wok;
        }
        named_barrier_sync(1 + team, a.team_threads);
        const float w = lane < team_warps ? red[par * 32 + first_warp + lane] : 0.f;
        const int o = lane < team_warps ? okf[par * 32 + first_warp + lane] : 1;
        const float part = warp_sum(w);
        if (!__all_sync(0xffffffffu, o)) {
            failed = true;
            break;
        }

        // dx = wdy*rstd + x*b with b = -rstd^2*c1 (+ dres); partial += dy*x_hat
        const float c1 = rs * part * a.inv_n;
        const float b = -rs * rs * c1;
        const f32x2 rs2 = f2_make(rs, rs), b2 = f2_make(b, b);
#pragma unroll
        for (int k = 0; k < J; ++k) {
            if (own[k]) {
                const uint32_t c16 = 16u * (uint32_t)(c0 + lane + 32 * k);
                const uint4 r = HAS_DRES ? ld_shared_v4(sm + 2 * a.tensor_bytes + c16)
                                         : make_uint4(0, 0, 0, 0);
                const uint4 out = RowMath<T>::template pass2<HAS_DRES>(
                    ld_shared_v4(sm + c16), ld_shared_v4(sm + a.tensor_bytes + c16), r, gp[k],
                    kGammaF ? g2[kGammaF ? k : 0] : nullptr, rs2, b2, acc2[k]);
                st_global_v4(dxr + col[k], out);
            }
        }
        if (e_own) {
            float d = fmaf(xe, b, (de * ge) * rs);
            if (HAS_DRES) d += re;
            dxr[je] = from_f<T>(d);
            dwe = fmaf(xe * de, rs, dwe);
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
            atomicOr(&g_device_status, 1u);
        }
    }
    __syncthreads();  // every copy has landed; the ring is free
    if (cta_failed) return;

    // team t's partial into region t, by padded column
    float *reg = reinterpret_cast<float *>(smem + a.ring_off);
    {
        float *mine = reg + (size_t)team * a.region_words;
#pragma unroll
        for (int k = 0; k < J; ++k)
            if (own[k])
#pragma unroll
                for (int q = 0; q < P2; ++q)
                    f2_split(acc2[k][q], mine[vpad(col[k] + 2 * q)], mine[vpad(col[k] + 2 * q + 1)]);
        if (e_own) mine[vpad(je)] = dwe;
    }
    __syncthreads();
    const int nthr = a.teams * a.team_threads;
    const size_t rw = a.region_words;
    if (ATOMIC) {
        pdl_wait();  // the zeroing kernel is done with dweight_f32
        const int n4 = N >> 2;
        for (int i = tid; i < n4; i += nthr) {
            const int c = 4 * i;
            float4 v = make_float4(reg[vpad(c)], reg[vpad(c + 1)], reg[vpad(c + 2)], reg[vpad(c + 3)]);
            for (int t = 1; t < a.teams; ++t) {
                const float *o = reg + t * rw;
                v.x += o[vpad(c)];
                v.y += o[vpad(c + 1)];
                v.z += o[vpad(c + 2)];
                v.w += o[vpad(c + 3)];
            }
            atomicAdd(reinterpret_cast<float4 *>(a.dw_out) + i, v);
        }
        for (int c = (n4 << 2) + tid; c < N; c += nthr) {
            float v = reg[vpad(c)];
            for (int t = 1; t < a.teams; ++t) v += reg[t * rw + vpad(c)];
            atomicAdd(a.dw_out + c, v);
        }
    } else {
        float *out = a.dw_out + (size_t)blockIdx.x * N;
        for (int c = tid; c < N; c += nthr) {
            float v = reg[vpad(c)];
            for (int t = 1; t < a.teams; ++t) v += reg[t * rw + vpad(c)];
            out[c] = v;
        }
    }
}

size_t stage_smem_bytes(int N, int dtype, bool dres, int teams, int slots, int cpt,
                        int team_threads, uint32_t *tensor_bytes, uint32_t *region_words) {
    const int V = 16 / elem_bytes(dtype);
    const int64_t maxnv = (int64_t)N / V;  // whole chunks of any class's row
    (void)cpt;
    (void)team_threads;
    // a tensor's slot: the head block, the whole chunks, the tail block
    const uint32_t tb = (uint32_t)((kMid + (maxnv + 1) * 16 + 127) / 128 * 128);
    const uint32_t rwords = (uint32_t)((vec_words(N) + 31) / 32 * 32);
    if (tensor_bytes) *tensor_bytes = tb;
    if (region_words) *region_words = rwords;
    const size_t ring = (size_t)teams * slots * (dres ? 3 : 2) * tb;
    const size_t regions = (size_t)teams * rwords * 4;
    return stage_ring_offset(slots) + (ring > regions ? ring : regions);
}

template <typename T, bool HAS_DRES, bool ATOMIC, int J>
static cudaError_t launch_stage_t(const StageArgs &args, const StagePlan &plan, cudaStream_t s,
                                  bool pdl) {
    auto kern = bwd_stage_kernel<T, HAS_DRES, ATOMIC, J>;
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

template <typename T, bool HAS_DRES, bool ATOMIC>
static cudaError_t launch_stage_j(const StageArgs &args, const StagePlan &plan, cudaStream_t s,
                                  bool pdl) {
    switch (plan.cpt) {
    case 1: return launch_stage_t<T, HAS_DRES, ATOMIC, 1>(args, plan, s, pdl);
    case 2: return launch_stage_t<T, HAS_DRES, ATOMIC, 2>(args, plan, s, pdl);
    case 4: return launch_stage_t<T, HAS_DRES, ATOMIC, 4>(args, plan, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
static cudaError_t launch_stage_dt(const StageArgs &args, const StagePlan &plan, bool has_dres,
                                   cudaStream_t s, bool pdl) {
    if (plan.atomic)
        return has_dres ? launch_stage_j<T, true, true>(args, plan, s, pdl)
                        : launch_stage_j<T, false, true>(args, plan, s, pdl);
    return has_dres ? launch_stage_j<T, true, false>(args, plan, s, pdl)
                    : launch_stage_j<T, false, false>(args, plan, s, pdl);
}

cudaError_t launch_bwd_stage(const BwdProblem &p, const StagePlan &plan, cudaStream_t s,
                             bool pdl_after_zero) {
    StageArgs a;
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
    a.teams = plan.teams;
    a.team_threads = plan.team_threads;
    a.slots = plan.slots;
    a.skip_row = plan.skip_row;
    const int V = 16 / elem_bytes(p.dtype);
    const bool has_dres = p.dres != nullptr;
    const size_t need = stage_smem_bytes(p.N, p.dtype, has_dres, plan.teams, plan.slots, plan.cpt,
                                         plan.team_threads, &a.tensor_bytes, &a.region_words);
    a.stage_bytes = (has_dres ? 3 : 2) * a.tensor_bytes;
    a.ring_off = stage_ring_offset(plan.slots);
    // the launch shape the kernel relies on: every chunk owned, named barrier IDs 1..15, the
    // head and tail elements in the team's first warp, two or more slots, every residue
    // class with a CTA, and the shared memory it indexes
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
    case kF32: return launch_stage_dt<float>(a, plan, has_dres, s, pdl_after_zero);
    case kF16: return launch_stage_dt<__half>(a, plan, has_dres, s, pdl_after_zero);
    case kBF16: return launch_stage_dt<__nv_bfloat16>(a, plan, has_dres, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
static const void *stage_kernel_ptr(bool dres, bool atomic, int cpt) {
    if (cpt == 4)
        return dres ? (atomic ? (const void *)bwd_stage_kernel<T, true, true, 4>
                              : (const void *)bwd_stage_kernel<T, true, false, 4>)
                    : (atomic ? (const void *)bwd_stage_kernel<T, false, true, 4>
                              : (const void *)bwd_stage_kernel<T, false, false, 4>);
    if (cpt == 2)
        return dres ? (atomic ? (const void *)bwd_stage_kernel<T, true, true, 2>
                              : (const void *)bwd_stage_kernel<T, true, false, 2>)
                    : (atomic ? (const void *)bwd_stage_kernel<T, false, true, 2>
                              : (const void *)bwd_stage_kernel<T, false, false, 2>);
    return dres ? (atomic ? (const void *)bwd_stage_kernel<T, true, true, 1>
                          : (const void *)bwd_stage_kernel<T, true, false, 1>)
                : (atomic ? (const void *)bwd_stage_kernel<T, false, true, 1>
                          : (const void *)bwd_stage_kernel<T, false, false, 1>);
}

int stage_blocks_per_sm(int dtype, bool dres, bool atomic, int cpt, int threads, size_t smem) {
    const void *k = dtype == kF32 ? stage_kernel_ptr<float>(dres, atomic, cpt)
                  : dtype == kF16 ? stage_kernel_ptr<__half>(dres, atomic, cpt)
                                  : stage_kernel_ptr<__nv_bfloat16>(dres, atomic, cpt);
    int n = 0;
    if (ensure_smem_attr(k, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess ||
        n < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    return n;
}

cudaError_t take_device_status(unsigned int *status) {
    unsigned int v = 0, zero = 0, ln = 0, fw = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
    e = take_ln_device_status(&ln);  // the LayerNorm staged kernel's word
    if (e != cudaSuccess) return e;
    e = take_fwd_device_status(&fw);  // the forward staged kernel's word
    if (e != cudaSuccess) return e;
    *status = v | ln | fw;
    return cudaSuccess;
}

}  // namespace rn
