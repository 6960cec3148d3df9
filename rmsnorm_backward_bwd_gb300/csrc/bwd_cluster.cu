// Backward cluster engine: RMSNorm (and fused-add) backward for rows too long
// for one CTA's tile of the row engine (more than 2048 16-byte chunks).
//
// Same math as the row engine (FlyDSL issue #769 "Math"; PR #800 "What's
// included"), with a row split across a thread-block cluster of C CTAs
// (C = 2..16):
//   * CTA r of a cluster owns chunks [r*slice, (r+1)*slice) of every row its
//     cluster handles; its threads own chunks tid + k*blockDim.x of that slice.
//     Clusters walk rows with a stride of the cluster count.
//   * Each thread streams its chunks of the next rows into its own
//     shared-memory ring with 16-byte cp.async (as in the row engine: no
//     barrier or mbarrier guards the ring).
//   * Pass 1 sums x*dy*gamma over the CTA's slice; each warp's sum goes to
//     shared memory; one cluster barrier per row (barrier.cluster, a hardware
//     barrier every thread of the cluster reaches) publishes them; then lane
//     l of every warp reads partial l of the cluster's C x warps partials
//     through distributed shared memory and a warp butterfly adds them, so
//     every warp of every CTA gets the same bits. The partial slots are
//     double-buffered by row parity.
//   * (Pipelining rows around a split arrive/wait of the barrier was measured
//     slower: keeping two rows resident leaves one row fewer in flight.)
//   * Pass 2 stores dx for the slice and adds dy*x_hat into fp32 registers;
//     at the end each CTA writes its slice of the weight-gradient partial
//     (scratch: one partial row per cluster; atomic: fp32 vector atomics).
//   * A last cluster barrier keeps every CTA alive until its peers have read
//     its partial slots.
#include "cluster.cuh"
#include "common.cuh"
#include "launch.h"
#include "row_math.cuh"

namespace rn {

constexpr int kClusterRingOffset = 256;  // [2 parities][16 warps] fp32 warp sums first

size_t cluster_smem_bytes(int stages, int ntensors, int cpt, int threads) {
    return (size_t)kClusterRingOffset + (size_t)stages * ntensors * cpt * threads * 16;
}

struct ClusterArgs {
    const uint8_t *x;
    const uint8_t *gamma;
    const uint8_t *dy;
    const float *rstd;
    const uint8_t *dres;
    uint8_t *dx;
    float *dw_out;  // scratch: partial rows [clusters][N]; atomic: dweight_f32
    int64_t M;
    int N;
    int nchunks;
    int row_bytes;
    int slice;      // chunks per CTA slice
    int stages;
    float inv_n;
};

template <typename T, int CPT, bool HAS_DRES, bool ATOMIC>
__global__ void __launch_bounds__(512, 1) bwd_cluster_kernel(const ClusterArgs a) {
    constexpr int V = Traits<T>::kVec;
    constexpr int P = RowMath<T>::kPairs;
    constexpr int NT = HAS_DRES ? 3 : 2;
    constexpr bool kGammaF = RowMath<T>::kNeedsGammaF || CPT * V <= 8;
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    uint8_t *ring = smem + kClusterRingOffset;

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
    const uint32_t slot_bytes = NT * tensor_bytes;
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
        if (j < nrows) issue(cid + j * ncl, j);
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

    const int64_t ahead = (int64_t)(S - 1) * ncl;
    const int nparts = csize * nwarps;  // <= 16 x 16
    float rs_next = nrows > 0 ? __ldg(a.rstd + cid) : 0.f;
    int slot = 0, fill = S - 1;
    int64_t row = cid;
    for (int64_t k = 0; k < nrows; ++k, row += ncl) {
        // refill the slot finished in the previous row, then wait for this row
        if (k + S - 1 < nrows) issue(row + ahead, fill);
        cp_async_commit();
        const float rs = rs_next;
        if (k + 1 < nrows) rs_next = __ldg(a.rstd + row + ncl);
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
        const float wsum = warp_sum(plo + phi);
        const int par = (int)(k & 1) * 16;
        if (lane == 0) red[par + warp] = wsum;
        cluster_sync_all();
        float t = 0.f;
        for (int i = lane; i < nparts; i += 32) {
            const int r = i / nwarps, w = i - r * nwarps;
            t += ld_peer_f32(red_addr + 4u * (par + w), (uint32_t)r);
        }
        const float part = warp_sum(t);

        const float c1v = rs * part * a.inv_n;
        const float b = -rs * rs * c1v;
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
    // peers may still read this CTA's partial slots of the last row
    cluster_sync_all();

    pdl_launch_dependents();
    if (ATOMIC) pdl_wait();  // the zeroing kernel ahead of this one has finished
    float *out_row = ATOMIC ? a.dw_out : a.dw_out + (size_t)cid * a.N;
#pragma unroll
    for (int kk = 0; kk < CPT; ++kk) {
        if (cok[kk]) {
            const int c = c0 + tid + kk * nthr;
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
}

template <typename T, int CPT, bool HAS_DRES, bool ATOMIC>
static const void *cluster_kernel_ptr() {
    return (const void *)bwd_cluster_kernel<T, CPT, HAS_DRES, ATOMIC>;
}

template <typename T, int CPT, bool HAS_DRES, bool ATOMIC>
static cudaError_t launch_cluster_t(const ClusterArgs &args, const ClusterPlan &plan,
                                    cudaStream_t s, bool pdl) {
    auto kern = bwd_cluster_kernel<T, CPT, HAS_DRES, ATOMIC>;
    cudaError_t e = ensure_smem_attr((const void *)kern, plan.smem);
    if (e != cudaSuccess) return e;
    if (plan.csize > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
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

template <typename T, int CPT>
static cudaError_t launch_cluster_cpt(const ClusterArgs &args, const ClusterPlan &plan,
                                      bool has_dres, cudaStream_t s, bool pdl) {
    if (plan.atomic)
        return has_dres ? launch_cluster_t<T, CPT, true, true>(args, plan, s, pdl)
                        : launch_cluster_t<T, CPT, false, true>(args, plan, s, pdl);
    return has_dres ? launch_cluster_t<T, CPT, true, false>(args, plan, s, pdl)
                    : launch_cluster_t<T, CPT, false, false>(args, plan, s, pdl);
}

template <typename T>
static cudaError_t launch_cluster_dt(const ClusterArgs &args, const ClusterPlan &plan,
                                     bool has_dres, cudaStream_t s, bool pdl) {
    switch (plan.cpt) {
    case 1: return launch_cluster_cpt<T, 1>(args, plan, has_dres, s, pdl);
    case 2: return launch_cluster_cpt<T, 2>(args, plan, has_dres, s, pdl);
    case 4: return launch_cluster_cpt<T, 4>(args, plan, has_dres, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
static const void *cluster_kernel_for(int cpt, bool has_dres, bool atomic) {
    // the (cpt, dres, atomic) instance the launcher would pick
    if (cpt == 1)
        return has_dres ? (atomic ? cluster_kernel_ptr<T, 1, true, true>() : cluster_kernel_ptr<T, 1, true, false>())
                        : (atomic ? cluster_kernel_ptr<T, 1, false, true>() : cluster_kernel_ptr<T, 1, false, false>());
    if (cpt == 2)
        return has_dres ? (atomic ? cluster_kernel_ptr<T, 2, true, true>() : cluster_kernel_ptr<T, 2, true, false>())
                        : (atomic ? cluster_kernel_ptr<T, 2, false, true>() : cluster_kernel_ptr<T, 2, false, false>());
    return has_dres ? (atomic ? cluster_kernel_ptr<T, 4, true, true>() : cluster_kernel_ptr<T, 4, true, false>())
                    : (atomic ? cluster_kernel_ptr<T, 4, false, true>() : cluster_kernel_ptr<T, 4, false, false>());
}

cudaError_t cluster_max_active(const BwdProblem &p, const ClusterPlan &plan, int *clusters) {
    const void *kern = nullptr;
    switch (p.dtype) {
    case kF32: kern = cluster_kernel_for<float>(plan.cpt, p.dres != nullptr, plan.atomic); break;
    case kF16: kern = cluster_kernel_for<__half>(plan.cpt, p.dres != nullptr, plan.atomic); break;
    case kBF16: kern = cluster_kernel_for<__nv_bfloat16>(plan.cpt, p.dres != nullptr, plan.atomic); break;
    default: return cudaErrorInvalidValue;
    }
    cudaError_t e = ensure_smem_attr(kern, plan.smem);
    if (e != cudaSuccess) return e;
    if (plan.csize > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
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

cudaError_t launch_bwd_cluster(const BwdProblem &p, const ClusterPlan &plan, cudaStream_t s,
                               bool pdl_after_zero) {
    ClusterArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.dy = static_cast<const uint8_t *>(p.dy);
    a.rstd = p.rstd;
    a.dres = static_cast<const uint8_t *>(p.dres);
    a.dx = static_cast<uint8_t *>(p.dx);
    a.dw_out = plan.atomic ? p.dw_f32 : reinterpret_cast<float *>(p.ws + kWsHeaderBytes);
    a.M = p.M;
    a.N = p.N;
    a.row_bytes = p.N * elem_bytes(p.dtype);
    a.nchunks = a.row_bytes / 16;
    a.slice = plan.slice;
    a.stages = plan.stages;
    a.inv_n = 1.0f / (float)p.N;
    const bool has_dres = p.dres != nullptr;
    switch (p.dtype) {
    case kF32: return launch_cluster_dt<float>(a, plan, has_dres, s, pdl_after_zero);
    case kF16: return launch_cluster_dt<__half>(a, plan, has_dres, s, pdl_after_zero);
    case kBF16: return launch_cluster_dt<__nv_bfloat16>(a, plan, has_dres, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
