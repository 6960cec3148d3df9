// Backward realigning engine: rows whose byte length is not a multiple of 16
// (so consecutive rows start at different offsets within a 16-byte line),
// with x, dy, dx and dresidual_out at one common alignment phase. Run only
// when asked for (RN_OPT_GENERIC_KERNEL = 3): the phase-class kernel covers
// its 16-32 KB rows faster.
//
// Same math as the row engine (FlyDSL issue #769 "Math"; fused-add from
// PR #800 "What's included"), and the same per-chunk arithmetic (RowMath).
// What differs is how a row reaches fixed columns:
//   - the row's aligned 16-byte chunks are loaded with 128-bit loads and
//     stored to a shared-memory row buffer at aligned offsets; the few
//     elements before the first 16-byte boundary (head) and after the last
//     whole chunk (tail) go element by element;
//   - a thread owns fixed column blocks (16 bytes of columns each, as in the
//     row engine) and reads a block back with two aligned 16-byte shared loads
//     and a funnel shift by the row's phase;
//   - dx blocks are written to a second, block-aligned shared buffer and go
//     out to global memory as aligned 16-byte chunks read back the same way
//     (head and tail element by element).
// With fixed columns, gamma is read once per thread and the weight-gradient
// partial stays in registers, as in the row engine. One CTA is one team;
// R rows are processed per iteration (the planner uses R = 1: its rows are
// 16 to 32 KB), and the next iteration's rows are fetched into registers
// while they are.
#include "common.cuh"
#include "unaligned.cuh"
#include "launch.h"
#include "row_math.cuh"

namespace rn {

namespace {

// [2 parities][2 rows][32 warps] fp32 warp sums, then the row buffers
constexpr int kRealignRedBytes = 512;

// 16 bytes of shared memory starting at byte offset `start` of the buffer at
// shared address `buf` (16-byte aligned; the buffer extends 16 bytes past
// the last window read).
__device__ __forceinline__ uint4 ld_shared_window(uint32_t buf, int start) {
    const uint32_t addr = buf + (uint32_t)(start & ~15);
    const int sh = start & 15;
    const uint4 lo = ld_shared_v4(addr);
    if (sh == 0) return lo;
    return shift_bytes(lo, ld_shared_v4(addr + 16), sh);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

template <typename T> __device__ __forceinline__ void st_shared_elem(uint32_t addr, T v) {
    if (sizeof(T) == 4)
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(__float_as_uint(to_f(v)))
                     : "memory");
    else
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr),
                     "h"(*reinterpret_cast<const unsigned short *>(&v))
                     : "memory");
}

template <typename T> __device__ __forceinline__ T ld_shared_elem(uint32_t addr) {
    if (sizeof(T) == 4) {
        uint32_t u;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(u) : "r"(addr) : "memory");
        return from_f<T>(__uint_as_float(u));
    } else {
        unsigned short u;
        asm volatile("ld.shared.b16 %0, [%1];" : "=h"(u) : "r"(addr) : "memory");
        return *reinterpret_cast<const T *>(&u);
    }
}

}  // namespace

struct RealignArgs {
    const uint8_t *x;
    const uint8_t *gamma;
    const uint8_t *dy;
    const float *rstd;
    const uint8_t *dres;
    uint8_t *dx;
    float *dw_out;   // scratch: partial rows [gridDim.x][N]; atomic: dweight_f32
    int64_t M;
    int N;
    int nb;          // column blocks of 16 bytes per row (the last may be partial)
    int buf;         // bytes of one row buffer (16 * nb + 32)
    float inv_n;
};

size_t realign_smem_bytes(int N, int dtype, int rows, bool dres) {
    const int nb = (int)(((int64_t)N * elem_bytes(dtype) + 15) / 16);
    const size_t buf = 16 * (size_t)nb + 32;
    return kRealignRedBytes + (size_t)rows * (dres ? 4 : 3) * buf;
}

template <typename T, int CPB, int R, bool HAS_DRES, bool ATOMIC>
__global__ void __launch_bounds__(512, 1) bwd_realign_kernel(const RealignArgs a) {
    constexpr int S = sizeof(T);
    constexpr int V = 16 / S;
    constexpr int P = RowMath<T>::kPairs;
    constexpr int NB = HAS_DRES ? 4 : 3;  // buffers per row: x, dy, [dres], dx
    constexpr bool kGammaF = RowMath<T>::kNeedsGammaF || CPB * V <= 8;
    extern __shared__ __align__(16) uint8_t smem[];
    float *red = reinterpret_cast<float *>(smem);
    const uint32_t bufs = smem_addr(smem) + kRealignRedBytes;

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
    const int N = a.N, nb = a.nb;
    const T *x = reinterpret_cast<const T *>(a.x);
    const T *dy = reinterpret_cast<const T *>(a.dy);
    const T *dres = reinterpret_cast<const T *>(a.dres);
    const T *gam = reinterpret_cast<const T *>(a.gamma);
    T *dx = reinterpret_cast<T *>(a.dx);
    // shared address of buffer b (0 x, 1 dy, 2 dres, NB-1 dx) of in-flight row r
    auto buf_of = [&](int r, int b) { return bufs + (uint32_t)((r * NB + b) * a.buf); };

    // this thread's column blocks and gamma (zero past N)
    uint4 gp[CPB];
    f32x2 g2[kGammaF ? CPB : 1][kGammaF ? P : 1];
#pragma unroll
    for (int k = 0; k < CPB; ++k) {
        const int c = tid + k * nthr;
        float gf[V];
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const int j = c * V + e;
            gf[e] = (c < nb && j < N) ? to_f(gam[j]) : 0.f;
        }
        gp[k] = float_to_chunk<T>(gf);
        if (kGammaF) {
#pragma unroll
            for (int q = 0; q < P; ++q)
                g2[kGammaF ? k : 0][kGammaF ? q : 0] = f2_make(gf[2 * q], gf[2 * q + 1]);
        }
    }
    f32x2 acc2[CPB][P];
#pragma unroll
    for (int k = 0; k < CPB; ++k)
#pragma unroll
        for (int q = 0; q < P; ++q) acc2[k][q] = f2_make(0.f, 0.f);

    // Geometry of the group of R rows starting at g0: head bytes, whole
    // chunks, tail elements, rstd (zeros for rows past M).
    auto geom = [&](int64_t g0, int (&hs_)[R], int (&nv_)[R], int (&nt_)[R], float (&rs_)[R]) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int64_t row = g0 + r;
            hs_[r] = nv_[r] = nt_[r] = 0;
            rs_[r] = 0.f;
            if (row < a.M) {
                const uintptr_t ad = reinterpret_cast<uintptr_t>(x + (size_t)row * N);
                int h = (int)(((16u - (unsigned)(ad & 15u)) & 15u) / S);
                if (h > N) h = N;
                hs_[r] = h * S;
                nv_[r] = (N - h) / V;
                nt_[r] = N - h - nv_[r] * V;
                rs_[r] = __ldg(a.rstd + row);
            }
        }
    };
    // This thread's part of a group's rows, fetched into registers: its
    // whole chunks, and its head or tail element (threads below h + tail).
    uint4 lx[R][CPB], ld[R][CPB], lr[HAS_DRES ? R : 1][HAS_DRES ? CPB : 1];
    T ex[R], ed[R], er[R];
    auto fetch = [&](int64_t g0, const int (&hs_)[R], const int (&nv_)[R], const int (&nt_)[R]) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const size_t base = (size_t)(g0 + r) * N;
#pragma unroll
            for (int k = 0; k < CPB; ++k) {
                const int i = tid + k * nthr;
                if (i < nv_[r]) {
                    const size_t e0 = base + hs_[r] / S + (size_t)i * V;
                    lx[r][k] = ld_global_nc_v4(x + e0);
                    ld[r][k] = ld_global_nc_v4(dy + e0);
                    if (HAS_DRES)
                        lr[HAS_DRES ? r : 0][HAS_DRES ? k : 0] =
                            *reinterpret_cast<const uint4 *>(dres + e0);
                }
            }
            const int h = hs_[r] / S;
            if (g0 + r < a.M && tid < h + nt_[r]) {
                const int j = tid < h ? tid : h + nv_[r] * V + (tid - h);
                ex[r] = x[base + j];
                ed[r] = dy[base + j];
                if (HAS_DRES) er[r] = dres[base + j];
            }
        }
    };

    int hs[R], nv[R], nt[R];  // the current group's head bytes, whole chunks, tail elements
    float rs[R];
    const int64_t gstride = (int64_t)gridDim.x * R;
    int64_t row0 = (int64_t)blockIdx.x * R;
    if (row0 < a.M) {
        geom(row0, hs, nv, nt, rs);
        fetch(row0, hs, nv, nt);
    }
    int parity = 0;
    for (; row0 < a.M; row0 += gstride) {
        // 1. the fetched rows into the row buffers (element j at byte
        //    16 + (j - h)*S: chunk i at the aligned offset 16*(i+1))
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r >= a.M) continue;
#pragma unroll
            for (int k = 0; k < CPB; ++k) {
                const int i = tid + k * nthr;
                if (i < nv[r]) {
                    const uint32_t off = 16u * (uint32_t)(i + 1);
                    st_shared_v4(buf_of(r, 0) + off, lx[r][k]);
                    st_shared_v4(buf_of(r, 1) + off, ld[r][k]);
                    if (HAS_DRES)
                        st_shared_v4(buf_of(r, 2) + off, lr[HAS_DRES ? r : 0][HAS_DRES ? k : 0]);
                }
            }
            const int h = hs[r] / S;
            // head and tail elements (fewer than V each)
            if (tid < h + nt[r]) {
                const int j = tid < h ? tid : h + nv[r] * V + (tid - h);
                const uint32_t off = (uint32_t)(16 + (j - h) * S);
                st_shared_elem<T>(buf_of(r, 0) + off, ex[r]);
                st_shared_elem<T>(buf_of(r, 1) + off, ed[r]);
                if (HAS_DRES) st_shared_elem<T>(buf_of(r, 2) + off, er[r]);
            }
            // zeros after the last element, up to the end of the last block's
            // window (at most 15 bytes): the partial block's extra columns
            // then contribute nothing
            const int pad0 = 16 + (N - h) * S, pad1 = 16 * (nb + 1) - hs[r];
            for (int pb = pad0 + tid * S; pb < pad1; pb += nthr * S) {
                st_shared_elem<T>(buf_of(r, 0) + pb, from_f<T>(0.f));
                st_shared_elem<T>(buf_of(r, 1) + pb, from_f<T>(0.f));
                if (HAS_DRES) st_shared_elem<T>(buf_of(r, 2) + pb, from_f<T>(0.f));
            }
        }
        // the next group's rows are fetched while this group is processed
        int nhs[R], nnv[R], nnt[R];
        float nrs[R];
        const int64_t nxt = row0 + gstride;
        if (nxt < a.M) {
            geom(nxt, nhs, nnv, nnt, nrs);
            fetch(nxt, nhs, nnv, nnt);
        }
        __syncthreads();

        // 2. pass 1 on fixed column blocks (read back by the row's phase)
        f32x2 part2[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            part2[r] = f2_make(0.f, 0.f);
            if (row0 + r >= a.M) continue;  // (uniform) no row: its buffers hold stale bytes
#pragma unroll
            for (int k = 0; k < CPB; ++k) {
                const int c = tid + k * nthr;
                if (c < nb) {
                    const int start = 16 * (c + 1) - hs[r];
                    part2[r] = RowMath<T>::pass1(ld_shared_window(buf_of(r, 0), start),
                                                 ld_shared_window(buf_of(r, 1), start), gp[k],
                                                 kGammaF ? g2[kGammaF ? k : 0] : nullptr,
                                                 part2[r]);
                }
            }
        }
        float *slot = red + parity * (2 * 32);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float lo, hi;
            f2_split(part2[r], lo, hi);
            const float w = warp_sum(lo + hi);
            if (lane == 0) slot[r * 32 + warp] = w;
        }
        __syncthreads();
        float b[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float v = lane < nwarps ? slot[r * 32 + lane] : 0.f;
            const float tot = warp_sum(v);
            // dx = (wdy - x_hat*c1)*rstd = wdy*rstd + x*b with b = -rstd^2*c1
            const float c1 = rs[r] * tot * a.inv_n;
            b[r] = -rs[r] * rs[r] * c1;
        }
        parity ^= 1;

        // 3. pass 2: dx blocks into the block-aligned dx buffer (element j at
        //    byte j*S), weight-gradient partial in registers
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r >= a.M) continue;
            const f32x2 rs2 = f2_make(rs[r], rs[r]), b2 = f2_make(b[r], b[r]);
#pragma unroll
            for (int k = 0; k < CPB; ++k) {
                const int c = tid + k * nthr;
                if (c < nb) {
                    const int start = 16 * (c + 1) - hs[r];
                    const uint4 rv = HAS_DRES ? ld_shared_window(buf_of(r, 2), start)
                                              : make_uint4(0, 0, 0, 0);
                    const uint4 o = RowMath<T>::template pass2<HAS_DRES>(
                        ld_shared_window(buf_of(r, 0), start), ld_shared_window(buf_of(r, 1), start),
                        rv, gp[k], kGammaF ? g2[kGammaF ? k : 0] : nullptr, rs2, b2, acc2[k]);
                    st_shared_v4(buf_of(r, NB - 1) + 16u * (uint32_t)c, o);
                }
            }
        }
        __syncthreads();

        // 4. dx out: aligned chunks (window at byte h*S + 16*i of the dx
        //    buffer), head and tail element by element
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r >= a.M) continue;
            const int h = hs[r] / S;
            const size_t base = (size_t)(row0 + r) * N;
#pragma unroll
            for (int k = 0; k < CPB; ++k) {
                const int i = tid + k * nthr;
                if (i < nv[r])
                    st_global_v4(dx + base + h + (size_t)i * V,
                                 ld_shared_window(buf_of(r, NB - 1), hs[r] + 16 * i));
            }
            if (tid < h + nt[r]) {
                const int j = tid < h ? tid : h + nv[r] * V + (tid - h);
                dx[base + j] = ld_shared_elem<T>(buf_of(r, NB - 1) + (uint32_t)(j * S));
            }
        }
        // (the next rows' buffer writes come after this iteration's last
        // barrier; their dx-buffer writes after the next two)
        if (nxt < a.M) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                hs[r] = nhs[r];
                nv[r] = nnv[r];
                nt[r] = nnt[r];
                rs[r] = nrs[r];
            }
        }
    }

    // the CTA's weight-gradient partial: each thread owns its columns
    pdl_launch_dependents();
    if (ATOMIC) pdl_wait();  // the zeroing kernel ahead of this one has finished
    float *dst = ATOMIC ? a.dw_out : a.dw_out + (size_t)blockIdx.x * N;
#pragma unroll
    for (int k = 0; k < CPB; ++k) {
        const int c = tid + k * nthr;
        if (c >= nb) continue;
        float v[2 * P];
#pragma unroll
        for (int q = 0; q < P; ++q) f2_split(acc2[k][q], v[2 * q], v[2 * q + 1]);
#pragma unroll
        for (int e = 0; e < V; ++e) {
            const int j = c * V + e;
            if (j < N) {
                if (ATOMIC) atomicAdd(dst + j, v[e]);
                else dst[j] = v[e];
            }
        }
    }
}

template <typename T, int CPB, int R, bool HAS_DRES, bool ATOMIC>
static cudaError_t launch_realign_t(const RealignArgs &args, const GenericPlan &plan,
                                    cudaStream_t s, bool pdl) {
    auto kern = bwd_realign_kernel<T, CPB, R, HAS_DRES, ATOMIC>;
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
static cudaError_t launch_realign_c(const RealignArgs &args, const GenericPlan &plan,
                                    cudaStream_t s, bool pdl) {
    switch (plan.cpb) {
    case 2: return launch_realign_t<T, 2, 1, HAS_DRES, ATOMIC>(args, plan, s, pdl);
    case 4: return launch_realign_t<T, 4, 1, HAS_DRES, ATOMIC>(args, plan, s, pdl);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
static cudaError_t launch_realign_dt(const RealignArgs &args, const GenericPlan &plan,
                                     bool has_dres, cudaStream_t s, bool pdl) {
    if (plan.atomic)
        return has_dres ? launch_realign_c<T, true, true>(args, plan, s, pdl)
                        : launch_realign_c<T, false, true>(args, plan, s, pdl);
    return has_dres ? launch_realign_c<T, true, false>(args, plan, s, pdl)
                    : launch_realign_c<T, false, false>(args, plan, s, pdl);
}

cudaError_t launch_bwd_realign(const BwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                               bool pdl_after_zero) {
    RealignArgs a;
    a.x = static_cast<const uint8_t *>(p.x);
    a.gamma = static_cast<const uint8_t *>(p.gamma);
    a.dy = static_cast<const uint8_t *>(p.dy);
    a.rstd = p.rstd;
    a.dres = static_cast<const uint8_t *>(p.dres);
    a.dx = static_cast<uint8_t *>(p.dx);
    a.dw_out = plan.atomic ? p.dw_f32 : reinterpret_cast<float *>(p.ws + kWsHeaderBytes);
    a.M = p.M;
    a.N = p.N;
    a.nb = (int)(((int64_t)p.N * elem_bytes(p.dtype) + 15) / 16);
    a.buf = 16 * a.nb + 32;
    a.inv_n = 1.0f / (float)p.N;
    const bool has_dres = p.dres != nullptr;
    switch (p.dtype) {
    case kF32: return launch_realign_dt<float>(a, plan, has_dres, s, pdl_after_zero);
    case kF16: return launch_realign_dt<__half>(a, plan, has_dres, s, pdl_after_zero);
    case kBF16: return launch_realign_dt<__nv_bfloat16>(a, plan, has_dres, s, pdl_after_zero);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
