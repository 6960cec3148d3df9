// Cross-CTA weight-gradient steps (the pages count the fp32 zero and the
// cast to the parameter dtype inside the backward call -- FlyDSL PR #854,
// "Benchmark contract"; the dweight reduction choice between fp32 atomics and
// scratch partials + a finalizer -- FlyDSL issue #769, "dweight reduction
// experiment").
//
//  * finalize: dweight_f32[j] = sum over the G partial rows, in a fixed
//    order (deterministic), and the cast to the I/O dtype in the same pass
//    (either output may be absent).
//    A CTA covers 32 columns with 32 x 32 threads: thread (cx, gy) sums rows
//    gy, gy+32, ... of column cx; a fixed-shape tree in shared memory then
//    adds the 32 column sums.
//  * zero / cast: the two ends of the atomic mode.
// Each handles an optional second output of the same length (LayerNorm's
// dbeta beside dgamma) in the same launch.
// All three use programmatic dependent launch so that their launch overlaps
// the tail of the kernel before them.
#include "common.cuh"
#include "launch.h"

namespace rn {

template <typename T>
__global__ void __launch_bounds__(1024) finalize_kernel(const float *__restrict__ partials, int G,
                                                        int ld, int N, float *__restrict__ dw_f32,
                                                        T *__restrict__ dw_cast,
                                                        float *__restrict__ dw2_f32,
                                                        T *__restrict__ dw2_cast) {
    // columns [0, N) of the partial rows go to dw_f32 / dw_cast; with a second
    // output, columns [N, 2N) go to dw2_f32 / dw2_cast. Rows are ld floats apart.
    __shared__ float sm[32][33];
    const int cx = threadIdx.x, gy = threadIdx.y;
    const int col = blockIdx.x * 32 + cx;
    const int ncols = (dw2_f32 || dw2_cast) ? 2 * N : N;
    pdl_wait();  // the row pass has finished writing its partial rows
    float s = 0.f;
    if (col < ncols) {
        int g = gy;
        for (; g + 3 * 32 < G; g += 4 * 32) {
            const float a0 = partials[(size_t)g * ld + col];
            const float a1 = partials[(size_t)(g + 32) * ld + col];
            const float a2 = partials[(size_t)(g + 64) * ld + col];
            const float a3 = partials[(size_t)(g + 96) * ld + col];
            s += a0;
            s += a1;
            s += a2;
            s += a3;
        }
        for (; g < G; g += 32) s += partials[(size_t)g * ld + col];
    }
    sm[gy][cx] = s;
    __syncthreads();
#pragma unroll
    for (int h = 16; h > 0; h >>= 1) {
        if (gy < h) sm[gy][cx] += sm[gy + h][cx];
        __syncthreads();
    }
    if (gy == 0 && col < ncols) {
        const float v = sm[0][cx];
        if (col < N) {
            if (dw_f32) dw_f32[col] = v;
            if (dw_cast) dw_cast[col] = from_f<T>(v);
        } else {
            if (dw2_f32) dw2_f32[col - N] = v;
            if (dw2_cast) dw2_cast[col - N] = from_f<T>(v);
        }
    }
}

__global__ void zero_f32_kernel(float *p, float *p2, int N) {
    pdl_launch_dependents();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x) {
        p[i] = 0.f;
        if (p2) p2[i] = 0.f;
    }
}

template <typename T>
__global__ void cast_kernel(const float *__restrict__ src, T *__restrict__ dst,
                            const float *__restrict__ src2, T *__restrict__ dst2, int N) {
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x) {
        if (dst) dst[i] = from_f<T>(src[i]);
        if (dst2) dst2[i] = from_f<T>(src2[i]);
    }
}

template <typename K, typename... Args>
static cudaError_t launch_ex(K kern, dim3 grid, dim3 block, cudaStream_t s, bool pdl,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

cudaError_t launch_finalize2(const float *partials, int G, int ld, int N, float *dw_f32,
                             void *dw_cast, float *dw2_f32, void *dw2_cast, int dtype,
                             cudaStream_t s, bool pdl) {
    const int ncols = (dw2_f32 || dw2_cast) ? 2 * N : N;
    dim3 grid((ncols + 31) / 32), block(32, 32);
    switch (dtype) {
    case kF32:
        return launch_ex(finalize_kernel<float>, grid, block, s, pdl, partials, G, ld, N, dw_f32,
                         static_cast<float *>(dw_cast), dw2_f32, static_cast<float *>(dw2_cast));
    case kF16:
        return launch_ex(finalize_kernel<__half>, grid, block, s, pdl, partials, G, ld, N, dw_f32,
                         static_cast<__half *>(dw_cast), dw2_f32,
                         static_cast<__half *>(dw2_cast));
    case kBF16:
        return launch_ex(finalize_kernel<__nv_bfloat16>, grid, block, s, pdl, partials, G, ld, N,
                         dw_f32, static_cast<__nv_bfloat16 *>(dw_cast), dw2_f32,
                         static_cast<__nv_bfloat16 *>(dw2_cast));
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_finalize(const float *partials, int G, int N, float *dw_f32, void *dw_cast,
                            int dtype, cudaStream_t s, bool pdl) {
    return launch_finalize2(partials, G, N, N, dw_f32, dw_cast, nullptr, nullptr, dtype, s, pdl);
}

cudaError_t launch_zero_f32(float *p, int N, cudaStream_t s, float *p2) {
    const int threads = 256;
    int blocks = (N + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    return launch_ex(zero_f32_kernel, dim3(blocks), dim3(threads), s, false, p, p2, N);
}

cudaError_t launch_cast(const float *dw_f32, void *dw_cast, int N, int dtype, cudaStream_t s,
                        bool pdl, const float *dw2_f32, void *dw2_cast) {
    const int threads = 256;
    int blocks = (N + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    switch (dtype) {
    case kF32:
        return launch_ex(cast_kernel<float>, dim3(blocks), dim3(threads), s, pdl, dw_f32,
                         static_cast<float *>(dw_cast), dw2_f32, static_cast<float *>(dw2_cast),
                         N);
    case kF16:
        return launch_ex(cast_kernel<__half>, dim3(blocks), dim3(threads), s, pdl, dw_f32,
                         static_cast<__half *>(dw_cast), dw2_f32,
                         static_cast<__half *>(dw2_cast), N);
    case kBF16:
        return launch_ex(cast_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), s, pdl,
                         dw_f32, static_cast<__nv_bfloat16 *>(dw_cast), dw2_f32,
                         static_cast<__nv_bfloat16 *>(dw2_cast), N);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
