// Cross-CTA weight-gradient steps (the pages count the fp32 zero and the
// cast to the parameter dtype inside the backward call -- FlyDSL PR #854,
// "Benchmark contract"; the dweight reduction choice between fp32 atomics and
// scratch partials + a finalizer -- FlyDSL issue #769, "dweight reduction
// experiment").
//
//  * finalize: dweight_f32[j] = sum over the G partial rows, in a fixed
//    order (deterministic), and the cast to the I/O dtype in the same pass.
//    A CTA covers 32 columns with 32 x 32 threads: thread (cx, gy) sums rows
//    gy, gy+32, ... of column cx; a fixed-shape tree in shared memory then
//    adds the 32 column sums.
//  * zero / cast: the two ends of the atomic mode.
// All three use programmatic dependent launch so that their launch overlaps
// the tail of the kernel before them.
#include "common.cuh"
#include "launch.h"

namespace rn {

template <typename T>
__global__ void __launch_bounds__(1024) finalize_kernel(const float *__restrict__ partials, int G,
                                                        int N, float *__restrict__ dw_f32,
                                                        T *__restrict__ dw_cast) {
    __shared__ float sm[32][33];
    const int cx = threadIdx.x, gy = threadIdx.y;
    const int col = blockIdx.x * 32 + cx;
    pdl_wait();  // the row pass has finished writing its partial rows
    float s = 0.f;
    if (col < N) {
        int g = gy;
        for (; g + 3 * 32 < G; g += 4 * 32) {
            const float a0 = partials[(size_t)g * N + col];
            const float a1 = partials[(size_t)(g + 32) * N + col];
            const float a2 = partials[(size_t)(g + 64) * N + col];
            const float a3 = partials[(size_t)(g + 96) * N + col];
            s += a0;
            s += a1;
            s += a2;
            s += a3;
        }
        for (; g < G; g += 32) s += partials[(size_t)g * N + col];
    }
    sm[gy][cx] = s;
    __syncthreads();
#pragma unroll
    for (int h = 16; h > 0; h >>= 1) {
        if (gy < h) sm[gy][cx] += sm[gy + h][cx];
        __syncthreads();
    }
    if (gy == 0 && col < N) {
        const float v = sm[0][cx];
        dw_f32[col] = v;
        if (dw_cast) dw_cast[col] = from_f<T>(v);
    }
}

__global__ void zero_f32_kernel(float *p, int N) {
    pdl_launch_dependents();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
        p[i] = 0.f;
}

template <typename T>
__global__ void cast_kernel(const float *__restrict__ src, T *__restrict__ dst, int N) {
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
        dst[i] = from_f<T>(src[i]);
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

cudaError_t launch_finalize(const float *partials, int G, int N, float *dw_f32, void *dw_cast,
                            int dtype, cudaStream_t s, bool pdl) {
    dim3 grid((N + 31) / 32), block(32, 32);
    switch (dtype) {
    case kF32:
        return launch_ex(finalize_kernel<float>, grid, block, s, pdl, partials, G, N, dw_f32,
                         static_cast<float *>(dw_cast));
    case kF16:
        return launch_ex(finalize_kernel<__half>, grid, block, s, pdl, partials, G, N, dw_f32,
                         static_cast<__half *>(dw_cast));
    case kBF16:
        return launch_ex(finalize_kernel<__nv_bfloat16>, grid, block, s, pdl, partials, G, N,
                         dw_f32, static_cast<__nv_bfloat16 *>(dw_cast));
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_zero_f32(float *p, int N, cudaStream_t s) {
    const int threads = 256;
    int blocks = (N + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    return launch_ex(zero_f32_kernel, dim3(blocks), dim3(threads), s, false, p, N);
}

cudaError_t launch_cast(const float *dw_f32, void *dw_cast, int N, int dtype, cudaStream_t s,
                        bool pdl) {
    const int threads = 256;
    int blocks = (N + threads - 1) / threads;
    if (blocks > 1024) blocks = 1024;
    switch (dtype) {
    case kF32:
        return launch_ex(cast_kernel<float>, dim3(blocks), dim3(threads), s, pdl, dw_f32,
                         static_cast<float *>(dw_cast), N);
    case kF16:
        return launch_ex(cast_kernel<__half>, dim3(blocks), dim3(threads), s, pdl, dw_f32,
                         static_cast<__half *>(dw_cast), N);
    case kBF16:
        return launch_ex(cast_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), s, pdl,
                         dw_f32, static_cast<__nv_bfloat16 *>(dw_cast), N);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace rn
