// Allocation-free variant of the plain RMSNorm backward.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: code that executes while a memory pool or allocator is locked or
// being torn down, runtimes whose allocator is owned by someone else and
// must not be re-entered from inside a step, and embedders that budget every
// device byte up front. For them this file provides rn_rmsnorm_bwd_noalloc:
// the same computation as rn_rmsnorm_bwd, with its scratch (the per-CTA
// weight-gradient partials) taken from a fixed array that lives in this
// library's device image instead of a caller-provided workspace.
//
// The array below is a file-scope __device__ symbol: every GPU that loads the
// library holds it until the process exits. In host code its name is only a
// host-side handle, not a device address, so the device address is looked up
// with cudaGetSymbolAddress once per device (with that device current) and
// cached; that lookup happens on the first call on each device. The cache
// assumes the device image stays loaded: a cudaDeviceReset while this library
// is loaded would reload it at another address, so a reset is not supported
// (the header says so).
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/rmsnorm_gb300.h"
#include "launch.h"

namespace {

constexpr size_t kNoallocScratchBytes = 16u << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" rn_status rn_rmsnorm_bwd_noalloc(const void *x, const void *gamma, const void *dy,
                                            const float *rstd, void *dx, float *dweight_f32,
                                            void *dweight, int64_t M, int64_t N, int dtype,
                                            void *stream) {
    char msg[256];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
        rn::set_last_error(msg);
        return RN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "device %d out of range", dev);
        rn::set_last_error(msg);
        return RN_ERR_UNSUPPORTED;
    }
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess || p == nullptr) {
                snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the scratch array failed: %s",
                         cudaGetErrorString(e));
                rn::set_last_error(msg);
                return RN_ERR_CUDA;
            }
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    // The scratch this problem needs on this device; too large -> refuse.
    size_t need = 0;
    rn_status st = rn_bwd_workspace_bytes(M, N, dtype, &need);  // sets the message on failure
    if (st != RN_OK) return st;
    if (need > kNoallocScratchBytes) {
        snprintf(msg, sizeof(msg),
                 "rn_rmsnorm_bwd_noalloc: N=%lld needs %zu bytes of scratch, more than its fixed "
                 "%zu; call rn_rmsnorm_bwd with a caller workspace instead",
                 (long long)N, need, kNoallocScratchBytes);
        rn::set_last_error(msg);
        return RN_ERR_UNSUPPORTED;
    }
    return rn_rmsnorm_bwd(x, gamma, dy, rstd, dx, dweight_f32, dweight, scratch,
                          kNoallocScratchBytes, M, N, dtype, stream);
}
