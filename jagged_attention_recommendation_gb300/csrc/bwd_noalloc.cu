// bwd_noalloc.cu -- jattn_bwd_noalloc: the backward pass with its device
// scratch taken from a fixed array inside this library instead of a
// caller-provided workspace, so that callers that cannot allocate device
// memory can still run it.  The array is a file-scope __device__ object: every
// GPU that loads the library holds it until the process exits.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "jattn.h"

namespace jattn {
int plan_device(const jattn_plan *plan);  // api.cpp
}

namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on `dev`, looked up once per device with that
// device current.  In host code the array's name is only a host-side stand-in;
// kernels must be given this address.  The caller's current device is put back
// afterwards; if that fails, the call fails too (and caches nothing), so a
// success never leaves the caller on another device.
cudaError_t scratch_address(int dev, void **addr) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        int prev = -1;
        cudaError_t e = cudaGetDevice(&prev);
        if (e != cudaSuccess) return e;
        if (prev != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return e;
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_bwd_scratch);
        if (prev != dev) {
            const cudaError_t r = cudaSetDevice(prev);
            if (e == cudaSuccess) e = r;
        }
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" jattn_status jattn_bwd_noalloc(const jattn_plan *plan, const void *dout, const void *q, const void *k,
                                          const void *v, const float *bias, const void *out, const float *lse,
                                          void *dq, void *dk, void *dv, float *dbias, void *stream) {
    if (plan == nullptr) return JATTN_ERR_INVALID_ARG;
    const int dev = jattn::plan_device(plan);
    if (dev < 0) return JATTN_ERR_NO_DEVICE;
    if (dev >= kMaxDevices) return JATTN_ERR_UNSUPPORTED;
    const size_t need = jattn_bwd_workspace_bytes_min(plan);
    if (need > kNoAllocScratchBytes) return JATTN_ERR_WORKSPACE;  // batch too large for the fixed array
    // the array goes to jattn_bwd whenever any path could use scratch; jattn_bwd
    // takes its dS-chunk path when the whole size fits, else the recomputing one
    const bool give = jattn_bwd_workspace_bytes(plan) > 0;
    void *scratch = nullptr;
    if (give && scratch_address(dev, &scratch) != cudaSuccess) return JATTN_ERR_CUDA;
    return jattn_bwd(plan, dout, q, k, v, bias, out, lse, dq, dk, dv, dbias, give ? scratch : nullptr,
                     give ? kNoAllocScratchBytes : 0, stream);
}
