// kernels.h -- host-side entry points of the CUDA kernels (one per .cu file).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "common.h"

namespace jattn {

// Per-device record of a kernel's shared-memory opt-in.  Atomic, because host
// threads driving different plans may launch the same kernel for the first
// time at once; the opt-in itself is idempotent, so two threads that both find
// it unset both make it, and either result stands.
struct SmemOnce {
    std::atomic<bool> done[64];
    SmemOnce() {
        for (auto &d : done) d.store(false, std::memory_order_relaxed);
    }
};

// Opt a kernel into `bytes` of dynamic shared memory, once per device.
template <typename K>
inline cudaError_t ensure_smem(K kern, uint32_t bytes, SmemOnce &once) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    const bool cacheable = dev >= 0 && dev < 64;
    if (cacheable && once.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && cacheable) once.done[dev].store(true, std::memory_order_release);
    return e;
}

// TMA descriptors of the bf16 [T, H*D] operand views a kernel reads.
struct TmapSet {
    CUtensorMap q, k, v, dout;
};

// forward: D in {64, 128}; act selects the GDPA activation path
cudaError_t launch_fwd(int D, bool act, const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream);

// test build of the forward whose first bounded wait runs out after a.g.wait_ns
// (softmax, no bias, no window, D in {64, 128})
cudaError_t launch_fwd_stall(int D, const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream);

// forward with rotary position embedding of Q and K (a.g.rope_cos / rope_sin set, no window)
cudaError_t launch_fwd_rope(int D, bool act, const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream);

// backward, full attention: dQ pass (query-major tiles) and dK/dV pass (key-major tiles)
cudaError_t launch_bwd_dq(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t stream);

// backward with dS chunks: dQ = scale * dS K over query-major tiles, from the
// chunks the dK/dV pass wrote (a.g.ds, a.g.ds_base); tm.k in 128-row boxes
cudaError_t launch_bwd_dq_gemm(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t stream);

// backward, BlockAttention: one fused pass over query-major tiles (with
// rotary position embedding when a.g.rope_cos is set)
cudaError_t launch_bwd_block(int D, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t stream);

// Delta_i = <dO_i, O_i> (fp32) for every row and head: delta[h * Tq + t]
cudaError_t launch_delta(const void *out, const void *dout, int f32, int64_t Tq, int H, int D, float *delta,
                         cudaStream_t stream);

// MXFP8 quantisation (32 local rows x 32 features per block) of up to four
// tensors x [T, H, D] bf16: job j quantises x[j] into xq[j] over the plan's
// device tile list tiles[j] (ntiles[j] tiles of 128 rows; kv_side[j]: the
// tiles' key rows, else their query rows).  D is 64 or 128.
struct MxJobs {
    const void *x[4];  // bf16
    void *xq[4];       // bf16
    const Tile *tiles[4];
    int32_t ntiles[4];
    int32_t kv_side[4];
    int32_t n;
};
cudaError_t launch_mx_quant(const MxJobs &jobs, int H, int D, cudaStream_t stream);

// src [rows, D] (bf16 or fp32) -> dst [rows, Dp] bf16, zero-padded columns D..Dp-1
cudaError_t launch_stage(const void *src, int f32, int64_t rows, int D, int Dp, void *dst, cudaStream_t stream);

// broadcast Q: dq [n, HD] bf16 = sum over the B samples of ws [B * n, HD] float32, in a fixed order
cudaError_t launch_bcast_reduce(const float *ws, int B, int n, int64_t HD, void *dq, cudaStream_t stream);

// device-side planner: tile lists and zigzag schedule from device offsets
constexpr int kDevPlanMaxSeqs = 8192;  // sequences per batch the one-CTA sort takes
struct DevPlanArgs {
    const int32_t *q_off, *kv_off;  // DEVICE [B + 1]
    int32_t B, H, block, window;
    int32_t n_ctas;                 // CTAs the kernels launch (each list gets n_ctas + 1 range entries)
    int32_t Tq, Tk;                 // expected last offsets
    Tile *tiles_q, *tiles_kv;
    int32_t *cta_q, *cta_kv;
    int32_t cap_q, cap_kv;          // capacities in tiles
    int *status;                    // device status word (bad offsets or capacity: kStatusDeviceCheck)
    int32_t sort_len;               // power of two >= B, <= kDevPlanMaxSeqs
    int32_t bcast_n;                // broadcast Q: every sequence must have this many queries (0: off)
};
cudaError_t launch_plan_device(const DevPlanArgs &a, cudaStream_t stream);

}  // namespace jattn
