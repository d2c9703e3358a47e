// aux.cu -- small memory-bound helpers of the attention passes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.h"

namespace jattn {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
    return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

// Delta_i = <dO_i, O_i> for every (token, head) row: one warp per row, fp32
// accumulation; rows are [T, H, D] and the result is laid out [H, T].
template <typename T>
__global__ void delta_kernel(const T *__restrict__ out, const T *__restrict__ dout, int64_t Tq, int H, int D,
                             float *__restrict__ delta) {
    const int64_t nrows = Tq * H;
    const int lane = threadIdx.x & 31;
    int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    for (; r < nrows; r += stride) {
        const T *o = out + r * D;
        const T *d = dout + r * D;
        float acc = 0.0f;
        for (int c = lane; c < D; c += 32) acc = fmaf(to_f(o[c]), to_f(d[c]), acc);
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
        if (lane == 0) {
            const int64_t t = r / H;
            const int h = static_cast<int>(r % H);
            delta[static_cast<int64_t>(h) * Tq + t] = acc;
        }
    }
}

// src [rows, D] -> dst [rows, Dp] bf16 (columns D..Dp-1 zero).
template <typename T>
__global__ void stage_kernel(const T *__restrict__ src, int64_t rows, int D, int Dp, __nv_bfloat16 *__restrict__ dst) {
    const int64_t n = rows * Dp;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / Dp;
        const int c = static_cast<int>(i - r * Dp);
        dst[i] = c < D ? __float2bfloat16_rn(to_f(src[r * D + c])) : __float2bfloat16_rn(0.0f);
    }
}

static int grid_for(int64_t work, int per_block) {
    int64_t g = (work + per_block - 1) / per_block;
    if (g > 152 * 16) g = 152 * 16;
    return g < 1 ? 1 : static_cast<int>(g);
}

cudaError_t launch_delta(const void *out, const void *dout, int f32, int64_t Tq, int H, int D, float *delta,
                         cudaStream_t stream) {
    if (Tq <= 0) return cudaSuccess;
    const int grid = grid_for(Tq * H, 8);  // 8 warps of 32 per block
    if (f32)
        delta_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float *>(out),
                                                       static_cast<const float *>(dout), Tq, H, D, delta);
    else
        delta_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(out),
                                                               static_cast<const __nv_bfloat16 *>(dout), Tq, H, D,
                                                               delta);
    return cudaGetLastError();
}

cudaError_t launch_stage(const void *src, int f32, int64_t rows, int D, int Dp, void *dst, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int grid = grid_for(rows * Dp, 256);
    if (f32)
        stage_kernel<float><<<grid, 256, 0, stream>>>(static_cast<const float *>(src), rows, D, Dp,
                                                       static_cast<__nv_bfloat16 *>(dst));
    else
        stage_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(src), rows, D, Dp,
                                                               static_cast<__nv_bfloat16 *>(dst));
    return cudaGetLastError();
}

}  // namespace jattn
