// aux.cu -- small memory-bound helpers of the attention passes.
#include <cuda_bf16.h>

#include <algorithm>
#include <cuda_runtime.h>

#include "attn.cuh"
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

// Delta_i = <dO_i, O_i> for every (token, head) row, fp32 accumulation; rows
// are [T, H, D] and the result is laid out [H, T].  Every thread reads 16-byte
// vectors of both rows; TPR = D / (elements per vector) consecutive lanes share
// a row and reduce with shuffles.
template <typename T>
__device__ __forceinline__ float dot16(const uint4 &a, const uint4 &b);
template <>
__device__ __forceinline__ float dot16<float>(const uint4 &a, const uint4 &b) {
    return __uint_as_float(a.x) * __uint_as_float(b.x) + __uint_as_float(a.y) * __uint_as_float(b.y) +
           __uint_as_float(a.z) * __uint_as_float(b.z) + __uint_as_float(a.w) * __uint_as_float(b.w);
}
template <>
__device__ __forceinline__ float dot16<__nv_bfloat16>(const uint4 &a, const uint4 &b) {
    const __nv_bfloat162 *x = reinterpret_cast<const __nv_bfloat162 *>(&a);
    const __nv_bfloat162 *y = reinterpret_cast<const __nv_bfloat162 *>(&b);
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 u = __bfloat1622float2(x[k]), w = __bfloat1622float2(y[k]);
        acc = fmaf(u.x, w.x, fmaf(u.y, w.y, acc));
    }
    return acc;
}

template <typename T>
__global__ void delta_kernel(const T *__restrict__ out, const T *__restrict__ dout, int64_t Tq, int H, int D,
                             float *__restrict__ delta) {
    constexpr int E = 16 / sizeof(T);  // elements per 16-byte vector
    const int tpr = D / E;             // lanes per row (4..32, a power of two)
    const int64_t nrows = Tq * H;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int sub = threadIdx.x & (tpr - 1);
    // whole warps stay in the loop together so the shuffles see every lane
    for (int64_t base = (gtid / tpr) - ((threadIdx.x & 31) / tpr); base < nrows; base += nthreads / tpr) {
        const int64_t r = base + (threadIdx.x & 31) / tpr;
        float acc = 0.0f;
        if (r < nrows) {
            const uint4 *o = reinterpret_cast<const uint4 *>(out + r * D);
            const uint4 *d = reinterpret_cast<const uint4 *>(dout + r * D);
            acc = dot16<T>(__ldg(o + sub), __ldg(d + sub));
        }
        for (int k = tpr >> 1; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
        if (sub == 0 && r < nrows) {
            const int64_t t = r / H;
            const int h = static_cast<int>(r - t * H);
            delta[static_cast<int64_t>(h) * Tq + t] = acc;
        }
    }
}

// MXFP8 quantisation of x [T, H, D] (bf16) per sequence and head, in blocks of
// 32 local rows x 32 features: xq receives the values the quantised blocks
// stand for (bf16, exact).  A CTA takes one (sequence, head) at a time; each
// warp takes one block: lane = row, the block's largest magnitude by a warp
// reduction.
__global__ void mx_quant_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ off, int B, int H,
                                int D, __nv_bfloat16 *__restrict__ xq) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int fbs = D / 32;
    for (int64_t bh = blockIdx.x; bh < static_cast<int64_t>(B) * H; bh += gridDim.x) {
        const int b = static_cast<int>(bh / H), h = static_cast<int>(bh - static_cast<int64_t>(b) * H);
        const int r0 = off[b], L = off[b + 1] - r0;
        const int ntask = ((L + 31) / 32) * fbs;
        for (int task = warp; task < ntask; task += nw) {
            const int rb = task / fbs, fb = task - rb * fbs;
            const int row = rb * 32 + lane;
            const bool ok = row < L;
            const int64_t base = (static_cast<int64_t>(r0 + row) * H + h) * D + fb * 32;
            float v[32];
            if (ok) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(x + base) + k);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        v[8 * k + 2 * j] = __uint_as_float(ws[j] << 16);
                        v[8 * k + 2 * j + 1] = __uint_as_float(ws[j] & 0xffff0000u);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            }
            const int e = dev::mx_exponent(dev::warp_max_nonneg(dev::amax32(v)));
            dev::mx_qdq32(v, e);
            if (ok) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    reinterpret_cast<uint4 *>(xq + base)[k] =
                        make_uint4(dev::pack_bf16x2(v[8 * k], v[8 * k + 1]), dev::pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                                   dev::pack_bf16x2(v[8 * k + 4], v[8 * k + 5]),
                                   dev::pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
            }
        }
    }
}

cudaError_t launch_mx_quant(const void *x, const int32_t *off, int B, int H, int D, void *xq, cudaStream_t stream) {
    if (B <= 0 || D % 32 != 0) return B <= 0 ? cudaSuccess : cudaErrorInvalidValue;
    const int64_t want = static_cast<int64_t>(B) * H;
    const int blocks = static_cast<int>(std::min<int64_t>(want, 152 * 8));
    mx_quant_kernel<<<blocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(x), off, B, H, D,
                                                static_cast<__nv_bfloat16 *>(xq));
    return cudaGetLastError();
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
    const int per_vec = f32 ? 4 : 8;
    if (D % per_vec != 0 || D / per_vec > 32 || ((D / per_vec) & (D / per_vec - 1)) != 0) return cudaErrorInvalidValue;
    const int grid = grid_for(Tq * H * (D / per_vec), 256);
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

// Broadcast Q: dq[i, c] = sum over b of ws[b * n + i, c] (fp32), stored as
// bf16.  ws: [B * n, HD] float32; dq: [n, HD] bf16.  A block takes 32
// consecutive elements; its warp g sums the sequences b = g, g + 8, g + 16, ...
// in order (lane = element, so every load of a warp is one 128-byte row piece),
// and the eight partial sums are added in the order g = 0..7.  The order is
// fixed, so the result is reproducible bit for bit.
constexpr int kReduceGroups = 8;

__global__ void __launch_bounds__(32 * kReduceGroups)
    bcast_reduce_kernel(const float *__restrict__ ws, int B, int n, int64_t HD, __nv_bfloat16 *__restrict__ dq) {
    __shared__ float part[kReduceGroups][32];
    const int64_t total = static_cast<int64_t>(n) * HD;
    const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
    for (int64_t e0 = static_cast<int64_t>(blockIdx.x) * 32; e0 < total; e0 += static_cast<int64_t>(gridDim.x) * 32) {
        const int64_t e = e0 + lane;
        float acc = 0.0f;
        if (e < total)
            for (int b = grp; b < B; b += kReduceGroups) acc += ws[static_cast<int64_t>(b) * total + e];
        part[grp][lane] = acc;
        __syncthreads();
        if (grp == 0 && e < total) {
            float s_ = part[0][lane];
#pragma unroll
            for (int k = 1; k < kReduceGroups; ++k) s_ += part[k][lane];
            dq[e] = __float2bfloat16_rn(s_);
        }
        __syncthreads();
    }
}

cudaError_t launch_bcast_reduce(const float *ws, int B, int n, int64_t HD, void *dq, cudaStream_t stream) {
    const int64_t total = static_cast<int64_t>(n) * HD;
    if (total <= 0 || B <= 0) return cudaSuccess;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (total + 31) / 32;
    const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 8));
    bcast_reduce_kernel<<<blocks, 32 * kReduceGroups, 0, stream>>>(ws, B, n, HD, static_cast<__nv_bfloat16 *>(dq));
    return cudaGetLastError();
}

}  // namespace jattn
