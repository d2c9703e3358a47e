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
    // Two rows per lane group and pass, both rows' loads issued before either
    // sum.  Whole warps stay in the loop together so the shuffles see every lane.
    const int64_t rstep = nthreads / tpr;
    for (int64_t base = (gtid / tpr) - ((threadIdx.x & 31) / tpr); base < nrows; base += 2 * rstep) {
        const int64_t r[2] = {base + (threadIdx.x & 31) / tpr, base + (threadIdx.x & 31) / tpr + rstep};
        uint4 o[2], d[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            o[j] = d[j] = make_uint4(0u, 0u, 0u, 0u);
            if (r[j] < nrows) {
                o[j] = __ldg(reinterpret_cast<const uint4 *>(out + r[j] * D) + sub);
                d[j] = __ldg(reinterpret_cast<const uint4 *>(dout + r[j] * D) + sub);
            }
        }
        float acc[2] = {dot16<T>(o[0], d[0]), dot16<T>(o[1], d[1])};
        for (int k = tpr >> 1; k > 0; k >>= 1) {
            acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], k);
            acc[1] += __shfl_xor_sync(0xffffffffu, acc[1], k);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (sub == 0 && r[j] < nrows) {
                const int64_t t = r[j] / H;
                const int h = static_cast<int>(r[j] - t * H);
                delta[static_cast<int64_t>(h) * Tq + t] = acc[j];
            }
        }
    }
}

// MXFP8 quantisation of up to four tensors x [T, H, D] (bf16) per sequence and
// head, in blocks of 32 local rows x 32 features: xq receives the values the
// quantised blocks stand for (bf16, exact).  The work items are the plan's
// 128-row tiles of each tensor's side (every tile is one sequence and head,
// and starts at a multiple of 128 local rows, so its 32-row slices are the
// blocks' rows).  A CTA takes one tile, each of its four warps one 32-row
// slice, all D features: a warp instruction reads whole rows' D features (16
// bytes a lane, D / 8 lanes a row), so every load and store is row-contiguous.
// A block's largest magnitude comes from the four lanes of its 32 features
// over the slice's rows, by butterfly shuffles.  Each lane holds its 32 rows'
// loads at once (D = 128: 64 registers), so the launch bound keeps three CTAs
// on an SM without spilling.
__device__ __forceinline__ uint32_t mx_qdq_bf16x2(uint32_t w, float down, float up) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(make_float2(lo * down, hi * down), __NV_SATFINITE, __NV_E4M3);
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(q, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
    return dev::pack_bf16x2(f.x * up, f.y * up);
}

__device__ __forceinline__ float amax_bf16x2(float a, uint32_t w) {
    return fmaxf(a, fmaxf(fabsf(__uint_as_float(w << 16)), fabsf(__uint_as_float(w & 0xffff0000u))));
}

template <int D>
__global__ void __launch_bounds__(128, 3) mx_quant_kernel(const __grid_constant__ MxJobs jobs, int H) {
    constexpr int LPR = D / 8;     // lanes per row, 16 bytes each
    constexpr int RPI = 32 / LPR;  // rows per warp instruction
    constexpr int NI = 32 / RPI;   // instructions per 32-row slice
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / LPR, c = lane % LPR;
    int total = 0;
    for (int j = 0; j < jobs.n; ++j) total += jobs.ntiles[j];
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        int j = 0, i = t;
        while (j + 1 < jobs.n && i >= jobs.ntiles[j]) i -= jobs.ntiles[j++];
        const Tile tile = jobs.tiles[j][i];
        const int start = jobs.kv_side[j] ? tile.kv_start : tile.q_start;
        const int n = min(32, (jobs.kv_side[j] ? tile.kv_len : tile.q_len) - 32 * warp);
        if (n <= 0) continue;
        const int64_t rs = static_cast<int64_t>(H) * D;
        const int64_t base = (static_cast<int64_t>(start + 32 * warp) * H + tile.h) * D + c * 8;
        const __nv_bfloat16 *src = static_cast<const __nv_bfloat16 *>(jobs.x[j]) + base;
        uint4 w[NI];
        float a = 0.0f;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int row = k * RPI + sub;
            w[k] = row < n ? __ldg(reinterpret_cast<const uint4 *>(src + row * rs)) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < NI; ++k) a = amax_bf16x2(amax_bf16x2(amax_bf16x2(amax_bf16x2(a, w[k].x), w[k].y), w[k].z), w[k].w);
        // the block's lanes: the four of its features (lane bits 0, 1) on every row group
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
#pragma unroll
        for (int m = LPR; m < 32; m <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
        const int e = dev::mx_exponent(a);
        const float down = dev::pow2i(-e), up = dev::pow2i(e);
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(jobs.xq[j]) + base;
#pragma unroll
        for (int k = 0; k < NI; ++k) {
            const int row = k * RPI + sub;
            if (row < n)
                *reinterpret_cast<uint4 *>(dst + row * rs) =
                    make_uint4(mx_qdq_bf16x2(w[k].x, down, up), mx_qdq_bf16x2(w[k].y, down, up),
                               mx_qdq_bf16x2(w[k].z, down, up), mx_qdq_bf16x2(w[k].w, down, up));
        }
    }
}

cudaError_t launch_mx_quant(const MxJobs &jobs, int H, int D, cudaStream_t stream) {
    int64_t total = 0;
    for (int j = 0; j < jobs.n; ++j) total += jobs.ntiles[j];
    if (total == 0) return cudaSuccess;
    if (jobs.n < 1 || jobs.n > 4 || (D != 64 && D != 128)) return cudaErrorInvalidValue;
    // about one tile per CTA: the hardware hands tiles to SMs as CTAs finish
    const int blocks = static_cast<int>(std::min<int64_t>(total, 152 * 64));
    if (D == 128)
        mx_quant_kernel<128><<<blocks, 128, 0, stream>>>(jobs, H);
    else
        mx_quant_kernel<64><<<blocks, 128, 0, stream>>>(jobs, H);
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
