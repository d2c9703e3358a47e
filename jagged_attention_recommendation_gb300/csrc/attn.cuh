// attn.cuh -- pieces shared by the attention kernels: tile records, bias
// lookup, swizzled shared-memory row writes, result stores, activations.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "common.h"
#include "device.cuh"

namespace jattn {
namespace dev {

__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int round_up16(int a) { return (a + 15) & ~15; }

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Reads tile record `idx` and checks it against the batch geometry.  A record
// that fails the checks is reported on the status word and skipped by every
// role of the CTA alike (they all read the same record).
__device__ __forceinline__ bool load_tile(const Geom &g, int idx, Tile &t, const ErrCtx &e, bool report) {
    t = g.tiles[idx];
    bool ok = t.b >= 0 && t.b < g.B && t.h >= 0 && t.h < g.H && t.q_len >= 0 && t.q_len <= g.max_q_len &&
              t.kv_len >= 0 && t.kv_len <= g.max_kv_len && t.q_start >= 0 && t.kv_start >= 0 &&
              static_cast<int64_t>(t.q_start) + t.q_len <= g.Tq &&
              static_cast<int64_t>(t.kv_start) + t.kv_len <= g.Tk;
    if (!ok && report) raise_error(e, kStatusDeviceCheck);
    return ok;
}

// Copy the whole bias table [H, nb] into shared memory, times `mul`
// (all threads of the CTA, before the roles split; a __syncthreads follows).
__device__ __forceinline__ void stage_bias(const Geom &g, float *sbias, float mul) {
    if (g.nb <= 0) return;
    for (int i = threadIdx.x; i < g.H * g.nb; i += blockDim.x) sbias[i] = g.bias[i] * mul;
}

// Bias for the 32 keys kv0..kv0+31 of local query position q: T[min(|q - kv|, nb-1)].
// `bt` is the head's table row in shared memory, already scaled.
__device__ __forceinline__ void bias32(const float *bt, int nb, int q, int kv0, float (&bv)[32]) {
    const int lo = q - (kv0 + 31), hi = kv0 - q;  // distance bounds when the chunk lies left / right of q
    const int dmin = lo > 0 ? lo : (hi > 0 ? hi : 0);
    if (dmin >= nb - 1) {
        const float c = bt[nb - 1];
#pragma unroll
        for (int i = 0; i < 32; ++i) bv[i] = c;
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            int d = q - (kv0 + i);
            d = d < 0 ? -d : d;
            bv[i] = bt[d < nb - 1 ? d : nb - 1];
        }
    }
}

// Write 32 values of one row as bf16 into a 128B-swizzled tile (sub-tiles of
// 64 columns, `sub_bytes` apart), columns c0..c0+31 (c0 a multiple of 32).
__device__ __forceinline__ void st_row32_bf16(uint32_t tile, uint32_t sub_bytes, uint32_t row, uint32_t c0,
                                              const float (&v)[32]) {
    const uint32_t base = tile + (c0 >> 6) * sub_bytes;
    const uint32_t k0 = (c0 & 63u) >> 3;  // first 16-byte chunk within the 128-byte row
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        st_shared_v4(base + sw128_offset(row, k0 + k), pack_bf16x2(v[8 * k + 0], v[8 * k + 1]),
                     pack_bf16x2(v[8 * k + 2], v[8 * k + 3]), pack_bf16x2(v[8 * k + 4], v[8 * k + 5]),
                     pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
    }
}

// Same, splitting every value into a bf16 high part and a bf16 remainder, so
// that hi + lo carries ~16 significant bits into the tensor-core product.
__device__ __forceinline__ void st_row32_bf16_hilo(uint32_t tile_hi, uint32_t tile_lo, uint32_t sub_bytes,
                                                   uint32_t row, uint32_t c0, const float (&v)[32]) {
    const uint32_t off = (c0 >> 6) * sub_bytes;
    const uint32_t k0 = (c0 & 63u) >> 3;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = v[8 * k + 2 * e], b = v[8 * k + 2 * e + 1];
            __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
            const float ra = a - __bfloat162float(h2.x), rb = b - __bfloat162float(h2.y);
            hi[e] = *reinterpret_cast<uint32_t *>(&h2);
            lo[e] = pack_bf16x2(ra, rb);
        }
        const uint32_t o = off + sw128_offset(row, k0 + k);
        st_shared_v4(tile_hi + o, hi[0], hi[1], hi[2], hi[3]);
        st_shared_v4(tile_lo + o, lo[0], lo[1], lo[2], lo[3]);
    }
}

__device__ __forceinline__ void st_row32_zero(uint32_t tile, uint32_t sub_bytes, uint32_t row, uint32_t c0) {
    const uint32_t base = tile + (c0 >> 6) * sub_bytes;
    const uint32_t k0 = (c0 & 63u) >> 3;
#pragma unroll
    for (int k = 0; k < 4; ++k) st_shared_v4(base + sw128_offset(row, k0 + k), 0u, 0u, 0u, 0u);
}

// Store columns c0..c0+31 (times `mul`) of result row `row`, head h.
__device__ __forceinline__ void store_out32(const OutDesc &o, int64_t row, int h, int c0, const float (&v)[32],
                                            float mul) {
    const int n = o.cols - c0;
    if (n <= 0) return;
    if (o.f32) {
        float *p = static_cast<float *>(o.ptr) + row * o.ld + static_cast<int64_t>(h) * o.cols + c0;
        if (n >= 32) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                reinterpret_cast<float4 *>(p)[k] =
                    make_float4(v[4 * k] * mul, v[4 * k + 1] * mul, v[4 * k + 2] * mul, v[4 * k + 3] * mul);
        } else {
            for (int i = 0; i < n; ++i) p[i] = v[i] * mul;
        }
    } else {
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(o.ptr) + row * o.ld + static_cast<int64_t>(h) * o.cols + c0;
        if (n >= 32) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint4 w;
                w.x = pack_bf16x2(v[8 * k + 0] * mul, v[8 * k + 1] * mul);
                w.y = pack_bf16x2(v[8 * k + 2] * mul, v[8 * k + 3] * mul);
                w.z = pack_bf16x2(v[8 * k + 4] * mul, v[8 * k + 5] * mul);
                w.w = pack_bf16x2(v[8 * k + 6] * mul, v[8 * k + 7] * mul);
                reinterpret_cast<uint4 *>(p)[k] = w;
            }
        } else {
            for (int i = 0; i < n; ++i) p[i] = __float2bfloat16_rn(v[i] * mul);
        }
    }
}

// act(x) = x * sigmoid(z) with z = x (SiLU) or z = 2 sqrt(2/pi) (x + 0.044715 x^3)
// (tanh-GELU, since (1 + tanh(u)) / 2 = sigmoid(2u)).
constexpr float kGeluC2 = 1.5957691216057308f;  // 2 * sqrt(2 / pi)
constexpr float kGeluA = 0.044715f;

__device__ __forceinline__ float act_fwd(int act, float x) {
    const float z = act == kSilu ? x : kGeluC2 * fmaf(kGeluA * x, x * x, x);
    return x * sigmoid_f(z);
}

// act'(x) = sigmoid(z) + x sigmoid(z) (1 - sigmoid(z)) z'(x); also returns act(x).
__device__ __forceinline__ float act_bwd(int act, float x, float &a) {
    float z, dz;
    if (act == kSilu) {
        z = x;
        dz = 1.0f;
    } else {
        z = kGeluC2 * fmaf(kGeluA * x, x * x, x);
        dz = kGeluC2 * fmaf(3.0f * kGeluA, x * x, 1.0f);
    }
    const float sg = sigmoid_f(z);
    a = x * sg;
    return fmaf(x * sg * (1.0f - sg), dz, sg);
}

template <int N>
__device__ __forceinline__ float (&sub32(float (&a)[N], int c))[32] {
    return *reinterpret_cast<float(*)[32]>(&a[32 * c]);
}

}  // namespace dev
}  // namespace jattn
