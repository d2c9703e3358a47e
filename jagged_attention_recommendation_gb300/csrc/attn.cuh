// attn.cuh -- pieces shared by the attention kernels: tile records, bias
// lookup, swizzled shared-memory row writes, result stores, activations.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
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

// Checks a tile record against the batch geometry.  A record that fails is
// reported on the status word and skipped by every role of the CTA alike (they
// all read the same record).
__device__ __forceinline__ bool check_tile(const Geom &g, const Tile &t, const ErrCtx &e, bool report) {
    bool ok = t.b >= 0 && t.b < g.B && t.h >= 0 && t.h < g.H && t.q_len >= 0 && t.q_len <= g.max_q_len &&
              t.kv_len >= 0 && t.kv_len <= g.max_kv_len && t.q_start >= 0 && t.kv_start >= 0 &&
              t.q_loc0 >= 0 && t.kv_loc0 >= 0 && static_cast<int64_t>(t.q_start) + t.q_len <= g.Tq &&
              static_cast<int64_t>(t.kv_start) + t.kv_len <= g.Tk &&
              (g.rope_cos == nullptr ||
               (t.q_loc0 + t.q_len <= g.rope_rows && t.kv_loc0 + t.kv_len <= g.rope_rows));
    if (!ok && report) raise_error(e, kStatusDeviceCheck);
    return ok;
}

// A CTA's tile range, read one record ahead so that the global load of the
// next record overlaps the current tile's work.
struct TileStream {
    const Tile *p;
    int i, end;
    Tile nxt;
    __device__ __forceinline__ TileStream(const Geom &g, int begin, int stop) : p(g.tiles), i(begin), end(stop) {
        if (i < end) nxt = p[i];
    }
    __device__ __forceinline__ bool next(Tile &t) {
        if (i >= end) return false;
        t = nxt;
        if (++i < end) nxt = p[i];
        return true;
    }
};

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

// Sliding window |p - o| < W on local positions: bit k is set when position
// o0 + k of the other side is inside row p's band (all bits when W == 0).
__device__ __forceinline__ uint32_t window_bits32(int W, int p, int o0) {
    if (W <= 0) return 0xffffffffu;
    const int lo = p - W + 1 - o0, hi = p + W - 1 - o0;  // allowed k in [lo, hi]
    if (lo <= 0 && hi >= 31) return 0xffffffffu;
    if (hi < 0 || lo > 31) return 0u;
    const int a = lo < 0 ? 0 : lo, b = hi > 31 ? 31 : hi;
    const uint32_t upto = b == 31 ? 0xffffffffu : ((1u << (b + 1)) - 1u);
    return upto & ~((1u << a) - 1u);
}
// False when none of rows p0..p0+31 has o0..o0+31 in its band (a warp-uniform test).
__device__ __forceinline__ bool window_chunk_live(int W, int p0, int o0) {
    return W <= 0 || (o0 <= p0 + 31 + W - 1 && o0 + 31 >= p0 - W + 1);
}
// Entries of a 32-wide chunk outside the band take `fill`.
__device__ __forceinline__ void window_fill32(float (&x)[32], uint32_t bits, float fill) {
    if (bits == 0xffffffffu) return;
#pragma unroll
    for (int k = 0; k < 32; ++k)
        if (!((bits >> k) & 1u)) x[k] = fill;
}

// Row-contiguous output through shared memory.  With one thread per result
// row, a direct 16-byte store per thread touches 32 rows per instruction; a
// warp instead stages W columns of its 32 rows as bf16 in a buffer of 32 x W
// values (the 16-byte chunks of a row XOR-swizzled by row, so that neither the
// per-row writes nor the row-contiguous reads have bank conflicts) and then
// writes W-column row pieces, W / 8 lanes per row.
template <int W>
__device__ __forceinline__ void stage_row32_bf16(uint32_t stg, int lane, int c0, const uint32_t (&w)[16]) {
    static_assert(W == 64 || W == 128, "staged width");
    const uint32_t rowb = stg + static_cast<uint32_t>(lane) * (W * 2);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t ch = static_cast<uint32_t>((c0 >> 3) + k) ^ static_cast<uint32_t>(lane & 7);
        st_shared_v4(rowb + ch * 16, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
}
// Rows 0..nrows-1 of the staged block to base + r * ld (bf16 elements); call
// after a __syncwarp that follows the last stage_row32_bf16 of the block.
template <int W>
__device__ __forceinline__ void store_rows_bf16(uint32_t stg, int lane, __nv_bfloat16 *base, int64_t ld, int nrows) {
    constexpr int CPR = W / 8;     // 16-byte chunks per row
    constexpr int RPI = 32 / CPR;  // rows per instruction
    const int ch = lane % CPR, rsub = lane / CPR;
#pragma unroll
    for (int it = 0; it < 32 / RPI; ++it) {
        const int r = it * RPI + rsub;
        const uint4 v = ld_shared_v4(stg + static_cast<uint32_t>(r * (W * 2) + ((ch ^ (r & 7)) * 16)));
        if (r < nrows) *reinterpret_cast<uint4 *>(base + r * ld + ch * 8) = v;
    }
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
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < n) p[i] = v[i] * mul;
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
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < n) p[i] = __float2bfloat16_rn(v[i] * mul);
        }
    }
}

// Copy a warp's 32 staged rows (row0 .. row0+31 of a 128B-swizzled bf16 tile,
// sub-tiles of 64 columns `sub_bytes` apart) to the bf16 result rows
// grow0 + row, head h; rows >= nvalid are skipped.  Consecutive lanes write
// consecutive 16-byte pieces of a row, so every store is a full row segment.
template <int D>
__device__ __forceinline__ void copy_rows_out(uint32_t tile, uint32_t sub_bytes, int row0, int nvalid,
                                              const OutDesc &o, int64_t grow0, int h, uint32_t lane) {
    constexpr int CPR = D / 8;      // 16-byte pieces per row
    constexpr int RPI = 32 / CPR;   // rows per warp instruction
    const int cc = static_cast<int>(lane) % CPR, rsub = static_cast<int>(lane) / CPR;
    uint4 v[32 / RPI];
#pragma unroll
    for (int k = 0; k < 32 / RPI; ++k)
        v[k] = ld_shared_v4(tile + (cc >> 3) * sub_bytes + sw128_offset(row0 + k * RPI + rsub, cc & 7));
#pragma unroll
    for (int k = 0; k < 32 / RPI; ++k) {
        const int r = row0 + k * RPI + rsub;
        if (r < nvalid) {
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(o.ptr) + (grow0 + r) * o.ld +
                                 static_cast<int64_t>(h) * D + cc * 8;
            *reinterpret_cast<uint4 *>(dst) = v[k];
        }
    }
}

// Copy a warp's 32 staged rows of one 64-column sub-tile (128B-swizzled bf16,
// rows row0 .. row0+31) to columns gcol0 .. gcol0+63 of the bf16 result rows
// grow0 + row, head h; rows >= nvalid are skipped.  Eight lanes cover one
// 128-byte row segment, so each warp store writes four whole segments.
template <int D>
__device__ __forceinline__ void copy_seg64(uint32_t sub, int row0, int nvalid, const OutDesc &o, int64_t grow0,
                                           int h, int gcol0, uint32_t lane) {
    const int cc = static_cast<int>(lane) & 7, rsub = static_cast<int>(lane) >> 3;
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = ld_shared_v4(sub + sw128_offset(row0 + 4 * k + rsub, cc));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int r = row0 + 4 * k + rsub;
        if (r < nvalid) {
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(o.ptr) + (grow0 + r) * o.ld +
                                 static_cast<int64_t>(h) * D + gcol0 + cc * 8;
            *reinterpret_cast<uint4 *>(dst) = v[k];
        }
    }
}

// Same, for a W-column slice [c0, c0 + W) of rows of width D: lanes write
// consecutive 16-byte pieces of each row slice.
template <int W, int D>
__device__ __forceinline__ void copy_rows_cols(uint32_t tile, uint32_t sub_bytes, int c0, int row0, int nvalid,
                                               const OutDesc &o, int64_t grow0, int h, uint32_t lane) {
    constexpr int CPR = W / 8;
    constexpr int RPI = 32 / CPR;
    const int cc = static_cast<int>(lane) % CPR, rsub = static_cast<int>(lane) / CPR;
    const int col = c0 + cc * 8;
    const uint32_t src = tile + (col >> 6) * sub_bytes;
    uint4 v[32 / RPI];
#pragma unroll
    for (int k = 0; k < 32 / RPI; ++k) v[k] = ld_shared_v4(src + sw128_offset(row0 + k * RPI + rsub, (col & 63) >> 3));
#pragma unroll
    for (int k = 0; k < 32 / RPI; ++k) {
        const int r = row0 + k * RPI + rsub;
        if (r < nvalid) {
            __nv_bfloat16 *dst =
                static_cast<__nv_bfloat16 *>(o.ptr) + (grow0 + r) * o.ld + static_cast<int64_t>(h) * D + col;
            *reinterpret_cast<uint4 *>(dst) = v[k];
        }
    }
}

// True when results can be staged and written as whole bf16 rows of width D.
template <int D>
__device__ __forceinline__ bool rows_fast(const OutDesc &o) {
    return o.f32 == 0 && o.cols == D;
}

// act(x) = x * sigmoid(z) with z = x (SiLU) or z = 2 sqrt(2/pi) (x + 0.044715 x^3)
// (tanh-GELU, since (1 + tanh(u)) / 2 = sigmoid(2u)).
constexpr float kGeluC2 = 1.5957691216057308f;  // 2 * sqrt(2 / pi)
constexpr float kGeluA = 0.044715f;

__device__ __forceinline__ float act_fwd(int act, float x) {
    const float z = act == kSilu ? x : kGeluC2 * fmaf(kGeluA * x, x * x, x);
    return x * sigmoid_f(z);
}

// The same with the activation fixed at compile time, so that a loop over
// many elements carries no per-element test and its exponential / reciprocal
// chains overlap.
template <int AF>
__device__ __forceinline__ float act_fwd_t(float x) {
    if constexpr (AF == kSilu) {
        return x * sigmoid_f(x);
    } else {
        return x * sigmoid_f(kGeluC2 * fmaf(kGeluA * x, x * x, x));
    }
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

// The same with the activation fixed at compile time.
template <int AF>
__device__ __forceinline__ float act_bwd_t(float x, float &a) {
    float z, dz;
    if constexpr (AF == kSilu) {
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

// ---------------------------------------------------------------------------
// packed fp32 pairs (sm_100 family f32x2 arithmetic) and 3-input max
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk(uint64_t r, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
// (a0, a1) <- (a0, a1) * (b0, b1) + (c0, c1)
__device__ __forceinline__ void fma2(float &a0, float &a1, float b0, float b1, float c0, float c1) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk(a0, a1)), "l"(pk(b0, b1)), "l"(pk(c0, c1)));
    upk(r, a0, a1);
}
// (a0, a1) <- (a0, a1) + (b0, b1)
__device__ __forceinline__ void add2(float &a0, float &a1, float b0, float b1) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a0, a1)), "l"(pk(b0, b1)));
    upk(r, a0, a1);
}
// (a0, a1) <- (a0, a1) * (b0, b1)
__device__ __forceinline__ void mul2(float &a0, float &a1, float b0, float b1) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a0, a1)), "l"(pk(b0, b1)));
    upk(r, a0, a1);
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Maximum of 32 values with a tree of 3-input max operations.
__device__ __forceinline__ float max32(const float (&v)[32]) {
    float m[11];
#pragma unroll
    for (int k = 0; k < 10; ++k) m[k] = max3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
    m[10] = fmaxf(v[30], v[31]);
    const float a = max3(m[0], m[1], m[2]), b = max3(m[3], m[4], m[5]), c = max3(m[6], m[7], m[8]);
    return max3(max3(a, b, c), m[9], m[10]);
}

// Sum of 32 values with four independent packed accumulators.
__device__ __forceinline__ float sum32(const float (&v)[32]) {
    float a0 = v[0], a1 = v[1], b0 = v[2], b1 = v[3];
#pragma unroll
    for (int k = 4; k < 32; k += 4) {
        add2(a0, a1, v[k], v[k + 1]);
        add2(b0, b1, v[k + 2], v[k + 3]);
    }
    add2(a0, a1, b0, b1);
    return a0 + a1;
}

// ---------------------------------------------------------------------------
// MXFP8 ("Training GEM at LLM scale", section "Low Precision Flash Attention"):
// FP8 E4M3 elements with one power-of-two (E8M0) scale per block.  The scale
// exponent of a block with largest magnitude amax is floor(log2 amax) - 8 (8 =
// the exponent of E4M3's largest normal, 448), clamped to [-127, 127], read
// from the float's exponent bits; an element x becomes E4M3(x 2^-e) 2^e, the
// E4M3 rounding to nearest even and saturating at +-448.
// ---------------------------------------------------------------------------
// 2^k as a float, k in [-149, 127]
__device__ __forceinline__ float pow2i(int k) {
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}
// block exponent of a non-negative amax
__device__ __forceinline__ int mx_exponent(float amax) {
    const int e = ((__float_as_int(amax) >> 23) & 0xFF) - 127 - 8;  // zero / subnormal: below -127
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}
// the values of 32 elements' MXFP8 quantisation with block exponent e, in place
__device__ __forceinline__ void mx_qdq32(float (&x)[32], int e) {
    const float down = pow2i(-e), up = pow2i(e);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const __nv_fp8x2_storage_t q =
            __nv_cvt_float2_to_fp8x2(make_float2(x[i] * down, x[i + 1] * down), __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(q, __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
        x[i] = f.x * up;
        x[i + 1] = f.y * up;
    }
}
// largest magnitude of 32 values
__device__ __forceinline__ float amax32(const float (&x)[32]) {
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(x[i]));
    return a;
}
// largest of a non-negative value over the warp (non-negative floats order as
// their bit patterns)
__device__ __forceinline__ float warp_max_nonneg(float a) {
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(a)));
}

// ---------------------------------------------------------------------------
// relative-position bias as a reflected table: ext[x + kExtPad] =
// T[min(|x|, nb-1)] * mul for |x| <= nb - 1 + 31, so that the 32 biases of a
// chunk that touches the band are a contiguous (reversed) window.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int ext_pad(int nb) { return nb - 1 + 31; }
__host__ __device__ constexpr int ext_len(int nb) { return 2 * ext_pad(nb) + 1; }

__device__ __forceinline__ void stage_bias_ext(const Geom &g, float *sext, float mul) {
    if (g.nb <= 0) return;
    const int pad = ext_pad(g.nb), len = ext_len(g.nb);
    for (int i = threadIdx.x; i < g.H * len; i += blockDim.x) {
        const int h = i / len;
        int x = i - h * len - pad;
        x = x < 0 ? -x : x;
        sext[i] = g.bias[h * g.nb + (x < g.nb - 1 ? x : g.nb - 1)] * mul;
    }
}

// Bias of keys kv0..kv0+31 for local query position q (or, symmetrically, of
// queries for a key): returns false and a constant when the chunk lies
// entirely beyond the last bucket, else fills bv from the reflected table.
__device__ __forceinline__ bool bias32_ext(const float *ext_h, int nb, int q, int kv0, float (&bv)[32], float &cst) {
    const int lo = q - (kv0 + 31), hi = kv0 - q;
    const int dmin = lo > 0 ? lo : (hi > 0 ? hi : 0);
    if (dmin >= nb - 1) {
        cst = ext_h[0];  // |x| = pad >= nb - 1: the last bucket
        return false;
    }
    const float *p = ext_h + ext_pad(nb) + (q - kv0);  // p[-i] = bias of key kv0 + i
#pragma unroll
    for (int i = 0; i < 32; ++i) bv[i] = p[-i];
    return true;
}

// One accumulator row of D fp32 columns from TMEM (one round trip).
template <int D>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, float (&v)[D]) {
    if constexpr (D == 128) {
        tmem_ld128(taddr, v);
    } else if constexpr (D == 64) {
        tmem_ld64(taddr, v);
    } else {
        static_assert(D == 32, "32, 64 or 128 columns");
        tmem_ld32(taddr, v);
    }
}

// x[i] = x[i] * sc + bias(key kv0 + i) for a 32-column chunk, bias read straight
// from the reflected table (or the constant last bucket when the chunk is past it).
__device__ __forceinline__ void scale_bias32(float (&x)[32], float sc, const float *ext_h, int nb, int q, int kv0) {
    const int lo = q - (kv0 + 31), hi = kv0 - q;
    const int dmin = lo > 0 ? lo : (hi > 0 ? hi : 0);
    if (dmin >= nb - 1) {
        const float c = ext_h[0];
#pragma unroll
        for (int i = 0; i < 32; i += 2) fma2(x[i], x[i + 1], sc, sc, c, c);
    } else {
        const float *p = ext_h + ext_pad(nb) + (q - kv0);
#pragma unroll
        for (int i = 0; i < 32; i += 2) fma2(x[i], x[i + 1], sc, sc, p[-i], p[-i - 1]);
    }
}

// Scale and relative-position bias of a 32-wide chunk, plus a constant offset:
// x[i] = x[i] * sc + bias(position p, other positions o0 .. o0+31) + off.
// BIAS: 0 none, 1 reflected table ext_h, 2 plain table bt (see the kernels).
template <int BIAS>
__device__ __forceinline__ void scale_bias_off32(float (&x)[32], float sc, float off, const float *ext_h,
                                                 const float *bt, int nb, int p, int o0) {
    if constexpr (BIAS == 0) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) fma2(x[i], x[i + 1], sc, sc, off, off);
    } else {
        float bv[32], cst = 0.0f;
        bool band = true;
        if constexpr (BIAS == 1) {
            band = bias32_ext(ext_h, nb, p, o0, bv, cst);
        } else {
            bias32(bt, nb, p, o0, bv);
        }
        if (band) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                add2(bv[i], bv[i + 1], off, off);
                fma2(x[i], x[i + 1], sc, sc, bv[i], bv[i + 1]);
            }
        } else {
            const float o2 = cst + off;
#pragma unroll
            for (int i = 0; i < 32; i += 2) fma2(x[i], x[i + 1], sc, sc, o2, o2);
        }
    }
}

template <int N>
__device__ __forceinline__ float (&sub64(float (&a)[N], int c))[64] {
    return *reinterpret_cast<float(*)[64]>(&a[64 * c]);
}

template <int N>
__device__ __forceinline__ float (&sub32(float (&a)[N], int c))[32] {
    return *reinterpret_cast<float(*)[32]>(&a[32 * c]);
}

// Rotary position embedding, in place, of rows [0, nrows) of one or two
// [128, D] bf16 operand tiles in 128B-swizzled shared memory (D/64 sub-tiles of
// 128 rows x 64 columns, sub_bytes apart; tile2 = 0: one tile).  Row r of
// both tiles sits at the same position, whose cos and sin rows (D/2 floats
// each) start at tc + r * D/2 and ts + r * D/2 (generic pointers: shared or
// global memory).  Feature pair (d, d + D/2), d < D/2, with c = cos, s = sin:
//   x[d] <- x[d] c - x[d + D/2] s,   x[d + D/2] <- x[d + D/2] c + x[d] s,
// each product rounded to float32, then one fused multiply-add, then bf16.
// One warp: a lane takes four feature pairs (16 bytes of table row, 8 of each
// bf16 half) of one row per pass; D/8 lanes cover a row.  With D = 64 a pass
// covers rows {0, 4, 1, 5} or {2, 6, 3, 7} of an 8-row band, so that both the
// swizzled 8-byte tile accesses and the 16-byte table accesses of a warp spread
// evenly over the shared-memory banks.
__device__ __forceinline__ void rope_pairs4(uint32_t alo, uint32_t ahi, const float4 &c, const float4 &s) {
    const uint2 x = ld_shared_v2(alo), y = ld_shared_v2(ahi);
    float x0 = __uint_as_float(x.x << 16), x1 = __uint_as_float(x.x & 0xffff0000u);
    float x2 = __uint_as_float(x.y << 16), x3 = __uint_as_float(x.y & 0xffff0000u);
    float y0 = __uint_as_float(y.x << 16), y1 = __uint_as_float(y.x & 0xffff0000u);
    float y2 = __uint_as_float(y.y << 16), y3 = __uint_as_float(y.y & 0xffff0000u);
    // t = -y s, u = x s (rounded), then a = x c + t, b = y c + u
    float t0 = y0, t1 = y1, t2 = y2, t3 = y3, u0 = x0, u1 = x1, u2 = x2, u3 = x3;
    mul2(t0, t1, -s.x, -s.y);
    mul2(t2, t3, -s.z, -s.w);
    mul2(u0, u1, s.x, s.y);
    mul2(u2, u3, s.z, s.w);
    fma2(x0, x1, c.x, c.y, t0, t1);
    fma2(x2, x3, c.z, c.w, t2, t3);
    fma2(y0, y1, c.x, c.y, u0, u1);
    fma2(y2, y3, c.z, c.w, u2, u3);
    st_shared_v2(alo, pack_bf16x2(x0, x1), pack_bf16x2(x2, x3));
    st_shared_v2(ahi, pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
}

template <int D, int UNROLL>
__device__ __forceinline__ int rope_row(int k, int grp) {
    constexpr int RP = 32 / (D / 8);  // rows per pass
    if (RP == 4) {
        const int i = (k & 1) * 4 + grp;                 // 0..7
        return (k >> 1) * 8 + ((i >> 1) | ((i & 1) << 2));  // rows 0, 4, 1, 5 | 2, 6, 3, 7 of the band
    }
    return k * RP + grp;
}

// UNROLL passes at a time: their table loads are all issued before the first
// rotation touches shared memory, so their latencies overlap.
template <int D, int UNROLL>
__device__ __forceinline__ void rope_tile(uint32_t tile, uint32_t tile2, uint32_t sub_bytes, int nrows,
                                          const float *tc, const float *ts, int lane) {
    constexpr int PPR = D / 8;       // lanes per row (four feature pairs each)
    constexpr int RP = 32 / PPR;     // rows per pass
    const int piece = lane % PPR, grp = lane / PPR;
    const uint32_t lo_col = piece * 4, hi_col = piece * 4 + D / 2;
    const uint32_t lo_off = (lo_col >> 6) * sub_bytes + (piece & 1) * 8u;
    const uint32_t hi_off = (hi_col >> 6) * sub_bytes + (piece & 1) * 8u;
    const uint32_t lo_chunk = (lo_col & 63u) >> 3, hi_chunk = (hi_col & 63u) >> 3;
    // passes that reach row nrows - 1 (with RP = 4, two passes cover an 8-row band);
    // rows at or past nrows in the last batch are skipped
    const int npass = RP == 4 ? 2 * ((nrows + 7) / 8) : (nrows + RP - 1) / RP;
#pragma unroll 1
    for (int k0 = 0; k0 < npass; k0 += UNROLL) {
        float4 c[UNROLL], s[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int r = rope_row<D, UNROLL>(k0 + u, grp);
            if (r < nrows) {
                c[u] = *reinterpret_cast<const float4 *>(tc + r * (D / 2) + piece * 4);
                s[u] = *reinterpret_cast<const float4 *>(ts + r * (D / 2) + piece * 4);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int r = rope_row<D, UNROLL>(k0 + u, grp);
            if (r < nrows) {
                const uint32_t olo = lo_off + sw128_offset(r, lo_chunk), ohi = hi_off + sw128_offset(r, hi_chunk);
                rope_pairs4(tile + olo, tile + ohi, c[u], s[u]);
                if (tile2 != 0u) rope_pairs4(tile2 + olo, tile2 + ohi, c[u], s[u]);
            }
        }
    }
}

// rope_tile with the table rows in shared memory (tc, ts: shared addresses).
template <int D, int UNROLL>
__device__ __forceinline__ void rope_tile_s(uint32_t tile, uint32_t tile2, uint32_t sub_bytes, int nrows, uint32_t tc,
                                            uint32_t ts, int lane) {
    constexpr int PPR = D / 8;
    constexpr int RP = 32 / PPR;
    const int piece = lane % PPR, grp = lane / PPR;
    const uint32_t lo_col = piece * 4, hi_col = piece * 4 + D / 2;
    const uint32_t lo_off = (lo_col >> 6) * sub_bytes + (piece & 1) * 8u;
    const uint32_t hi_off = (hi_col >> 6) * sub_bytes + (piece & 1) * 8u;
    const uint32_t lo_chunk = (lo_col & 63u) >> 3, hi_chunk = (hi_col & 63u) >> 3;
    const int npass = RP == 4 ? 2 * ((nrows + 7) / 8) : (nrows + RP - 1) / RP;
#pragma unroll 1
    for (int k0 = 0; k0 < npass; k0 += UNROLL) {
        float4 c[UNROLL], s[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int r = rope_row<D, UNROLL>(k0 + u, grp);
            if (r < nrows) {
                const uint32_t o = (r * (D / 2) + piece * 4) * 4;
                const uint4 cv = ld_shared_v4(tc + o), sv = ld_shared_v4(ts + o);
                c[u] = make_float4(__uint_as_float(cv.x), __uint_as_float(cv.y), __uint_as_float(cv.z),
                                   __uint_as_float(cv.w));
                s[u] = make_float4(__uint_as_float(sv.x), __uint_as_float(sv.y), __uint_as_float(sv.z),
                                   __uint_as_float(sv.w));
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int r = rope_row<D, UNROLL>(k0 + u, grp);
            if (r < nrows) {
                const uint32_t olo = lo_off + sw128_offset(r, lo_chunk), ohi = hi_off + sw128_offset(r, hi_chunk);
                rope_pairs4(tile + olo, tile + ohi, c[u], s[u]);
                if (tile2 != 0u) rope_pairs4(tile2 + olo, tile2 + ohi, c[u], s[u]);
            }
        }
    }
}

// rope_grad32 on values i0..i0+15 with their cos and sin in registers.
__device__ __forceinline__ void rope_grad16_regs(float (&lo)[32], float (&hi)[32], int i0, const float (&c)[16],
                                                 const float (&s)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float x = lo[i0 + i], y = hi[i0 + i];
        lo[i0 + i] = __fmaf_rn(x, c[i], __fmul_rn(y, s[i]));
        hi[i0 + i] = __fmaf_rn(y, c[i], __fmul_rn(-x, s[i]));
    }
}

// The transposed rotation of 32 + 32 float32 values of one row (features
// d0..d0+31 in lo, d0+D/2.. in hi), which carries a gradient with respect to
// the rotated row back to the unrotated one:
//   g[d] = c x[d] + s x[d + D/2],   g[d + D/2] = c x[d + D/2] - s x[d].
// tc, ts: the row's cos and sin from feature d0 on (global memory).
__device__ __forceinline__ void rope_grad32(float (&lo)[32], float (&hi)[32], const float *tc, const float *ts) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 c = *reinterpret_cast<const float4 *>(tc + i);
        const float4 s = *reinterpret_cast<const float4 *>(ts + i);
        const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x = lo[i + e], y = hi[i + e];
            lo[i + e] = __fmaf_rn(x, cc[e], __fmul_rn(y, ss[e]));
            hi[i + e] = __fmaf_rn(y, cc[e], __fmul_rn(-x, ss[e]));
        }
    }
}

}  // namespace dev
}  // namespace jattn
