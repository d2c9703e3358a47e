// bwd_common.cuh -- what the two backward passes (bwd.cu: dQ, bwd_dkdv.cu:
// dK / dV) share: the bias forms, the register split of the four-warpgroup
// layout and the packing of a row's results into TMEM operands.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#define JATTN_INLINE_WAITS 1
#include "attn.cuh"
#include "kernels.h"

namespace jattn {
using namespace dev;

namespace {
enum : int { kBiasNone = 0, kBiasExt = 1, kBiasTable = 2 };

// which bias form a launch takes (the kernels are specialised on it)
inline int bias_form(const Geom &g) {
    if (g.nb <= 0) return kBiasNone;
    return g.H * ext_len(g.nb) <= kMaxBiasExtFloats ? kBiasExt : kBiasTable;
}

// registers per thread after the split (launch: 512 threads x 128)
constexpr uint32_t kRegCtrl = 56, kRegCompute = 176, kRegOut = 104;
static_assert(kRegCtrl * 128 + kRegCompute * 256 + kRegOut * 128 <= 128 * 512, "register split");

// Packs 32 results of one row for a TMEM operand: bf16 pairs (16 words) or,
// with the remainder, hi / lo pairs interleaved per 16-column MMA step (hi at
// words 16k..16k+7, lo at 16k+8..16k+15 for step k of the chunk).
__device__ __forceinline__ void pack16(const float (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
}
__device__ __forceinline__ void pack_hilo32(const float (&v)[32], uint32_t (&w)[32]) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[i], v[i + 1]);
        const int k = i >> 4, e = (i & 15) >> 1;
        w[16 * k + e] = *reinterpret_cast<uint32_t *>(&h2);
        w[16 * k + 8 + e] = pack_bf16x2(v[i] - __bfloat162float(h2.x), v[i + 1] - __bfloat162float(h2.y));
    }
}
}  // namespace
}  // namespace jattn
