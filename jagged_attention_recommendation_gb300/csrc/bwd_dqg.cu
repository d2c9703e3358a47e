// bwd_dqg.cu -- jagged attention backward, dQ as a streaming product of the dS
// chunks that the dK/dV pass wrote ("Training GEM at LLM scale", section
// "Jagged Sequence Flash Attention": the backward computes dQ without atomic
// adds and without recomputing the scores for it).
//
// Per 128-row query tile of one (sequence, head): dQ = scale * sum over the
// sequence's 128-key tiles t of dS(t) K(t), where dS(t) is the 128-query x
// 128-key block of two 16 KB chunks (the tile's two 64-query blocks; the
// activation modes carry a bf16 hi and lo chunk each).  Nothing is
// recomputed: a producer thread bulk-copies the chunks (already laid out as a
// 128-byte-swizzled operand tile) and TMA-loads the K rows, one thread issues
// the products into a double-buffered TMEM accumulator, and four warps read it
// out, scale it and write the rows.  Each dQ row has one writer and a fixed
// summation order (key tiles in order, 16 keys per product step), so results
// are reproducible bit for bit.
//   warp 0      producer (chunks + K rows, NS-deep ring)
//   warp 1      TMEM allocation; one thread issues every product
//   warps 4-7   output: dQ rows from TMEM, times the score scale
#define JATTN_INLINE_WAITS 1
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.cuh"
#include "kernels.h"

namespace jattn {
using namespace dev;
namespace {

template <int D, int PLANES>
struct DqgCfg {
    static constexpr int BM = 128, BK = 128;
    static constexpr int NKB = D / 64;
    static constexpr uint32_t A_BYTES = PLANES * 2 * kDsChunkBytes;  // [plane][query block 0 | 1]
    static constexpr uint32_t SUB_K = BK * 128;                       // 16 KB: 128 keys x 64 features
    static constexpr uint32_t K_BYTES = BK * D * 2;
    static constexpr uint32_t STAGE = A_BYTES + K_BYTES;
    static constexpr int NS = (3 * STAGE <= 200 * 1024) ? 3 : 2;
    static constexpr uint32_t OFF_BAR = NS * STAGE;
    // full[NS], empty[NS], acc_full[2], acc_empty[2], drain
    static constexpr int NBAR = 2 * NS + 5;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    // per output warp: 32 rows x 64 bf16 staging for row-contiguous stores
    static constexpr int STG_W = 64;
    static constexpr uint32_t OFF_STG = (OFF_MISC + 16 + 127) & ~127u;
    static constexpr uint32_t SMEM = OFF_STG + 4 * 32 * STG_W * 2;
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 2 * D < 32 ? 32 : 2 * D;  // dQ[2]
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(STAGE % 1024 == 0 && A_BYTES % 1024 == 0, "operand alignment");
};

template <int D, int PLANES>
__global__ void __launch_bounds__(256, 1)
    dqg_kernel(const __grid_constant__ CUtensorMap tmK, const BwdArgs a) {
    using C = DqgCfg<D, PLANES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = full + C::NS;
    uint64_t *acc_full = empty + C::NS;   // [2]
    uint64_t *acc_empty = acc_full + 2;   // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    const uint32_t sbase = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&tmK);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const ErrCtx err{g.status, abort_flag, g.wait_ns};
    const int tbeg = g.cta_begin[blockIdx.x];
    const int tend = g.cta_begin[blockIdx.x + 1];

    // a query tile's key tiles, and where its chunks start
    struct Span {
        int nkt;        // key tiles of the sequence
        int64_t c0;     // chunk of (key tile 0, the tile's first 64-query block)
        int nqb;        // 64-query blocks of the sequence (chunk stride between key tiles)
    };
    auto span = [&](const Tile &t) {
        const int lq = g.q_off[t.b + 1] - g.q_off[t.b], lk = g.kv_off[t.b + 1] - g.kv_off[t.b];
        Span s;
        s.nkt = cdiv(lk, C::BK);
        s.nqb = cdiv(lq, 64);
        s.c0 = g.ds_base[t.b] + static_cast<int64_t>(t.h) * s.nkt * s.nqb + t.q_loc0 / 64;
        return s;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------------- producer
            uint32_t it = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, true)) continue;
                const Span sp = span(t);
                const int nblk = t.q_len > 64 ? 2 : 1;  // the tile's 64-query blocks
                const int lk = g.kv_off[t.b + 1] - g.kv_off[t.b];
                for (int kt = 0; kt < sp.nkt; ++kt, ++it) {
                    const uint32_t slot = it % C::NS, use = it / C::NS;
                    if (!(ok = mbar_wait(&empty[slot], (use & 1) ^ 1, err))) break;
                    // only the key rows the products read (a partial last key tile's
                    // rows past round_up16 are never touched)
                    const uint32_t rows = round_up16(min(C::BK, lk - kt * C::BK));
                    const uint32_t cbytes = rows * 128u;
                    mbar_arrive_expect_tx(&full[slot], PLANES * nblk * cbytes + C::K_BYTES);
                    uint8_t *st = smem + slot * C::STAGE;
                    for (int p = 0; p < PLANES; ++p)
                        for (int q = 0; q < nblk; ++q) {
                            const int64_t chunk = sp.c0 + static_cast<int64_t>(kt) * sp.nqb + q;
                            bulk_load(st + (p * 2 + q) * kDsChunkBytes,
                                      static_cast<const uint8_t *>(g.ds) + (chunk * PLANES + p) * kDsChunkBytes,
                                      cbytes, &full[slot]);
                        }
                    for (int kb = 0; kb < C::NKB; ++kb)
                        tma_load_2d(st + C::A_BYTES + kb * C::SUB_K, &tmK, &full[slot], t.h * D + kb * 64,
                                    t.kv_start + kt * C::BK);
                }
            }
            // the last copy into every slot has landed before the CTA leaves
            for (uint32_t s = 0; s < C::NS && s < it; ++s) {
                const uint32_t last = it - 1 - ((it - 1 - s) % C::NS);
                mbar_drain(&full[last % C::NS], (last / C::NS) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------------- MMA issuer
            // dQ (128 queries x D) += dS (128 queries x 16 keys) K (16 keys x D) per
            // step: A is MN-major (rows = keys, 64 queries per 128-byte row, the
            // second 64-query block 16 KB on), B is the K tile MN-major over D.
            const uint32_t idesc = idesc_bf16(128, D, true, true);
            uint32_t it = 0, tn = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                const Span sp = span(t);
                const uint32_t b = tn & 1;
                if (!(ok = mbar_wait(&acc_empty[b], ((tn >> 1) & 1) ^ 1, err))) break;
                const uint32_t dq = tmem + b * D;
                const int lk = g.kv_off[t.b + 1] - g.kv_off[t.b];
                for (int kt = 0; kt < sp.nkt; ++kt, ++it) {
                    const uint32_t slot = it % C::NS, use = it / C::NS;
                    if (!(ok = mbar_wait(&full[slot], use & 1, err))) break;
                    tc_fence_after();
                    const uint32_t st = sbase + slot * C::STAGE;
                    const uint64_t bd0 = sdesc_sw128(st + C::A_BYTES, C::SUB_K, 1024);
                    const int ksteps = (min(C::BK, lk - kt * C::BK) + 15) >> 4;
                    const uint32_t acc0 = kt > 0 ? 1u : 0u;
                    const uint64_t ad0 = sdesc_sw128(st, kDsChunkBytes, 1024);
                    // fully unrolled with a guard per step (constant operand offsets), so
                    // the products issue as fast as the tensor pipe takes them
#pragma unroll
                    for (int k = 0; k < C::BK / 16; ++k) {
                        if (k < ksteps) {
                            const uint32_t acc = k > 0 ? 1u : acc0;
                            const uint64_t bd = sdesc_add(bd0, k * 2048);
#pragma unroll
                            for (int p = 0; p < PLANES; ++p)
                                mma_bf16_ss(dq, sdesc_add(ad0, p * 2 * kDsChunkBytes + k * 2048), bd, idesc, p > 0 ? 1u : acc);
                        }
                    }
                    mma_commit(&empty[slot]);
                }
                if (!ok) break;
                mma_commit(&acc_full[b]);
                ++tn;
            }
            // every MMA this thread issued is done before TMEM is released
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ output
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t stg = sbase + C::OFF_STG + static_cast<uint32_t>(quad) * (32 * C::STG_W * 2);
        const bool staged = !a.dq.f32 && a.dq.cols == D;
        uint32_t tn = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const bool has_keys = g.kv_off[t.b + 1] > g.kv_off[t.b];
            const uint32_t b = tn & 1;
            if (!(ok = mbar_wait_warp(&acc_full[b], (tn >> 1) & 1, err))) break;
            ++tn;
            if (quad * 32 >= t.q_len) {  // no row of this warp is stored
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
                continue;
            }
            tc_fence_after();
            const bool row_ok = row < t.q_len;
            const int64_t qrow = static_cast<int64_t>(t.q_start) + row;
            const uint32_t tq = tmem + lane_base + b * D;
            if (staged) {
                // 32 columns per TMEM round trip, packed to bf16 into the warp's staging
                // rows; each 64-column half then goes out as whole 128-byte row pieces
                constexpr int W = C::STG_W;
                const int nrows = min(32, t.q_len - quad * 32);
                __nv_bfloat16 *dst0 = static_cast<__nv_bfloat16 *>(a.dq.ptr) +
                                      (static_cast<int64_t>(t.q_start) + quad * 32) * a.dq.ld + static_cast<int64_t>(t.h) * D;
#pragma unroll
                for (int col = 0; col < D; col += 32) {
                    float o[32];
                    if (has_keys) {
                        tmem_ld32(tq + col, o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0.0f;
                    }
                    if (col + 32 >= D) {  // every TMEM read of this tile is done
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&acc_empty[b]);
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2) mul2(o[i], o[i + 1], g.scale, g.scale);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
                    stage_row32_bf16<W>(stg, lane, col % W, w);
                    if ((col + 32) % W == 0) {
                        __syncwarp();
                        store_rows_bf16<W>(stg, lane, dst0 + (col + 32 - W), a.dq.ld, nrows);
                        __syncwarp();
                    }
                }
                continue;
            }
#pragma unroll 1
            for (int col = 0; col < D; col += 32) {
                float o[32];
                if (has_keys) {
                    tmem_ld32(tq + col, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.0f;
                }
                if (col + 32 >= D) {  // every TMEM read of this tile is done
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[b]);
                }
                if (row_ok) store_out32(a.dq, qrow, t.h, col, o, g.scale);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, int PLANES>
cudaError_t launch_dqg_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = DqgCfg<D, PLANES>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(dqg_kernel<D, PLANES>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    dqg_kernel<D, PLANES><<<n_ctas, 256, C::SMEM_ALLOC, st>>>(tm.k, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_gemm(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (a.g.ds == nullptr || a.g.ds_base == nullptr) return cudaErrorInvalidValue;
    if (D == 128) return act ? launch_dqg_t<128, 2>(tm, a, n_ctas, st) : launch_dqg_t<128, 1>(tm, a, n_ctas, st);
    if (D == 64) return act ? launch_dqg_t<64, 2>(tm, a, n_ctas, st) : launch_dqg_t<64, 1>(tm, a, n_ctas, st);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
