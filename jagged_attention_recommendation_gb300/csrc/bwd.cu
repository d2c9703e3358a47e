// bwd.cu -- jagged attention backward for sm_103a, full (non-block) attention.
//
// "Training GEM at LLM scale", section "Jagged Sequence Flash Attention",
// backward parallelisation: accumulating dQ across key tiles normally needs
// atomic adds; for recommendation shapes (many batch x head pairs) a
// non-sequence-parallel scheme that computes dQ in a separate pass removes the
// atomics.  Here:
//   pass 1 (dq_kernel, query-major tiles): per 128-row query tile, loop over the
//     sequence's keys in 64-row blocks: S = Q K^T, dP = dO V^T (TMEM),
//     dS = P (dP - Delta) or act'(S) dP, dQ += dS K (TMEM); one writer per dQ row.
//   pass 2 (dkdv_kernel, key-major tiles): per 128-row key tile, loop over the
//     sequence's queries in 64-row blocks: S^T = K Q^T, dP^T = V dO^T,
//     dV += P^T dO, dK += dS^T Q (TMEM); one writer per dK / dV row.
// Softmax mode recomputes P from the forward's lse; Delta_i = <dO_i, O_i> comes
// from a small pre-pass.  Activation mode needs neither; its dS and P reach the
// tensor cores as a bf16 hi + lo pair (reductions over long key or query ranges
// would otherwise lose the tolerance to bf16 rounding).
//
// Both passes share one layout, 16 warps (four warpgroups):
//   warpgroup 0  warp 0: TMA producer of the looped-over blocks (K / V, or
//                Q / dO with lse and Delta); warp 1: TMEM allocation and the
//                thread that issues the accumulating products (dQ, or dV and
//                dK); warp 2: TMA producer of the tile's own rows (Q / dO, or
//                K / V); warp 3: the thread that issues the two score-side
//                products of every block (S and dP, or S^T and dP^T).
//   warpgroups 1, 2  two compute groups; the CTA numbers its blocks n across
//                tile boundaries and group g takes the blocks with n % 2 == g,
//                one thread per tile row (TMEM lane), 32 columns at a time.
//   warpgroup 3  output group: reads the accumulators and writes the rows.
// A block's two products land in its group's TMEM columns; the compute group
// overwrites them in place with bf16 dS (and P^T) and the accumulating product
// reads that operand from TMEM.  Two issuing threads, because any wait of the
// issuing thread (an mbarrier, a shared-memory load, a named barrier) holds it
// until its queued MMAs have drained, which leaves the tensor pipe idle; with
// two, one thread's products run while the other waits.  Block n + 2 reuses
// block n's columns, so the score-side issuer waits for block n's accumulating
// product to finish (an mbarrier committed by the other thread) before it
// issues block n + 2; the accumulators have a single issuer, so their
// summation order is fixed and results are reproducible.
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

// ============================================================================
// pass 1: dQ
// ============================================================================
template <int D, bool ACT, int BIAS>
struct DqCfg {
    static constexpr int BM = 128, BN = 64;
    static constexpr int NKB = D / 64;
    static constexpr int NSK = (D == 64) ? 4 : 3;  // K ring: S, then dQ, read each block
    static constexpr int NSV = (D == 64) ? 3 : 2;  // V ring: dP only
    static constexpr uint32_t SUB_Q = BM * 128;    // 16 KB sub-tile (128 rows x 64 cols)
    static constexpr uint32_t SUB_KV = BN * 128;   // 8 KB sub-tile (64 rows x 64 cols)
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;
    static constexpr uint32_t OFF_Q = 0;  // [2 slots][Q | dO]
    static constexpr uint32_t OFF_K = OFF_Q + 4 * Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NSK * KV_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + NSV * KV_BYTES;
    // qd_full[2], qd_empty[2], k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV],
    // s_full[2], ds_full[2], dq_full[2], dq_empty[2], dq_done[2], drain[2]
    static constexpr int NBAR = 4 + 2 * NSK + 2 * NSV + 8 + 2 + 2;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;
    static constexpr uint32_t OFF_BEXT = OFF_BIAS + (BIAS == kBiasTable ? kMaxBiasFloats * 4 : 0);
    static constexpr uint32_t SMEM = OFF_BEXT + (BIAS == kBiasExt ? kMaxBiasExtFloats * 4 : 0);
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    // group g: S at 128 g, dP at 128 g + 64 (dS over S); dQ[b] at 256 + b D
    static constexpr uint32_t COL_DQ = 256;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "operand alignment");
    static_assert(COL_DQ + 2 * D <= TMEM_COLS, "TMEM budget");
};

// WIN: sliding window on (compile time, so kernels without one carry no band test)
template <int D, bool ACT, int BIAS, bool WIN>
__global__ void __launch_bounds__(512, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const BwdArgs a) {
    using C = DqCfg<D, ACT, BIAS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *qd_full = bars + 0;   // [2]
    uint64_t *qd_empty = bars + 2;  // [2]
    uint64_t *k_full = bars + 4;
    uint64_t *k_empty = k_full + C::NSK;
    uint64_t *v_full = k_empty + C::NSK;
    uint64_t *v_empty = v_full + C::NSV;
    uint64_t *s_full = v_empty + C::NSV;  // [2] per compute group
    uint64_t *ds_full = s_full + 2;       // [2] per compute group
    uint64_t *dq_full = ds_full + 2;      // [2] per dQ buffer
    uint64_t *dq_empty = dq_full + 2;     // [2] per dQ buffer
    uint64_t *dq_done = dq_empty + 2;     // [2] per compute group: its block's dQ product finished
    uint64_t *drain = dq_done + 2;        // [2] per MMA-issuing thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qd_full[s], 1);
            mbar_init(&qd_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&ds_full[s], 4);
            mbar_init(&dq_full[s], 1);
            mbar_init(&dq_empty[s], 4);
            mbar_init(&dq_done[s], 1);
            mbar_init(&drain[s], 1);
        }
        for (int s = 0; s < C::NSK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < C::NSV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (BIAS == kBiasTable) stage_bias(g, sbias, ACT ? 1.0f : kLog2e);
    if (BIAS == kBiasExt) stage_bias_ext(g, sext, ACT ? 1.0f : kLog2e);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const ErrCtx err{g.status, abort_flag};
    const int tbeg = g.cta_begin[blockIdx.x];
    const int tend = g.cta_begin[blockIdx.x + 1];

    const int wgi = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 7, 0);
    if (wgi == 0) {
        regs_release<kRegCtrl>();
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------------- K / V producer
            uint32_t k_it = 0, v_it = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, true)) continue;
                const int nkv = cdiv(t.kv_len, C::BN);
                for (int j = 0; j < nkv; ++j) {
                    const int y = t.kv_start + j * C::BN;
                    const uint32_t ks = k_it % C::NSK, ku = k_it / C::NSK;
                    if (!(ok = mbar_wait(&k_empty[ks], (ku & 1) ^ 1, err))) break;
                    mbar_arrive_expect_tx(&k_full[ks], C::KV_BYTES);
                    for (int kb = 0; kb < C::NKB; ++kb)
                        tma_load_2d(smem + C::OFF_K + ks * C::KV_BYTES + kb * C::SUB_KV, &tmK, &k_full[ks],
                                    t.h * D + kb * 64, y);
                    ++k_it;
                    const uint32_t vs = v_it % C::NSV, vu = v_it / C::NSV;
                    if (!(ok = mbar_wait(&v_empty[vs], (vu & 1) ^ 1, err))) break;
                    mbar_arrive_expect_tx(&v_full[vs], C::KV_BYTES);
                    for (int kb = 0; kb < C::NKB; ++kb)
                        tma_load_2d(smem + C::OFF_V + vs * C::KV_BYTES + kb * C::SUB_KV, &tmV, &v_full[vs],
                                    t.h * D + kb * 64, y);
                    ++v_it;
                }
            }
            if (!ok) {
                for (uint32_t s = 0; s < C::NSK && s < k_it; ++s) {
                    const uint32_t last = k_it - 1 - ((k_it - 1 - s) % C::NSK);
                    mbar_drain(&k_full[last % C::NSK], (last / C::NSK) & 1);
                }
                for (uint32_t s = 0; s < C::NSV && s < v_it; ++s) {
                    const uint32_t last = v_it - 1 - ((v_it - 1 - s) % C::NSV);
                    mbar_drain(&v_full[last % C::NSV], (last / C::NSV) & 1);
                }
            }
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------------------- Q / dO producer
            uint32_t t_local = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                const uint32_t s = t_local & 1, use = t_local >> 1;
                if (!(ok = mbar_wait(&qd_empty[s], (use & 1) ^ 1, err))) break;
                mbar_arrive_expect_tx(&qd_full[s], 2 * C::Q_BYTES);
                uint8_t *base = smem + C::OFF_Q + s * 2 * C::Q_BYTES;
                for (int kb = 0; kb < C::NKB; ++kb) {
                    tma_load_2d(base + kb * C::SUB_Q, &tmQ, &qd_full[s], t.h * D + kb * 64, t.q_start);
                    tma_load_2d(base + C::Q_BYTES + kb * C::SUB_Q, &tmDO, &qd_full[s], t.h * D + kb * 64, t.q_start);
                }
                ++t_local;
            }
            if (!ok) {
                for (uint32_t i = (t_local > 2 ? t_local - 2 : 0); i < t_local; ++i)
                    mbar_drain(&qd_full[i & 1], (i >> 1) & 1);
            }
        } else if (warp == 3 && lane == 0) {
            // -------------------------------------------------------- S / dP issuer
            // Two issuing threads keep the tensor pipe fed (a thread's own waits
            // stall its queued MMAs): this one issues every S = Q K^T and
            // dP = dO V^T, the other every dQ product.  Block n (the CTA's blocks
            // in order, across tiles) reuses the TMEM columns of block n - 2, its
            // compute group's previous block, once that block's dQ product is done.
            bool ok = true;
            TileStream tsa(g, tbeg, tend);
            Tile ta;
            uint32_t ta_n = 0, ns = 0;
            while (ok && tsa.next(ta)) {
                if (!check_tile(g, ta, err, false)) continue;
                const int na = cdiv(ta.kv_len, C::BN);
                const uint32_t qs = ta_n & 1;
                if (!(ok = mbar_wait(&qd_full[qs], (ta_n >> 1) & 1, err))) break;
                const uint32_t qb = sQ + qs * 2 * C::Q_BYTES;
                const uint64_t dq0 = sdesc_sw128(qb, 16, 1024), ddo0 = sdesc_sw128(qb + C::Q_BYTES, 16, 1024);
                for (int ja = 0; ja < na; ++ja, ++ns) {
                    const uint32_t grp = ns & 1;
                    if (ns >= 2 && !(ok = mbar_wait(&dq_done[grp], ((ns - 2) >> 1) & 1, err))) break;
                    const uint32_t ks = ns % C::NSK, vs = ns % C::NSV;
                    if (!(ok = mbar_wait(&k_full[ks], (ns / C::NSK) & 1, err))) break;
                    if (!(ok = mbar_wait(&v_full[vs], (ns / C::NSV) & 1, err))) break;
                    tc_fence_after();
                    const int ncols = round_up16(min(C::BN, ta.kv_len - ja * C::BN));
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint64_t dk0 = sdesc_sw128(sK + ks * C::KV_BYTES, 16, 1024);
                    const uint64_t dv0 = sdesc_sw128(sV + vs * C::KV_BYTES, 16, 1024);
                    const uint32_t dS = tmem + grp * 128, dDP = dS + 64;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t ao = (k >> 2) * C::SUB_Q + (k & 3) * 32;
                        const uint32_t bo = (k >> 2) * C::SUB_KV + (k & 3) * 32;
                        mma_bf16_ss(dS, sdesc_add(dq0, ao), sdesc_add(dk0, bo), idesc, k > 0);
                        mma_bf16_ss(dDP, sdesc_add(ddo0, ao), sdesc_add(dv0, bo), idesc, k > 0);
                    }
                    mma_commit(&s_full[grp]);
                    mma_commit(&v_empty[vs]);  // dP was the V slot's only reader
                }
                if (!ok) break;
                mma_commit(&qd_empty[qs]);  // the last reads of this Q / dO slot are in flight
                ++ta_n;
            }
            // every MMA this thread issued is done before TMEM is released
            mma_commit(&drain[0]);
            mbar_drain(&drain[0], 0);
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- dQ issuer
            // dQ += dS K, dS (bf16; activation: hi and lo parts) read from TMEM, into
            // the tile's dQ buffer (two, so the output group reads one while the
            // next tile accumulates); one thread, so the accumulation order is fixed.
            const uint32_t idesc_dq = idesc_bf16(128, D, false, true);
            bool ok = true;
            TileStream tsb(g, tbeg, tend);
            Tile tb;
            uint32_t tb_n = 0, np = 0;
            while (ok && tsb.next(tb)) {
                if (!check_tile(g, tb, err, false)) continue;
                const int nbk = cdiv(tb.kv_len, C::BN);
                const uint32_t b = tb_n & 1;
                // dQ buffer b must have been read out for tile tb_n - 2
                if (!(ok = mbar_wait(&dq_empty[b], ((tb_n >> 1) & 1) ^ 1, err))) break;
                const uint32_t dq = tmem + C::COL_DQ + b * D;
                for (int jb = 0; jb < nbk; ++jb, ++np) {
                    const uint32_t grp = np & 1;
                    if (!(ok = mbar_wait(&ds_full[grp], (np >> 1) & 1, err))) break;
                    tc_fence_after();
                    const int ksteps = round_up16(min(C::BN, tb.kv_len - jb * C::BN)) / 16;
                    const uint32_t ks = np % C::NSK;
                    const uint64_t bd0 = sdesc_sw128(sK + ks * C::KV_BYTES, C::SUB_KV, 1024);
                    const uint32_t aS = tmem + grp * 128;
                    for (int k = 0; k < ksteps; ++k) {
                        const uint64_t bd = sdesc_add(bd0, k * 2048);
                        const uint32_t acc = (jb > 0 || k > 0) ? 1u : 0u;
                        if (ACT) {  // hi at columns 16 k .. +7, lo at 16 k + 8 .. +15
                            mma_bf16_ts(dq, aS + k * 16, bd, idesc_dq, acc);
                            mma_bf16_ts(dq, aS + k * 16 + 8, bd, idesc_dq, 1u);
                        } else {
                            mma_bf16_ts(dq, aS + k * 8, bd, idesc_dq, acc);
                        }
                    }
                    mma_commit(&k_empty[ks]);     // S and dQ were the K slot's readers
                    mma_commit(&dq_done[grp]);    // the group's columns may take block np + 2
                }
                if (!ok) break;
                mma_commit(&dq_full[b]);
                ++tb_n;
            }
            mma_commit(&drain[1]);
            mbar_drain(&drain[1], 0);
        }
    } else if (wgi < 3) {
        regs_claim<kRegCompute>();
        // ------------------------------------------------------------ compute groups
        // One thread per query row (TMEM lane): dS of the group's key blocks,
        // 32 keys at a time, written as bf16 over the block's S columns
        // (chunk c: columns 16c..16c+15, or 32c..32c+31 as hi / lo pairs).
        const int grp = wgi - 1;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + grp * 128, tDP = tS + 64;
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        uint32_t s_it = 0, n0 = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nkv = cdiv(t.kv_len, C::BN);
            const float *bt = sbias + t.h * g.nb;
            const float *ext_h = sext + t.h * ext_len(g.nb);
            const int q_loc = t.q_loc0 + row;
            const bool row_ok = row < t.q_len;
            const bool warp_live = quad * 32 < t.q_len;  // else its rows reach nothing that is stored
            const int j0 = (grp - static_cast<int>(n0 & 1)) & 1;
            float lse2 = 0.0f, dlt = 0.0f;  // log2 units / Delta of this row
            if (!ACT && row_ok && j0 < nkv) {
                const int64_t idx = static_cast<int64_t>(t.h) * g.Tq + t.q_start + row;
                lse2 = a.lse[idx] * kLog2e;
                dlt = a.delta[idx];
            }
            auto blocks = [&](auto af) {
                constexpr int AF = decltype(af)::value;
                for (int j = j0; j < nkv; j += 2) {
                    if (!(ok = mbar_wait_warp(&s_full[grp], s_it & 1, err))) return;
                    ++s_it;
                    if (warp_live) {
                        tc_fence_after();
                        const int nvalid = min(C::BN, t.kv_len - j * C::BN);
                        const int kvb = t.kv_loc0 + j * C::BN;
#pragma unroll 1
                        for (int c = 0; c < 2 && c * 32 < nvalid; ++c) {
                            float x[32], dp[32];
                            tmem_ld32x2(tS + 32 * c, tDP + 32 * c, x, dp);
                            // x = scale * s + bias (softmax: minus lse, log2 units)
                            scale_bias_off32<BIAS>(x, sc, ACT ? 0.0f : -lse2, ext_h, bt, g.nb, q_loc, kvb + c * 32);
                            if constexpr (ACT) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    float av;
                                    x[i] = act_bwd_t<AF>(x[i], av) * dp[i];
                                }
                            } else {
                                const float nd = -dlt;
#pragma unroll
                                for (int i = 0; i < 32; ++i) x[i] = ex2_approx(x[i]);
#pragma unroll
                                for (int i = 0; i < 32; i += 2) {
                                    add2(dp[i], dp[i + 1], nd, nd);
                                    mul2(x[i], x[i + 1], dp[i], dp[i + 1]);
                                }
                            }
                            if (c * 32 + 32 > nvalid) {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (c * 32 + i >= nvalid) x[i] = 0.0f;
                            }
                            // keys outside the row's window
                            if constexpr (WIN) window_fill32(x, window_bits32(g.window, q_loc, kvb + c * 32), 0.0f);
                            if constexpr (ACT) {
                                uint32_t w[32];
                                pack_hilo32(x, w);
                                tmem_st32_u32(tS + 32 * c, w);
                            } else {
                                uint32_t w[16];
                                pack16(x, w);
                                tmem_st16_u32(tS + 16 * c, w);
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ds_full[grp]);
                }
            };
            if (!ACT || g.act == kSilu) {
                blocks(std::integral_constant<int, kSilu>{});
            } else {
                blocks(std::integral_constant<int, kGeluTanh>{});
            }
            if (!ok) break;
            n0 += nkv;
        }
    } else {
        regs_release<kRegOut>();
        // ------------------------------------------------------------ output
        // One thread per query row: dQ (TMEM, fp32) times the score scale ->
        // the row of dq (each thread stores whole 64-byte pieces of its row).
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t t_local = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nkv = cdiv(t.kv_len, C::BN);
            const uint32_t b = t_local & 1;
            if (!(ok = mbar_wait_warp(&dq_full[b], (t_local >> 1) & 1, err))) break;
            ++t_local;
            if (quad * 32 >= t.q_len) {  // no row of this warp is stored
                __syncwarp();
                if (lane == 0) mbar_arrive(&dq_empty[b]);
                continue;
            }
            tc_fence_after();
            const bool row_ok = row < t.q_len;
            const int64_t qrow = static_cast<int64_t>(t.q_start) + row;
            const uint32_t tq = tmem + lane_base + C::COL_DQ + b * D;
#pragma unroll 1
            for (int col = 0; col < D; col += 32) {
                float o[32];
                if (nkv > 0) {
                    tmem_ld32(tq + col, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.0f;
                }
                if (col + 32 >= D) {  // every TMEM read of this tile is done
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dq_empty[b]);
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

// ============================================================================
// pass 2: dK, dV
// ============================================================================
template <int D, bool ACT, int BIAS>
struct DkvCfg {
    static constexpr int BKV = 128, BQ = 64;
    static constexpr int NKB = D / 64;
    static constexpr int NSQ = (D == 64) ? 6 : 4;   // Q / dO / lse / Delta ring
    static constexpr uint32_t SUB_KV = BKV * 128;  // 16 KB
    static constexpr uint32_t SUB_Q = BQ * 128;    // 8 KB
    static constexpr uint32_t KV_BYTES = BKV * D * 2;
    static constexpr uint32_t Q_BYTES = BQ * D * 2;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = KV_BYTES;
    static constexpr uint32_t OFF_Q = 2 * KV_BYTES;  // [NSQ][Q | dO]
    static constexpr uint32_t OFF_LD = OFF_Q + NSQ * 2 * Q_BYTES;  // [NSQ][-lse log2 e | -Delta][64] floats
    static constexpr uint32_t OFF_BAR = OFF_LD + NSQ * 2 * BQ * 4;
    // kv_full, kv_empty, qs_full[NSQ], qs_empty[NSQ], st_full[2], p_full[2], acc_full, acc_empty,
    // acc_done[2], drain[2]
    static constexpr int NBAR = 2 + 2 * NSQ + 4 + 2 + 2 + 2;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;
    static constexpr uint32_t OFF_BEXT = OFF_BIAS + (BIAS == kBiasTable ? kMaxBiasFloats * 4 : 0);
    // per output warp: 32 rows x 64 bf16 staging for row-contiguous stores
    static constexpr int STG_W = 64;
    static constexpr uint32_t OFF_STG = (OFF_BEXT + (BIAS == kBiasExt ? kMaxBiasExtFloats * 4 : 0) + 127) & ~127u;
    static constexpr uint32_t SMEM = OFF_STG + 4 * 32 * STG_W * 2;
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    // group g: S^T at 128 g (P^T over it), dP^T at 128 g + 64 (dS^T over it); dV, dK
    static constexpr uint32_t COL_DV = 256;
    static constexpr uint32_t COL_DK = 256 + D;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(OFF_Q % 1024 == 0 && Q_BYTES % 1024 == 0, "operand alignment");
    static_assert(OFF_STG % 16 == 0, "16-byte shared-memory vectors");
    static_assert(COL_DK + D <= TMEM_COLS, "TMEM budget");
};

template <int D, bool ACT, int BIAS, bool WIN>
__global__ void __launch_bounds__(512, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const BwdArgs a) {
    using C = DkvCfg<D, ACT, BIAS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *kv_full = bars + 0;
    uint64_t *kv_empty = bars + 1;
    uint64_t *qs_full = bars + 2;
    uint64_t *qs_empty = qs_full + C::NSQ;
    uint64_t *st_full = qs_empty + C::NSQ;  // [2] per compute group
    uint64_t *p_full = st_full + 2;         // [2] per compute group
    uint64_t *acc_full = p_full + 2;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *acc_done = acc_empty + 1;  // [2] per compute group: its block's dV / dK products finished
    uint64_t *drain = acc_done + 2;      // [2] per MMA-issuing thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    float *sLD = reinterpret_cast<float *>(smem + C::OFF_LD);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < C::NSQ; ++s) {
            mbar_init(&qs_full[s], 1);
            mbar_init(&qs_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&st_full[b], 1);
            mbar_init(&p_full[b], 4);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_done[b], 1);
            mbar_init(&drain[b], 1);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (BIAS == kBiasTable) stage_bias(g, sbias, ACT ? 1.0f : kLog2e);
    if (BIAS == kBiasExt) stage_bias_ext(g, sext, ACT ? 1.0f : kLog2e);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmDO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const ErrCtx err{g.status, abort_flag};
    const int tbeg = g.cta_begin[blockIdx.x];
    const int tend = g.cta_begin[blockIdx.x + 1];

    const int wgi = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 7, 0);
    if (wgi == 0) {
        regs_release<kRegCtrl>();
        if (warp == 0) {
            // -------------------------------------------------------- Q / dO producer
            // lane 0 issues the copies; all lanes first write lse / Delta of the
            // block's queries (negated, lse in log2 units) into the stage's slot.
            uint32_t q_it = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, lane == 0)) continue;
                const int nq = cdiv(t.q_len, C::BQ);
                for (int i = 0; i < nq; ++i, ++q_it) {
                    const uint32_t slot = q_it % C::NSQ, use = q_it / C::NSQ;
                    if (!(ok = mbar_wait_warp(&qs_empty[slot], (use & 1) ^ 1, err))) break;
                    if (!ACT) {
                        float *ld = sLD + slot * 2 * C::BQ;
                        for (int k = lane; k < C::BQ; k += 32) {
                            const int qi = i * C::BQ + k;
                            float l2 = 0.0f, dl = 0.0f;
                            if (qi < t.q_len) {
                                const int64_t idx = static_cast<int64_t>(t.h) * g.Tq + t.q_start + qi;
                                l2 = -a.lse[idx] * kLog2e;
                                dl = -a.delta[idx];
                            }
                            ld[k] = l2;
                            ld[C::BQ + k] = dl;
                        }
                        __syncwarp();
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&qs_full[slot], 2 * C::Q_BYTES);
                        const int y = t.q_start + i * C::BQ;
                        uint8_t *base = smem + C::OFF_Q + slot * 2 * C::Q_BYTES;
                        for (int kb = 0; kb < C::NKB; ++kb) {
                            tma_load_2d(base + kb * C::SUB_Q, &tmQ, &qs_full[slot], t.h * D + kb * 64, y);
                            tma_load_2d(base + C::Q_BYTES + kb * C::SUB_Q, &tmDO, &qs_full[slot], t.h * D + kb * 64,
                                        y);
                        }
                    }
                }
            }
            if (!ok && lane == 0) {
                for (uint32_t s = 0; s < C::NSQ && s < q_it; ++s) {
                    const uint32_t last = q_it - 1 - ((q_it - 1 - s) % C::NSQ);
                    mbar_drain(&qs_full[last % C::NSQ], (last / C::NSQ) & 1);
                }
            }
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------------------- K / V producer
            // one buffer: the tile's K and V are last read by its final S^T / dP^T,
            // two blocks before the tile ends, so the next tile's rows load early
            uint32_t t_local = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                if (!(ok = mbar_wait(kv_empty, (t_local & 1) ^ 1, err))) break;
                ++t_local;
                mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
                for (int kb = 0; kb < C::NKB; ++kb) {
                    tma_load_2d(smem + C::OFF_K + kb * C::SUB_KV, &tmK, kv_full, t.h * D + kb * 64, t.kv_start);
                    tma_load_2d(smem + C::OFF_V + kb * C::SUB_KV, &tmV, kv_full, t.h * D + kb * 64, t.kv_start);
                }
            }
            if (!ok && t_local > 0) mbar_drain(kv_full, (t_local - 1) & 1);
        } else if (warp == 3 && lane == 0) {
            // -------------------------------------------------------- S^T / dP^T issuer
            // Two issuing threads keep the tensor pipe fed: a thread's own waits
            // (any shared-memory access) stall its queued MMAs, so this thread
            // issues every S^T = K Q^T and dP^T = V dO^T and the other every
            // dV / dK product.  Block n (the CTA's blocks in order, across tiles)
            // reuses the TMEM columns of block n - 2, its compute group's previous
            // block, once that block's dV / dK products have finished.
            bool ok = true;
            TileStream tsa(g, tbeg, tend);
            Tile ta;
            uint32_t ta_n = 0, ns = 0;
            const uint64_t dk0 = sdesc_sw128(sK, 16, 1024), dv0 = sdesc_sw128(sV, 16, 1024);
            while (ok && tsa.next(ta)) {
                if (!check_tile(g, ta, err, false)) continue;
                const int na = cdiv(ta.q_len, C::BQ);
                if (!(ok = mbar_wait(kv_full, ta_n & 1, err))) break;
                for (int ia = 0; ia < na; ++ia, ++ns) {
                    const uint32_t grp = ns & 1;
                    if (ns >= 2 && !(ok = mbar_wait(&acc_done[grp], ((ns - 2) >> 1) & 1, err))) break;
                    const uint32_t slot = ns % C::NSQ;
                    if (!(ok = mbar_wait(&qs_full[slot], (ns / C::NSQ) & 1, err))) break;
                    tc_fence_after();
                    const int ncols = round_up16(min(C::BQ, ta.q_len - ia * C::BQ));
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint32_t qb = sQ + slot * 2 * C::Q_BYTES;
                    const uint64_t dqq = sdesc_sw128(qb, 16, 1024), ddo = sdesc_sw128(qb + C::Q_BYTES, 16, 1024);
                    const uint32_t dS = tmem + grp * 128, dDP = dS + 64;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t ao = (k >> 2) * C::SUB_KV + (k & 3) * 32;
                        const uint32_t bo = (k >> 2) * C::SUB_Q + (k & 3) * 32;
                        mma_bf16_ss(dS, sdesc_add(dk0, ao), sdesc_add(dqq, bo), idesc, k > 0);
                        mma_bf16_ss(dDP, sdesc_add(dv0, ao), sdesc_add(ddo, bo), idesc, k > 0);
                    }
                    mma_commit(&st_full[grp]);
                }
                if (!ok) break;
                mma_commit(kv_empty);  // the tile's last reads of K and V are in flight
                ++ta_n;
            }
            // every MMA this thread issued is done before TMEM is released
            mma_commit(&drain[0]);
            mbar_drain(&drain[0], 0);
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- dV / dK issuer
            // dV += P^T dO and dK += dS^T Q, P^T and dS^T (bf16; activation: hi and
            // lo parts) read from TMEM; one thread, so the accumulation order is fixed.
            const uint32_t idesc_acc = idesc_bf16(128, D, false, true);
            bool ok = true;
            TileStream tsb(g, tbeg, tend);
            Tile tb;
            uint32_t tb_n = 0, np = 0;
            while (ok && tsb.next(tb)) {
                if (!check_tile(g, tb, err, false)) continue;
                const int nbq = cdiv(tb.q_len, C::BQ);
                // the output group must have read dV / dK of the previous tile
                if (!(ok = mbar_wait(acc_empty, (tb_n & 1) ^ 1, err))) break;
                for (int ib = 0; ib < nbq; ++ib, ++np) {
                    const uint32_t grp = np & 1;
                    if (!(ok = mbar_wait(&p_full[grp], (np >> 1) & 1, err))) break;
                    tc_fence_after();
                    const int ksteps = round_up16(min(C::BQ, tb.q_len - ib * C::BQ)) / 16;
                    const uint32_t slot = np % C::NSQ;
                    const uint32_t qb = sQ + slot * 2 * C::Q_BYTES;
                    const uint64_t bq0 = sdesc_sw128(qb, C::SUB_Q, 1024);
                    const uint64_t bdo0 = sdesc_sw128(qb + C::Q_BYTES, C::SUB_Q, 1024);
                    const uint32_t aP = tmem + grp * 128, aDS = aP + 64;
                    for (int k = 0; k < ksteps; ++k) {
                        const uint32_t acc = (ib > 0 || k > 0) ? 1u : 0u;
                        const uint64_t bdo = sdesc_add(bdo0, k * 2048);
                        const uint64_t bq = sdesc_add(bq0, k * 2048);
                        if (ACT) {  // hi at columns 16 k .. +7, lo at 16 k + 8 .. +15
                            mma_bf16_ts(tmem + C::COL_DV, aP + k * 16, bdo, idesc_acc, acc);
                            mma_bf16_ts(tmem + C::COL_DV, aP + k * 16 + 8, bdo, idesc_acc, 1u);
                            mma_bf16_ts(tmem + C::COL_DK, aDS + k * 16, bq, idesc_acc, acc);
                            mma_bf16_ts(tmem + C::COL_DK, aDS + k * 16 + 8, bq, idesc_acc, 1u);
                        } else {
                            mma_bf16_ts(tmem + C::COL_DV, aP + k * 8, bdo, idesc_acc, acc);
                            mma_bf16_ts(tmem + C::COL_DK, aDS + k * 8, bq, idesc_acc, acc);
                        }
                    }
                    mma_commit(&qs_empty[slot]);  // last reads of the Q / dO slot
                    mma_commit(&acc_done[grp]);   // the group's columns may take block np + 2
                }
                if (!ok) break;
                mma_commit(acc_full);
                ++tb_n;
            }
            mma_commit(&drain[1]);
            mbar_drain(&drain[1], 0);
        }
    } else if (wgi < 3) {
        regs_claim<kRegCompute>();
        // ------------------------------------------------------------ compute groups
        // One thread per key row (TMEM lane): P^T and dS^T of the group's query
        // blocks, 32 queries at a time, written as bf16 over the block's S^T and
        // dP^T columns (chunk c: columns 16c..16c+15, or 32c..32c+31 as hi / lo).
        const int grp = wgi - 1;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + grp * 128, tDP = tS + 64;
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        uint32_t s_it = 0, n0 = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nq = cdiv(t.q_len, C::BQ);
            const float *bt = sbias + t.h * g.nb;
            const float *ext_h = sext + t.h * ext_len(g.nb);
            const int kv_loc = t.kv_loc0 + row;
            const bool warp_live = quad * 32 < t.kv_len;
            const int i0 = (grp - static_cast<int>(n0 & 1)) & 1;
            auto blocks = [&](auto af) {
                constexpr int AF = decltype(af)::value;
                for (int i = i0; i < nq; i += 2) {
                    if (!(ok = mbar_wait_warp(&st_full[grp], s_it & 1, err))) return;
                    ++s_it;
                    if (warp_live) {
                        tc_fence_after();
                        const int nvalid = min(C::BQ, t.q_len - i * C::BQ);
                        const int qb = t.q_loc0 + i * C::BQ;
                        // [-lse log2 e | -Delta] of the block's queries (shared by all rows)
                        const float *ld = sLD + ((n0 + i) % C::NSQ) * 2 * C::BQ;
#pragma unroll 1
                        for (int c = 0; c < 2 && c * 32 < nvalid; ++c) {
                            float x[32], dp[32];
                            tmem_ld32x2(tS + 32 * c, tDP + 32 * c, x, dp);
                            scale_bias_off32<BIAS>(x, sc, 0.0f, ext_h, bt, g.nb, kv_loc, qb + c * 32);
                            if constexpr (ACT) {
#pragma unroll
                                for (int k = 0; k < 32; ++k) {
                                    float pv;
                                    dp[k] = act_bwd_t<AF>(x[k], pv) * dp[k];
                                    x[k] = pv;
                                }
                            } else {
                                const float4 *l4 = reinterpret_cast<const float4 *>(ld + c * 32);
                                const float4 *d4 = reinterpret_cast<const float4 *>(ld + C::BQ + c * 32);
#pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    const float4 lz = l4[k], dz = d4[k];
                                    add2(x[4 * k], x[4 * k + 1], lz.x, lz.y);
                                    add2(x[4 * k + 2], x[4 * k + 3], lz.z, lz.w);
                                    add2(dp[4 * k], dp[4 * k + 1], dz.x, dz.y);
                                    add2(dp[4 * k + 2], dp[4 * k + 3], dz.z, dz.w);
                                }
#pragma unroll
                                for (int k = 0; k < 32; ++k) x[k] = ex2_approx(x[k]);
#pragma unroll
                                for (int k = 0; k < 32; k += 2) mul2(dp[k], dp[k + 1], x[k], x[k + 1]);
                            }
                            if (c * 32 + 32 > nvalid) {
#pragma unroll
                                for (int k = 0; k < 32; ++k)
                                    if (c * 32 + k >= nvalid) {
                                        x[k] = 0.0f;
                                        dp[k] = 0.0f;
                                    }
                            }
                            if constexpr (WIN) {  // queries whose window does not reach this key
                                const uint32_t wb = window_bits32(g.window, kv_loc, qb + c * 32);
                                window_fill32(x, wb, 0.0f);
                                window_fill32(dp, wb, 0.0f);
                            }
                            if constexpr (ACT) {
                                uint32_t w[32];
                                pack_hilo32(x, w);
                                tmem_st32_u32(tS + 32 * c, w);
                                pack_hilo32(dp, w);
                                tmem_st32_u32(tDP + 32 * c, w);
                            } else {
                                uint32_t w[16];
                                pack16(x, w);
                                tmem_st16_u32(tS + 16 * c, w);
                                pack16(dp, w);
                                tmem_st16_u32(tDP + 16 * c, w);
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[grp]);
                }
            };
            if (!ACT || g.act == kSilu) {
                blocks(std::integral_constant<int, kSilu>{});
            } else {
                blocks(std::integral_constant<int, kGeluTanh>{});
            }
            if (!ok) break;
            n0 += nq;
        }
    } else {
        regs_release<kRegOut>();
        // ------------------------------------------------------------ output
        // One thread per key row reads dV and dK (times the score scale) from
        // TMEM.  bf16 outputs go out row-contiguous through the warp's staging
        // buffer: dV is staged and dK packed into registers before the
        // accumulators are handed back, so the next tile's products wait only
        // for the TMEM reads, not for the stores.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tDV = tmem + lane_base + C::COL_DV, tDK = tmem + lane_base + C::COL_DK;
        constexpr int W = C::STG_W;
        const uint32_t stg = smem_u32(smem + C::OFF_STG) + static_cast<uint32_t>(quad) * (32 * W * 2);
        const bool staged = !a.dv.f32 && !a.dk.f32 && a.dv.cols == D && a.dk.cols == D;
        uint32_t t_local = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nq = cdiv(t.q_len, C::BQ);
            if (!(ok = mbar_wait_warp(acc_full, t_local & 1, err))) break;
            ++t_local;
            if (quad * 32 >= t.kv_len) {  // no row of this warp is stored
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
                continue;
            }
            tc_fence_after();
            if (staged) {
                const int nrows = min(32, t.kv_len - quad * 32);
                const int64_t r0 = static_cast<int64_t>(t.kv_start) + quad * 32;
                __nv_bfloat16 *dv0 = static_cast<__nv_bfloat16 *>(a.dv.ptr) + r0 * a.dv.ld + t.h * D;
                __nv_bfloat16 *dk0 = static_cast<__nv_bfloat16 *>(a.dk.ptr) + r0 * a.dk.ld + t.h * D;
                // dV: W columns at a time through the staging buffer
#pragma unroll
                for (int h0 = 0; h0 < D; h0 += W) {
#pragma unroll
                    for (int c = 0; c < W / 32; ++c) {
                        float v[32];
                        uint32_t w[16];
                        if (nq > 0) {
                            tmem_ld32(tDV + h0 + 32 * c, v);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                        }
                        pack16(v, w);
                        stage_row32_bf16<W>(stg, lane, 32 * c, w);
                    }
                    __syncwarp();
                    store_rows_bf16<W>(stg, lane, dv0 + h0, a.dv.ld, nrows);
                    __syncwarp();
                }
                // dK (times the score scale) packed into registers
                uint32_t kw[D / 32][16];
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    if (nq > 0) {
                        tmem_ld32(tDK + 32 * c, v);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                    }
#pragma unroll
                    for (int i = 0; i < 32; i += 2) mul2(v[i], v[i + 1], g.scale, g.scale);
                    pack16(v, kw[c]);
                }
                // every TMEM read of this tile is done
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
#pragma unroll
                for (int h0 = 0; h0 < D; h0 += W) {
#pragma unroll
                    for (int c = 0; c < W / 32; ++c) stage_row32_bf16<W>(stg, lane, 32 * c, kw[h0 / 32 + c]);
                    __syncwarp();
                    store_rows_bf16<W>(stg, lane, dk0 + h0, a.dk.ld, nrows);
                    __syncwarp();
                }
                continue;
            }
            const bool row_ok = row < t.kv_len;
            const int64_t krow = static_cast<int64_t>(t.kv_start) + row;
#pragma unroll 1
            for (int col = 0; col < D; col += 32) {
                float ov[32], ok_[32];
                if (nq > 0) {
                    tmem_ld32x2(tDV + col, tDK + col, ov, ok_);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = ok_[i] = 0.0f;
                }
                if (col + 32 >= D) {  // every TMEM read of this tile is done
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty);
                }
                if (row_ok) {
                    store_out32(a.dv, krow, t.h, col, ov, 1.0f);
                    store_out32(a.dk, krow, t.h, col, ok_, g.scale);
                }
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

// ============================================================================
// launchers
// ============================================================================
template <int D, bool ACT, int BIAS, bool WIN>
static cudaError_t launch_dq_w(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = DqCfg<D, ACT, BIAS>;
    static bool done[64] = {};
    cudaError_t e = ensure_smem(dq_kernel<D, ACT, BIAS, WIN>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    dq_kernel<D, ACT, BIAS, WIN><<<n_ctas, 512, C::SMEM_ALLOC, st>>>(tm.q, tm.k, tm.v, tm.dout, a);
    return cudaGetLastError();
}

template <int D, bool ACT, int BIAS, bool WIN>
static cudaError_t launch_dkdv_w(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = DkvCfg<D, ACT, BIAS>;
    static bool done[64] = {};
    cudaError_t e = ensure_smem(dkdv_kernel<D, ACT, BIAS, WIN>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    dkdv_kernel<D, ACT, BIAS, WIN><<<n_ctas, 512, C::SMEM_ALLOC, st>>>(tm.q, tm.k, tm.v, tm.dout, a);
    return cudaGetLastError();
}

template <int D, bool ACT, int BIAS>
static cudaError_t launch_dq_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    return a.g.window > 0 ? launch_dq_w<D, ACT, BIAS, true>(tm, a, n_ctas, st)
                          : launch_dq_w<D, ACT, BIAS, false>(tm, a, n_ctas, st);
}

template <int D, bool ACT, int BIAS>
static cudaError_t launch_dkdv_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    return a.g.window > 0 ? launch_dkdv_w<D, ACT, BIAS, true>(tm, a, n_ctas, st)
                          : launch_dkdv_w<D, ACT, BIAS, false>(tm, a, n_ctas, st);
}

static int bias_form(const Geom &g) {
    if (g.nb <= 0) return kBiasNone;
    return g.H * ext_len(g.nb) <= kMaxBiasExtFloats ? kBiasExt : kBiasTable;
}

template <int D, bool ACT>
static cudaError_t launch_dq_b(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    switch (bias_form(a.g)) {
    case kBiasNone: return launch_dq_t<D, ACT, kBiasNone>(tm, a, n_ctas, st);
    case kBiasExt: return launch_dq_t<D, ACT, kBiasExt>(tm, a, n_ctas, st);
    default: return launch_dq_t<D, ACT, kBiasTable>(tm, a, n_ctas, st);
    }
}

template <int D, bool ACT>
static cudaError_t launch_dkdv_b(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    switch (bias_form(a.g)) {
    case kBiasNone: return launch_dkdv_t<D, ACT, kBiasNone>(tm, a, n_ctas, st);
    case kBiasExt: return launch_dkdv_t<D, ACT, kBiasExt>(tm, a, n_ctas, st);
    default: return launch_dkdv_t<D, ACT, kBiasTable>(tm, a, n_ctas, st);
    }
}

cudaError_t launch_bwd_dq(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (D == 128) return act ? launch_dq_b<128, true>(tm, a, n_ctas, st) : launch_dq_b<128, false>(tm, a, n_ctas, st);
    if (D == 64) return act ? launch_dq_b<64, true>(tm, a, n_ctas, st) : launch_dq_b<64, false>(tm, a, n_ctas, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dkdv(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (D == 128)
        return act ? launch_dkdv_b<128, true>(tm, a, n_ctas, st) : launch_dkdv_b<128, false>(tm, a, n_ctas, st);
    if (D == 64) return act ? launch_dkdv_b<64, true>(tm, a, n_ctas, st) : launch_dkdv_b<64, false>(tm, a, n_ctas, st);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
