// bwd.cu -- jagged attention backward for sm_103a, full (non-block) attention.
//
// "Training GEM at LLM scale", section "Jagged Sequence Flash Attention",
// backward parallelisation: accumulating dQ across key tiles normally needs
// atomic adds; for recommendation shapes (many batch x head pairs) a
// non-sequence-parallel scheme that computes dQ in a separate pass removes both
// the atomics and the redundant recompute.  Here:
//   pass 1 (dq_kernel, query-major tiles): per 128-row query tile, loop over the
//     sequence's keys in 64-row blocks: S = Q K^T, dP = dO V^T (TMEM),
//     dS = P (dP - Delta) or act'(S) dP, dQ += dS K (TMEM); one writer per dQ row.
//   pass 2 (dkdv_kernel, key-major tiles): per 128-row key tile, loop over the
//     sequence's queries in 64-row blocks: S^T = K Q^T, dP^T = V dO^T,
//     dV += P^T dO, dK += dS^T Q (TMEM); one writer per dK / dV row.
// Softmax mode recomputes P from the forward's lse; Delta_i = <dO_i, O_i> is
// computed by a small pre-pass.  Activation mode needs neither; its dS and P
// reach the tensor cores as a bf16 hi + lo pair (reductions over long key or
// query ranges would otherwise lose the tolerance to bf16 rounding).
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.cuh"
#include "kernels.h"

namespace jattn {
using namespace dev;

// ============================================================================
// pass 1: dQ
// ============================================================================
template <int D, bool ACT>
struct DqCfg {
    static constexpr int BM = 128, BN = 64;
    static constexpr int NKB = D / 64;
    static constexpr int NST = 3;
    static constexpr uint32_t SUB_Q = BM * 128;  // 16 KB sub-tile (128 rows x 64 cols)
    static constexpr uint32_t SUB_KV = BN * 128; // 8 KB sub-tile (64 rows x 64 cols)
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;
    static constexpr uint32_t DS_BYTES = BM * BN * 2;  // one 16 KB sub-tile
    static constexpr int NDS = ACT ? 2 : 1;            // hi (+ lo) planes
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_DO = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_K = OFF_DO + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NST * KV_BYTES;
    static constexpr uint32_t OFF_DS = OFF_V + NST * KV_BYTES;  // [2 buffers][NDS planes]
    static constexpr uint32_t OFF_BAR = OFF_DS + 2 * NDS * DS_BYTES;
    // qd_full, qd_empty, kv_full[NST], kv_empty[NST], s_full[2], s_empty[2], ds_full[2], ds_empty[2],
    // dq_full, dq_empty, drain
    static constexpr int NBAR = 2 + 2 * NST + 8 + 3;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;
    static constexpr uint32_t OFF_BEXT = OFF_BIAS + kMaxBiasFloats * 4;
    static constexpr uint32_t SMEM = OFF_BEXT + (ACT ? 0 : kMaxBiasExtFloats * 4);
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0;     // S[2]:  0, 64
    static constexpr uint32_t COL_DP = 128;  // dP[2]: 128, 192
    static constexpr uint32_t COL_DQ = 256;  // dQ: D columns
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

template <int D, bool ACT>
__global__ void __launch_bounds__(192, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const BwdArgs a) {
    using C = DqCfg<D, ACT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *qd_full = bars + 0;
    uint64_t *qd_empty = bars + 1;
    uint64_t *kv_full = bars + 2;
    uint64_t *kv_empty = kv_full + C::NST;
    uint64_t *s_full = kv_empty + C::NST;
    uint64_t *s_empty = s_full + 2;
    uint64_t *ds_full = s_empty + 2;
    uint64_t *ds_empty = ds_full + 2;
    uint64_t *dq_full = ds_empty + 2;
    uint64_t *dq_empty = dq_full + 1;
    uint64_t *drain = dq_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    const bool use_ext = !ACT && g.nb > 0 && g.H * ext_len(g.nb) <= kMaxBiasExtFloats;
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sDO = smem_u32(smem + C::OFF_DO);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);
    const uint32_t sDS = smem_u32(smem + C::OFF_DS);

    if (threadIdx.x == 0) {
        mbar_init(qd_full, 1);
        mbar_init(qd_empty, 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], 4);
            mbar_init(&ds_full[b], 4);
            mbar_init(&ds_empty[b], 1);
        }
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    stage_bias(g, sbias, ACT ? 1.0f : kLog2e);
    if (use_ext) stage_bias_ext(g, sext, kLog2e);
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

    if (warp == 0) {
        if (lane == 0) {
            uint32_t kv_it = 0, t_local = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, true)) continue;
                if (!(ok = mbar_wait(qd_empty, (t_local & 1) ^ 1, err))) break;
                ++t_local;
                mbar_arrive_expect_tx(qd_full, 2 * C::Q_BYTES);
                for (int kb = 0; kb < C::NKB; ++kb) {
                    tma_load_2d(smem + C::OFF_Q + kb * C::SUB_Q, &tmQ, qd_full, t.h * D + kb * 64, t.q_start);
                    tma_load_2d(smem + C::OFF_DO + kb * C::SUB_Q, &tmDO, qd_full, t.h * D + kb * 64, t.q_start);
                }
                const int nkv = cdiv(t.kv_len, C::BN);
                for (int j = 0; j < nkv; ++j, ++kv_it) {
                    const uint32_t slot = kv_it % C::NST, use = kv_it / C::NST;
                    if (!(ok = mbar_wait(&kv_empty[slot], (use & 1) ^ 1, err))) break;
                    mbar_arrive_expect_tx(&kv_full[slot], 2 * C::KV_BYTES);
                    const int y = t.kv_start + j * C::BN;
                    for (int kb = 0; kb < C::NKB; ++kb) {
                        tma_load_2d(smem + C::OFF_K + slot * C::KV_BYTES + kb * C::SUB_KV, &tmK, &kv_full[slot],
                                    t.h * D + kb * 64, y);
                        tma_load_2d(smem + C::OFF_V + slot * C::KV_BYTES + kb * C::SUB_KV, &tmV, &kv_full[slot],
                                    t.h * D + kb * 64, y);
                    }
                }
            }
            if (!ok) {
                if (t_local > 0) mbar_drain(qd_full, (t_local - 1) & 1);
                for (uint32_t s = 0; s < C::NST && s < kv_it; ++s) {
                    const uint32_t last = kv_it - 1 - ((kv_it - 1 - s) % C::NST);
                    mbar_drain(&kv_full[last % C::NST], (last / C::NST) & 1);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t kv_it = 0, s_it = 0, ds_it = 0, t_local = 0;
            const uint32_t idesc_dq = idesc_bf16(128, D, false, true);
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                const int nkv = cdiv(t.kv_len, C::BN);
                if (!(ok = mbar_wait(qd_full, t_local & 1, err))) break;
                if (!(ok = mbar_wait(dq_empty, (t_local & 1) ^ 1, err))) break;
                tc_fence_after();

                auto issue_sdp = [&](int j) -> bool {
                    const uint32_t it = kv_it + j, slot = it % C::NST, use = it / C::NST;
                    if (!mbar_wait(&kv_full[slot], use & 1, err)) return false;
                    const uint32_t sb = s_it & 1, suse = s_it >> 1;
                    if (!mbar_wait(&s_empty[sb], (suse & 1) ^ 1, err)) return false;
                    tc_fence_after();
                    const int ncols = round_up16(min(C::BN, t.kv_len - j * C::BN));
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint32_t kb = sK + slot * C::KV_BYTES, vb = sV + slot * C::KV_BYTES;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ao = (ks >> 2) * C::SUB_Q + (ks & 3) * 32;
                        const uint32_t bo = (ks >> 2) * C::SUB_KV + (ks & 3) * 32;
                        mma_bf16_ss(tmem + C::COL_S + sb * C::BN, sdesc_sw128(sQ + ao, 16, 1024),
                                    sdesc_sw128(kb + bo, 16, 1024), idesc, ks > 0);
                        mma_bf16_ss(tmem + C::COL_DP + sb * C::BN, sdesc_sw128(sDO + ao, 16, 1024),
                                    sdesc_sw128(vb + bo, 16, 1024), idesc, ks > 0);
                    }
                    mma_commit(&s_full[sb]);
                    ++s_it;
                    return true;
                };

                if (nkv > 0) ok = issue_sdp(0);
                for (int j = 0; ok && j < nkv; ++j) {
                    if (j + 1 < nkv) {
                        if (!(ok = issue_sdp(j + 1))) break;
                    } else {
                        mma_commit(qd_empty);
                    }
                    const uint32_t db = ds_it & 1, duse = ds_it >> 1;
                    if (!(ok = mbar_wait(&ds_full[db], duse & 1, err))) break;
                    tc_fence_after();
                    const uint32_t slot = (kv_it + j) % C::NST;
                    const int ksteps = round_up16(min(C::BN, t.kv_len - j * C::BN)) / 16;
                    const uint32_t kb = sK + slot * C::KV_BYTES;
                    const uint32_t dsb = sDS + db * C::NDS * C::DS_BYTES;
                    for (int ks = 0; ks < ksteps; ++ks) {
                        const uint64_t bd = sdesc_sw128(kb + ks * 2048, C::SUB_KV, 1024);
                        mma_bf16_ss(tmem + C::COL_DQ, sdesc_sw128(dsb + ks * 32, 16, 1024), bd, idesc_dq,
                                    (j > 0 || ks > 0) ? 1u : 0u);
                        if (ACT)
                            mma_bf16_ss(tmem + C::COL_DQ, sdesc_sw128(dsb + C::DS_BYTES + ks * 32, 16, 1024), bd,
                                        idesc_dq, 1u);
                    }
                    mma_commit(&kv_empty[slot]);
                    mma_commit(&ds_empty[db]);
                    ++ds_it;
                }
                if (!ok) break;
                if (nkv == 0) mma_commit(qd_empty);
                mma_commit(dq_full);
                kv_it += nkv;
                ++t_local;
            }
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        uint32_t s_it = 0, ds_it = 0, t_local = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nkv = cdiv(t.kv_len, C::BN);
            const float *bt = sbias + t.h * g.nb;
            const float *ext_h = sext + t.h * ext_len(g.nb);
            const int q_loc = t.q_loc0 + row;
            const int kv_loc0 = t.kv_loc0;
            const bool row_ok = row < t.q_len;
            const int64_t qrow = static_cast<int64_t>(t.q_start) + row;
            float lse2 = 0.0f, dlt = 0.0f;
            if (!ACT && row_ok) {
                lse2 = a.lse[static_cast<int64_t>(t.h) * g.Tq + qrow] * kLog2e;
                dlt = a.delta[static_cast<int64_t>(t.h) * g.Tq + qrow];
            }
            for (int j = 0; j < nkv; ++j) {
                const uint32_t sb = s_it & 1, suse = s_it >> 1;
                if (!(ok = mbar_wait_warp(&s_full[sb], suse & 1, err))) break;
                tc_fence_after();
                const int nvalid = min(C::BN, t.kv_len - j * C::BN);
                const int ncols = round_up16(nvalid);
                float s[C::BN], dp[C::BN];
                bool live[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) live[c] = c * 32 < nvalid;
                tmem_ld64x2(tmem + lane_base + C::COL_S + sb * C::BN, tmem + lane_base + C::COL_DP + sb * C::BN, s,
                            dp);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                ++s_it;

                const int kvb = kv_loc0 + j * C::BN;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (!live[c]) continue;
                    float(&xs)[32] = sub32(s, c);
                    float(&dpc)[32] = sub32(dp, c);
                    // x = scale * s + bias (softmax: minus lse, in log2 units)
                    const float off = ACT ? 0.0f : -lse2;
                    float bv[32], cst = 0.0f;
                    bool band = false;
                    if (g.nb > 0) {
                        if (use_ext) {
                            band = bias32_ext(ext_h, g.nb, q_loc, kvb + c * 32, bv, cst);
                        } else {
                            bias32(bt, g.nb, q_loc, kvb + c * 32, bv);
                            band = true;
                        }
                    }
                    if (band) {
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            add2(bv[i], bv[i + 1], off, off);
                            fma2(xs[i], xs[i + 1], sc, sc, bv[i], bv[i + 1]);
                        }
                    } else {
                        const float o2 = cst + off;
#pragma unroll
                        for (int i = 0; i < 32; i += 2) fma2(xs[i], xs[i + 1], sc, sc, o2, o2);
                    }
                    if (ACT) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            float av;
                            xs[i] = act_bwd(g.act, xs[i], av) * dpc[i];
                        }
                    } else {
                        const float nd = -dlt;
#pragma unroll
                        for (int i = 0; i < 32; ++i) xs[i] = ex2_approx(xs[i]);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            add2(dpc[i], dpc[i + 1], nd, nd);
                            mul2(xs[i], xs[i + 1], dpc[i], dpc[i + 1]);
                        }
                    }
                    if (c * 32 + 32 > nvalid) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c * 32 + i >= nvalid) xs[i] = 0.0f;
                    }
                }
                const uint32_t db = ds_it & 1, duse = ds_it >> 1;
                if (!(ok = mbar_wait_warp(&ds_empty[db], (duse & 1) ^ 1, err))) break;
                const uint32_t dsb = sDS + db * C::NDS * C::DS_BYTES;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (c * 32 >= ncols) continue;
                    if (!live[c]) {
                        st_row32_zero(dsb, C::DS_BYTES, row, c * 32);
                        if (ACT) st_row32_zero(dsb + C::DS_BYTES, C::DS_BYTES, row, c * 32);
                    } else if (ACT) {
                        st_row32_bf16_hilo(dsb, dsb + C::DS_BYTES, C::DS_BYTES, row, c * 32, sub32(s, c));
                    } else {
                        st_row32_bf16(dsb, C::DS_BYTES, row, c * 32, sub32(s, c));
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ds_full[db]);
                ++ds_it;
            }
            if (!ok) break;
            if (!(ok = mbar_wait_warp(dq_full, t_local & 1, err))) break;
            tc_fence_after();
            const bool fast = rows_fast<D>(a.dq);
            float oa[D];
            if (nkv > 0) {
                tmem_ld_row<D>(tmem + lane_base + C::COL_DQ, oa);
            } else {
#pragma unroll
                for (int i = 0; i < D; ++i) oa[i] = 0.0f;
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float(&o)[32] = sub32(oa, c);
                if (fast) {
                    // stage in this warp's rows of the two dS buffers (every dQ MMA is done)
#pragma unroll
                    for (int i = 0; i < 32; i += 2) mul2(o[i], o[i + 1], g.scale, g.scale);
                    st_row32_bf16(sDS, C::NDS * C::DS_BYTES, row, c * 32, o);
                } else if (row_ok) {
                    store_out32(a.dq, qrow, t.h, c * 32, o, g.scale);
                }
            }
            if (fast) {
                __syncwarp();
                copy_rows_out<D>(sDS, C::NDS * C::DS_BYTES, quad * 32, t.q_len, a.dq, t.q_start, t.h, lane);
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dq_empty);
            ++t_local;
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
template <int D, bool ACT>
struct DkvCfg {
    static constexpr int BKV = 128, BQ = 64;
    static constexpr int NKB = D / 64;
    static constexpr int NST = (ACT && D == 128) ? 2 : 3;
    static constexpr uint32_t SUB_KV = BKV * 128;  // 16 KB
    static constexpr uint32_t SUB_Q = BQ * 128;    // 8 KB
    static constexpr uint32_t KV_BYTES = BKV * D * 2;
    static constexpr uint32_t Q_BYTES = BQ * D * 2;
    static constexpr uint32_t PT_BYTES = BKV * BQ * 2;  // 16 KB
    static constexpr int NPL = ACT ? 2 : 1;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = KV_BYTES;
    static constexpr uint32_t OFF_Q = 2 * KV_BYTES;
    static constexpr uint32_t OFF_DO = OFF_Q + NST * Q_BYTES;
    static constexpr uint32_t OFF_PT = OFF_DO + NST * Q_BYTES;    // P^T planes
    static constexpr uint32_t OFF_DST = OFF_PT + NPL * PT_BYTES;  // dS^T planes
    static constexpr uint32_t OFF_LD = OFF_DST + NPL * PT_BYTES;  // [NST][lse | delta][64] floats
    static constexpr uint32_t OFF_BAR = OFF_LD + NST * 2 * BQ * 4;
    // kv_full, kv_empty, qs_full[NST], qs_empty[NST], st_full[2], st_empty[2], p_full, p_empty,
    // acc_full, acc_empty, drain
    static constexpr int NBAR = 2 + 2 * NST + 4 + 2 + 2 + 1;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;
    static constexpr uint32_t OFF_BEXT = OFF_BIAS + kMaxBiasFloats * 4;
    static constexpr uint32_t SMEM = OFF_BEXT + (ACT ? 0 : kMaxBiasExtFloats * 4);
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_ST = 0;
    static constexpr uint32_t COL_DPT = 128;
    static constexpr uint32_t COL_DV = 256;
    static constexpr uint32_t COL_DK = 256 + D;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

template <int D, bool ACT>
__global__ void __launch_bounds__(192, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const BwdArgs a) {
    using C = DkvCfg<D, ACT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *kv_full = bars + 0;
    uint64_t *kv_empty = bars + 1;
    uint64_t *qs_full = bars + 2;
    uint64_t *qs_empty = qs_full + C::NST;
    uint64_t *st_full = qs_empty + C::NST;
    uint64_t *st_empty = st_full + 2;
    uint64_t *p_full = st_empty + 2;
    uint64_t *p_empty = p_full + 1;
    uint64_t *acc_full = p_empty + 1;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *drain = acc_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    const bool use_ext = !ACT && g.nb > 0 && g.H * ext_len(g.nb) <= kMaxBiasExtFloats;
    float *sLD = reinterpret_cast<float *>(smem + C::OFF_LD);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sDO = smem_u32(smem + C::OFF_DO);
    const uint32_t sPT = smem_u32(smem + C::OFF_PT);
    const uint32_t sDST = smem_u32(smem + C::OFF_DST);

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&qs_full[s], 1);
            mbar_init(&qs_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&st_full[b], 1);
            mbar_init(&st_empty[b], 4);
        }
        mbar_init(p_full, 4);
        mbar_init(p_empty, 1);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    stage_bias(g, sbias, ACT ? 1.0f : kLog2e);
    if (use_ext) stage_bias_ext(g, sext, kLog2e);
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

    if (warp == 0) {
        // producer warp: lane 0 issues TMA; all lanes copy lse / Delta of each
        // query block into the stage's shared-memory slot before it is published.
        uint32_t q_it = 0, t_local = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, lane == 0)) continue;
            if (!(ok = mbar_wait_warp(kv_empty, (t_local & 1) ^ 1, err))) break;
            ++t_local;
            if (lane == 0) {
                mbar_arrive_expect_tx(kv_full, 2 * C::KV_BYTES);
                for (int kb = 0; kb < C::NKB; ++kb) {
                    tma_load_2d(smem + C::OFF_K + kb * C::SUB_KV, &tmK, kv_full, t.h * D + kb * 64, t.kv_start);
                    tma_load_2d(smem + C::OFF_V + kb * C::SUB_KV, &tmV, kv_full, t.h * D + kb * 64, t.kv_start);
                }
            }
            const int nq = cdiv(t.q_len, C::BQ);
            for (int i = 0; i < nq; ++i, ++q_it) {
                const uint32_t slot = q_it % C::NST, use = q_it / C::NST;
                if (!(ok = mbar_wait_warp(&qs_empty[slot], (use & 1) ^ 1, err))) break;
                if (!ACT) {
                    float *ld = sLD + slot * 2 * C::BQ;
                    for (int k = lane; k < C::BQ; k += 32) {
                        const int qi = i * C::BQ + k;
                        float l2 = 0.0f, dl = 0.0f;  // stored negated: the consumer adds them
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
                    for (int kb = 0; kb < C::NKB; ++kb) {
                        tma_load_2d(smem + C::OFF_Q + slot * C::Q_BYTES + kb * C::SUB_Q, &tmQ, &qs_full[slot],
                                    t.h * D + kb * 64, y);
                        tma_load_2d(smem + C::OFF_DO + slot * C::Q_BYTES + kb * C::SUB_Q, &tmDO, &qs_full[slot],
                                    t.h * D + kb * 64, y);
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            if (t_local > 0) mbar_drain(kv_full, (t_local - 1) & 1);
            for (uint32_t s = 0; s < C::NST && s < q_it; ++s) {
                const uint32_t last = q_it - 1 - ((q_it - 1 - s) % C::NST);
                mbar_drain(&qs_full[last % C::NST], (last / C::NST) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t q_it = 0, st_it = 0, p_it = 0, t_local = 0;
            const uint32_t idesc_acc = idesc_bf16(128, D, false, true);
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                const int nq = cdiv(t.q_len, C::BQ);
                if (!(ok = mbar_wait(kv_full, t_local & 1, err))) break;
                if (!(ok = mbar_wait(acc_empty, (t_local & 1) ^ 1, err))) break;
                tc_fence_after();

                auto issue_st = [&](int i) -> bool {
                    const uint32_t it = q_it + i, slot = it % C::NST, use = it / C::NST;
                    if (!mbar_wait(&qs_full[slot], use & 1, err)) return false;
                    const uint32_t sb = st_it & 1, suse = st_it >> 1;
                    if (!mbar_wait(&st_empty[sb], (suse & 1) ^ 1, err)) return false;
                    tc_fence_after();
                    const int ncols = round_up16(min(C::BQ, t.q_len - i * C::BQ));
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint32_t qb = sQ + slot * C::Q_BYTES, dob = sDO + slot * C::Q_BYTES;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ao = (ks >> 2) * C::SUB_KV + (ks & 3) * 32;
                        const uint32_t bo = (ks >> 2) * C::SUB_Q + (ks & 3) * 32;
                        mma_bf16_ss(tmem + C::COL_ST + sb * C::BQ, sdesc_sw128(sK + ao, 16, 1024),
                                    sdesc_sw128(qb + bo, 16, 1024), idesc, ks > 0);
                        mma_bf16_ss(tmem + C::COL_DPT + sb * C::BQ, sdesc_sw128(sV + ao, 16, 1024),
                                    sdesc_sw128(dob + bo, 16, 1024), idesc, ks > 0);
                    }
                    mma_commit(&st_full[sb]);
                    ++st_it;
                    return true;
                };

                if (nq > 0) ok = issue_st(0);
                for (int i = 0; ok && i < nq; ++i) {
                    if (i + 1 < nq) {
                        if (!(ok = issue_st(i + 1))) break;
                    }
                    if (!(ok = mbar_wait(p_full, p_it & 1, err))) break;
                    tc_fence_after();
                    const uint32_t slot = (q_it + i) % C::NST;
                    const int ksteps = round_up16(min(C::BQ, t.q_len - i * C::BQ)) / 16;
                    const uint32_t qb = sQ + slot * C::Q_BYTES, dob = sDO + slot * C::Q_BYTES;
                    for (int ks = 0; ks < ksteps; ++ks) {
                        const uint32_t acc = (i > 0 || ks > 0) ? 1u : 0u;
                        const uint64_t bdo = sdesc_sw128(dob + ks * 2048, C::SUB_Q, 1024);
                        const uint64_t bq = sdesc_sw128(qb + ks * 2048, C::SUB_Q, 1024);
                        mma_bf16_ss(tmem + C::COL_DV, sdesc_sw128(sPT + ks * 32, 16, 1024), bdo, idesc_acc, acc);
                        mma_bf16_ss(tmem + C::COL_DK, sdesc_sw128(sDST + ks * 32, 16, 1024), bq, idesc_acc, acc);
                        if (ACT) {
                            mma_bf16_ss(tmem + C::COL_DV, sdesc_sw128(sPT + C::PT_BYTES + ks * 32, 16, 1024), bdo,
                                        idesc_acc, 1u);
                            mma_bf16_ss(tmem + C::COL_DK, sdesc_sw128(sDST + C::PT_BYTES + ks * 32, 16, 1024), bq,
                                        idesc_acc, 1u);
                        }
                    }
                    mma_commit(&qs_empty[slot]);
                    mma_commit(p_empty);
                    ++p_it;
                }
                if (!ok) break;
                mma_commit(kv_empty);
                mma_commit(acc_full);
                q_it += nq;
                ++t_local;
            }
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;  // key row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        uint32_t q_it = 0, st_it = 0, p_it = 0, t_local = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nq = cdiv(t.q_len, C::BQ);
            const float *bt = sbias + t.h * g.nb;
            const float *ext_h = sext + t.h * ext_len(g.nb);
            const int kv_loc = t.kv_loc0 + row;
            const int q_loc0 = t.q_loc0;
            for (int i = 0; i < nq; ++i, ++q_it) {
                const uint32_t slot = q_it % C::NST;
                const uint32_t sb = st_it & 1, suse = st_it >> 1;
                if (!(ok = mbar_wait_warp(&st_full[sb], suse & 1, err))) break;
                tc_fence_after();
                const int nvalid = min(C::BQ, t.q_len - i * C::BQ);
                const int ncols = round_up16(nvalid);
                float st[C::BQ], dpt[C::BQ];
                bool live[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) live[c] = c * 32 < nvalid;
                tmem_ld64x2(tmem + lane_base + C::COL_ST + sb * C::BQ, tmem + lane_base + C::COL_DPT + sb * C::BQ, st,
                            dpt);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&st_empty[sb]);
                ++st_it;

                const float *ld = sLD + slot * 2 * C::BQ;  // [-lse * log2 e | -Delta] of the 64 queries
                const int qb = q_loc0 + i * C::BQ;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (!live[c]) continue;
                    float(&xs)[32] = sub32(st, c);
                    float(&dpc)[32] = sub32(dpt, c);
                    float bv[32], cst = 0.0f;
                    bool band = false;
                    if (g.nb > 0) {
                        if (use_ext) {
                            band = bias32_ext(ext_h, g.nb, kv_loc, qb + c * 32, bv, cst);
                        } else {
                            bias32(bt, g.nb, kv_loc, qb + c * 32, bv);
                            band = true;
                        }
                    }
                    if (band) {
#pragma unroll
                        for (int k = 0; k < 32; k += 2) fma2(xs[k], xs[k + 1], sc, sc, bv[k], bv[k + 1]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; k += 2) fma2(xs[k], xs[k + 1], sc, sc, cst, cst);
                    }
                    if (ACT) {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            float pv;
                            dpc[k] = act_bwd(g.act, xs[k], pv) * dpc[k];
                            xs[k] = pv;
                        }
                    } else {
                        const float4 *l4 = reinterpret_cast<const float4 *>(ld + c * 32);
                        const float4 *d4 = reinterpret_cast<const float4 *>(ld + C::BQ + c * 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float4 lz = l4[k], dz = d4[k];
                            add2(xs[4 * k], xs[4 * k + 1], lz.x, lz.y);
                            add2(xs[4 * k + 2], xs[4 * k + 3], lz.z, lz.w);
                            add2(dpc[4 * k], dpc[4 * k + 1], dz.x, dz.y);
                            add2(dpc[4 * k + 2], dpc[4 * k + 3], dz.z, dz.w);
                        }
#pragma unroll
                        for (int k = 0; k < 32; ++k) xs[k] = ex2_approx(xs[k]);
#pragma unroll
                        for (int k = 0; k < 32; k += 2) mul2(dpc[k], dpc[k + 1], xs[k], xs[k + 1]);
                    }
                    if (c * 32 + 32 > nvalid) {
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (c * 32 + k >= nvalid) {
                                xs[k] = 0.0f;
                                dpc[k] = 0.0f;
                            }
                    }
                }
                if (!(ok = mbar_wait_warp(p_empty, (p_it & 1) ^ 1, err))) break;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (c * 32 >= ncols) continue;
                    if (!live[c]) {
                        for (int pl = 0; pl < C::NPL; ++pl) {
                            st_row32_zero(sPT + pl * C::PT_BYTES, C::PT_BYTES, row, c * 32);
                            st_row32_zero(sDST + pl * C::PT_BYTES, C::PT_BYTES, row, c * 32);
                        }
                    } else if (ACT) {
                        st_row32_bf16_hilo(sPT, sPT + C::PT_BYTES, C::PT_BYTES, row, c * 32, sub32(st, c));
                        st_row32_bf16_hilo(sDST, sDST + C::PT_BYTES, C::PT_BYTES, row, c * 32, sub32(dpt, c));
                    } else {
                        st_row32_bf16(sPT, C::PT_BYTES, row, c * 32, sub32(st, c));
                        st_row32_bf16(sDST, C::PT_BYTES, row, c * 32, sub32(dpt, c));
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
                ++p_it;
            }
            if (!ok) break;
            if (!(ok = mbar_wait_warp(acc_full, t_local & 1, err))) break;
            tc_fence_after();
            const bool row_ok = row < t.kv_len;
            const int64_t krow = static_cast<int64_t>(t.kv_start) + row;
            if (rows_fast<D>(a.dv)) {
                // stage dV, then dK, in this warp's rows of the P^T / dS^T planes (all MMAs are done)
                for (int pass = 0; pass < 2; ++pass) {
                    const float mul = pass == 0 ? 1.0f : g.scale;
                    float oa[D];
                    if (nq > 0) {
                        tmem_ld_row<D>(tmem + lane_base + (pass == 0 ? C::COL_DV : C::COL_DK), oa);
                    } else {
#pragma unroll
                        for (int k = 0; k < D; ++k) oa[k] = 0.0f;
                    }
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float(&o)[32] = sub32(oa, c);
#pragma unroll
                        for (int k = 0; k < 32; k += 2) mul2(o[k], o[k + 1], mul, mul);
                        st_row32_bf16(sPT, C::PT_BYTES, row, c * 32, o);
                    }
                    __syncwarp();
                    copy_rows_out<D>(sPT, C::PT_BYTES, quad * 32, t.kv_len, pass == 0 ? a.dv : a.dk, t.kv_start,
                                     t.h, lane);
                    __syncwarp();
                }
            } else {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    if (nq > 0) {
                        tmem_ld32(tmem + lane_base + C::COL_DV + c * 32, o);
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = 0.0f;
                    }
                    if (row_ok) store_out32(a.dv, krow, t.h, c * 32, o, 1.0f);
                    if (nq > 0) tmem_ld32(tmem + lane_base + C::COL_DK + c * 32, o);
                    if (row_ok) store_out32(a.dk, krow, t.h, c * 32, o, g.scale);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            ++t_local;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}


template <int D, bool ACT>
static cudaError_t launch_dq_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = DqCfg<D, ACT>;
    static bool done[64] = {};
    cudaError_t e = ensure_smem(dq_kernel<D, ACT>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    dq_kernel<D, ACT><<<n_ctas, 192, C::SMEM_ALLOC, st>>>(tm.q, tm.k, tm.v, tm.dout, a);
    return cudaGetLastError();
}

template <int D, bool ACT>
static cudaError_t launch_dkdv_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = DkvCfg<D, ACT>;
    static bool done[64] = {};
    cudaError_t e = ensure_smem(dkdv_kernel<D, ACT>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    dkdv_kernel<D, ACT><<<n_ctas, 192, C::SMEM_ALLOC, st>>>(tm.q, tm.k, tm.v, tm.dout, a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (D == 128) return act ? launch_dq_t<128, true>(tm, a, n_ctas, st) : launch_dq_t<128, false>(tm, a, n_ctas, st);
    if (D == 64) return act ? launch_dq_t<64, true>(tm, a, n_ctas, st) : launch_dq_t<64, false>(tm, a, n_ctas, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dkdv(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (D == 128)
        return act ? launch_dkdv_t<128, true>(tm, a, n_ctas, st) : launch_dkdv_t<128, false>(tm, a, n_ctas, st);
    if (D == 64) return act ? launch_dkdv_t<64, true>(tm, a, n_ctas, st) : launch_dkdv_t<64, false>(tm, a, n_ctas, st);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
