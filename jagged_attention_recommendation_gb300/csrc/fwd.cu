// fwd.cu -- jagged attention forward for sm_103a.
//
// "Training GEM at LLM scale", section "Jagged Sequence Flash Attention":
// FlashAttention directly on jagged tensors (no padding), with custom biases and
// asymmetric query/key-value lengths, TMA loads, warp specialisation and a
// persistent schedule; section "Generalized Dot-Product Attention (GDPA)": the
// softmax replaced by GELU / SiLU with no normalisation (no max, no rescale);
// section "BlockAttention": each 64-token query block sees only its own block.
//
// One CTA = 6 warps, persistent over the tiles the planner gave it:
//   warp 0     TMA producer: Q tile (128 rows) once per tile, then K/V tiles
//              (128 rows each) through an NST-deep ring.
//   warp 1     allocates TMEM; one thread issues every tcgen05.mma:
//              S_j = Q K_j^T into one of two TMEM score buffers, then
//              O += P_j V_j into one of two TMEM output buffers.
//   warps 2-5  one thread per query row (TMEM lane): scores -> bias, mask,
//              online softmax (or activation) -> P (bf16, 128B-swizzled smem),
//              rare O rescales in TMEM, epilogue O / l -> global, lse.
// Rows past a sequence's end are loaded (they belong to the next sequence or
// are zero-filled past the tensor end) but masked as keys and never stored as
// queries; the last key block of a sequence runs a narrower MMA (N rounded up
// to 16), so no tensor-core work is spent on whole masked column groups.
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.cuh"
#include "kernels.h"

namespace jattn {
using namespace dev;

template <int D, bool ACT>
struct FwdCfg {
    static constexpr int BM = 128, BN = 128;
    static constexpr int NKB = D / 64;  // 64-column sub-tiles along D
    static constexpr int NST = (D == 64) ? 4 : 2;
    static constexpr uint32_t SUB_Q = BM * 128;   // bytes of one 64-column sub-tile
    static constexpr uint32_t SUB_KV = BN * 128;
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;
    static constexpr uint32_t P_BYTES = BM * BN * 2;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NST * KV_BYTES;
    static constexpr uint32_t OFF_P = OFF_V + NST * KV_BYTES;
    static constexpr uint32_t OFF_PLO = OFF_P + P_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_PLO + (ACT ? P_BYTES : 0);
    // q_full, q_empty, kv_full[NST], kv_empty[NST], s_full[2], s_empty[2], p_full, pv_done,
    // o_full[2], o_empty[2], drain, xbar[4]
    static constexpr int NBAR = 2 + 2 * NST + 4 + 2 + 4 + 1 + 4;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;
    static constexpr uint32_t OFF_BEXT = OFF_BIAS + kMaxBiasFloats * 4;  // reflected table (softmax only)
    static constexpr uint32_t OFF_XCHG = OFF_BEXT + (ACT ? 0 : kMaxBiasExtFloats * 4);  // [2][2][128] floats
    static constexpr uint32_t SMEM = OFF_XCHG + (ACT ? 0 : 2 * 2 * 128 * 4);
    static constexpr int THREADS = 320;  // producer, MMA issuer, two softmax warpgroups
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;  // slack to align the base to 1024
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0;    // two score buffers of BN columns
    static constexpr uint32_t COL_O = 256;  // two output buffers of D columns
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

template <int D, bool ACT>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
    using C = FwdCfg<D, ACT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *q_full = bars + 0;
    uint64_t *q_empty = bars + 1;
    uint64_t *kv_full = bars + 2;
    uint64_t *kv_empty = bars + 2 + C::NST;
    uint64_t *s_full = bars + 2 + 2 * C::NST;
    uint64_t *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2;
    uint64_t *pv_done = p_full + 1;
    uint64_t *o_full = pv_done + 1;
    uint64_t *o_empty = o_full + 2;
    uint64_t *drain = o_empty + 2;
    uint64_t *xbar = drain + 1;  // [4]: the two groups' warps of one TMEM lane quadrant
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    float *xchg = reinterpret_cast<float *>(smem + C::OFF_XCHG);
    const bool use_ext = !ACT && g.nb > 0 && g.H * ext_len(g.nb) <= kMaxBiasExtFloats;

    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);
    const uint32_t sP = smem_u32(smem + C::OFF_P);
    const uint32_t sPlo = smem_u32(smem + C::OFF_PLO);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], 8);
            mbar_init(&o_full[b], 1);
            mbar_init(&o_empty[b], 8);
        }
        for (int q = 0; q < 4; ++q) mbar_init(&xbar[q], 2);
        mbar_init(p_full, 8);
        mbar_init(pv_done, 1);
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const ErrCtx err{g.status, abort_flag};
    const int tbeg = g.cta_begin[blockIdx.x];
    const int tend = g.cta_begin[blockIdx.x + 1];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t kv_it = 0, t_local = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, true)) continue;
                if (!(ok = mbar_wait(q_empty, (t_local & 1) ^ 1, err))) break;
                ++t_local;
                mbar_arrive_expect_tx(q_full, C::Q_BYTES);
                for (int kb = 0; kb < C::NKB; ++kb)
                    tma_load_2d(smem + C::OFF_Q + kb * C::SUB_Q, &tmQ, q_full, t.h * D + kb * 64, t.q_start);
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
            // Do not leave the CTA with copies still landing in shared memory.
            if (!ok) {
                if (t_local > 0) mbar_drain(q_full, (t_local - 1) & 1);
                for (uint32_t s = 0; s < C::NST && s < kv_it; ++s) {
                    const uint32_t last = kv_it - 1 - ((kv_it - 1 - s) % C::NST);  // last iteration using slot s
                    mbar_drain(&kv_full[last % C::NST], (last / C::NST) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t kv_it = 0, s_it = 0, p_it = 0, t_local = 0;
            const uint32_t idesc_pv = idesc_bf16(128, D, false, true);
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                const int nkv = cdiv(t.kv_len, C::BN);
                const uint32_t ob = t_local & 1, ouse = t_local >> 1;
                if (!(ok = mbar_wait(q_full, t_local & 1, err))) break;
                if (!(ok = mbar_wait(&o_empty[ob], (ouse & 1) ^ 1, err))) break;
                tc_fence_after();

                auto issue_S = [&](int j) -> bool {
                    const uint32_t it = kv_it + j, slot = it % C::NST, use = it / C::NST;
                    if (!mbar_wait(&kv_full[slot], use & 1, err)) return false;
                    const uint32_t sb = s_it & 1, suse = s_it >> 1;
                    if (!mbar_wait(&s_empty[sb], (suse & 1) ^ 1, err)) return false;
                    tc_fence_after();
                    const int ncols = round_up16(min(C::BN, t.kv_len - j * C::BN));
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint32_t kbase = sK + slot * C::KV_BYTES;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t ad = sdesc_sw128(sQ + (ks >> 2) * C::SUB_Q + (ks & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(kbase + (ks >> 2) * C::SUB_KV + (ks & 3) * 32, 16, 1024);
                        mma_bf16_ss(tmem + C::COL_S + sb * C::BN, ad, bd, idesc, ks > 0);
                    }
                    mma_commit(&s_full[sb]);
                    ++s_it;
                    return true;
                };

                if (nkv > 0) ok = issue_S(0);
                for (int j = 0; ok && j < nkv; ++j) {
                    if (j + 1 < nkv) {
                        if (!(ok = issue_S(j + 1))) break;
                    } else {
                        mma_commit(q_empty);  // last read of Q for this tile is in flight
                    }
                    if (!(ok = mbar_wait(p_full, p_it & 1, err))) break;
                    tc_fence_after();
                    const uint32_t slot = (kv_it + j) % C::NST;
                    const int ksteps = round_up16(min(C::BN, t.kv_len - j * C::BN)) / 16;
                    const uint32_t vbase = sV + slot * C::KV_BYTES;
                    const uint32_t dcol = tmem + C::COL_O + ob * D;
                    for (int ks = 0; ks < ksteps; ++ks) {
                        const uint64_t bd = sdesc_sw128(vbase + ks * 2048, C::SUB_KV, 1024);
                        const uint64_t ad = sdesc_sw128(sP + (ks >> 2) * (C::BM * 128) + (ks & 3) * 32, 16, 1024);
                        mma_bf16_ss(dcol, ad, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
                        if (ACT) {
                            const uint64_t al =
                                sdesc_sw128(sPlo + (ks >> 2) * (C::BM * 128) + (ks & 3) * 32, 16, 1024);
                            mma_bf16_ss(dcol, al, bd, idesc_pv, 1u);
                        }
                    }
                    mma_commit(&kv_empty[slot]);
                    mma_commit(pv_done);
                    ++p_it;
                }
                if (!ok) break;
                if (nkv == 0) mma_commit(q_empty);
                mma_commit(&o_full[ob]);
                kv_it += nkv;
                ++t_local;
            }
            // wait for every MMA this thread issued before TMEM is released
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        // ------------------------------------------------------------ softmax / epilogue
        // Two warpgroups share every score row: group wg handles key columns
        // [64 wg, 64 wg + 64) of each 128-key block and output columns
        // [wg D/2, (wg + 1) D/2).  Per key block they exchange their partial row
        // maxima through shared memory (one bounded mbarrier per TMEM lane
        // quadrant); their partial row sums are added once per tile.
        constexpr int HC = C::BN / 2;  // key columns per group
        constexpr int HD = D / 2;      // output columns per group
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;            // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;     // query row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        const int cbase = wg * HC;            // first key column of this group in a block
        uint32_t s_it = 0, p_it = 0, t_local = 0, x_it = 0;
        bool ok = true;
        // Swap one value per row with the partner warp (same quadrant, other group).
        auto exchange = [&](float mine, float &theirs) -> bool {
            const uint32_t slot = x_it & 1;
            xchg[(slot * 2 + wg) * 128 + row] = mine;
            __syncwarp();
            if (lane == 0) mbar_arrive(&xbar[quad]);
            if (!mbar_wait_warp(&xbar[quad], x_it & 1, err)) return false;
            theirs = xchg[(slot * 2 + (wg ^ 1)) * 128 + row];
            ++x_it;
            return true;
        };
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nkv = cdiv(t.kv_len, C::BN);
            const float *bt = sbias + t.h * g.nb;
            const float *ext_h = sext + t.h * ext_len(g.nb);
            const int q_loc = t.q_loc0 + row;
            float m = -INFINITY, l = 0.0f;  // l: this group's partial row sum

            for (int j = 0; j < nkv; ++j) {
                const uint32_t sb = s_it & 1, suse = s_it >> 1;
                if (!(ok = mbar_wait_warp(&s_full[sb], suse & 1, err))) break;
                tc_fence_after();
                const int nvalid = min(C::BN, t.kv_len - j * C::BN);
                const int ncols = round_up16(nvalid);
                float x[HC];
                bool live[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int cg = cbase + c * 32;
                    live[c] = (cg < nvalid) && (g.block == 0 || (cg >> 6) == (row >> 6));
                }
                if (cbase < ncols) tmem_ld64(tmem + lane_base + C::COL_S + sb * C::BN + cbase, x);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                ++s_it;

                // scores with bias and key mask (softmax: log2 units; without a
                // bias the scale is folded into the exponent's FMA below)
                const int kvb = t.kv_loc0 + j * C::BN + cbase;
                const bool scaled = ACT || g.nb > 0;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (!live[c]) continue;
                    float(&xc)[32] = sub32(x, c);
                    if (g.nb > 0) {
                        if (use_ext) {
                            scale_bias32(xc, sc, ext_h, g.nb, q_loc, kvb + c * 32);
                        } else {
                            float bv[32];
                            bias32(bt, g.nb, q_loc, kvb + c * 32, bv);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) fma2(xc[i], xc[i + 1], sc, sc, bv[i], bv[i + 1]);
                        }
                    } else if (ACT) {
#pragma unroll
                        for (int i = 0; i < 32; i += 2) mul2(xc[i], xc[i + 1], sc, sc);
                    }
                    const int cg = cbase + c * 32;
                    if (cg + 32 > nvalid) {  // the sequence's last keys end inside this chunk
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (cg + i >= nvalid) xc[i] = ACT ? 0.0f : -INFINITY;
                    }
                }
                float mloc = -INFINITY;
                if (!ACT) {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        if (live[c]) mloc = fmaxf(mloc, max32(sub32(x, c)));
                    if (!scaled) mloc *= sc;
                    float mo;
                    if (!(ok = exchange(mloc, mo))) break;
                    mloc = fmaxf(mloc, mo);
                }
                // the previous P @ V must be done before P is overwritten or O touched
                if (p_it > 0) {
                    if (!(ok = mbar_wait_warp(pv_done, (p_it - 1) & 1, err))) break;
                }
                if (!ACT) {
                    const float m_new = fmaxf(m, mloc);
                    if (j == 0) {
                        m = m_new;
                    } else {
                        // both groups see the same maxima, so they take the same decision
                        const bool need = m_new > m + kRescaleThreshold;
                        if (__any_sync(0xffffffffu, need)) {
                            const float alpha = ex2_approx(m - m_new);
                            tc_fence_after();
                            const uint32_t ta = tmem + lane_base + C::COL_O + (t_local & 1) * D + wg * HD;
                            if constexpr (HD == 64) {
                                float o[64];
                                tmem_ld64(ta, o);
#pragma unroll
                                for (int i = 0; i < 64; i += 2) mul2(o[i], o[i + 1], alpha, alpha);
                                tmem_st32(ta, sub32(o, 0));
                                tmem_st32(ta + 32, sub32(o, 1));
                            } else {
                                float o[32];
                                tmem_ld32(ta, o);
#pragma unroll
                                for (int i = 0; i < 32; i += 2) mul2(o[i], o[i + 1], alpha, alpha);
                                tmem_st32(ta, o);
                            }
                            l *= alpha;
                            m = m_new;
                        }
                    }
                    const float nm = (m == -INFINITY) ? 0.0f : -m;
                    float rs = 0.0f;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int cg = cbase + c * 32;
                        if (cg >= ncols) continue;
                        if (!live[c]) {
                            st_row32_zero(sP, C::BM * 128, row, cg);
                            continue;
                        }
                        float(&xc)[32] = sub32(x, c);
                        if (scaled) {
#pragma unroll
                            for (int i = 0; i < 32; i += 2) add2(xc[i], xc[i + 1], nm, nm);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 2) fma2(xc[i], xc[i + 1], sc, sc, nm, nm);
                        }
#pragma unroll
                        for (int i = 0; i < 32; ++i) xc[i] = ex2_approx(xc[i]);
                        rs += sum32(xc);
                        st_row32_bf16(sP, C::BM * 128, row, cg, xc);
                    }
                    l += rs;
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int cg = cbase + c * 32;
                        if (cg >= ncols) continue;
                        if (!live[c]) {
                            st_row32_zero(sP, C::BM * 128, row, cg);
                            st_row32_zero(sPlo, C::BM * 128, row, cg);
                            continue;
                        }
                        float(&xc)[32] = sub32(x, c);
#pragma unroll
                        for (int i = 0; i < 32; ++i) xc[i] = cg + i < nvalid ? act_fwd(g.act, xc[i]) : 0.0f;
                        st_row32_bf16_hilo(sP, sPlo, C::BM * 128, row, cg, xc);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
                ++p_it;
            }
            if (!ok) break;

            // ---- epilogue: this group's half of O (/ l) -> global; lse from group 0
            const uint32_t ob = t_local & 1, ouse = t_local >> 1;
            if (!(ok = mbar_wait_warp(&o_full[ob], ouse & 1, err))) break;
            tc_fence_after();
            float lt = l;
            if (!ACT) {
                float lo_;
                if (!(ok = exchange(l, lo_))) break;
                lt = wg == 0 ? l + lo_ : lo_ + l;  // same order in both groups
            }
            const bool row_ok = row < t.q_len;
            const int64_t orow = static_cast<int64_t>(t.q_start) + row;
            const float mul = ACT ? 1.0f : (lt > 0.0f ? 1.0f / lt : 0.0f);
            const bool fast = rows_fast<D>(a.out);
            float oa[HD];
            if (nkv > 0) {
                tmem_ld_row<HD>(tmem + lane_base + C::COL_O + ob * D + wg * HD, oa);
            } else {
#pragma unroll
                for (int i = 0; i < HD; ++i) oa[i] = 0.0f;
            }
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                float(&o)[32] = sub32(oa, c);
                const int col = wg * HD + c * 32;
                if (fast) {
                    // stage the row in this warp's own rows of the P tile (all P @ V are done)
#pragma unroll
                    for (int i = 0; i < 32; i += 2) mul2(o[i], o[i + 1], mul, mul);
                    st_row32_bf16(sP, C::BM * 128, row, col, o);
                } else if (row_ok) {
                    store_out32(a.out, orow, t.h, col, o, mul);
                }
            }
            if (fast) {
                __syncwarp();
                copy_rows_cols<HD, D>(sP, C::BM * 128, wg * HD, quad * 32, t.q_len, a.out, t.q_start, t.h, lane);
                __syncwarp();
            }
            if (!ACT && wg == 0 && a.lse != nullptr && row_ok) {
                a.lse[static_cast<int64_t>(t.h) * g.Tq + orow] =
                    (nkv > 0 && lt > 0.0f) ? (m + __log2f(lt)) * kLn2 : -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[ob]);
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
static cudaError_t launch_fwd_t(const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    using C = FwdCfg<D, ACT>;
    auto kern = fwd_kernel<D, ACT>;
    static bool done[64] = {};
    cudaError_t e = ensure_smem(kern, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    kern<<<n_ctas, C::THREADS, C::SMEM_ALLOC, stream>>>(tm.q, tm.k, tm.v, a);
    return cudaGetLastError();
}

cudaError_t launch_fwd(int D, bool act, const TmapSet &tm, const FwdArgs &a, int n_ctas, cudaStream_t stream) {
    if (D == 128) return act ? launch_fwd_t<128, true>(tm, a, n_ctas, stream) : launch_fwd_t<128, false>(tm, a, n_ctas, stream);
    if (D == 64) return act ? launch_fwd_t<64, true>(tm, a, n_ctas, stream) : launch_fwd_t<64, false>(tm, a, n_ctas, stream);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
