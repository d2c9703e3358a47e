// bwd_block.cu -- BlockAttention backward for sm_103a.
//
// "Training GEM at LLM scale", section "BlockAttention": with fixed 64-token
// blocks every query block attends only to its own key/value block, so the
// problem splits into independent 64x64 attentions and a dedicated kernel
// needs no online-softmax correction, no logsumexp traffic and no separate
// Delta pre-processing.  Here one CTA pass handles a 128-row chunk (two
// blocks) of one head:
//   S = Q K^T and dP = dO V^T (128x128, block-diagonal part used),
//   P = softmax over the row's own 64-block (recomputed, exact within the tile),
//   Delta_i = sum_j P_ij dP_ij (= <dO_i, O_i>), dS = P (dP - Delta)
//   (activation mode: P = act(S), dS = act'(S) dP),
//   dV = P^T dO, dK = dS^T Q, dQ = dS K   (all in TMEM; dQ reuses the S columns).
// P and dS are written once to shared memory as 128x128 bf16 tiles (zeros off
// the diagonal blocks) and read by the tensor cores both as K-major and as
// MN-major operands, so no transpose is ever materialised.  In activation mode
// P and dS are unnormalised and both get a bf16 remainder (hi + lo) in one
// shared lo plane: P's first, read by the dV products, then dS's, read by the
// dK and dQ products (a second hand-off, lo_free / dslo_full).
// With rotary position embedding (ROPE; same section: RoPE's backward fused
// into the attention epilogue) two more warps rotate each chunk's Q and K rows
// in shared memory as they arrive, the products run on the rotated operands,
// and the epilogue applies the transposed rotation to dQ and dK in float32,
// before the bf16 store, so the gradients leave for the unrotated inputs and
// no separate rotary kernel reads or writes them.
// OVL (D = 64, softmax, bf16 results, no RoPE): the compute warps write a
// chunk's results one chunk late, after they have handed the next chunk's P
// and dS to the products, so the epilogue overlaps the products of the next
// chunk.  dQ then has its own TMEM columns (the S columns take the next
// chunk's scores at once); the MMA thread waits only for the compute warps to
// have read S and dP (sp_free) before the next scores, and for the previous
// chunk's results to be read out (acc_empty) before the next chunk's dV / dK /
// dQ products; the compute warps wait for the previous chunk's products to be
// done with the P / dS tiles (pd_free) before they overwrite them, and stage
// the results in the lo plane, which softmax leaves unused.  (A separate
// output warpgroup would overlap the epilogue with the softmax as well, but
// the compute warps' 255 registers leave no room for its registers.)
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "attn.cuh"
#include "kernels.h"

namespace jattn {
using namespace dev;

template <int D>
struct BlkCfg {
    static constexpr int BM = 128;
    static constexpr int NKB = D / 64;
    static constexpr int NBUF = (D == 64) ? 2 : 1;
    static constexpr uint32_t SUB = BM * 128;          // 16 KB sub-tile
    static constexpr uint32_t T_BYTES = BM * D * 2;    // one [128, D] operand
    static constexpr uint32_t IN_BYTES = 4 * T_BYTES;  // Q, K, V, dO
    static constexpr uint32_t M_BYTES = BM * BM * 2;   // P or dS (two 16 KB sub-tiles)
    static constexpr uint32_t OFF_IN = 0;
    static constexpr uint32_t OFF_P = NBUF * IN_BYTES;
    static constexpr uint32_t OFF_DS = OFF_P + M_BYTES;
    static constexpr uint32_t OFF_DSLO = OFF_DS + M_BYTES;  // bf16 remainder of dS (activation mode)
    static constexpr uint32_t OFF_BAR = OFF_DSLO + M_BYTES;
    // in_full[NBUF], in_empty[NBUF], s_full, pd_full, acc_full, acc_empty, drain, rot_full[NBUF],
    // lo_free, dslo_full, sp_free, pd_free
    static constexpr int NBAR = 3 * NBUF + 9;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;
    static constexpr uint32_t SMEM = OFF_BIAS + kMaxBiasFloats * 4;
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0;  // S, later dQ
    static constexpr uint32_t COL_DP = 128;
    static constexpr uint32_t COL_DK = 256;
    static constexpr uint32_t COL_DV = 256 + D;
    static constexpr uint32_t COL_DQ_OVL = 256 + 2 * D;  // OVL: dQ's own columns (D = 64)
    // RoPE, D = 64: the epilogue's cos / sin row per lane (columns past dV)
    static constexpr uint32_t COL_TAB = D == 64 ? 256 + 2 * D : 0;
    // operand offsets inside one input buffer
    static constexpr uint32_t IQ = 0, IK = T_BYTES, IV = 2 * T_BYTES, IDO = 3 * T_BYTES;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

template <int D, bool ROPE, bool OVL>
__global__ void __launch_bounds__(ROPE ? 256 : 192, 1)
    bwd_block_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                     const BwdArgs a) {
    using C = BlkCfg<D>;
    static_assert(!OVL || (D == 64 && !ROPE), "the overlapped epilogue: D = 64 without RoPE");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *in_full = bars;
    uint64_t *in_empty = bars + C::NBUF;
    uint64_t *s_full = bars + 2 * C::NBUF;
    uint64_t *pd_full = s_full + 1;
    uint64_t *acc_full = pd_full + 1;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *drain = acc_empty + 1;
    uint64_t *rot_full = drain + 1;  // [NBUF] RoPE: the buffer's Q and K rows are rotated
    uint64_t *lo_free = rot_full + C::NBUF;  // activation: the dV products are done with P's lo plane
    uint64_t *dslo_full = lo_free + 1;       // activation: dS's lo plane is written
    uint64_t *sp_free = dslo_full + 1;       // OVL: the compute warps have read S and dP
    uint64_t *pd_free = sp_free + 1;         // OVL: the chunk's products are done with the P / dS tiles
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    const uint32_t sIn = smem_u32(smem + C::OFF_IN);
    const uint32_t sP = smem_u32(smem + C::OFF_P);
    const uint32_t sDS = smem_u32(smem + C::OFF_DS);
    const uint32_t sDSlo = smem_u32(smem + C::OFF_DSLO);
    const bool ACT = g.act != kSoftmax;

    if (threadIdx.x == 0) {
        for (int b = 0; b < C::NBUF; ++b) {
            mbar_init(&in_full[b], 1);
            mbar_init(&in_empty[b], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(pd_full, 4);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain, 1);
        for (int b = 0; b < C::NBUF; ++b) mbar_init(&rot_full[b], 2);  // the two rotation warps
        mbar_init(lo_free, 1);
        mbar_init(dslo_full, 4);
        mbar_init(sp_free, 4);
        mbar_init(pd_free, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    stage_bias(g, sbias, ACT ? 1.0f : kLog2e);
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
    const ErrCtx err{g.status, abort_flag, g.wait_ns};
    const int tbeg = g.cta_begin[blockIdx.x];
    const int tend = g.cta_begin[blockIdx.x + 1];

    // OVL: chunk n's dV, dQ, dK from TMEM through this warp's rows of the
    // staging tile (the lo plane) to whole 128-byte result rows; TMEM goes
    // back after the last read, before the last stores
    auto drain_ovl = [&](const Tile &pt, uint32_t n, int row, int quad, uint32_t lane_base) -> bool {
        if (!mbar_wait_warp(acc_full, n & 1, err)) return false;
        tc_fence_after();
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {  // dV, dQ, dK
            const uint32_t col = pass == 0 ? C::COL_DV : (pass == 1 ? C::COL_DQ_OVL : C::COL_DK);
            const float mul = pass == 0 ? 1.0f : g.scale;
            float oa[64];
            tmem_ld64(tmem + lane_base + col, oa);
            if (pass == 2) {  // every TMEM read of the chunk is done
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
#pragma unroll
            for (int i = 0; i < 64; i += 2) mul2(oa[i], oa[i + 1], mul, mul);
            st_row32_bf16(sDSlo, C::SUB, row, 0, sub32(oa, 0));
            st_row32_bf16(sDSlo, C::SUB, row, 32, sub32(oa, 1));
            __syncwarp();
            copy_rows_out<D>(sDSlo, C::SUB, quad * 32, pt.q_len, pass == 0 ? a.dv : (pass == 1 ? a.dq : a.dk),
                             pass == 1 ? pt.q_start : pt.kv_start, pt.h, lane);
            __syncwarp();
        }
        return true;
    };
    if (warp == 0) {
        if (lane == 0) {
            uint32_t t_local = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, true)) continue;
                const uint32_t buf = t_local % C::NBUF, use = t_local / C::NBUF;
                if (!(ok = mbar_wait(&in_empty[buf], (use & 1) ^ 1, err))) break;
                ++t_local;
                mbar_arrive_expect_tx(&in_full[buf], C::IN_BYTES);
                uint8_t *base = smem + C::OFF_IN + buf * C::IN_BYTES;
                for (int kb = 0; kb < C::NKB; ++kb) {
                    const int x = t.h * D + kb * 64;
                    tma_load_2d(base + C::IQ + kb * C::SUB, &tmQ, &in_full[buf], x, t.q_start);
                    tma_load_2d(base + C::IK + kb * C::SUB, &tmK, &in_full[buf], x, t.kv_start);
                    tma_load_2d(base + C::IV + kb * C::SUB, &tmV, &in_full[buf], x, t.kv_start);
                    tma_load_2d(base + C::IDO + kb * C::SUB, &tmDO, &in_full[buf], x, t.q_start);
                }
            }
            {  // the last copy into every buffer has landed before the CTA leaves (also after an abort)
                for (uint32_t b = 0; b < C::NBUF && b < t_local; ++b) {
                    const uint32_t last = t_local - 1 - ((t_local - 1 - b) % C::NBUF);
                    mbar_drain(&in_full[last % C::NBUF], (last / C::NBUF) & 1);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && OVL) {
            // one chunk ahead: the next chunk's S and dP are issued as soon as the
            // compute warps have read this chunk's, before this chunk's dV / dK / dQ
            const uint32_t idesc_mn = idesc_bf16(128, D, true, true);   // dV, dK
            const uint32_t idesc_kmn = idesc_bf16(128, D, false, true); // dQ
            TileStream ts(g, tbeg, tend);
            auto next_valid = [&](Tile &x) -> bool {
                while (ts.next(x))
                    if (check_tile(g, x, err, false)) return true;
                return false;
            };
            auto issue_s = [&](const Tile &x, uint32_t n) -> bool {  // chunk n's S and dP
                const uint32_t buf = n % C::NBUF, use = n / C::NBUF;
                if (!mbar_wait(&in_full[buf], use & 1, err)) return false;
                if (n > 0 && !mbar_wait(sp_free, (n - 1) & 1, err)) return false;  // chunk n - 1's read out
                tc_fence_after();
                const uint32_t base = sIn + buf * C::IN_BYTES;
                const uint32_t idesc_s = idesc_bf16(128, round_up16(x.q_len), false, false);
                const uint64_t kQ = sdesc_sw128(base + C::IQ, 16, 1024), kK = sdesc_sw128(base + C::IK, 16, 1024);
                const uint64_t kDO = sdesc_sw128(base + C::IDO, 16, 1024), kV = sdesc_sw128(base + C::IV, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t o = (ks >> 2) * C::SUB + (ks & 3) * 32;
                    mma_bf16_ss(tmem + C::COL_S, sdesc_add(kQ, o), sdesc_add(kK, o), idesc_s, ks > 0);
                    mma_bf16_ss(tmem + C::COL_DP, sdesc_add(kDO, o), sdesc_add(kV, o), idesc_s, ks > 0);
                }
                mma_commit(s_full);
                return true;
            };
            auto issue_acc = [&](const Tile &x, uint32_t n) -> bool {  // chunk n's dV, dK, dQ
                const uint32_t buf = n % C::NBUF;
                if (!mbar_wait(pd_full, n & 1, err)) return false;
                if (!mbar_wait(acc_empty, (n & 1) ^ 1, err)) return false;  // chunk n - 1's results read out
                tc_fence_after();
                const uint32_t base = sIn + buf * C::IN_BYTES;
                const int ksteps = round_up16(x.q_len) / 16;
                const uint64_t mP = sdesc_sw128(sP, C::SUB, 1024), mDS = sdesc_sw128(sDS, C::SUB, 1024);
                const uint64_t kDS = sdesc_sw128(sDS, 16, 1024);
                const uint64_t mDO = sdesc_sw128(base + C::IDO, C::SUB, 1024), mQ = sdesc_sw128(base + C::IQ, C::SUB, 1024);
                const uint64_t mK = sdesc_sw128(base + C::IK, C::SUB, 1024);
#pragma unroll
                for (int ks = 0; ks < C::BM / 16; ++ks) {
                    if (ks < ksteps) {
                        const uint32_t acc = ks > 0 ? 1u : 0u;
                        mma_bf16_ss(tmem + C::COL_DV, sdesc_add(mP, ks * 2048), sdesc_add(mDO, ks * 2048), idesc_mn, acc);
                        mma_bf16_ss(tmem + C::COL_DK, sdesc_add(mDS, ks * 2048), sdesc_add(mQ, ks * 2048), idesc_mn, acc);
                        mma_bf16_ss(tmem + C::COL_DQ_OVL, sdesc_add(kDS, (ks >> 2) * C::SUB + (ks & 3) * 32),
                                    sdesc_add(mK, ks * 2048), idesc_kmn, acc);
                    }
                }
                mma_commit(&in_empty[buf]);
                mma_commit(pd_free);
                mma_commit(acc_full);
                return true;
            };
            Tile cur, nxt;
            bool have = next_valid(cur), ok = true;
            if (have) ok = issue_s(cur, 0);
            for (uint32_t n = 0; ok && have; ++n) {
                const bool have_next = next_valid(nxt);
                if (have_next && !(ok = issue_s(nxt, n + 1))) break;
                if (!(ok = issue_acc(cur, n))) break;
                cur = nxt;
                have = have_next;
            }
            mma_commit(drain);
            mbar_drain(drain, 0);
        } else if (lane == 0) {
            uint32_t t_local = 0;
            const uint32_t idesc_mn = idesc_bf16(128, D, true, true);   // dV, dK
            const uint32_t idesc_kmn = idesc_bf16(128, D, false, true); // dQ
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                const uint32_t buf = t_local % C::NBUF, use = t_local / C::NBUF;
                if (!(ok = mbar_wait(ROPE ? &rot_full[buf] : &in_full[buf], use & 1, err))) break;
                // the S / dP columns: read out by the compute warps (OVL), or the whole
                // previous chunk written out (dQ reuses them otherwise)
                if (!(ok = mbar_wait(OVL ? sp_free : acc_empty, (t_local & 1) ^ 1, err))) break;
                tc_fence_after();
                const uint32_t base = sIn + buf * C::IN_BYTES;
                const int n16 = round_up16(t.q_len);
                const uint32_t idesc_s = idesc_bf16(128, n16, false, false);
                // Descriptors are built once per tile and the product runs are fully
                // unrolled (a guard per step where the count varies): constant offsets
                // and nothing else between two products, so this one thread issues them
                // as fast as the tensor pipe takes them.
                const uint64_t kQ = sdesc_sw128(base + C::IQ, 16, 1024), kK = sdesc_sw128(base + C::IK, 16, 1024);
                const uint64_t kDO = sdesc_sw128(base + C::IDO, 16, 1024), kV = sdesc_sw128(base + C::IV, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t o = (ks >> 2) * C::SUB + (ks & 3) * 32;
                    mma_bf16_ss(tmem + C::COL_S, sdesc_add(kQ, o), sdesc_add(kK, o), idesc_s, ks > 0);
                    mma_bf16_ss(tmem + C::COL_DP, sdesc_add(kDO, o), sdesc_add(kV, o), idesc_s, ks > 0);
                }
                mma_commit(s_full);
                if (!(ok = mbar_wait(pd_full, t_local & 1, err))) break;
                // OVL: the previous chunk's dV, dK, dQ have been read out before these
                // products start over in their columns
                if (OVL && !(ok = mbar_wait(acc_empty, (t_local & 1) ^ 1, err))) break;
                tc_fence_after();
                const int ksteps = n16 / 16;
                const uint64_t mP = sdesc_sw128(sP, C::SUB, 1024), mDS = sdesc_sw128(sDS, C::SUB, 1024);
                const uint64_t mDSlo = sdesc_sw128(sDSlo, C::SUB, 1024), kDS = sdesc_sw128(sDS, 16, 1024);
                const uint64_t kDSlo = sdesc_sw128(sDSlo, 16, 1024);
                const uint64_t mDO = sdesc_sw128(base + C::IDO, C::SUB, 1024), mQ = sdesc_sw128(base + C::IQ, C::SUB, 1024);
                const uint64_t mK = sdesc_sw128(base + C::IK, C::SUB, 1024);
#pragma unroll
                for (int ks = 0; ks < C::BM / 16; ++ks) {
                    if (ks < ksteps) {
                        // dV += P^T dO and dK += dS^T Q: reduction over query rows ks*16..+15
                        const uint32_t acc = ks > 0 ? 1u : 0u;
                        mma_bf16_ss(tmem + C::COL_DV, sdesc_add(mP, ks * 2048), sdesc_add(mDO, ks * 2048), idesc_mn, acc);
                        if (ACT)  // unnormalised P: its bf16 remainder, in the lo plane for now
                            mma_bf16_ss(tmem + C::COL_DV, sdesc_add(mDSlo, ks * 2048), sdesc_add(mDO, ks * 2048),
                                        idesc_mn, 1u);
                        mma_bf16_ss(tmem + C::COL_DK, sdesc_add(mDS, ks * 2048), sdesc_add(mQ, ks * 2048), idesc_mn, acc);
                        // dQ += dS K: reduction over key rows ks*16..+15
                        mma_bf16_ss(tmem + (OVL ? C::COL_DQ_OVL : C::COL_S),
                                    sdesc_add(kDS, (ks >> 2) * C::SUB + (ks & 3) * 32), sdesc_add(mK, ks * 2048),
                                    idesc_kmn, acc);
                    }
                }
                if (ACT) {  // unnormalised dS: add its bf16 remainder to dK and dQ
                    mma_commit(lo_free);
                    if (!(ok = mbar_wait(dslo_full, t_local & 1, err))) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < C::BM / 16; ++ks) {
                        if (ks < ksteps) {
                            mma_bf16_ss(tmem + C::COL_DK, sdesc_add(mDSlo, ks * 2048), sdesc_add(mQ, ks * 2048),
                                        idesc_mn, 1u);
                            mma_bf16_ss(tmem + C::COL_S, sdesc_add(kDSlo, (ks >> 2) * C::SUB + (ks & 3) * 32),
                                        sdesc_add(mK, ks * 2048), idesc_kmn, 1u);
                        }
                    }
                }
                mma_commit(&in_empty[buf]);
                if (OVL) mma_commit(pd_free);
                mma_commit(acc_full);
                ++t_local;
            }
            mma_commit(drain);
            mbar_drain(drain, 0);
        }
    } else if (ROPE && warp >= 6) {
        // RoPE: rotate the chunk's Q and K rows (the same positions) in place as
        // soon as they land, warp 6 rows 0..63 and warp 7 rows 64..127 (two
        // sub-partitions share the extra issue load); the products wait for
        // rot_full.
        uint32_t t_local = 0;
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const uint32_t buf = t_local % C::NBUF, use = t_local / C::NBUF;
            if (!(ok = mbar_wait_warp(&in_full[buf], use & 1, err))) break;
            const int h0 = (warp - 6) * 64, nrows = min(64, t.q_len - h0);
            if (nrows > 0) {
                const uint32_t base = sIn + buf * C::IN_BYTES + h0 * 128;
                const int64_t r0 = static_cast<int64_t>(t.q_loc0 + h0) * (D / 2);
                rope_tile<D, 8>(base + C::IQ, base + C::IK, C::SUB, nrows, g.rope_cos + r0, g.rope_sin + r0, lane);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&rot_full[buf]);
            ++t_local;
        }
    } else if (warp >= 2 && warp < 6) {
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int half = row >> 6;  // which 64-block of the chunk this row belongs to
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        uint32_t t_local = 0;
        bool ok = true;
        Tile prev{};  // OVL: the chunk whose results are written next
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const float *bt = sbias + t.h * g.nb;
            const int len = t.q_len;
            const int q_loc = t.q_loc0 + row;
            const int kv_loc0 = t.kv_loc0 + half * 64;  // first key of this row's block
            const int nvalid = min(64, max(0, len - half * 64));          // valid keys in the block
            // Query rows past the sequence end must contribute nothing to dK / dV.
            const bool row_valid = row < len;
            if (!(ok = mbar_wait_warp(s_full, t_local & 1, err))) break;
            tc_fence_after();
            float s[64], dp[64];
            bool live[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) live[c] = c * 32 < nvalid;  // uniform: one warp lies in one block
            if (nvalid > 0)
                tmem_ld64x2(tmem + lane_base + C::COL_S + half * 64, tmem + lane_base + C::COL_DP + half * 64, s, dp);
            if constexpr (OVL) {  // S and dP are in registers: the next chunk's scores may start
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sp_free);
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                if (!live[c]) continue;
                float bv[32];
                if (g.nb > 0) {
                    bias32(bt, g.nb, q_loc, kv_loc0 + c * 32, bv);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) bv[i] = 0.0f;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int cc = c * 32 + i;
                    s[cc] = (row_valid && cc < nvalid) ? fmaf(s[cc], sc, bv[i]) : (ACT ? 0.0f : -INFINITY);
                }
            }
            if (!ACT) {
                float m = -INFINITY;
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    if (live[c]) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) m = fmaxf(m, s[c * 32 + i]);
                    }
                if (m == -INFINITY) m = 0.0f;
                float l = 0.0f;
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    if (live[c]) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float p = ex2_approx(s[c * 32 + i] - m);
                            s[c * 32 + i] = p;
                            l += p;
                        }
                    }
                const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                float delta = 0.0f;
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    if (live[c]) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            s[c * 32 + i] *= inv;
                            delta = fmaf(s[c * 32 + i], dp[c * 32 + i], delta);
                        }
                    }
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    if (live[c]) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) dp[c * 32 + i] = s[c * 32 + i] * (dp[c * 32 + i] - delta);
                    }
            } else {
                // the activation fixed per loop (a run-time choice per element
                // would put a branch around every element)
                auto act_rows = [&](auto af) {
                    constexpr int AF = decltype(af)::value;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        if (live[c]) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int cc = c * 32 + i;
                                float av;
                                const float dv = act_bwd_t<AF>(s[cc], av) * dp[cc];
                                const bool in = row_valid && cc < nvalid;
                                s[cc] = in ? av : 0.0f;
                                dp[cc] = in ? dv : 0.0f;
                            }
                        }
                };
                if (g.act == kSilu)
                    act_rows(std::integral_constant<int, kSilu>{});
                else
                    act_rows(std::integral_constant<int, kGeluTanh>{});
            }
            // OVL: the previous chunk's products have read the P / dS tiles
            if (OVL && !(ok = mbar_wait_warp(pd_free, (t_local & 1) ^ 1, err))) break;
            // P and dS rows: this row's block gets values, the other block zeros
            // (activation: the lo plane takes P's remainder first)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const uint32_t col = half * 64 + c * 32;
                if (live[c] && row_valid) {
                    if (ACT)
                        st_row32_bf16_hilo(sP, sDSlo, C::SUB, row, col, sub32(s, c));
                    else
                        st_row32_bf16(sP, C::SUB, row, col, sub32(s, c));
                    st_row32_bf16(sDS, C::SUB, row, col, sub32(dp, c));
                } else {
                    st_row32_zero(sP, C::SUB, row, col);
                    st_row32_zero(sDS, C::SUB, row, col);
                    if (ACT) st_row32_zero(sDSlo, C::SUB, row, col);
                }
                const uint32_t ocol = (1 - half) * 64 + c * 32;
                st_row32_zero(sP, C::SUB, row, ocol);
                st_row32_zero(sDS, C::SUB, row, ocol);
                if (ACT) st_row32_zero(sDSlo, C::SUB, row, ocol);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pd_full);
            if constexpr (OVL) {  // the previous chunk's results, now that this chunk's products may run
                if (t_local > 0 && !(ok = drain_ovl(prev, t_local - 1, row, quad, lane_base))) break;
                prev = t;
                ++t_local;
                continue;
            }
            if (ACT) {
                // once the dV products are done with P's remainder, the lo plane
                // takes dS's (hi was rounded from the same values above); the rest
                // of the plane is still zero from P's
                if (!(ok = mbar_wait_warp(lo_free, t_local & 1, err))) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (live[c] && row_valid) {
                        float lo[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float x = dp[c * 32 + i];
                            lo[i] = x - __bfloat162float(__float2bfloat16_rn(x));
                        }
                        st_row32_bf16(sDSlo, C::SUB, row, half * 64 + c * 32, lo);
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dslo_full);
            }

            // RoPE, D = 64: this row's cos / sin (its query and its key share the
            // position) go to free TMEM columns while the products run, so the
            // epilogue reads them without a global-memory wait
            const bool tab_tmem = ROPE && C::COL_TAB > 0 && t.q_loc0 == t.kv_loc0;
            if (tab_tmem) {
                const int64_t pr = static_cast<int64_t>(t.q_loc0 + (row < len ? row : 0)) * (D / 2);
#pragma unroll 1
                for (int part = 0; part < 2; ++part) {
                    const float *src = (part == 0 ? g.rope_cos : g.rope_sin) + pr;
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 x = *reinterpret_cast<const float4 *>(src + i);
                        v[i] = x.x, v[i + 1] = x.y, v[i + 2] = x.z, v[i + 3] = x.w;
                    }
                    tmem_st32(tmem + lane_base + C::COL_TAB + part * 32, v);
                }
                tmem_wait_st();
            }
            if (!(ok = mbar_wait_warp(acc_full, t_local & 1, err))) break;
            tc_fence_after();
            const bool row_ok = row < len;
            const int64_t qrow = static_cast<int64_t>(t.q_start) + row;
            const int64_t krow = static_cast<int64_t>(t.kv_start) + row;
            if (rows_fast<D>(a.dq)) {
                // stage dV, dQ, dK in turn in this warp's rows of the P tile (every MMA is done)
#pragma unroll 1
                for (int pp = 0; pp < 3; ++pp) {
                    const int pass = pp == 0 ? 2 : pp - 1;
                    const uint32_t col = pass == 0 ? C::COL_S : (pass == 1 ? C::COL_DK : C::COL_DV);
                    const float mul = pass == 2 ? 1.0f : g.scale;
                    if (ROPE && pass < 2) {
                        // dQ / dK of the rotated rows -> of the unrotated ones: the
                        // transposed rotation at the row's position, in float32
                        const int64_t pr = static_cast<int64_t>((pass == 0 ? t.q_loc0 : t.kv_loc0) + (row_ok ? row : 0));
                        const float *tc = g.rope_cos + pr * (D / 2), *tsn = g.rope_sin + pr * (D / 2);
#pragma unroll 1
                        for (int cp = 0; cp < D / 64; ++cp) {
                            float lo[32], hi[32];
                            tmem_ld32x2(tmem + lane_base + col + cp * 32, tmem + lane_base + col + D / 2 + cp * 32,
                                        lo, hi);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                mul2(lo[i], lo[i + 1], mul, mul);
                                mul2(hi[i], hi[i + 1], mul, mul);
                            }
                            if (tab_tmem) {
#pragma unroll
                                for (int h = 0; h < 2; ++h) {  // 16 cos and 16 sin at a time
                                    float c[16], sn[16];
                                    tmem_ld16x2(tmem + lane_base + C::COL_TAB + h * 16,
                                                tmem + lane_base + C::COL_TAB + 32 + h * 16, c, sn);
                                    rope_grad16_regs(lo, hi, h * 16, c, sn);
                                }
                            } else {
                                rope_grad32(lo, hi, tc + cp * 32, tsn + cp * 32);
                            }
                            st_row32_bf16(sP, C::SUB, row, cp * 32, lo);
                            st_row32_bf16(sP, C::SUB, row, D / 2 + cp * 32, hi);
                        }
                    } else {
#pragma unroll
                        for (int hc = 0; hc < D / 64; ++hc) {
                            float oa[64];
                            tmem_ld64(tmem + lane_base + col + hc * 64, oa);
#pragma unroll
                            for (int i = 0; i < 64; i += 2) mul2(oa[i], oa[i + 1], mul, mul);
                            st_row32_bf16(sP, C::SUB, row, hc * 64, sub32(oa, 0));
                            st_row32_bf16(sP, C::SUB, row, hc * 64 + 32, sub32(oa, 1));
                        }
                    }
                    __syncwarp();
                    copy_rows_out<D>(sP, C::SUB, quad * 32, len, pass == 0 ? a.dq : (pass == 1 ? a.dk : a.dv),
                                     pass == 0 ? t.q_start : t.kv_start, t.h, lane);
                    __syncwarp();
                }
            } else if (ROPE) {
                // the same with direct stores (bf16 data with D in {64, 128}
                // takes the staged path above; this keeps the kernel whole)
                for (int pass = 0; pass < 2; ++pass) {
                    const uint32_t col = pass == 0 ? C::COL_S : C::COL_DK;
                    const int64_t pr = static_cast<int64_t>((pass == 0 ? t.q_loc0 : t.kv_loc0) + (row_ok ? row : 0));
                    const float *tc = g.rope_cos + pr * (D / 2), *tsn = g.rope_sin + pr * (D / 2);
#pragma unroll 1
                    for (int cp = 0; cp < D / 64; ++cp) {
                        float lo[32], hi[32];
                        tmem_ld32x2(tmem + lane_base + col + cp * 32, tmem + lane_base + col + D / 2 + cp * 32, lo,
                                    hi);
                        rope_grad32(lo, hi, tc + cp * 32, tsn + cp * 32);
                        if (row_ok) {
                            store_out32(pass == 0 ? a.dq : a.dk, pass == 0 ? qrow : krow, t.h, cp * 32, lo, g.scale);
                            store_out32(pass == 0 ? a.dq : a.dk, pass == 0 ? qrow : krow, t.h, D / 2 + cp * 32, hi,
                                        g.scale);
                        }
                    }
                }
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tmem + lane_base + C::COL_DV + c * 32, o);
                    if (row_ok) store_out32(a.dv, krow, t.h, c * 32, o, 1.0f);
                }
            } else {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tmem + lane_base + C::COL_S + c * 32, o);
                    if (row_ok) store_out32(a.dq, qrow, t.h, c * 32, o, g.scale);
                    tmem_ld32(tmem + lane_base + C::COL_DK + c * 32, o);
                    if (row_ok) store_out32(a.dk, krow, t.h, c * 32, o, g.scale);
                    tmem_ld32(tmem + lane_base + C::COL_DV + c * 32, o);
                    if (row_ok) store_out32(a.dv, krow, t.h, c * 32, o, 1.0f);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            ++t_local;
        }
        if (OVL && ok && t_local > 0) drain_ovl(prev, t_local - 1, row, quad, lane_base);  // the last chunk
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, bool ROPE, bool OVL = false>
static cudaError_t launch_block_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = BlkCfg<D>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(bwd_block_kernel<D, ROPE, OVL>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    bwd_block_kernel<D, ROPE, OVL><<<n_ctas, ROPE ? 256 : 192, C::SMEM_ALLOC, st>>>(tm.q, tm.k, tm.v, tm.dout, a);
    return cudaGetLastError();
}

cudaError_t launch_bwd_block(int D, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    const bool rope = a.g.rope_cos != nullptr;
    // the rotation is offered with softmax only (checked by the host first)
    if (rope && (a.g.rope_sin == nullptr || a.g.act != kSoftmax)) return cudaErrorInvalidValue;
    if (D == 128) return rope ? launch_block_t<128, true>(tm, a, n_ctas, st) : launch_block_t<128, false>(tm, a, n_ctas, st);
    if (D == 64) {
        if (rope) return launch_block_t<64, true>(tm, a, n_ctas, st);
        // softmax with bf16 results of width D: the epilogue runs on its own warps
        const bool rows = !a.dq.f32 && !a.dk.f32 && !a.dv.f32 && a.dq.cols == D && a.dk.cols == D && a.dv.cols == D;
        if (a.g.act == kSoftmax && rows) return launch_block_t<64, false, true>(tm, a, n_ctas, st);
        return launch_block_t<64, false>(tm, a, n_ctas, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace jattn
