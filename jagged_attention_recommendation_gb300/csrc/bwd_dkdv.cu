// bwd_dkdv.cu -- jagged attention backward, pass 2 (dK, dV over key-major
// tiles); the layout, the roles and the reasoning behind them are described at
// the top of bwd.cu (pass 1, dQ), which shares this file's helpers through
// bwd_common.cuh. Here both compute groups work on every query block, group g
// on its 32 queries 32 g .. 32 g + 31, so a block's P^T / dS^T take half the
// time of one group doing all 64; the hand-off to the dV / dK issuer waits for
// all eight compute warps.
#include "bwd_common.cuh"

namespace jattn {
using namespace dev;
namespace {
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
    // kv_full, kv_empty, qs_full[NSQ], qs_empty[NSQ], st_full[2], p_full[2], acc_full, dv_empty,
    // acc_done[2], drain[2], dk_empty
    static constexpr int NBAR = 2 + 2 * NSQ + 4 + 2 + 2 + 2 + 1;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;
    static constexpr uint32_t OFF_BEXT = OFF_BIAS + (BIAS == kBiasTable ? kMaxBiasFloats * 4 : 0);
    // per output warp: 32 rows x 64 bf16 staging for row-contiguous stores
    static constexpr int STG_W = 64;
    static constexpr uint32_t OFF_STG = (OFF_BEXT + (BIAS == kBiasExt ? kMaxBiasExtFloats * 4 : 0) + 127) & ~127u;
    // the CTA's share of the bias-table gradient [H, nb] (dS chunk mode with a bias)
    static constexpr uint32_t OFF_DT = OFF_STG + 4 * 32 * STG_W * 2;
    // per compute warp: 16 rows x 64 bytes of its dS piece, for row-grouped
    // stores (softmax with a bias, where the compute warps bound the block rate)
    static constexpr bool DS_STAGED = !ACT && BIAS != kBiasNone;
    static constexpr uint32_t OFF_DSS = OFF_DT + (BIAS != kBiasNone ? kMaxBiasFloats * 4 : 0);
    static constexpr uint32_t SMEM = OFF_DSS + (DS_STAGED ? 8 * 1024 : 0);
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    // group g: S^T at 128 g (P^T over it), dP^T at 128 g + 64 (dS^T over it); dV, dK
    static constexpr uint32_t COL_DV = 256;
    static constexpr uint32_t COL_DK = 256 + D;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(OFF_Q % 1024 == 0 && Q_BYTES % 1024 == 0, "operand alignment");
    static_assert(OFF_STG % 16 == 0, "16-byte shared-memory vectors");
    static_assert(COL_DK + D <= TMEM_COLS, "TMEM budget");
    // registers per thread after the split (launch: 512 threads x 128).  The
    // reflected-bias compute path needs 176; the others fit in 160, which
    // leaves the output group enough to read 64 accumulator columns per TMEM
    // round trip instead of 32.
    static constexpr uint32_t REG_CTRL = 56;
    static constexpr uint32_t REG_COMPUTE = BIAS == kBiasExt ? 176 : 160;
    static constexpr uint32_t REG_OUT = (128 * 512 - REG_CTRL * 128 - REG_COMPUTE * 256) / 128;
    static constexpr int DRAIN_COLS = REG_OUT >= 136 ? 64 : 32;
    static_assert(REG_CTRL * 128 + REG_COMPUTE * 256 + REG_OUT * 128 <= 128 * 512, "register split");
    static_assert(REG_OUT % 8 == 0, "setmaxnreg granularity");
};

// WIN: sliding window on.  DS: every block's dS (bf16; activation mode: the
// bf16 hi and lo parts) also goes to the workspace, one 16 KB chunk per
// (key tile, 64-query block): rows are the tile's 128 keys, each row the
// block's 64 queries, 16-byte pieces XOR-swizzled by row (the 128-byte swizzle
// of an MMA operand tile, so that a plain bulk copy into shared memory gives
// the dQ product's A operand); rows past the tile's keys are zero.  DT (with
// DS): this pass also sums the bias-table gradient.  All three are compile
// time switches, so kernels without them carry none of their work.
// MX (with DS): MXFP8 attention ("Training GEM at LLM scale", section "Low
// Precision Flash Attention"): Q, K, V, dO arrive quantised, and P and dS are
// quantised in 32 x 32 blocks before the products that take them (dV, and dK
// with the dS chunks for dQ).  A compute warp's chunk of a block, 32 keys (its
// lanes) x 32 queries, is exactly one such block of the sequence's local
// positions; its scale comes from a warp-wide maximum.
template <int D, bool ACT, int BIAS, bool WIN, bool DS, bool DT, bool MX = false>
__global__ void __launch_bounds__(512, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO, const BwdArgs a) {
    using C = DkvCfg<D, ACT, BIAS>;
    static_assert(!(DS && WIN), "dS chunks are written for full attention only");
    static_assert(DS || !DT, "the bias gradient is summed here only with dS chunks");
    static_assert(!MX || (DS && !ACT && BIAS == kBiasNone && !DT), "MXFP8: softmax, dS chunks, no bias");
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
    uint64_t *st_full = qs_empty + C::NSQ;  // [2] per TMEM buffer (blocks alternate)
    uint64_t *p_full = st_full + 2;         // [2] per TMEM buffer, both compute groups arrive
    uint64_t *acc_full = p_full + 2;
    uint64_t *dv_empty = acc_full + 1;   // the output group has read dV (its columns are free)
    uint64_t *acc_done = dv_empty + 1;   // [2] per TMEM buffer: its block's dV / dK products finished
    uint64_t *drain = acc_done + 2;      // [2] per MMA-issuing thread
    uint64_t *dk_empty = drain + 2;      // the output group has read dK
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    float *sLD = reinterpret_cast<float *>(smem + C::OFF_LD);
    float *sdt = reinterpret_cast<float *>(smem + C::OFF_DT);
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
            mbar_init(&p_full[b], 8);  // both compute groups' warps
        }
        mbar_init(acc_full, 1);
        mbar_init(dv_empty, 4);
        mbar_init(dk_empty, 4);
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
    constexpr bool want_dt = DT && BIAS != kBiasNone;
    if constexpr (want_dt)
        for (int i = threadIdx.x; i < g.H * g.nb; i += blockDim.x) sdt[i] = 0.0f;
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

    const int wgi = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 7, 0);
    if (wgi == 0) {
        regs_to<C::REG_CTRL, 128>();
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
                        const int yq = (g.q_bcast ? t.q_loc0 : t.q_start) + i * C::BQ;  // shared Q: the local row
                        uint8_t *base = smem + C::OFF_Q + slot * 2 * C::Q_BYTES;
                        for (int kb = 0; kb < C::NKB; ++kb) {
                            tma_load_2d(base + kb * C::SUB_Q, &tmQ, &qs_full[slot], t.h * D + kb * 64, yq);
                            tma_load_2d(base + C::Q_BYTES + kb * C::SUB_Q, &tmDO, &qs_full[slot], t.h * D + kb * 64,
                                        y);
                        }
                    }
                }
            }
            if (lane == 0) {  // the last copy into every slot has landed before the CTA leaves
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
            if (t_local > 0) mbar_drain(kv_full, (t_local - 1) & 1);  // also after an abort
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
                    const uint32_t buf = ns & 1;  // TMEM buffer of block ns
                    if (ns >= 2 && !(ok = mbar_wait(&acc_done[buf], ((ns - 2) >> 1) & 1, err))) break;
                    const uint32_t slot = ns % C::NSQ;
                    if (!(ok = mbar_wait(&qs_full[slot], (ns / C::NSQ) & 1, err))) break;
                    tc_fence_after();
                    const int ncols = round_up16(min(C::BQ, ta.q_len - ia * C::BQ));
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint32_t qb = sQ + slot * 2 * C::Q_BYTES;
                    const uint64_t dqq = sdesc_sw128(qb, 16, 1024), ddo = sdesc_sw128(qb + C::Q_BYTES, 16, 1024);
                    const uint32_t dS = tmem + buf * 128, dDP = dS + 64;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t ao = (k >> 2) * C::SUB_KV + (k & 3) * 32;
                        const uint32_t bo = (k >> 2) * C::SUB_Q + (k & 3) * 32;
                        mma_bf16_ss(dS, sdesc_add(dk0, ao), sdesc_add(dqq, bo), idesc, k > 0);
                        mma_bf16_ss(dDP, sdesc_add(dv0, ao), sdesc_add(ddo, bo), idesc, k > 0);
                    }
                    mma_commit(&st_full[buf]);
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
            // A block's dV products go first: the output group hands the dV columns
            // back before the dK columns, so a tile's first dV products may start
            // while the previous tile's dK is still being read.
            const uint32_t idesc_acc = idesc_bf16(128, D, false, true);
            bool ok = true;
            TileStream tsb(g, tbeg, tend);
            Tile tb;
            uint32_t tb_n = 0, np = 0;
            while (ok && tsb.next(tb)) {
                if (!check_tile(g, tb, err, false)) continue;
                const int nbq = cdiv(tb.q_len, C::BQ);
                // the output group must have read dV of the previous tile
                if (!(ok = mbar_wait(dv_empty, (tb_n & 1) ^ 1, err))) break;
                for (int ib = 0; ib < nbq; ++ib, ++np) {
                    const uint32_t buf = np & 1;
                    if (!(ok = mbar_wait(&p_full[buf], (np >> 1) & 1, err))) break;
                    tc_fence_after();
                    const int ksteps = (min(C::BQ, tb.q_len - ib * C::BQ) + 15) >> 4;
                    const uint32_t slot = np % C::NSQ;
                    const uint32_t qb = sQ + slot * 2 * C::Q_BYTES;
                    const uint64_t bq0 = sdesc_sw128(qb, C::SUB_Q, 1024);
                    const uint64_t bdo0 = sdesc_sw128(qb + C::Q_BYTES, C::SUB_Q, 1024);
                    const uint32_t aP = tmem + buf * 128, aDS = aP + 64;
                    const uint32_t acc0 = ib > 0 ? 1u : 0u;
                    // Both product runs are fully unrolled with a guard per step: constant
                    // operand offsets and nothing else between two products, so this one
                    // thread issues them as fast as the tensor pipe takes them.
#pragma unroll
                    for (int k = 0; k < C::BQ / 16; ++k) {
                        if (k < ksteps) {
                            const uint32_t acc = k > 0 ? 1u : acc0;
                            const uint64_t bdo = sdesc_add(bdo0, k * 2048);
                            if (ACT) {  // hi at columns 16 k .. +7, lo at 16 k + 8 .. +15
                                mma_bf16_ts(tmem + C::COL_DV, aP + k * 16, bdo, idesc_acc, acc);
                                mma_bf16_ts(tmem + C::COL_DV, aP + k * 16 + 8, bdo, idesc_acc, 1u);
                            } else {
                                // 32-query chunk k / 2 keeps its bf16 pairs in its own first 16 columns
                                mma_bf16_ts(tmem + C::COL_DV, aP + (k >> 1) * 32 + (k & 1) * 8, bdo, idesc_acc, acc);
                            }
                        }
                    }
                    // ... and dK of the previous tile before the tile's first dK product
                    if (ib == 0 && !(ok = mbar_wait(dk_empty, (tb_n & 1) ^ 1, err))) break;
#pragma unroll
                    for (int k = 0; k < C::BQ / 16; ++k) {
                        if (k < ksteps) {
                            const uint32_t acc = k > 0 ? 1u : acc0;
                            const uint64_t bq = sdesc_add(bq0, k * 2048);
                            if (ACT) {
                                mma_bf16_ts(tmem + C::COL_DK, aDS + k * 16, bq, idesc_acc, acc);
                                mma_bf16_ts(tmem + C::COL_DK, aDS + k * 16 + 8, bq, idesc_acc, 1u);
                            } else {
                                mma_bf16_ts(tmem + C::COL_DK, aDS + (k >> 1) * 32 + (k & 1) * 8, bq, idesc_acc, acc);
                            }
                        }
                    }
                    mma_commit(&qs_empty[slot]);  // last reads of the Q / dO slot
                    mma_commit(&acc_done[buf]);   // the buffer may take block np + 2
                }
                if (!ok) break;
                mma_commit(acc_full);
                ++tb_n;
            }
            mma_commit(&drain[1]);
            mbar_drain(&drain[1], 0);
        }
    } else if (wgi < 3) {
        regs_to<C::REG_COMPUTE, 128>();
        // ------------------------------------------------------------ compute groups
        // One thread per key row (TMEM lane): P^T and dS^T of the group's query
        // blocks, 32 queries at a time, written as bf16 over the block's S^T and
        // dP^T columns (chunk c: columns 16c..16c+15, or 32c..32c+31 as hi / lo).
        const int grp = wgi - 1;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS0 = tmem + lane_base;  // buffer b of a block: S^T at 128 b, dP^T at 128 b + 64
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        uint32_t n0 = 0;
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
            // dS chunks: the tile's first chunk; block i of the tile is chunk ds0 + i
            int64_t ds0 = 0;
            if constexpr (DS) {
                const int lq = g.q_off[t.b + 1] - g.q_off[t.b], lk = g.kv_off[t.b + 1] - g.kv_off[t.b];
                const int nqb = cdiv(lq, C::BQ);
                ds0 = g.ds_base[t.b] + (static_cast<int64_t>(t.h) * cdiv(lk, C::BKV) + t.kv_loc0 / C::BKV) * nqb +
                      t.q_loc0 / C::BQ;
            }
            float dt_far = 0.0f;  // this row's dS in the last bias bucket, per tile
            auto blocks = [&](auto af) {
                constexpr int AF = decltype(af)::value;
                // every block of the tile; this group takes its 32-query chunk c = grp
                for (int i = 0; i < nq; ++i) {
                    const uint32_t n = n0 + i, b = n & 1;
                    if (!(ok = mbar_wait_warp(&st_full[b], (n >> 1) & 1, err))) return;
                    const int nvalid = min(C::BQ, t.q_len - i * C::BQ);
                    const int c = grp;
                    if (warp_live && c * 32 < nvalid) {
                        tc_fence_after();
                        const uint32_t tS = tS0 + b * 128, tDP = tS + 64;
                        const int qb = t.q_loc0 + i * C::BQ;
                        // [-lse log2 e | -Delta] of the block's queries (shared by all rows)
                        const float *ld = sLD + (n % C::NSQ) * 2 * C::BQ;
                        {
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
                            if constexpr (DS) {
                                // a row past the tile's keys adds nothing to dQ (its dK row is
                                // not stored, so zeroing it here changes no stored result)
                                if (row >= t.kv_len) {
#pragma unroll
                                    for (int k = 0; k < 32; ++k) dp[k] = MX ? (x[k] = 0.0f) : 0.0f;
                                }
                            }
                            if constexpr (MX) {  // this warp's 32 x 32 block of P and of dS
                                mx_qdq32(x, mx_exponent(warp_max_nonneg(amax32(x))));
                                mx_qdq32(dp, mx_exponent(warp_max_nonneg(amax32(dp))));
                            }
                            // bias-table gradient: dT[h, min(|i - j|, nb - 1)] += dS_ij; the far
                            // bucket in a register, the few near ones in shared memory
                            if constexpr (want_dt) {
                                if (row < t.kv_len) {
                                    const int i0 = qb + c * 32, nbm = g.nb - 1;
                                    const int dmin = kv_loc < i0 ? i0 - kv_loc : (kv_loc > i0 + 31 ? kv_loc - i0 - 31 : 0);
                                    if (dmin >= nbm) {
                                        dt_far += sum32(dp);
                                    } else {
#pragma unroll
                                        for (int k = 0; k < 32; ++k) {
                                            const int d = abs(kv_loc - (i0 + k));
                                            if (d >= nbm)
                                                dt_far += dp[k];
                                            else
                                                atomicAdd(&sdt[t.h * g.nb + d], dp[k]);
                                        }
                                    }
                                }
                            }
                            // this row's 64-byte piece of the block's dS chunk (plane p at
                            // 16 KB p): 16-byte pieces 4 c .. 4 c + 3 of the 128-byte row,
                            // XOR-swizzled by row.  Stored straight from the lanes, each
                            // 16-byte warp store touches 32 rows; staged (16 rows at a time
                            // through the warp's 1 KB of shared memory, pieces rotated by
                            // row pair so that neither side has bank conflicts), four lanes
                            // write one row's 64 contiguous bytes and a store touches 8 rows.
                            auto ds_store = [&](const uint32_t *wp, int plane) {
                                uint8_t *chunk = static_cast<uint8_t *>(g.ds) +
                                                 ((ds0 + i) * (ACT ? 2 : 1) + plane) * static_cast<int64_t>(kDsChunkBytes);
                                if constexpr (C::DS_STAGED) {
                                    const uint32_t sb = smem_u32(smem + C::OFF_DSS) +
                                                        static_cast<uint32_t>((grp * 4 + quad) * 1024);
                                    const int pc = lane & 3, jr = lane >> 2;  // piece, row within 8
#pragma unroll
                                    for (int r = 0; r < 2; ++r) {
                                        if ((lane >> 4) == r) {
                                            const int lr = lane & 15;
#pragma unroll
                                            for (int k = 0; k < 4; ++k)
                                                st_shared_v4(sb + lr * 64 + ((k ^ ((lr >> 1) & 3)) << 4), wp[4 * k],
                                                             wp[4 * k + 1], wp[4 * k + 2], wp[4 * k + 3]);
                                        }
                                        __syncwarp();
#pragma unroll
                                        for (int i2 = 0; i2 < 2; ++i2) {
                                            const int lr = 8 * i2 + jr;
                                            const uint4 v = ld_shared_v4(sb + lr * 64 + ((pc ^ ((lr >> 1) & 3)) << 4));
                                            const int grow = quad * 32 + 16 * r + lr;
                                            *reinterpret_cast<uint4 *>(chunk + grow * 128 +
                                                                       (((4 * c + pc) ^ (grow & 7)) << 4)) = v;
                                        }
                                        __syncwarp();  // the buffer is rewritten next
                                    }
                                } else {
                                    uint8_t *rowp = chunk + row * 128;
#pragma unroll
                                    for (int k = 0; k < 4; ++k)
                                        *reinterpret_cast<uint4 *>(rowp + (((4 * c + k) ^ (row & 7)) << 4)) =
                                            make_uint4(wp[4 * k], wp[4 * k + 1], wp[4 * k + 2], wp[4 * k + 3]);
                                }
                            };
                            if constexpr (ACT) {
                                uint32_t w[32];
                                pack_hilo32(x, w);
                                tmem_st32_u32(tS + 32 * c, w);
                                pack_hilo32(dp, w);
                                tmem_st32_u32(tDP + 32 * c, w);
                                if constexpr (DS) {  // hi words: 0..7, 16..23; lo words: 8..15, 24..31
                                    uint32_t hw[16], lw[16];
#pragma unroll
                                    for (int k = 0; k < 8; ++k) {
                                        hw[k] = w[k];
                                        hw[8 + k] = w[16 + k];
                                        lw[k] = w[8 + k];
                                        lw[8 + k] = w[24 + k];
                                    }
                                    ds_store(hw, 0);
                                    ds_store(lw, 1);
                                }
                            } else {
                                uint32_t w[16];
                                pack16(x, w);  // over the chunk's own first 16 columns
                                tmem_st16_u32(tS + 32 * c, w);
                                pack16(dp, w);
                                tmem_st16_u32(tDP + 32 * c, w);
                                if constexpr (DS) ds_store(w, 0);
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[b]);
                }
            };
            if (!ACT || g.act == kSilu) {
                blocks(std::integral_constant<int, kSilu>{});
            } else {
                blocks(std::integral_constant<int, kGeluTanh>{});
            }
            if constexpr (want_dt) {
                {  // the tile's far-bucket sums: one shared-memory add per warp
                    float f = dt_far;
#pragma unroll
                    for (int k = 16; k > 0; k >>= 1) f += __shfl_xor_sync(0xffffffffu, f, k);
                    if (lane == 0 && f != 0.0f) atomicAdd(&sdt[t.h * g.nb + g.nb - 1], f);
                    dt_far = 0.0f;
                }
            }
            if (!ok) break;
            n0 += nq;
        }
    } else {
        regs_to<C::REG_OUT, 128>();
        // ------------------------------------------------------------ output
        // One thread per key row reads dV and dK (times the score scale) from
        // TMEM, 64 columns per round trip.  bf16 outputs go out row-contiguous
        // through the warp's staging buffer.  dV's columns are handed back as
        // soon as they have been read (the next tile's dV products may start),
        // then dK's.
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
        // one accumulator (dV or dK, times mul) W = 64 columns at a time: read
        // (C::DRAIN_COLS per TMEM round trip), hand the columns back after the
        // last read, stage, store
        auto drain_acc = [&](uint32_t tacc, uint64_t *empty_bar, const OutDesc &o, float mul, bool has, int nrows,
                             int64_t r0, int h) {
            __nv_bfloat16 *dst0 = static_cast<__nv_bfloat16 *>(o.ptr) + r0 * o.ld + h * D;
            constexpr int RC = C::DRAIN_COLS;
#pragma unroll
            for (int h0 = 0; h0 < D; h0 += W) {
#pragma unroll
                for (int c0 = 0; c0 < W; c0 += RC) {
                    float v[RC];
                    if (has) {
                        if constexpr (RC == 64) {
                            tmem_ld32x2(tacc + h0 + c0, tacc + h0 + c0 + 32, sub32(v, 0), sub32(v, 1));
                        } else {
                            tmem_ld32(tacc + h0 + c0, v);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < RC; ++i) v[i] = 0.0f;
                    }
                    if (h0 + c0 + RC >= D) {  // every TMEM read of this accumulator is done
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(empty_bar);
                    }
                    if (mul != 1.0f) {
#pragma unroll
                        for (int i = 0; i < RC; i += 2) mul2(v[i], v[i + 1], mul, mul);
                    }
#pragma unroll
                    for (int c = 0; c < RC / 32; ++c) {
                        uint32_t w[16];
                        pack16(sub32(v, c), w);
                        stage_row32_bf16<W>(stg, lane, c0 + 32 * c, w);
                    }
                }
                __syncwarp();
                store_rows_bf16<W>(stg, lane, dst0 + h0, o.ld, nrows);
                __syncwarp();
            }
        };
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nq = cdiv(t.q_len, C::BQ);
            if (!(ok = mbar_wait_warp(acc_full, t_local & 1, err))) break;
            ++t_local;
            if (quad * 32 >= t.kv_len) {  // no row of this warp is stored
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(dv_empty);
                    mbar_arrive(dk_empty);
                }
                continue;
            }
            tc_fence_after();
            if (staged) {
                const int nrows = min(32, t.kv_len - quad * 32);
                const int64_t r0 = static_cast<int64_t>(t.kv_start) + quad * 32;
                drain_acc(tDV, dv_empty, a.dv, 1.0f, nq > 0, nrows, r0, t.h);
                drain_acc(tDK, dk_empty, a.dk, g.scale, nq > 0, nrows, r0, t.h);
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
                    if (lane == 0) {
                        mbar_arrive(dv_empty);
                        mbar_arrive(dk_empty);
                    }
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
    if constexpr (want_dt) {  // the CTA's share of the bias-table gradient
        for (int i = threadIdx.x; i < g.H * g.nb; i += blockDim.x)
            if (sdt[i] != 0.0f) atomicAdd(&a.dbias[i], sdt[i]);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace

// ============================================================================
// launcher
// ============================================================================
template <int D, bool ACT, int BIAS, bool WIN, bool DS, bool DT, bool MX = false>
static cudaError_t launch_dkdv_w(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = DkvCfg<D, ACT, BIAS>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(dkdv_kernel<D, ACT, BIAS, WIN, DS, DT, MX>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    dkdv_kernel<D, ACT, BIAS, WIN, DS, DT, MX><<<n_ctas, 512, C::SMEM_ALLOC, st>>>(tm.q, tm.k, tm.v, tm.dout, a);
    return cudaGetLastError();
}

// the variant a launch takes: window, dS chunks (a.g.ds set), bias gradient with
// them, MXFP8 (softmax, dS chunks, no bias)
template <int D, bool ACT, int BIAS>
static cudaError_t launch_dkdv_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (a.g.mxfp8) {
        if constexpr (!ACT && BIAS == kBiasNone) {
            if (a.g.ds == nullptr || a.g.window > 0 || a.dbias != nullptr) return cudaErrorInvalidValue;
            return launch_dkdv_w<D, false, kBiasNone, false, true, false, true>(tm, a, n_ctas, st);
        }
        return cudaErrorInvalidValue;
    }
    if (a.g.ds != nullptr) {
        if (a.g.window > 0) return cudaErrorInvalidValue;
        if constexpr (BIAS != kBiasNone) {
            if (a.dbias != nullptr) return launch_dkdv_w<D, ACT, BIAS, false, true, true>(tm, a, n_ctas, st);
        }
        return launch_dkdv_w<D, ACT, BIAS, false, true, false>(tm, a, n_ctas, st);
    }
    return a.g.window > 0 ? launch_dkdv_w<D, ACT, BIAS, true, false, false>(tm, a, n_ctas, st)
                          : launch_dkdv_w<D, ACT, BIAS, false, false, false>(tm, a, n_ctas, st);
}

template <int D, bool ACT>
static cudaError_t launch_dkdv_b(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    switch (bias_form(a.g)) {
    case kBiasNone: return launch_dkdv_t<D, ACT, kBiasNone>(tm, a, n_ctas, st);
    case kBiasExt: return launch_dkdv_t<D, ACT, kBiasExt>(tm, a, n_ctas, st);
    default: return launch_dkdv_t<D, ACT, kBiasTable>(tm, a, n_ctas, st);
    }
}

cudaError_t launch_bwd_dkdv(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (D == 128)
        return act ? launch_dkdv_b<128, true>(tm, a, n_ctas, st) : launch_dkdv_b<128, false>(tm, a, n_ctas, st);
    if (D == 64) return act ? launch_dkdv_b<64, true>(tm, a, n_ctas, st) : launch_dkdv_b<64, false>(tm, a, n_ctas, st);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
