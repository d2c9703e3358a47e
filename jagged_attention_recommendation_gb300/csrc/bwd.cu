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
//   warpgroups 1, 2  two compute groups, one thread per tile row (TMEM lane).
//                The CTA numbers its blocks n across tile boundaries; block n
//                uses TMEM buffer n % 2. Both groups take every block, group g
//                its 32-column half g (keys in the dQ pass, queries in the dK/dV
//                pass); a block's hand-off waits for all eight compute warps.
//   warpgroup 3  output group: reads the accumulators and writes the rows.
// A block's two products land in its buffer's TMEM columns; the compute groups
// overwrite them in place with bf16 dS (and P^T), each 32-column chunk in its
// own columns, and the accumulating product reads that operand from TMEM.  Two issuing threads, because any wait of the
// issuing thread (an mbarrier, a shared-memory load, a named barrier) holds it
// until its queued MMAs have drained, which leaves the tensor pipe idle; with
// two, one thread's products run while the other waits.  Block n + 2 reuses
// block n's columns, so the score-side issuer waits for block n's accumulating
// product to finish (an mbarrier committed by the other thread) before it
// issues block n + 2; the accumulators have a single issuer, so their
// summation order is fixed and results are reproducible.
#include "bwd_common.cuh"

namespace jattn {
using namespace dev;
namespace {

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
    // the CTA's share of the bias-table gradient [H, nb] (with a bias)
    static constexpr uint32_t OFF_DT = OFF_BEXT + (BIAS == kBiasExt ? kMaxBiasExtFloats * 4 : 0);
    static constexpr uint32_t SMEM = OFF_DT + (BIAS != kBiasNone ? kMaxBiasFloats * 4 : 0);
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    // group g: S at 128 g, dP at 128 g + 64 (dS over S); dQ[b] at 256 + b D
    static constexpr uint32_t COL_DQ = 256;
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "operand alignment");
    static_assert(COL_DQ + 2 * D <= TMEM_COLS, "TMEM budget");
};

// WIN: sliding window on; DT: bias-table gradient wanted (both compile time, so
// kernels without them carry none of their work)
template <int D, bool ACT, int BIAS, bool WIN, bool DT>
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
    uint64_t *s_full = v_empty + C::NSV;  // [2] per TMEM buffer (blocks alternate)
    uint64_t *ds_full = s_full + 2;       // [2] per TMEM buffer, both compute groups arrive
    uint64_t *dq_full = ds_full + 2;      // [2] per dQ buffer
    uint64_t *dq_empty = dq_full + 2;     // [2] per dQ buffer
    uint64_t *dq_done = dq_empty + 2;     // [2] per TMEM buffer: its block's dQ product finished
    uint64_t *drain = dq_done + 2;        // [2] per MMA-issuing thread
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    float *sdt = reinterpret_cast<float *>(smem + C::OFF_DT);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&qd_full[s], 1);
            mbar_init(&qd_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&ds_full[s], 8);  // both compute groups' warps
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
            {  // the last copy into every slot has landed before the CTA leaves (also after an abort)
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
                const int qrow = g.q_bcast ? t.q_loc0 : t.q_start;  // shared Q: the local row
                for (int kb = 0; kb < C::NKB; ++kb) {
                    tma_load_2d(base + kb * C::SUB_Q, &tmQ, &qd_full[s], t.h * D + kb * 64, qrow);
                    tma_load_2d(base + C::Q_BYTES + kb * C::SUB_Q, &tmDO, &qd_full[s], t.h * D + kb * 64, t.q_start);
                }
                ++t_local;
            }
            // the last copy into each slot has landed before the CTA leaves
            for (uint32_t i = (t_local > 2 ? t_local - 2 : 0); i < t_local; ++i)
                mbar_drain(&qd_full[i & 1], (i >> 1) & 1);
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
                    const uint32_t buf = ns & 1;  // TMEM buffer of block ns
                    if (ns >= 2 && !(ok = mbar_wait(&dq_done[buf], ((ns - 2) >> 1) & 1, err))) break;
                    const uint32_t ks = ns % C::NSK, vs = ns % C::NSV;
                    if (!(ok = mbar_wait(&k_full[ks], (ns / C::NSK) & 1, err))) break;
                    if (!(ok = mbar_wait(&v_full[vs], (ns / C::NSV) & 1, err))) break;
                    tc_fence_after();
                    const int ncols = round_up16(min(C::BN, ta.kv_len - ja * C::BN));
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint64_t dk0 = sdesc_sw128(sK + ks * C::KV_BYTES, 16, 1024);
                    const uint64_t dv0 = sdesc_sw128(sV + vs * C::KV_BYTES, 16, 1024);
                    const uint32_t dS = tmem + buf * 128, dDP = dS + 64;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t ao = (k >> 2) * C::SUB_Q + (k & 3) * 32;
                        const uint32_t bo = (k >> 2) * C::SUB_KV + (k & 3) * 32;
                        mma_bf16_ss(dS, sdesc_add(dq0, ao), sdesc_add(dk0, bo), idesc, k > 0);
                        mma_bf16_ss(dDP, sdesc_add(ddo0, ao), sdesc_add(dv0, bo), idesc, k > 0);
                    }
                    mma_commit(&s_full[buf]);
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
                    const uint32_t buf = np & 1;
                    if (!(ok = mbar_wait(&ds_full[buf], (np >> 1) & 1, err))) break;
                    tc_fence_after();
                    const int ksteps = (min(C::BN, tb.kv_len - jb * C::BN) + 15) >> 4;
                    const uint32_t ks = np % C::NSK;
                    const uint64_t bd0 = sdesc_sw128(sK + ks * C::KV_BYTES, C::SUB_KV, 1024);
                    const uint32_t aS = tmem + buf * 128;
                    const uint32_t acc0 = jb > 0 ? 1u : 0u;
                    // fully unrolled with a guard per step (constant operand offsets), so
                    // the products issue as fast as the tensor pipe takes them
#pragma unroll
                    for (int k = 0; k < C::BN / 16; ++k) {
                        if (k < ksteps) {
                            const uint64_t bd = sdesc_add(bd0, k * 2048);
                            const uint32_t acc = k > 0 ? 1u : acc0;
                            if (ACT) {  // hi at columns 16 k .. +7, lo at 16 k + 8 .. +15
                                mma_bf16_ts(dq, aS + k * 16, bd, idesc_dq, acc);
                                mma_bf16_ts(dq, aS + k * 16 + 8, bd, idesc_dq, 1u);
                            } else {
                                // 32-key chunk k / 2 keeps its bf16 pairs in its own first 16 columns
                                mma_bf16_ts(dq, aS + (k >> 1) * 32 + (k & 1) * 8, bd, idesc_dq, acc);
                            }
                        }
                    }
                    mma_commit(&k_empty[ks]);     // S and dQ were the K slot's readers
                    mma_commit(&dq_done[buf]);    // the buffer may take block np + 2
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
        const uint32_t tS0 = tmem + lane_base;  // buffer b of a block: S at 128 b, dP at 128 b + 64
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        uint32_t n0 = 0;
        float dt_far = 0.0f;  // this row's dS in the last bias bucket, per tile
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
            float lse2 = 0.0f, dlt = 0.0f;  // log2 units / Delta of this row
            if (!ACT && row_ok && nkv > 0) {
                const int64_t idx = static_cast<int64_t>(t.h) * g.Tq + t.q_start + row;
                lse2 = a.lse[idx] * kLog2e;
                dlt = a.delta[idx];
            }
            auto blocks = [&](auto af) {
                constexpr int AF = decltype(af)::value;
                // every block of the tile; this group takes its 32-key chunk c = grp
                for (int j = 0; j < nkv; ++j) {
                    const uint32_t n = n0 + j, b = n & 1;
                    if (!(ok = mbar_wait_warp(&s_full[b], (n >> 1) & 1, err))) return;
                    const int nvalid = min(C::BN, t.kv_len - j * C::BN);
                    const int c = grp;
                    if (warp_live && c * 32 < nvalid) {
                        tc_fence_after();
                        const uint32_t tS = tS0 + b * 128, tDP = tS + 64;
                        const int kvb = t.kv_loc0 + j * C::BN;
                        {
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
                            // bias-table gradient: dT[h, min(|i - j|, nb - 1)] += dS_ij; the
                            // far bucket in a register, the few near ones in shared memory
                            if constexpr (want_dt) {
                                if (row_ok) {
                                    const int j0 = kvb + c * 32, nbm = g.nb - 1;
                                    const int dmin = q_loc < j0 ? j0 - q_loc : (q_loc > j0 + 31 ? q_loc - j0 - 31 : 0);
                                    if (dmin >= nbm) {
                                        dt_far += sum32(x);
                                    } else {
#pragma unroll
                                        for (int i = 0; i < 32; ++i) {
                                            const int d = abs(q_loc - (j0 + i));
                                            if (d >= nbm)
                                                dt_far += x[i];
                                            else
                                                atomicAdd(&sdt[t.h * g.nb + d], x[i]);
                                        }
                                    }
                                }
                            }
                            if constexpr (ACT) {
                                uint32_t w[32];
                                pack_hilo32(x, w);
                                tmem_st32_u32(tS + 32 * c, w);
                            } else {
                                uint32_t w[16];
                                pack16(x, w);
                                tmem_st16_u32(tS + 32 * c, w);  // over the chunk's own first 16 columns
                            }
                        }
                        tmem_wait_st();
                        tc_fence_before();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ds_full[b]);
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
template <int D, bool ACT, int BIAS, bool WIN, bool DT>
static cudaError_t launch_dq_w(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    using C = DqCfg<D, ACT, BIAS>;
    static SmemOnce done;
    cudaError_t e = ensure_smem(dq_kernel<D, ACT, BIAS, WIN, DT>, C::SMEM_ALLOC, done);
    if (e != cudaSuccess || n_ctas <= 0) return e;
    dq_kernel<D, ACT, BIAS, WIN, DT><<<n_ctas, 512, C::SMEM_ALLOC, st>>>(tm.q, tm.k, tm.v, tm.dout, a);
    return cudaGetLastError();
}

template <int D, bool ACT, int BIAS, bool DT>
static cudaError_t launch_dq_d(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    return a.g.window > 0 ? launch_dq_w<D, ACT, BIAS, true, DT>(tm, a, n_ctas, st)
                          : launch_dq_w<D, ACT, BIAS, false, DT>(tm, a, n_ctas, st);
}

template <int D, bool ACT, int BIAS>
static cudaError_t launch_dq_t(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if constexpr (BIAS != kBiasNone) {
        if (a.dbias != nullptr) return launch_dq_d<D, ACT, BIAS, true>(tm, a, n_ctas, st);
    }
    return launch_dq_d<D, ACT, BIAS, false>(tm, a, n_ctas, st);
}

template <int D, bool ACT>
static cudaError_t launch_dq_b(const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    switch (bias_form(a.g)) {
    case kBiasNone: return launch_dq_t<D, ACT, kBiasNone>(tm, a, n_ctas, st);
    case kBiasExt: return launch_dq_t<D, ACT, kBiasExt>(tm, a, n_ctas, st);
    default: return launch_dq_t<D, ACT, kBiasTable>(tm, a, n_ctas, st);
    }
}

cudaError_t launch_bwd_dq(int D, bool act, const TmapSet &tm, const BwdArgs &a, int n_ctas, cudaStream_t st) {
    if (D == 128) return act ? launch_dq_b<128, true>(tm, a, n_ctas, st) : launch_dq_b<128, false>(tm, a, n_ctas, st);
    if (D == 64) return act ? launch_dq_b<64, true>(tm, a, n_ctas, st) : launch_dq_b<64, false>(tm, a, n_ctas, st);
    return cudaErrorInvalidValue;
}

}  // namespace jattn
