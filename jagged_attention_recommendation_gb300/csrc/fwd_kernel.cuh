// fwd_kernel.cuh -- jagged attention forward kernel for sm_103a (the
// launchers are in fwd.cu and fwd_rope.cu).
//
// "Training GEM at LLM scale", section "Jagged Sequence Flash Attention":
// FlashAttention directly on jagged tensors (no padding), with custom biases and
// asymmetric query/key-value lengths, TMA loads, warp specialisation and a
// persistent schedule; section "Generalized Dot-Product Attention (GDPA)": the
// softmax replaced by GELU / SiLU with no normalisation (no max, no rescale);
// section "BlockAttention": each 64-token query block sees only its own block.
//
// One CTA = 16 warps (four warpgroups), persistent over the tiles the planner
// gave it.  A tile is 128 query rows of one (sequence, head) against all of its
// keys, in blocks of 128 keys.  The CTA numbers the key blocks of its tiles
// consecutively (block n), across tile boundaries.
//   warp 0      TMA producer for K and V (128-row tiles) through NST-deep rings
//               with separate release barriers: a K slot refills as soon as
//               its S = Q K^T is done, a V slot once its P V is done.
//   warp 1      allocates TMEM; one thread issues every P V product.
//   warp 2      TMA producer for Q, double-buffered so the next tile's rows
//               arrive while the current tile runs.
//   warp 3      one thread issues every S = Q K^T.
//   warps 4-7   softmax group 0: keys 0..63 of every key block.
//   warps 8-11  softmax group 1: keys 64..127 of every key block.
//   warps 12-15 output group: merges the two groups' partial results of a
//               tile, O / l -> global, lse.
// Each softmax group runs its own online softmax (row max m_g, row sum l_g)
// over its half of every block of a tile into its own TMEM accumulator O_g, so
// the groups never wait for each other and both have work on every block but
// a last one of at most 64 keys.  The output group combines
//   O = (2^(m_0-m) O_0 + 2^(m_1-m) O_1) / (2^(m_0-m) l_0 + 2^(m_1-m) l_1),
// m = max(m_0, m_1), over the groups that saw keys in the tile (in the
// activation modes simply O_0 + O_1).
// P never touches shared memory: the softmax writes it as bf16 over the
// group's own score columns in TMEM and P V reads it from there (the A operand
// of tcgen05.mma may live in TMEM).  Two threads issue the products, because
// any wait of an issuing thread (an mbarrier, a shared-memory load) holds it
// until its queued MMAs have drained, which idles the tensor pipe; with two,
// one thread's products run while the other waits.  The score columns are
// double-buffered by block parity: S_{n+2} overwrites P_n, so the S issuer
// waits for PV_n to finish (an mbarrier committed by the P V issuer) before it
// issues S_{n+2}, and S_{n+1} is computed during the softmax of block n.
// Rows past a sequence's end are loaded (they belong to the next sequence or
// are zero-filled past the tensor end) but masked as keys and never stored as
// queries; the last key block of a sequence runs a narrower MMA (N rounded up
// to 16), so no tensor-core work is spent on whole masked column groups.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#define JATTN_INLINE_WAITS 1
#include "attn.cuh"
#include "kernels.h"

namespace jattn {
using namespace dev;

// How the relative-position bias reaches the scores.
enum : int {
    kBiasNone = 0,
    kBiasExt = 1,    // reflected per-head table in shared memory (contiguous windows)
    kBiasTable = 2,  // the [H, nb] table in shared memory, bucket computed per element
};

template <int D, bool ACT, int BIAS, bool ROPE = false>
struct FwdCfg {
    static constexpr int BM = 128, BN = 128;
    static constexpr int NKB = D / 64;  // 64-column sub-tiles along D
    // depth of the K ring and of the V ring (D = 64 with RoPE: 2, to make room
    // for the staged rotation tables)
    static constexpr int NST = (D == 64 && !ROPE) ? 4 : 2;
    // RoPE with D = 64: the cos / sin rows of a tile's query positions travel
    // with its Q (one slot per Q buffer); D = 128 reads them from global memory
    static constexpr bool TAB = ROPE && D == 64;
    static constexpr uint32_t TAB_BYTES = TAB ? 2 * BM * (D / 2) * 4 : 0;  // cos + sin rows of one slot
    static constexpr uint32_t SUB_Q = BM * 128;    // bytes of one 64-column sub-tile
    static constexpr uint32_t SUB_KV = BN * 128;
    static constexpr uint32_t Q_BYTES = BM * D * 2;
    static constexpr uint32_t KV_BYTES = BN * D * 2;
    // q_full[2], q_empty[2], k_full[NST], k_empty[NST], v_full[NST], v_empty[NST],
    // s_full[2], p_full[2], o_full[2], o_empty[2], l_full[2], pv_done[2], drain[2]
    // (RoPE: q_rot[2], k_rot[NST])
    static constexpr int NBAR = 4 + 4 * NST + 2 + 2 + 2 + 2 + 2 + 2 + 2 + (ROPE ? 2 + NST : 0);
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + 2 * Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NST * KV_BYTES;
    static constexpr uint32_t OFF_TAB = OFF_V + NST * KV_BYTES;  // [2][cos | sin][BM][D/2] float32
    static constexpr uint32_t OFF_BAR = OFF_TAB + 2 * TAB_BYTES;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr uint32_t OFF_BIAS = OFF_MISC + 16;  // [H, nb] table (kBiasTable)
    static constexpr uint32_t OFF_BEXT = OFF_BIAS + (BIAS == kBiasTable ? kMaxBiasFloats * 4 : 0);
    static constexpr uint32_t OFF_ROWS = OFF_BEXT + (BIAS == kBiasExt ? kMaxBiasExtFloats * 4 : 0);
    // D = 128: per output warp 32 rows x 64 bf16 of staging for row-contiguous
    // stores (D = 64 and RoPE keep per-row stores: their output registers do not
    // fit both)
    static constexpr bool STAGE_OUT = D == 128 && !ROPE;
    static constexpr int STG_W = 64;
    static constexpr uint32_t OFF_STG = (OFF_ROWS + (ACT ? 0 : 2 * 4 * 128 * 4) + 127) & ~127u;  // after [2][m0 l0 m1 l1][128]
    static constexpr uint32_t SMEM = OFF_STG + (STAGE_OUT ? 4 * 32 * STG_W * 2 : 0);
    static constexpr int THREADS = 512;
    static constexpr uint32_t SMEM_ALLOC = SMEM + 1024;  // slack to align the base to 1024
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 0;    // S_g / P_g: BN columns per group
    static constexpr uint32_t COL_O = 256;  // O_g: D columns per group
    // D = 64: two sets of O_0 / O_1 by tile parity, so the next tile's P V
    // products need not wait for the output group to read this tile's
    static constexpr int OB = (D == 64) ? 2 : 1;
    // registers per thread after the split (launch: 512 threads x 128)
    // (the staged D = 128 softmax output without a bias needs 120 in the output
    // group; its softmax fits in 168)
    static constexpr bool WIDE_OUT = STAGE_OUT && !ACT && BIAS == kBiasNone;
    static constexpr uint32_t REG_CTRL = 56, REG_SOFTMAX = WIDE_OUT ? 168 : 176, REG_OUT = WIDE_OUT ? 120 : 104;
    static_assert(REG_CTRL * 128 + REG_SOFTMAX * 256 + REG_OUT * 128 <= 128 * 512, "register split");
    static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
    static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "operand alignment");
    static_assert(COL_O + OB * 2 * D <= TMEM_COLS, "TMEM budget");
};

// WIN: sliding window on (a compile-time switch, so that kernels without one
// carry no band test in their softmax passes).  ROPE: rotary position
// embedding of Q and K ("Training GEM at LLM scale", section "BlockAttention")
// in shared memory as the tiles arrive: the output warpgroup rotates each
// BlockAttention tile's Q rows and its one K block two tiles ahead, before the
// S issuer may use them (q_rot / k_rot).  STALL: a test build only (one
// instantiation, launched by jattn_test_fwd_stall): before its first product
// the S issuer waits on a barrier that nothing completes at that point, so
// the bounded wait runs out and the kernel takes its error path (status word,
// abort flag, drained copies, TMEM freed) on a real launch.
// MX: MXFP8 attention ("Training GEM at LLM scale", section "Low Precision
// Flash Attention"; softmax without bias, window or RoPE): Q, K, V arrive
// already quantised (their MXFP8 values, bf16), the running row max is kept
// as an integer in log2 units, so every rescale is an exact power of two,
// and each row's P is quantised online in its 32-key chunks (one E8M0 scale
// per chunk from the chunk's largest value) after the row sum has taken the
// unquantised values.
// TP: tile-parallel, for batches whose every query tile meets at most one
// 128-key block (short key sequences; BlockAttention): softmax group g takes
// the whole block of the CTA's tiles of parity g, into its own O_g, so the two
// groups run two tiles at once instead of splitting every block's keys (half
// of which are masked in such tiles), and a tile's P V never waits for the
// previous tile's output (the other group's O).  Every tile counts as one
// block, also a tile without keys, so that block and tile numbers agree.
template <int D, bool ACT, int BIAS, bool WIN, bool ROPE = false, bool STALL = false, bool MX = false,
          bool TP = false>
__global__ void __launch_bounds__(512, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
    using C = FwdCfg<D, ACT, BIAS, ROPE>;
    static_assert(!MX || (!ACT && BIAS == kBiasNone && !WIN && !ROPE), "MXFP8: softmax without bias, window, RoPE");
    static_assert(!TP || (!ACT && !WIN && !ROPE && !MX && !STALL), "tile-parallel: plain softmax");
    // block count of a tile (tile-parallel: exactly one)
    auto nblocks = [](const Tile &x) { return TP ? 1 : cdiv(x.kv_len, C::BN); };
    const int win = WIN ? a.g.window : 0;  // |i - j| < win, 0 = no window
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *q_full = bars + 0;   // [2]
    uint64_t *q_empty = bars + 2;  // [2]
    uint64_t *k_full = bars + 4;
    uint64_t *k_empty = k_full + C::NST;
    uint64_t *v_full = k_empty + C::NST;
    uint64_t *v_empty = v_full + C::NST;
    uint64_t *s_full = v_empty + C::NST;  // [2] per score buffer (blocks alternate)
    uint64_t *p_full = s_full + 2;        // [2] per score buffer, both softmax groups arrive
    uint64_t *o_full = p_full + 2;   // [2] per tile parity: the tile's last P V is done
    uint64_t *o_empty = o_full + 2;  // [2] per tile parity
    uint64_t *l_full = o_empty + 2;  // [2] per tile parity
    uint64_t *pv_done = l_full + 2;  // [2] per score buffer: its block's P V finished
    uint64_t *drain = pv_done + 2;   // [2] per MMA-issuing thread
    uint64_t *q_rot = drain + 2;     // [2] RoPE: Q slot rotated
    uint64_t *k_rot = q_rot + 2;     // [NST] RoPE: K slot rotated
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    float *sbias = reinterpret_cast<float *>(smem + C::OFF_BIAS);
    float *sext = reinterpret_cast<float *>(smem + C::OFF_BEXT);
    float *srows = reinterpret_cast<float *>(smem + C::OFF_ROWS);  // [tile & 1][m0 | l0 | m1 | l1][row]

    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], TP ? 4 : 8);  // both softmax groups' warps (TP: the tile's group)
            mbar_init(&o_empty[s], 4);
            mbar_init(&l_full[s], TP ? 4 : 8);
            mbar_init(&pv_done[s], 1);
            mbar_init(&drain[s], 1);
        }
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        if (ROPE) {  // the output warpgroup's four warps
            for (int s = 0; s < 2; ++s) mbar_init(&q_rot[s], 4);
            for (int s = 0; s < C::NST; ++s) mbar_init(&k_rot[s], 4);
        }
        for (int s = 0; s < 2; ++s) mbar_init(&o_full[s], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    // softmax works in log2 units: the bias goes in times log2(e)
    if (BIAS == kBiasTable) stage_bias(g, sbias, ACT ? 1.0f : kLog2e);
    if (BIAS == kBiasExt) stage_bias_ext(g, sext, ACT ? 1.0f : kLog2e);
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const ErrCtx err{g.status, abort_flag, g.wait_ns};
    const int tbeg = g.cta_begin[blockIdx.x];
    const int tend = g.cta_begin[blockIdx.x + 1];

    // Role of this warp's warpgroup, warp-uniform by construction; each role
    // sets its warpgroup's register budget first.
    const int wgi = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) >> 7, 0);
    if (wgi == 0) {
        regs_release<C::REG_CTRL>();
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------------- K/V producer
            // Issue order per key block: K_n, then V_{n-1}, so a V slot that still
            // waits for its P V never holds back the next S = Q K^T.
            uint32_t k_it = 0, v_it = 0;
            bool ok = true;
            bool v_pending = false;
            int v_col = 0, v_row = 0;
            auto load_v = [&]() -> bool {
                const uint32_t slot = v_it % C::NST, use = v_it / C::NST;
                if (!mbar_wait(&v_empty[slot], (use & 1) ^ 1, err)) return false;
                mbar_arrive_expect_tx(&v_full[slot], C::KV_BYTES);
                for (int kb = 0; kb < C::NKB; ++kb)
                    tma_load_2d(smem + C::OFF_V + slot * C::KV_BYTES + kb * C::SUB_KV, &tmV, &v_full[slot],
                                v_col + kb * 64, v_row);
                ++v_it;
                v_pending = false;
                return true;
            };
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, true)) continue;
                const int nkv = nblocks(t);
                for (int j = 0; j < nkv; ++j) {
                    const uint32_t slot = k_it % C::NST, use = k_it / C::NST;
                    if (!(ok = mbar_wait(&k_empty[slot], (use & 1) ^ 1, err))) break;
                    mbar_arrive_expect_tx(&k_full[slot], C::KV_BYTES);
                    const int y = t.kv_start + j * C::BN;
                    for (int kb = 0; kb < C::NKB; ++kb)
                        tma_load_2d(smem + C::OFF_K + slot * C::KV_BYTES + kb * C::SUB_KV, &tmK, &k_full[slot],
                                    t.h * D + kb * 64, y);
                    ++k_it;
                    if (v_pending && !(ok = load_v())) break;
                    v_pending = true;
                    v_col = t.h * D;
                    v_row = y;
                }
            }
            if (ok && v_pending) ok = load_v();
            // Do not leave the CTA with copies still landing in shared memory:
            // wait for the last copy into every slot.  In a normal run the
            // consumers have waited for them all; after an abort (here or in
            // another role) nobody else may.
            {
                for (uint32_t s = 0; s < C::NST && s < k_it; ++s) {
                    const uint32_t last = k_it - 1 - ((k_it - 1 - s) % C::NST);  // last load into slot s
                    mbar_drain(&k_full[last % C::NST], (last / C::NST) & 1);
                }
                for (uint32_t s = 0; s < C::NST && s < v_it; ++s) {
                    const uint32_t last = v_it - 1 - ((v_it - 1 - s) % C::NST);
                    mbar_drain(&v_full[last % C::NST], (last / C::NST) & 1);
                }
            }
        } else if (warp == 2 && lane == 0) {
            // -------------------------------------------------------- Q producer
            uint32_t t_local = 0;
            bool ok = true;
            TileStream ts(g, tbeg, tend);
            Tile t;
            while (ok && ts.next(t)) {
                if (!check_tile(g, t, err, false)) continue;
                const uint32_t s = t_local & 1, use = t_local >> 1;
                if (!(ok = mbar_wait(&q_empty[s], (use & 1) ^ 1, err))) break;
                // RoPE with D = 64: the cos / sin rows of the tile's query positions
                // travel with Q
                const uint32_t tab = C::TAB ? static_cast<uint32_t>(t.q_len) * (D / 2) * 4 : 0u;
                mbar_arrive_expect_tx(&q_full[s], C::Q_BYTES + 2 * tab);
                const int qrow = g.q_bcast ? t.q_loc0 : t.q_start;  // shared Q: the local row
                for (int kb = 0; kb < C::NKB; ++kb)
                    tma_load_2d(smem + C::OFF_Q + s * C::Q_BYTES + kb * C::SUB_Q, &tmQ, &q_full[s],
                                t.h * D + kb * 64, qrow);
                if (C::TAB) {
                    const int64_t r0 = static_cast<int64_t>(t.q_loc0) * (D / 2);
                    uint8_t *dst = smem + C::OFF_TAB + s * C::TAB_BYTES;
                    bulk_load(dst, g.rope_cos + r0, tab, &q_full[s]);
                    bulk_load(dst + C::TAB_BYTES / 2, g.rope_sin + r0, tab, &q_full[s]);
                }
                ++t_local;
            }
            // the last copy into each slot has landed before the CTA leaves
            for (uint32_t i = (t_local > 2 ? t_local - 2 : 0); i < t_local; ++i)
                mbar_drain(&q_full[i & 1], (i >> 1) & 1);
        } else if (warp == 3 && lane == 0) {
            // -------------------------------------------------------- S issuer
            // Two issuing threads keep the tensor pipe fed (a thread's own waits
            // stall its queued MMAs): this one issues every S = Q K^T, the other
            // every P V.  Block n (the CTA's blocks in order, across tiles) reuses
            // the score columns of block n - 2, its group's previous block, once
            // that block's P V has finished.  So when the softmax sees S_n, its
            // group's O already holds all of the group's earlier blocks, and a
            // rescale of O may touch it.
            bool ok = true;
            // test build: drain[0] completes only when this thread commits to it
            // after its loop, so this wait runs out (bounded by g.wait_ns)
            if constexpr (STALL) ok = mbar_wait(&drain[0], 0, err);
            TileStream tsa(g, tbeg, tend);
            Tile ta;
            uint32_t ta_n = 0, ns = 0;
            while (ok && tsa.next(ta)) {
                if (!check_tile(g, ta, err, false)) continue;
                const int na = nblocks(ta);
                const uint32_t qs = ta_n & 1;
                if (!(ok = mbar_wait(ROPE ? &q_rot[qs] : &q_full[qs], (ta_n >> 1) & 1, err))) break;
                const uint64_t ad0 = sdesc_sw128(sQ + qs * C::Q_BYTES, 16, 1024);
                for (int ja = 0; ja < na; ++ja, ++ns) {
                    const uint32_t buf = ns & 1;  // score buffer of block ns
                    if (ns >= 2 && !(ok = mbar_wait(&pv_done[buf], ((ns - 2) >> 1) & 1, err))) break;
                    const uint32_t slot = ns % C::NST, use = ns / C::NST;
                    if (!(ok = mbar_wait(ROPE ? &k_rot[slot] : &k_full[slot], use & 1, err))) break;
                    tc_fence_after();
                    const int ncols = round_up16(max(1, min(C::BN, ta.kv_len - ja * C::BN)));  // >= 16
                    const uint32_t idesc = idesc_bf16(128, ncols, false, false);
                    const uint64_t bd0 = sdesc_sw128(sK + slot * C::KV_BYTES, 16, 1024);
                    const uint32_t dS = tmem + C::COL_S + buf * C::BN;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_bf16_ss(dS, sdesc_add(ad0, (ks >> 2) * C::SUB_Q + (ks & 3) * 32),
                                    sdesc_add(bd0, (ks >> 2) * C::SUB_KV + (ks & 3) * 32), idesc, ks > 0);
                    mma_commit(&s_full[buf]);
                    mma_commit(&k_empty[slot]);
                }
                if (!ok) break;
                mma_commit(&q_empty[qs]);  // the last read of this Q slot is in flight
                ++ta_n;
            }
            // every MMA this thread issued is done before TMEM is released
            mma_commit(&drain[0]);
            mbar_drain(&drain[0], 0);
        } else if (warp == 1 && lane == 0) {
            // -------------------------------------------------------- P V issuer
            // O_g (+)= P_g V_g for softmax group g's 64 keys of every block, P
            // (bf16; activation: hi and lo parts) read from TMEM; one thread, so
            // the accumulation order is fixed.
            const uint32_t idesc_pv = idesc_bf16(128, D, false, true);
            bool ok = true;
            TileStream tsb(g, tbeg, tend);
            Tile tb;
            uint32_t tb_n = 0, np = 0;
            while (ok && tsb.next(tb)) {
                if (!check_tile(g, tb, err, false)) continue;
                const int nbk = nblocks(tb);
                // the output group must have read tile tb_n - 1 before O_0 / O_1 are
                // reused (a tile without keys hands over all-zero rows in order)
                // (D = 64, or tile-parallel: two O sets, so the tile before the previous one)
                constexpr uint32_t OBX = TP ? 2 : C::OB;
                if (tb_n >= OBX && !(ok = mbar_wait(&o_empty[(tb_n - OBX) & 1], ((tb_n - OBX) >> 1) & 1, err)))
                    break;
                for (int jb = 0; jb < nbk; ++jb, ++np) {
                    const uint32_t buf = np & 1;
                    if (!(ok = mbar_wait(&p_full[buf], (np >> 1) & 1, err))) break;
                    const uint32_t slot = np % C::NST, use = np / C::NST;
                    if (!(ok = mbar_wait(&v_full[slot], use & 1, err))) break;
                    tc_fence_after();
                    const int nvalid = min(C::BN, tb.kv_len - jb * C::BN);
                    const uint64_t bd0 = sdesc_sw128(sV + slot * C::KV_BYTES, C::SUB_KV, 1024);
                    const uint32_t aP = tmem + C::COL_S + buf * C::BN;
                    // Fully unrolled with a guard per step: every operand offset is a
                    // constant and nothing but the guard runs between two products, so
                    // one thread issues them as fast as the tensor pipe takes them (a
                    // loop with a run-time trip count throttles it to about half).
                    const uint32_t acc0 = jb > 0 ? 1u : 0u;  // the tile's first block starts O_grp
                    if constexpr (TP) {
                        // the tile's group has all of the block's keys, into its own O
                        const uint32_t dO = tmem + C::COL_O + (tb_n & 1) * D;
                        const int ksteps = (nvalid + 15) >> 4;
#pragma unroll
                        for (int st = 0; st < 8; ++st) {
                            if (st < ksteps)
                                mma_bf16_ts(dO, aP + (st >> 1) * 32 + (st & 1) * 8, sdesc_add(bd0, st * 2048), idesc_pv,
                                            st > 0 ? 1u : acc0);
                        }
                    } else {
#pragma unroll
                        for (int grp = 0; grp < 2; ++grp) {
                            // group grp's keys 64 grp .. of the block; its 16-key step ks is
                            // block step 4 grp + ks, whose P sits in 32-key chunk (4 grp + ks) / 2
                            const int ksteps = (min(64, nvalid - 64 * grp) + 15) >> 4;  // <= 0: none
                            const uint32_t dO = tmem + C::COL_O + (tb_n % C::OB) * 2 * D + grp * D;
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks) {
                                if (ks < ksteps) {
                                    const int st = 4 * grp + ks;
                                    const uint64_t bd = sdesc_add(bd0, st * 2048);
                                    const uint32_t acc = ks > 0 ? 1u : acc0;
                                    if (ACT) {  // hi at columns 16 st .. +7, lo at 16 st + 8 .. +15
                                        mma_bf16_ts(dO, aP + st * 16, bd, idesc_pv, acc);
                                        mma_bf16_ts(dO, aP + st * 16 + 8, bd, idesc_pv, 1u);
                                    } else {
                                        mma_bf16_ts(dO, aP + (st >> 1) * 32 + (st & 1) * 8, bd, idesc_pv, acc);
                                    }
                                }
                            }
                        }
                    }
                    mma_commit(&v_empty[slot]);
                    mma_commit(&pv_done[buf]);  // the buffer may take block np + 2; O_0 / O_1 hold block np
                }
                if (!ok) break;
                mma_commit(&o_full[tb_n & 1]);
                ++tb_n;
            }
            mma_commit(&drain[1]);
            mbar_drain(&drain[1], 0);
        }
        // warp 3 and the other lanes: idle
    } else if (wgi < 3) {
        regs_claim<C::REG_SOFTMAX>();
        // ------------------------------------------------------------ softmax
        // One thread per query row (TMEM lane) over the group's 64 columns of
        // every block: scores -> bias, mask, online softmax (or activation)
        // -> P as bf16 over the same TMEM columns; rare O rescales in TMEM; per
        // tile the row max and row sum go to the output group.
        const int grp = wgi - 1;                   // keys 64 grp .. 64 grp + 63 of every block
        const int quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;          // query row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tS0 = tmem + lane_base + C::COL_S;  // buffer b of block n = n % 2 at b BN
        const uint32_t tO_base = tmem + lane_base + C::COL_O + grp * D;
        const float sc = ACT ? g.scale : g.scale * kLog2e;
        constexpr bool scaled = ACT || BIAS != kBiasNone;  // else the scale is folded into the exponent
        uint32_t t_local = 0, n0 = 0;  // n0: global number of the tile's first block
        bool ok = true;
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            const int nkv = nblocks(t);
            if (TP && (t_local & 1) != static_cast<uint32_t>(grp)) {  // the other group's tile
                n0 += nkv;
                ++t_local;
                continue;
            }
            const float *bt = sbias + t.h * g.nb;
            const float *ext_h = sext + t.h * ext_len(g.nb);
            const int q_loc = t.q_loc0 + row;
            // A warp whose 32 rows all lie past the tile's end only keeps the hand-offs
            // going: rows are independent through both products, so whatever its TMEM
            // lanes hold reaches only output rows that are never stored.
            const bool warp_live = quad * 32 < t.q_len;
            float m = -INFINITY, l = 0.0f;

            for (int j = 0; j < nkv; ++j) {
                const uint32_t n = n0 + j, b = n & 1;
                if (!(ok = mbar_wait_warp(&s_full[b], (n >> 1) & 1, err))) break;
                const uint32_t tS = tS0 + b * C::BN;  // S, then P over it
                if (!warp_live) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[b]);
                    continue;
                }
                tc_fence_after();
                // The block is walked in 32-key chunks by compact loops (the whole
                // unrolled block would not stay in the instruction cache); TMEM
                // holds the scores between passes.
                const int nvalid = min(C::BN, t.kv_len - j * C::BN);
                const int kvb = t.kv_loc0 + j * C::BN;
                // chunk c holds keys this row may see (block mode: its own 64-block;
                // sliding window: some row of this warp has the chunk in its band)
                auto live = [&](int c) {
                    return c * 32 < nvalid && (g.block == 0 || ((c * 32) >> 6) == (row >> 6)) &&
                           window_chunk_live(win, t.q_loc0 + quad * 32, kvb + c * 32);
                };
                // scores of chunk c with scale, bias and key mask (softmax: log2 units;
                // without a bias the scale waits for the exponent's FMA)
                auto scores = [&](int c, float (&xc)[32]) {
                    if constexpr (BIAS == kBiasExt) {
                        scale_bias32(xc, sc, ext_h, g.nb, q_loc, kvb + c * 32);
                    } else if constexpr (BIAS == kBiasTable) {
                        float bv[32];
                        bias32(bt, g.nb, q_loc, kvb + c * 32, bv);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) fma2(xc[i], xc[i + 1], sc, sc, bv[i], bv[i + 1]);
                    } else if constexpr (ACT) {
#pragma unroll
                        for (int i = 0; i < 32; i += 2) mul2(xc[i], xc[i + 1], sc, sc);
                    }
                    if (c * 32 + 32 > nvalid) {  // the sequence's last keys end inside this chunk
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c * 32 + i >= nvalid) xc[i] = ACT ? 0.0f : -INFINITY;
                    }
                    // keys outside the row's window (activation: act(0) = 0)
                    if constexpr (WIN) window_fill32(xc, window_bits32(win, q_loc, kvb + c * 32), ACT ? 0.0f : -INFINITY);
                };

                if constexpr (!ACT) {
                    // pass 1: row max of the block (biased scores written back in place)
                    float mloc = -INFINITY;
#pragma unroll 1
                    for (int c = TP ? 0 : 2 * grp; c < (TP ? 4 : 2 * grp + 2); ++c) {
                        if (!live(c)) continue;
                        float xc[32];
                        tmem_ld32(tS + 32 * c, xc);
                        scores(c, xc);
                        mloc = fmaxf(mloc, max32(xc));
                        if constexpr (scaled) {
                            uint32_t w[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(xc[i]);
                            tmem_st32_u32(tS + 32 * c, w);
                        }
                    }
                    if constexpr (scaled) tmem_wait_st();
                    if (!scaled) mloc *= sc;
                    // MXFP8: the max is an integer (log2 units), so alpha is a power of two
                    const float m_new = MX ? ceilf(fmaxf(m, mloc)) : fmaxf(m, mloc);
                    // lazy rescale: keep the old max while it is within the threshold
                    float alpha = 1.0f;
                    bool resc = false;
                    if (j == 0) {
                        m = m_new;
                    } else if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
                        // the test is warp-wide: a row of the warp that has seen no
                        // key yet (m = m_new = -inf) keeps its zero l and O as they are
                        if constexpr (MX) {
                            alpha = m_new == -INFINITY ? 1.0f
                                    : (m == -INFINITY ? 0.0f : (m - m_new < -126.0f ? 0.0f : pow2i(static_cast<int>(m - m_new))));
                        } else {
                            alpha = m_new == -INFINITY ? 1.0f : ex2_approx(m - m_new);
                        }
                        resc = true;
                        l *= alpha;
                        m = m_new;
                    }
                    const float nm = (m == -INFINITY) ? 0.0f : -m;
                    // pass 2: P = 2^(s - m) as bf16; chunk c goes to its own first 16
                    // columns 32c..32c+15, scores already consumed
                    float rs = 0.0f;
#pragma unroll 1
                    for (int c = TP ? 0 : 2 * grp; c < (TP ? 4 : 2 * grp + 2); ++c) {
                        uint32_t pw[16];
                        if (!live(c)) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) pw[i] = 0u;
                        } else {
                            float xc[32];
                            tmem_ld32(tS + 32 * c, xc);
                            if constexpr (scaled) {
#pragma unroll
                                for (int i = 0; i < 32; i += 2) add2(xc[i], xc[i + 1], nm, nm);
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; i += 2) fma2(xc[i], xc[i + 1], sc, sc, nm, nm);
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) xc[i] = ex2_approx(xc[i]);
                            if (!scaled && c * 32 + 32 > nvalid) {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (c * 32 + i >= nvalid) xc[i] = 0.0f;
                            }
                            if constexpr (WIN && !scaled) window_fill32(xc, window_bits32(win, q_loc, kvb + c * 32), 0.0f);
                            rs += sum32(xc);
                            // MXFP8: the chunk's 32 keys of this row are one quantisation
                            // group (the row sum above took the unquantised values)
                            if constexpr (MX) mx_qdq32(xc, mx_exponent(amax32(xc)));
#pragma unroll
                            for (int i = 0; i < 16; ++i) pw[i] = pack_bf16x2(xc[2 * i], xc[2 * i + 1]);
                        }
                        tmem_st16_u32(tS + 32 * c, pw);
                    }
                    l += rs;
                    if (resc) {
                        // O_grp holds the tile's earlier blocks once P V of block n - 1 has
                        // finished (block n - 2's finished before S_n was issued, so the
                        // barrier is at most that one phase behind); then bring O_grp to
                        // the new max before this block's P V adds on
                        if (!(ok = mbar_wait_warp(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, err))) break;
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            float o[32];
                            tmem_ld32(tO_base + (t_local % C::OB) * 2 * D + c * 32, o);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) mul2(o[i], o[i + 1], alpha, alpha);
                            tmem_st32(tO_base + (t_local % C::OB) * 2 * D + c * 32, o);
                        }
                    }
                } else {
                    // P = act(s) as bf16 hi + lo parts, interleaved per 16-key MMA step:
                    // step k's hi at columns 16k..16k+7, its lo at 16k+8..16k+15, so
                    // chunk c lands exactly on its own score columns 32c..32c+31
                    auto act_block = [&](auto af) {
                        constexpr int AF = decltype(af)::value;
#pragma unroll 1
                        for (int c = 2 * grp; c < 2 * grp + 2; ++c) {
                            uint32_t w[32];
                            if (!live(c)) {
#pragma unroll
                                for (int i = 0; i < 32; ++i) w[i] = 0u;
                            } else {
                                float xc[32];
                                tmem_ld32(tS + 32 * c, xc);
                                scores(c, xc);
                                // keys past the sequence's end are 0 after scores(), and act(0) = 0:
                                // no per-element test (one around a larger activation would become
                                // a branch per element)
#pragma unroll
                                for (int i = 0; i < 32; i += 2) {
                                    const float a0 = act_fwd_t<AF>(xc[i]);
                                    const float a1 = act_fwd_t<AF>(xc[i + 1]);
                                    __nv_bfloat162 h2 = __floats2bfloat162_rn(a0, a1);
                                    const int k = i >> 4, e = (i & 15) >> 1;  // MMA step within the chunk, pair
                                    w[16 * k + e] = *reinterpret_cast<uint32_t *>(&h2);
                                    w[16 * k + 8 + e] =
                                        pack_bf16x2(a0 - __bfloat162float(h2.x), a1 - __bfloat162float(h2.y));
                                }
                            }
                            tmem_st32_u32(tS + 32 * c, w);
                        }
                    };
                    if (g.act == kSilu) {
                        act_block(std::integral_constant<int, kSilu>{});
                    } else {
                        act_block(std::integral_constant<int, kGeluTanh>{});
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            if (!ok) break;

            // ---- this group's row statistics for the output group
            if constexpr (!ACT) {
                const uint32_t sl = t_local & 1;
                // the output group must be done with the tile that last used this slot
                if (!(ok = mbar_wait_warp(&o_empty[sl], ((t_local >> 1) & 1) ^ 1, err))) break;
                srows[(sl * 4 + 2 * grp) * 128 + row] = m;
                srows[(sl * 4 + 2 * grp + 1) * 128 + row] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(&l_full[sl]);
            }
            n0 += nkv;
            ++t_local;
        }
    } else {
        regs_release<C::REG_OUT>();
        // ------------------------------------------------------------ output
        // One thread per query row: merge O_0 and O_1 (TMEM, fp32) of the groups
        // that had blocks in the tile with their row statistics, write the
        // output row (each thread stores whole 64-byte pieces of its row) and
        // lse = ln 2 (m + log2 L).  The accumulators are handed back as soon as
        // they have been read.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tO_base = tmem + lane_base + C::COL_O;  // + (tile % OB) 2 D: this tile's O set
        const uint32_t stg = smem_u32(smem + C::OFF_STG) + static_cast<uint32_t>(quad) * (32 * C::STG_W * 2);
        const bool staged = C::STAGE_OUT && !a.out.f32 && a.out.cols == D;
        uint32_t t_local = 0, n0 = 0;
        bool ok = true;
        // RoPE: this warpgroup rotates Q and K two tiles ahead of the one whose
        // output it writes (each warp its 32 rows), so the rotation of tile
        // t + 2, which only needs S_t done, never waits for this group's output
        // of tile t, and S_{t+2} finds it done.  Only BlockAttention tiles (one
        // K block at the Q rows' positions) are rotated here; any other tile
        // is a device error.
        TileStream rs(g, tbeg, tend);
        uint32_t r_local = 0, rk_it = 0;
        auto rotate_next = [&]() -> bool {
            Tile rt;
            bool found = false;
            while (!found && rs.next(rt)) found = check_tile(g, rt, err, false);
            if (!found) return true;
            const uint32_t qs = r_local & 1, slot = rk_it % C::NST;
            const bool joint = rt.kv_len == rt.q_len && rt.kv_loc0 == rt.q_loc0 && rt.kv_len <= C::BN;
            if (!joint) {
                if (lane == 0) raise_error(err, kStatusDeviceCheck);
                return false;
            }
            if (!mbar_wait_warp(&q_full[qs], (r_local >> 1) & 1, err)) return false;
            if (!mbar_wait_warp(&k_full[slot], (rk_it / C::NST) & 1, err)) return false;
            const int r0 = quad * 32, nrows = min(32, rt.q_len - r0);
            if (nrows > 0) {
                const float *qc = C::TAB ? reinterpret_cast<const float *>(smem + C::OFF_TAB + qs * C::TAB_BYTES)
                                         : g.rope_cos + static_cast<int64_t>(rt.q_loc0) * (D / 2);
                const float *qsn = C::TAB ? qc + C::BM * (D / 2) : g.rope_sin + static_cast<int64_t>(rt.q_loc0) * (D / 2);
                if (C::TAB)
                    rope_tile_s<D, 1>(sQ + qs * C::Q_BYTES + r0 * 128, sK + slot * C::KV_BYTES + r0 * 128, C::SUB_Q,
                                      nrows, smem_u32(qc + r0 * (D / 2)), smem_u32(qsn + r0 * (D / 2)), lane);
                else
                    rope_tile<D, 1>(sQ + qs * C::Q_BYTES + r0 * 128, sK + slot * C::KV_BYTES + r0 * 128, C::SUB_Q,
                                    nrows, qc + r0 * (D / 2), qsn + r0 * (D / 2), lane);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&q_rot[qs]);
                mbar_arrive(&k_rot[slot]);
            }
            ++r_local;
            ++rk_it;
            return true;
        };
        if (ROPE) ok = rotate_next() && rotate_next();
        TileStream ts(g, tbeg, tend);
        Tile t;
        while (ok && ts.next(t)) {
            if (!check_tile(g, t, err, false)) continue;
            if (ROPE && !(ok = rotate_next())) break;
            const int nkv = nblocks(t);
            // group g has keys in this tile when the tile has more than 64 g keys
            // (tile-parallel: the tile's group, read as group 0, has them all)
            const bool has0 = t.kv_len > 0;
            const bool has1 = !TP && t.kv_len > 64;
            const uint32_t sl = t_local & 1;
            if (!(ok = mbar_wait_warp(&o_full[t_local & 1], (t_local >> 1) & 1, err))) break;
            const uint32_t tO0 = TP ? tO_base + (t_local & 1) * D : tO_base + (t_local % C::OB) * 2 * D, tO1 = tO0 + D;
            float c0 = has0 ? 1.0f : 0.0f, c1 = has1 ? 1.0f : 0.0f, lse = -INFINITY;
            if constexpr (!ACT) {
                if (!(ok = mbar_wait_warp(&l_full[sl], (t_local >> 1) & 1, err))) break;
                // (tile-parallel: only the tile's group, g = sl, wrote its statistics)
                const float m0 = srows[(sl * 4 + (TP ? 2 * sl : 0)) * 128 + row];
                const float l0 = srows[(sl * 4 + (TP ? 2 * sl : 0) + 1) * 128 + row];
                const float m1 = TP ? -INFINITY : srows[(sl * 4 + 2) * 128 + row];
                const float l1 = TP ? 0.0f : srows[(sl * 4 + 3) * 128 + row];
                const float mm = fmaxf(m0, m1);
                const float w0 = l0 > 0.0f ? ex2_approx(m0 - mm) : 0.0f;
                const float w1 = l1 > 0.0f ? ex2_approx(m1 - mm) : 0.0f;
                const float L = l0 * w0 + l1 * w1;
                const float inv = L > 0.0f ? 1.0f / L : 0.0f;
                c0 = w0 * inv;
                c1 = w1 * inv;
                if (L > 0.0f) lse = (mm + __log2f(L)) * kLn2;
            }
            tc_fence_after();
            const bool row_ok = row < t.q_len;
            const int64_t orow = static_cast<int64_t>(t.q_start) + row;
            if (quad * 32 >= t.q_len) {  // no row of this warp is stored
                __syncwarp();
                if (lane == 0) mbar_arrive(&o_empty[sl]);
                n0 += nkv;
                ++t_local;
                continue;
            }
            if (C::STAGE_OUT && staged) {
                // each 64-column half of the warp's 32 rows goes out through the staging
                // rows as whole 128-byte row pieces (not 32 rows' 16-byte pieces per store)
                constexpr int W = C::STG_W;
                const int nrows = min(32, t.q_len - quad * 32);
                __nv_bfloat16 *dst0 = static_cast<__nv_bfloat16 *>(a.out.ptr) +
                                      (static_cast<int64_t>(t.q_start) + quad * 32) * a.out.ld +
                                      static_cast<int64_t>(t.h) * D;
#pragma unroll 1
                for (int col = 0; col < D; col += 32) {
                    float o[32];
                    if (has0) {
                        tmem_ld32(tO0 + col, o);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) mul2(o[i], o[i + 1], c0, c0);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0.0f;
                    }
                    if (has1) {
                        float o1[32];
                        tmem_ld32(tO1 + col, o1);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {  // o += c1 * o1
                            fma2(o1[i], o1[i + 1], c1, c1, o[i], o[i + 1]);
                            o[i] = o1[i];
                            o[i + 1] = o1[i + 1];
                        }
                    }
                    if (col + 32 >= D) {  // every TMEM read of this tile is done: O_0 / O_1 are free
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&o_empty[sl]);
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
                    stage_row32_bf16<W>(stg, lane, col % W, w);
                    if ((col + 32) % W == 0) {
                        __syncwarp();
                        store_rows_bf16<W>(stg, lane, dst0 + (col + 32 - W), a.out.ld, nrows);
                        __syncwarp();
                    }
                }
                if (!ACT && a.lse != nullptr && row_ok) a.lse[static_cast<int64_t>(t.h) * g.Tq + orow] = lse;
                n0 += nkv;
                ++t_local;
                continue;
            }
#pragma unroll 1
            for (int col = 0; col < D; col += 32) {
                float o[32];
                if (has0) {
                    tmem_ld32(tO0 + col, o);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) mul2(o[i], o[i + 1], c0, c0);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.0f;
                }
                if (has1) {
                    float o1[32];
                    tmem_ld32(tO1 + col, o1);
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {  // o += c1 * o1
                        fma2(o1[i], o1[i + 1], c1, c1, o[i], o[i + 1]);
                        o[i] = o1[i];
                        o[i + 1] = o1[i + 1];
                    }
                }
                if (col + 32 >= D) {
                    // every TMEM read of this tile is done: O_0 / O_1 are free
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&o_empty[sl]);
                }
                if (row_ok) store_out32(a.out, orow, t.h, col, o, 1.0f);
            }
            if (!ACT && a.lse != nullptr && row_ok) a.lse[static_cast<int64_t>(t.h) * g.Tq + orow] = lse;
            n0 += nkv;
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

}  // namespace jattn
