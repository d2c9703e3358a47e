// plan_device.cu -- the tile lists and the persistent schedule built on the GPU
// from offsets that are already in device memory.
//
// "Training GEM at LLM scale", section "Generalized Dot-Product Attention
// (GDPA)": the valid tiles of a jagged batch are precomputed and spread over
// the SMs in a zigzag so that no SM is left with the heavy tail.  The host
// planner (api.cpp) does this on the CPU from host offsets; here one CTA does it
// on the device, so a training loop whose offsets live on the GPU needs no
// device-to-host copy and no host work per step.
//
// The tile records are those of the host planner: query-major tiles of 128
// rows in the order (sequence, 128-row block, head), each with the key range
// its rows may see (all keys; its own 64-blocks in BlockAttention; the band of
// a sliding window), and, outside BlockAttention, key-major tiles likewise.
// Only the schedule differs.  Instead of the host's longest-first greedy
// assignment, the sequences are sorted by the cost of their tiles (descending,
// ties by index) and the tiles, in that order, are dealt to the CTAs in a
// zigzag (0, 1, .., C-1, C-1, .., 0, 0, 1, ..).  That places every tile and
// every CTA's range in closed form, with no serial step.  A tile's results do
// not depend on which CTA runs it, so the outputs equal those of the host plan
// bit for bit.
#include <cuda_runtime.h>

#include "attn.cuh"
#include "kernels.h"

namespace jattn {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ int cost_rows_d(int n) { return (n + 15) / 16; }

// Keys the tile's rows may see (query-major tile at row s of a sequence), as in
// the host planner: [lo, hi) within the sequence's keys.
__device__ __forceinline__ void q_tile_keys(int s, int ql, int Lk, int block, int win, int &lo, int &hi) {
    lo = 0;
    hi = Lk;
    if (block) {
        lo = s;
        hi = s + ql;
    } else if (win > 0) {
        lo = static_cast<int>(min(static_cast<int64_t>(Lk), max(int64_t{0}, static_cast<int64_t>(s) - win + 1)));
        hi = static_cast<int>(min(static_cast<int64_t>(Lk), static_cast<int64_t>(s) + ql + win - 1));
        if (hi < lo) hi = lo;
    }
}

// Block-wide exclusive scan of v[0..n) in shared memory (n <= kThreads * 8).
__device__ void scan_exclusive(int32_t *v, int n, int32_t *warp_sums, int32_t &total) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int per = (n + kThreads - 1) / kThreads;  // <= 8
    const int b0 = min(n, tid * per), b1 = min(n, b0 + per);
    int32_t run = 0;
    for (int i = b0; i < b1; ++i) run += v[i];
    int32_t x = run;  // inclusive warp scan of the per-thread sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int32_t w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    int32_t base = (wid > 0 ? warp_sums[wid - 1] : 0) + x - run;
    for (int i = b0; i < b1; ++i) {
        const int32_t c = v[i];
        v[i] = base;
        base += c;
    }
    total = warp_sums[31];
    __syncthreads();
}

// Slot of sorted tile g in the CTA-grouped list, and the first slot of CTA c,
// for N tiles dealt in a zigzag over C CTAs.
__device__ __forceinline__ int zigzag_cta(int64_t g, int C) {
    const int64_t r = g / C, w = g % C;
    return static_cast<int>((r & 1) ? C - 1 - w : w);
}
__device__ __forceinline__ int64_t zigzag_begin(int c, int64_t N, int C) {
    const int64_t nr = N / C, rem = N % C;
    const int64_t extra = (nr & 1) ? max(int64_t{0}, c - (C - rem)) : min(static_cast<int64_t>(c), rem);
    return c * nr + extra;
}

struct ListArgs {
    Tile *tiles;
    int32_t *cta;     // [C + 1]
    int32_t cap;      // capacity of tiles
    bool key_major;
};

__global__ void __launch_bounds__(kThreads, 1) plan_kernel(const DevPlanArgs a) {
    extern __shared__ uint8_t sm[];
    const int NS = a.sort_len;  // power of two >= B
    uint64_t *key = reinterpret_cast<uint64_t *>(sm);            // [NS] sort keys, then sequence order
    int32_t *first = reinterpret_cast<int32_t *>(key + NS);       // [NS + 1] first sorted tile of each sorted sequence
    __shared__ int32_t warp_sums[32];
    __shared__ int bad;
    const int tid = threadIdx.x;
    const int B = a.B, H = a.H, C = a.n_ctas;
    if (tid == 0) bad = 0;
    __syncthreads();
    // offsets: start at 0, nondecreasing, end at Tq / Tk; BlockAttention: equal lengths
    for (int b = tid; b < B; b += kThreads) {
        const int32_t q0 = a.q_off[b], q1 = a.q_off[b + 1], k0 = a.kv_off[b], k1 = a.kv_off[b + 1];
        bool ok = q1 >= q0 && k1 >= k0;
        if (b == 0) ok = ok && q0 == 0 && k0 == 0;
        if (b == B - 1) ok = ok && q1 == a.Tq && k1 == a.Tk;
        if (a.block) ok = ok && (q1 - q0) == (k1 - k0);
        if (a.bcast_n > 0) ok = ok && (q1 - q0) == a.bcast_n;
        if (!ok) bad = 1;
    }
    __syncthreads();
    const bool invalid = bad != 0;
    if (invalid && tid == 0) atomicCAS(a.status, 0, kStatusDeviceCheck);

    for (int which = 0; which < 2; ++which) {
        const ListArgs L = which == 0 ? ListArgs{a.tiles_q, a.cta_q, a.cap_q, false}
                                      : ListArgs{a.tiles_kv, a.cta_kv, a.cap_kv, true};
        const bool empty_list = invalid || (L.key_major && a.block);  // BlockAttention has no key-major pass
        // per-sequence tile count and cost of its tiles (span = the other side's rows)
        for (int i = tid; i < NS; i += kThreads) {
            uint64_t k = ~uint64_t{0};  // padding sorts last
            if (i < B && !empty_list) {
                const int Lq = a.q_off[i + 1] - a.q_off[i], Lk = a.kv_off[i + 1] - a.kv_off[i];
                int span = L.key_major ? Lq : Lk;
                if (a.block) span = min(Lq, 128);
                if (a.window > 0) span = min(span, 128 + 2 * a.window - 2);
                const uint32_t cost = 8u + static_cast<uint32_t>(cost_rows_d(span));
                k = (static_cast<uint64_t>(0xffffffffu - cost) << 32) | static_cast<uint32_t>(i);
            }
            key[i] = k;
        }
        __syncthreads();
        // bitonic sort, ascending: cost descending, then sequence index
        for (int size = 2; size <= NS; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < NS; i += kThreads) {
                    const int j = i ^ stride;
                    if (j > i) {
                        const bool up = (i & size) == 0;
                        const uint64_t x = key[i], y = key[j];
                        if ((x > y) == up) {
                            key[i] = y;
                            key[j] = x;
                        }
                    }
                }
                __syncthreads();
            }
        }
        // tiles of each sorted sequence, then their first sorted index
        for (int i = tid; i < NS; i += kThreads) {
            int32_t n = 0;
            if (i < B && !empty_list) {
                const int b = static_cast<int>(key[i] & 0xffffffffu);
                const int Lr = L.key_major ? a.kv_off[b + 1] - a.kv_off[b] : a.q_off[b + 1] - a.q_off[b];
                n = ((Lr + 127) / 128) * H;
            }
            first[i] = n;
        }
        __syncthreads();
        int32_t total = 0;
        scan_exclusive(first, NS, warp_sums, total);
        if (tid == 0) first[NS] = total;
        const bool over = total > L.cap;
        if (over && tid == 0) atomicCAS(a.status, 0, kStatusDeviceCheck);
        const int64_t N = over ? 0 : total;
        __syncthreads();
        // every tile: its sequence by binary search over first[], its record, its slot
        for (int64_t g = tid; g < N; g += kThreads) {
            int lo = 0, hi = min(B, NS) - 1;  // last i with first[i] <= g
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (first[mid] <= g) lo = mid;
                else hi = mid - 1;
            }
            const int b = static_cast<int>(key[lo] & 0xffffffffu);
            const int j = static_cast<int>(g - first[lo]);
            const int h = j % H, blk = j / H;
            const int q0 = a.q_off[b], k0 = a.kv_off[b];
            const int Lq = a.q_off[b + 1] - q0, Lk = a.kv_off[b + 1] - k0;
            Tile t;
            t.b = b;
            t.h = h;
            const int s = blk * 128;
            if (!L.key_major) {
                const int ql = min(128, Lq - s);
                int klo, khi;
                q_tile_keys(s, ql, Lk, a.block, a.window, klo, khi);
                t.q_start = q0 + s;
                t.q_len = ql;
                t.kv_start = k0 + klo;
                t.kv_len = khi - klo;
                t.q_loc0 = s;
                t.kv_loc0 = klo;
            } else {
                const int kl = min(128, Lk - s);
                int qlo = 0, qhi = Lq;  // queries whose window reaches the tile's keys
                if (a.window > 0) {
                    qlo = static_cast<int>(min(static_cast<int64_t>(Lq), max(int64_t{0}, static_cast<int64_t>(s) - a.window + 1)));
                    qhi = static_cast<int>(min(static_cast<int64_t>(Lq), static_cast<int64_t>(s) + kl + a.window - 1));
                    if (qhi < qlo) qhi = qlo;
                }
                t.q_start = q0 + qlo;
                t.q_len = qhi - qlo;
                t.kv_start = k0 + s;
                t.kv_len = kl;
                t.q_loc0 = qlo;
                t.kv_loc0 = s;
            }
            const int c = zigzag_cta(g, C);
            const int64_t slot = zigzag_begin(c, N, C) + g / C;
            L.tiles[slot] = t;
        }
        for (int c = tid; c <= C; c += kThreads) L.cta[c] = static_cast<int32_t>(zigzag_begin(c, N, C));
        __syncthreads();
    }
}

}  // namespace

static size_t plan_device_smem(int sort_len) { return static_cast<size_t>(sort_len) * 8 + (sort_len + 1) * 4; }

cudaError_t launch_plan_device(const DevPlanArgs &a, cudaStream_t stream) {
    if (a.sort_len < 2 || a.sort_len > kDevPlanMaxSeqs || (a.sort_len & (a.sort_len - 1)) != 0 || a.B > a.sort_len ||
        a.n_ctas < 1)
        return cudaErrorInvalidValue;
    const size_t smem = plan_device_smem(a.sort_len);
    static SmemOnce done;
    cudaError_t e = ensure_smem(plan_kernel, static_cast<uint32_t>(plan_device_smem(kDevPlanMaxSeqs)), done);
    if (e != cudaSuccess) return e;
    plan_kernel<<<1, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace jattn
