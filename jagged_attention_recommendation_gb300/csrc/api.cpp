// api.cpp -- the C ABI (include/jattn.h): argument checks, the jagged batch
// planner (tile lists + persistent-grid schedule), tensor-map construction and
// kernel dispatch.  Host code only; every step of the computation runs in the
// CUDA kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <queue>
#include <vector>

#include "common.h"
#include "jattn.h"
#include "kernels.h"

using namespace jattn;

static_assert(sizeof(jattn_tile) == 24, "tile record is 24 bytes");
static_assert(sizeof(Tile) == 32, "device tile record is 32 bytes");

namespace {

constexpr int kTileRows = 128;       // rows per query-major and key-major tile
constexpr int kDefaultSms = 152;     // schedule width of a host-only plan
constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

struct jattn_plan {
    int32_t B = 0, H = 0, D = 0, Dp = 0;
    jattn_mode mode{};
    float scale = 0.0f;
    int32_t device = -1;
    int32_t num_sms = kDefaultSms;
    bool staged = false;  // inputs are copied to bf16 [T, H, Dp] first (fp32 data or D = 32)
    // planned on the device (jattn_plan_update_device): the host tile lists and
    // offsets are stale until jattn_plan_tiles downloads them
    bool dev_planned = false;
    int32_t bcast_n = 0;  // broadcast Q: rows of the shared Q (every sequence's Lq)
    int64_t Tq = 0, Tk = 0;
    std::vector<int32_t> q_off, kv_off;
    // backward dS chunks (host plans): first chunk of every sequence, and the total
    std::vector<long long> ds_base;
    int64_t ds_chunks = 0;
    int32_t max_tile_kv = 0;  // largest key range of a query tile (host plans)
    std::vector<jattn_tile> tiles[2];
    std::vector<int32_t> cta[2];
    // device copies: one buffer holding both tile lists, both schedules and the offsets
    uint8_t *d_buf = nullptr;
    size_t d_cap = 0;
    size_t off_tiles[2] = {0, 0}, off_cta[2] = {0, 0}, off_qoff = 0, off_kvoff = 0, off_dsbase = 0;
    int *d_status = nullptr;
    // pinned staging for the asynchronous upload, double-buffered
    void *h_pin[2] = {nullptr, nullptr};
    size_t h_cap[2] = {0, 0};
    cudaEvent_t ev[2] = {nullptr, nullptr};
    bool ev_used[2] = {false, false};
    int pin_next = 0;
    // profiling hook and launch counter (mutable: updated by const calls)
    mutable std::vector<cudaEvent_t> prof_events;
    mutable int prof_next = 0;
    mutable int64_t launches = 0;
    // jattn_step_host: two device staging sets and the upload / compute /
    // download streams that overlap consecutive calls
    struct HostStep {
        bool init = false;
        cudaStream_t s_up = nullptr, s_comp = nullptr, s_down = nullptr;
        cudaEvent_t ev_start = nullptr;
        cudaEvent_t up_done[2] = {nullptr, nullptr}, comp_done[2] = {nullptr, nullptr},
                    down_done[2] = {nullptr, nullptr};
        bool used[2] = {false, false};
        uint8_t *dev[2] = {nullptr, nullptr};
        size_t cap[2] = {0, 0};
        int next = 0, last = -1;
    } hs;
};

namespace {

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

jattn_status check_offsets(const int32_t *qo, const int32_t *ko, int32_t B, bool block) {
    if (qo == nullptr || ko == nullptr || B < 1) return JATTN_ERR_INVALID_ARG;
    if (qo[0] != 0 || ko[0] != 0) return JATTN_ERR_INVALID_ARG;
    for (int32_t b = 0; b < B; ++b) {
        if (qo[b + 1] < qo[b] || ko[b + 1] < ko[b]) return JATTN_ERR_INVALID_ARG;
        if (block && (qo[b + 1] - qo[b]) != (ko[b + 1] - ko[b])) return JATTN_ERR_INVALID_ARG;
    }
    return JATTN_OK;
}

int cost_rows(int n) { return (n + 15) / 16; }

// Longest-processing-time-first assignment of tiles to n_ctas persistent CTAs:
// tiles in decreasing cost order, each to the currently least-loaded CTA (ties
// to the lower CTA id), then regrouped so CTA c runs list[cta[c] .. cta[c+1]).
void schedule(std::vector<jattn_tile> &list, std::vector<int32_t> &cta, int num_sms, bool kv_major, bool block) {
    const size_t n = list.size();
    const int n_ctas = static_cast<int>(std::min<size_t>(n, static_cast<size_t>(std::max(num_sms, 1))));
    cta.assign(static_cast<size_t>(n_ctas) + 1, 0);
    if (n == 0) return;
    std::vector<int64_t> cost(n);
    for (size_t i = 0; i < n; ++i) {
        const jattn_tile &t = list[i];
        const int span = block ? t.q_len : (kv_major ? t.q_len : t.kv_len);
        cost[i] = 8 + cost_rows(span);  // fixed per-tile work + 16-column MMA groups
    }
    std::vector<int32_t> order(n);
    for (size_t i = 0; i < n; ++i) order[i] = static_cast<int32_t>(i);
    std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return cost[x] > cost[y]; });
    using Slot = std::pair<int64_t, int32_t>;  // (load, cta)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t c = 0; c < n_ctas; ++c) heap.push({0, c});
    std::vector<int32_t> owner(n);
    std::vector<int32_t> count(static_cast<size_t>(n_ctas), 0);
    for (int32_t idx : order) {
        Slot s = heap.top();
        heap.pop();
        owner[idx] = s.second;
        ++count[s.second];
        heap.push({s.first + cost[idx], s.second});
    }
    for (int32_t c = 0; c < n_ctas; ++c) cta[c + 1] = cta[c] + count[c];
    std::vector<jattn_tile> out(n);
    std::vector<int32_t> fill(cta.begin(), cta.end() - 1);
    for (int32_t idx : order) out[fill[owner[idx]]++] = list[idx];
    list.swap(out);
}

void build_lists(jattn_plan *p) {
    const bool block = p->mode.block != 0;
    const int64_t win = p->mode.window;
    std::vector<jattn_tile> &tq = p->tiles[JATTN_TILES_Q];
    std::vector<jattn_tile> &tk = p->tiles[JATTN_TILES_KV];
    tq.clear();
    p->max_tile_kv = 0;
    tk.clear();
    for (int32_t b = 0; b < p->B; ++b) {
        const int32_t q0 = p->q_off[b], Lq = p->q_off[b + 1] - q0;
        const int32_t k0 = p->kv_off[b], Lk = p->kv_off[b + 1] - k0;
        for (int32_t s = 0; s < Lq; s += kTileRows) {
            const int32_t ql = std::min(kTileRows, Lq - s);
            // keys the tile's rows may see: all, the same chunk (block), or the
            // union of the rows' windows |i - j| < W (sliding window)
            int32_t lo = 0, hi = Lk;
            if (block) {
                lo = s;
                hi = s + ql;
            } else if (win > 0) {
                lo = static_cast<int32_t>(std::min<int64_t>(Lk, std::max<int64_t>(0, static_cast<int64_t>(s) - win + 1)));
                hi = static_cast<int32_t>(std::min<int64_t>(Lk, static_cast<int64_t>(s) + ql + win - 1));
                if (hi < lo) hi = lo;  // no key in reach: an empty range inside the sequence
            }
            for (int32_t h = 0; h < p->H; ++h) tq.push_back({b, h, q0 + s, ql, k0 + lo, hi - lo});
            p->max_tile_kv = std::max(p->max_tile_kv, hi - lo);
        }
    }
    if (!block) {
        for (int32_t b = 0; b < p->B; ++b) {
            const int32_t q0 = p->q_off[b], Lq = p->q_off[b + 1] - q0;
            const int32_t k0 = p->kv_off[b], Lk = p->kv_off[b + 1] - k0;
            for (int32_t s = 0; s < Lk; s += kTileRows) {
                const int32_t kl = std::min(kTileRows, Lk - s);
                int32_t lo = 0, hi = Lq;  // queries whose window reaches the tile's keys
                if (win > 0) {
                    lo = static_cast<int32_t>(std::min<int64_t>(Lq, std::max<int64_t>(0, static_cast<int64_t>(s) - win + 1)));
                    hi = static_cast<int32_t>(std::min<int64_t>(Lq, static_cast<int64_t>(s) + kl + win - 1));
                    if (hi < lo) hi = lo;  // no query in reach: an empty range inside the sequence
                }
                for (int32_t h = 0; h < p->H; ++h) tk.push_back({b, h, q0 + lo, hi - lo, k0 + s, kl});
            }
        }
    }
    schedule(tq, p->cta[JATTN_TILES_Q], p->num_sms, false, block);
    schedule(tk, p->cta[JATTN_TILES_KV], p->num_sms, true, block);
}

thread_local char g_last_cuda_error[256] = "";

// Map a CUDA result to a status, remembering the error text for jattn_last_cuda_error.
jattn_status cuda_status(cudaError_t e, const char *where = "") {
    if (e == cudaSuccess) return JATTN_OK;
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%s)", where, cudaGetErrorString(e),
                  cudaGetErrorName(e));
    return JATTN_ERR_CUDA;
}

#define CUDA_TRY(expr)                                      \
    do {                                                    \
        const cudaError_t e_ = (expr);                      \
        if (e_ != cudaSuccess) return cuda_status(e_, #expr); \
    } while (0)

// MXFP8 quantisation job over one side's tile list (host-planned plans only)
void add_mx_job(MxJobs &jobs, const jattn_plan *p, int which, const void *x, void *xq) {
    const int j = jobs.n++;
    jobs.x[j] = x;
    jobs.xq[j] = xq;
    jobs.tiles[j] = reinterpret_cast<const Tile *>(p->d_buf + p->off_tiles[which]);
    jobs.ntiles[j] = static_cast<int32_t>(p->tiles[which].size());
    jobs.kv_side[j] = which == JATTN_TILES_KV;
}

jattn_status note_error(const char *where) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s", where);
    return JATTN_ERR_CUDA;
}

// Lay out and upload tiles, schedules and offsets (asynchronously on `stream`).
jattn_status upload(jattn_plan *p, cudaStream_t stream) {
    size_t off = 0;
    for (int w = 0; w < 2; ++w) {
        p->off_tiles[w] = off;
        off = align_up(off + p->tiles[w].size() * sizeof(Tile), 16);
    }
    for (int w = 0; w < 2; ++w) {
        p->off_cta[w] = off;
        off = align_up(off + p->cta[w].size() * sizeof(int32_t), 16);
    }
    p->off_qoff = off;
    off = align_up(off + p->q_off.size() * sizeof(int32_t), 16);
    p->off_kvoff = off;
    off = align_up(off + p->kv_off.size() * sizeof(int32_t), 16);
    p->off_dsbase = off;
    off = align_up(off + p->ds_base.size() * sizeof(long long), 16);
    const size_t bytes = off;

    if (bytes > p->d_cap) {
        CUDA_TRY(cudaStreamSynchronize(stream));  // earlier launches may still read the old buffer
        if (p->d_buf) cudaFree(p->d_buf);
        p->d_buf = nullptr;
        p->d_cap = 0;
        const size_t cap = std::max(bytes + bytes / 2, static_cast<size_t>(4096));
        CUDA_TRY(cudaMalloc(&p->d_buf, cap));
        p->d_cap = cap;
    }
    const int k = p->pin_next;
    p->pin_next ^= 1;
    if (p->ev_used[k]) {
        CUDA_TRY(cudaEventSynchronize(p->ev[k]));
    }
    if (bytes > p->h_cap[k]) {
        if (p->h_pin[k]) cudaFreeHost(p->h_pin[k]);
        p->h_pin[k] = nullptr;
        p->h_cap[k] = 0;
        const size_t cap = std::max(bytes + bytes / 2, static_cast<size_t>(4096));
        CUDA_TRY(cudaMallocHost(&p->h_pin[k], cap));
        p->h_cap[k] = cap;
    }
    uint8_t *h = static_cast<uint8_t *>(p->h_pin[k]);
    for (int w = 0; w < 2; ++w) {
        Tile *dst = reinterpret_cast<Tile *>(h + p->off_tiles[w]);
        for (size_t i = 0; i < p->tiles[w].size(); ++i) {
            const jattn_tile &t = p->tiles[w][i];
            dst[i] = Tile{t.b, t.h, t.q_start, t.q_len, t.kv_start, t.kv_len, t.q_start - p->q_off[t.b],
                          t.kv_start - p->kv_off[t.b]};
        }
        std::memcpy(h + p->off_cta[w], p->cta[w].data(), p->cta[w].size() * sizeof(int32_t));
    }
    std::memcpy(h + p->off_qoff, p->q_off.data(), p->q_off.size() * sizeof(int32_t));
    std::memcpy(h + p->off_kvoff, p->kv_off.data(), p->kv_off.size() * sizeof(int32_t));
    std::memcpy(h + p->off_dsbase, p->ds_base.data(), p->ds_base.size() * sizeof(long long));
    CUDA_TRY(cudaMemcpyAsync(p->d_buf, h, bytes, cudaMemcpyHostToDevice, stream));
    CUDA_TRY(cudaEventRecord(p->ev[k], stream));
    p->ev_used[k] = true;
    return JATTN_OK;
}

jattn_status set_batch(jattn_plan *p, const int32_t *qo, const int32_t *ko, int32_t B) {
    jattn_status st = check_offsets(qo, ko, B, p->mode.block != 0);
    if (st != JATTN_OK) return st;
    if (p->mode.broadcast_q) {  // every sequence has the shared Q's rows
        for (int32_t b = 1; b < B; ++b)
            if (qo[b + 1] - qo[b] != qo[1] - qo[0]) return JATTN_ERR_INVALID_ARG;
        if (qo[1] - qo[0] < 1) return JATTN_ERR_INVALID_ARG;
        p->bcast_n = qo[1] - qo[0];
    }
    p->dev_planned = false;
    p->B = B;
    p->q_off.assign(qo, qo + B + 1);
    p->kv_off.assign(ko, ko + B + 1);
    p->Tq = qo[B];
    p->Tk = ko[B];
    build_lists(p);
    // dS chunks of the backward: per sequence, H x (key tiles of 128) x (query blocks of 64)
    p->ds_base.resize(static_cast<size_t>(B) + 1);
    int64_t c = 0;
    for (int32_t b = 0; b < B; ++b) {
        p->ds_base[b] = c;
        const int64_t lq = qo[b + 1] - qo[b], lk = ko[b + 1] - ko[b];
        c += static_cast<int64_t>(p->H) * ((lk + kTileRows - 1) / kTileRows) * ((lq + 63) / 64);
    }
    p->ds_base[B] = c;
    p->ds_chunks = c;
    return JATTN_OK;
}

// ---------------------------------------------------------------------------
// tensor maps
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// bf16 view [T, H*Dp] of a token-major tensor; boxes of 64 columns x box_rows rows,
// 128-byte swizzle (the layout the MMA descriptors expect).
bool make_tmap(CUtensorMap *m, const void *ptr, int64_t T, int H, int Dp, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H) * Dp, static_cast<cuuint64_t>(std::max<int64_t>(T, 1))};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * Dp * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t stage_bytes(const jattn_plan *p, int64_t rows) {
    return align_up(static_cast<size_t>(rows) * p->H * p->Dp * 2, kAlign);
}

bool softmax_full(const jattn_plan *p) { return p->mode.act == JATTN_SOFTMAX && p->mode.block == 0; }

// rows of the Q tensor a call reads: the shared rows with broadcast Q, else Tq
int64_t q_rows(const jattn_plan *p) { return p->mode.broadcast_q ? p->bcast_n : p->Tq; }

// broadcast Q: the dQ pass's per-sequence float32 rows, summed afterwards
size_t bcast_ws_bytes(const jattn_plan *p) {
    return p->mode.broadcast_q ? align_up(static_cast<size_t>(p->Tq) * p->H * p->D * 4, kAlign) : 0;
}

// The backward's dS chunks (full attention, host plans, no window): the dK/dV
// pass writes every block's dS and dQ becomes a streaming product of them.
// Device plans (lengths unknown on the host) and sliding windows use the dQ
// pass that recomputes the scores instead.
size_t ds_ws_bytes(const jattn_plan *p) {
    if (p->dev_planned || p->mode.block != 0 || p->mode.window > 0) return 0;
    const size_t planes = p->mode.act == JATTN_SOFTMAX ? 1 : 2;
    return align_up(static_cast<size_t>(p->ds_chunks) * planes * kDsChunkBytes, kAlign);
}

// the backward workspace's first part: Delta, staged inputs, broadcast-Q dQ
// rows, in that order
size_t bwd_ws_base(const jattn_plan *p) {
    size_t n = softmax_full(p) ? align_up(static_cast<size_t>(p->H) * p->Tq * 4, kAlign) : 0;
    if (p->staged) n += 2 * stage_bytes(p, p->Tq) + 2 * stage_bytes(p, p->Tk);
    return n + bcast_ws_bytes(p);
}

// MXFP8: the quantised copies (bf16 [T, H, D]) of q, k, v (forward) and of q,
// dout, k, v (backward, in that order after the base part)
size_t mx_copy_bytes(const jattn_plan *p, int64_t rows) {
    return align_up(static_cast<size_t>(rows) * p->H * p->D * 2, kAlign);
}
size_t mx_bwd_bytes(const jattn_plan *p) {
    return p->mode.mxfp8 ? 2 * mx_copy_bytes(p, p->Tq) + 2 * mx_copy_bytes(p, p->Tk) : 0;
}

// bytes the backward cannot run without: the base part, the MXFP8 copies and,
// for MXFP8 (whose dQ comes only from the dS chunks), the chunks
size_t bwd_ws_min(const jattn_plan *p) {
    return bwd_ws_base(p) + mx_bwd_bytes(p) + (p->mode.mxfp8 ? ds_ws_bytes(p) : 0);
}

Geom make_geom(const jattn_plan *p, int which) {
    Geom g{};
    g.tiles = reinterpret_cast<const Tile *>(p->d_buf + p->off_tiles[which]);
    g.cta_begin = reinterpret_cast<const int32_t *>(p->d_buf + p->off_cta[which]);
    g.q_off = reinterpret_cast<const int32_t *>(p->d_buf + p->off_qoff);
    g.kv_off = reinterpret_cast<const int32_t *>(p->d_buf + p->off_kvoff);
    g.n_tiles = static_cast<int32_t>(p->tiles[which].size());
    g.B = p->B;
    g.H = p->H;
    g.max_q_len = which == JATTN_TILES_Q ? kTileRows : INT_MAX;
    g.max_kv_len = which == JATTN_TILES_KV ? kTileRows : INT_MAX;
    g.Tq = static_cast<int32_t>(p->Tq);
    g.Tk = static_cast<int32_t>(p->Tk);
    g.act = p->mode.act;
    g.block = p->mode.block;
    g.window = std::min(p->mode.window, 1 << 30);  // wider than any sequence: same as no limit
    g.q_bcast = p->mode.broadcast_q;
    g.nb = p->mode.bias_buckets;
    g.scale = p->scale;
    g.bias = nullptr;
    g.status = p->d_status;
    g.wait_ns = kWaitTimeoutNs;
    g.ds = nullptr;
    g.ds_base = p->dev_planned ? nullptr : reinterpret_cast<const long long *>(p->d_buf + p->off_dsbase);
    g.mxfp8 = p->mode.mxfp8;
    g.tile_parallel = which == JATTN_TILES_Q && !p->dev_planned && p->mode.window == 0 && !p->mode.mxfp8 &&
                      p->max_tile_kv <= kTileRows;
    return g;
}

OutDesc out_desc(const jattn_plan *p, void *ptr) {
    OutDesc o;
    o.ptr = ptr;
    o.f32 = p->mode.dtype == JATTN_FP32 ? 1 : 0;
    o.cols = p->D;
    o.ld = static_cast<int64_t>(p->H) * p->D;
    return o;
}

int n_ctas(const jattn_plan *p, int which) { return static_cast<int>(p->cta[which].size()) - 1; }

// Rotary embedding: softmax BlockAttention plans on bf16 data with D in
// {64, 128}; the tables must cover the longest sequence of the batch.  The
// tensor cores take the rotated Q and K as bf16.  A softmax row is normalised,
// so that rounding stays inside the forward tolerance; an activation-mode row
// sums up to 64 unnormalised terms, which the rounding alone can move beyond
// it, so activation mode is not offered with the rotation.
jattn_status check_rope(const jattn_plan *p, const jattn_rope *r) {
    if (r == nullptr) return JATTN_OK;
    if (p->mode.block == 0 || p->staged || (p->D != 64 && p->D != 128) || p->mode.act != JATTN_SOFTMAX)
        return JATTN_ERR_UNSUPPORTED;
    if (r->cos == nullptr || r->sin == nullptr || r->rows < 1) return JATTN_ERR_INVALID_ARG;
    if (!aligned16(r->cos) || !aligned16(r->sin)) return JATTN_ERR_ALIGNMENT;
    if (p->dev_planned) return JATTN_OK;  // lengths unknown on the host: the kernels check the table bounds
    int32_t longest = 0;
    for (int32_t b = 0; b < p->B; ++b)
        longest = std::max({longest, p->q_off[b + 1] - p->q_off[b], p->kv_off[b + 1] - p->kv_off[b]});
    return r->rows < longest ? JATTN_ERR_INVALID_ARG : JATTN_OK;
}

void set_rope(Geom &g, const jattn_rope *r) {
    g.rope_cos = r ? r->cos : nullptr;
    g.rope_sin = r ? r->sin : nullptr;
    g.rope_rows = r ? r->rows : 0;
}

// Per-call launch bookkeeping: records the profiling events (if any) and counts kernels.
struct LaunchLog {
    const jattn_plan *p;
    cudaStream_t st;
    cudaError_t first = cudaSuccess;  // result of recording the call's first event
    LaunchLog(const jattn_plan *plan, cudaStream_t stream) : p(plan), st(stream) {
        p->prof_next = 0;
        first = mark();
    }
    cudaError_t mark() {
        if (p->prof_next < static_cast<int>(p->prof_events.size()))
            return cudaEventRecord(p->prof_events[p->prof_next++], st);
        return cudaSuccess;
    }
    // one kernel was launched (launch functions that skip an empty grid still count as one)
    cudaError_t done(cudaError_t e) {
        if (e == cudaSuccess && first != cudaSuccess) e = first;
        if (e == cudaSuccess) {
            ++p->launches;
            e = mark();
        }
        return e;
    }
};

}  // namespace

namespace jattn {
// Device ordinal of a plan (-1 for a host-only plan), for other translation units.
int plan_device(const jattn_plan *plan) { return plan == nullptr ? -1 : plan->device; }
}  // namespace jattn

extern "C" {

jattn_status jattn_plan_create(const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B, int32_t H, int32_t D,
                               const jattn_mode *mode, int32_t device, jattn_plan **out) {
    if (out == nullptr || mode == nullptr) return JATTN_ERR_INVALID_ARG;
    *out = nullptr;
    if (H < 1 || B < 1) return JATTN_ERR_INVALID_ARG;
    if (D != 32 && D != 64 && D != 128) return (D > 0) ? JATTN_ERR_UNSUPPORTED : JATTN_ERR_INVALID_ARG;
    if (mode->act < JATTN_SOFTMAX || mode->act > JATTN_GELU_TANH) return JATTN_ERR_INVALID_ARG;
    if (mode->block != 0 && mode->block != 64) return JATTN_ERR_UNSUPPORTED;
    if (mode->window < 0 || (mode->window > 0 && mode->block != 0)) return JATTN_ERR_INVALID_ARG;
    if (mode->broadcast_q != 0 && mode->broadcast_q != 1) return JATTN_ERR_INVALID_ARG;
    if (mode->broadcast_q && (mode->block != 0 || mode->dtype != JATTN_BF16 || D < 64))
        return JATTN_ERR_UNSUPPORTED;
    if (mode->dtype != JATTN_BF16 && mode->dtype != JATTN_FP32) return JATTN_ERR_INVALID_ARG;
    // float32 data enter the tensor cores rounded to bf16.  Normalised softmax
    // rows keep that rounding inside the tolerances; unnormalised activation
    // sums over many keys do not, so float32 is offered with softmax only.
    if (mode->dtype == JATTN_FP32 && mode->act != JATTN_SOFTMAX) return JATTN_ERR_UNSUPPORTED;
    // MXFP8 attention: softmax, full attention, bf16, D in {64, 128}, no bias, window or broadcast Q
    if (mode->mxfp8 != 0 && mode->mxfp8 != 1) return JATTN_ERR_INVALID_ARG;
    if (mode->mxfp8 && (mode->act != JATTN_SOFTMAX || mode->block != 0 || mode->window != 0 ||
                        mode->dtype != JATTN_BF16 || mode->broadcast_q || mode->bias_buckets > 0 || D < 64))
        return JATTN_ERR_UNSUPPORTED;
    if (mode->bias_buckets < 0) return JATTN_ERR_INVALID_ARG;
    if (mode->bias_buckets > 0 && H * mode->bias_buckets > kMaxBiasFloats) return JATTN_ERR_UNSUPPORTED;
    if (!(mode->scale >= 0.0f) || std::isinf(mode->scale)) return JATTN_ERR_INVALID_ARG;
    if (device < -1) return JATTN_ERR_INVALID_ARG;

    jattn_plan *p = new (std::nothrow) jattn_plan();
    if (p == nullptr) return JATTN_ERR_INVALID_ARG;
    p->H = H;
    p->D = D;
    p->Dp = D < 64 ? 64 : D;
    p->mode = *mode;
    p->scale = mode->scale > 0.0f ? mode->scale : 1.0f / std::sqrt(static_cast<float>(D));
    p->staged = mode->dtype == JATTN_FP32 || D == 32;
    p->device = device;
    if (device >= 0) {
        DeviceGuard g(device);
        int sms = 0;
        if (!g.ok || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
            delete p;
            return JATTN_ERR_CUDA;
        }
        p->num_sms = sms;
    }
    jattn_status st = set_batch(p, q_offsets, kv_offsets, B);
    if (st != JATTN_OK) {
        delete p;
        return st;
    }
    if (device >= 0) {
        DeviceGuard g(device);
        bool ok = cudaMalloc(&p->d_status, 16) == cudaSuccess && cudaMemset(p->d_status, 0, 16) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p->ev[0], cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p->ev[1], cudaEventDisableTiming) == cudaSuccess;
        if (ok) ok = upload(p, nullptr) == JATTN_OK && cudaStreamSynchronize(nullptr) == cudaSuccess;
        if (!ok) {
            jattn_plan_destroy(p);
            return JATTN_ERR_CUDA;
        }
    }
    *out = p;
    return JATTN_OK;
}

jattn_status jattn_plan_update(jattn_plan *plan, const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B,
                               void *stream) {
    if (plan == nullptr) return JATTN_ERR_INVALID_ARG;
    jattn_status st = check_offsets(q_offsets, kv_offsets, B, plan->mode.block != 0);
    if (st != JATTN_OK) return st;
    st = set_batch(plan, q_offsets, kv_offsets, B);
    if (st != JATTN_OK) return st;
    if (plan->device < 0) return JATTN_OK;
    DeviceGuard g(plan->device);
    if (!g.ok) return note_error("jattn_plan_update: cudaSetDevice failed");
    return upload(plan, static_cast<cudaStream_t>(stream));
}

jattn_status jattn_plan_update_device(jattn_plan *p, const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B,
                                      int64_t Tq, int64_t Tk, void *stream) {
    if (p == nullptr || q_offsets == nullptr || kv_offsets == nullptr) return JATTN_ERR_INVALID_ARG;
    if (p->device < 0) return JATTN_ERR_NO_DEVICE;
    if (B < 1 || Tq < 0 || Tk < 0 || Tq >= INT32_MAX || Tk >= INT32_MAX) return JATTN_ERR_INVALID_ARG;
    if (p->mode.block != 0 && Tq != Tk) return JATTN_ERR_INVALID_ARG;
    if (B > kDevPlanMaxSeqs) return JATTN_ERR_UNSUPPORTED;
    if (!aligned4(q_offsets) || !aligned4(kv_offsets)) return JATTN_ERR_ALIGNMENT;
    if (p->mode.broadcast_q && (Tq % B != 0 || Tq == 0)) return JATTN_ERR_INVALID_ARG;
    const int64_t H = p->H;
    const int64_t cap_q = H * ((Tq + kTileRows - 1) / kTileRows + B);
    const int64_t cap_kv = p->mode.block != 0 ? 0 : H * ((Tk + kTileRows - 1) / kTileRows + B);
    if (cap_q >= INT32_MAX || cap_kv >= INT32_MAX) return JATTN_ERR_INVALID_ARG;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_plan_update_device: cudaSetDevice failed");
    (void)cudaGetLastError();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int C = std::max(p->num_sms, 1);
    size_t off = 0;
    p->off_tiles[0] = off;
    off = align_up(off + static_cast<size_t>(cap_q) * sizeof(Tile), 16);
    p->off_tiles[1] = off;
    off = align_up(off + static_cast<size_t>(cap_kv) * sizeof(Tile), 16);
    for (int w = 0; w < 2; ++w) {
        p->off_cta[w] = off;
        off = align_up(off + static_cast<size_t>(C + 1) * sizeof(int32_t), 16);
    }
    p->off_qoff = off;
    off = align_up(off + static_cast<size_t>(B + 1) * sizeof(int32_t), 16);
    p->off_kvoff = off;
    off = align_up(off + static_cast<size_t>(B + 1) * sizeof(int32_t), 16);
    if (off > p->d_cap) {
        CUDA_TRY(cudaStreamSynchronize(st));  // earlier launches may still read the old buffer
        if (p->d_buf) cudaFree(p->d_buf);
        p->d_buf = nullptr;
        p->d_cap = 0;
        const size_t cap = std::max(off + off / 2, static_cast<size_t>(4096));
        CUDA_TRY(cudaMalloc(&p->d_buf, cap));
        p->d_cap = cap;
    }
    // the offsets are kept with the lists (for jattn_plan_tiles)
    CUDA_TRY(cudaMemcpyAsync(p->d_buf + p->off_qoff, q_offsets, (B + 1) * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
    CUDA_TRY(cudaMemcpyAsync(p->d_buf + p->off_kvoff, kv_offsets, (B + 1) * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                             st));
    DevPlanArgs a{};
    a.q_off = q_offsets;
    a.kv_off = kv_offsets;
    a.B = B;
    a.H = p->H;
    a.block = p->mode.block;
    a.window = std::min(p->mode.window, 1 << 30);
    a.n_ctas = C;
    a.Tq = static_cast<int32_t>(Tq);
    a.Tk = static_cast<int32_t>(Tk);
    a.tiles_q = reinterpret_cast<Tile *>(p->d_buf + p->off_tiles[0]);
    a.tiles_kv = reinterpret_cast<Tile *>(p->d_buf + p->off_tiles[1]);
    a.cta_q = reinterpret_cast<int32_t *>(p->d_buf + p->off_cta[0]);
    a.cta_kv = reinterpret_cast<int32_t *>(p->d_buf + p->off_cta[1]);
    a.cap_q = static_cast<int32_t>(cap_q);
    a.cap_kv = static_cast<int32_t>(cap_kv);
    a.status = p->d_status;
    a.sort_len = 2;
    while (a.sort_len < B) a.sort_len <<= 1;
    a.bcast_n = p->mode.broadcast_q ? static_cast<int32_t>(Tq / B) : 0;
    CUDA_TRY(launch_plan_device(a, st));
    ++p->launches;
    p->B = B;
    p->Tq = Tq;
    p->Tk = Tk;
    p->dev_planned = true;
    if (p->mode.broadcast_q) p->bcast_n = static_cast<int32_t>(Tq / B);
    for (int w = 0; w < 2; ++w) {
        p->tiles[w].clear();
        p->cta[w].assign(static_cast<size_t>(C) + 1, 0);
    }
    p->q_off.assign(static_cast<size_t>(B) + 1, 0);
    p->kv_off.assign(static_cast<size_t>(B) + 1, 0);
    return JATTN_OK;
}

jattn_status jattn_plan_tiles(const jattn_plan *plan, int32_t which, const jattn_tile **tiles, int64_t *n_tiles,
                              const int32_t **cta_begin, int32_t *n_ctas_out) {
    if (plan == nullptr || (which != JATTN_TILES_Q && which != JATTN_TILES_KV)) return JATTN_ERR_INVALID_ARG;
    if (plan->dev_planned) {
        // a device plan: wait for it and bring the lists, ranges and offsets to the host
        jattn_plan *p = const_cast<jattn_plan *>(plan);
        DeviceGuard guard(p->device);
        if (!guard.ok) return note_error("jattn_plan_tiles: cudaSetDevice failed");
        CUDA_TRY(cudaDeviceSynchronize());
        for (int w = 0; w < 2; ++w) {
            CUDA_TRY(cudaMemcpy(p->cta[w].data(), p->d_buf + p->off_cta[w], p->cta[w].size() * sizeof(int32_t),
                                cudaMemcpyDeviceToHost));
        }
        CUDA_TRY(cudaMemcpy(p->q_off.data(), p->d_buf + p->off_qoff, p->q_off.size() * sizeof(int32_t),
                            cudaMemcpyDeviceToHost));
        CUDA_TRY(cudaMemcpy(p->kv_off.data(), p->d_buf + p->off_kvoff, p->kv_off.size() * sizeof(int32_t),
                            cudaMemcpyDeviceToHost));
        for (int w = 0; w < 2; ++w) {
            const size_t n = static_cast<size_t>(std::max(p->cta[w].back(), 0));
            std::vector<Tile> dev(n);
            if (n > 0)
                CUDA_TRY(cudaMemcpy(dev.data(), p->d_buf + p->off_tiles[w], n * sizeof(Tile), cudaMemcpyDeviceToHost));
            p->tiles[w].resize(n);
            for (size_t i = 0; i < n; ++i)
                p->tiles[w][i] = jattn_tile{dev[i].b, dev[i].h, dev[i].q_start, dev[i].q_len, dev[i].kv_start,
                                            dev[i].kv_len};
        }
        p->dev_planned = false;
    }
    if (tiles) *tiles = plan->tiles[which].data();
    if (n_tiles) *n_tiles = static_cast<int64_t>(plan->tiles[which].size());
    if (cta_begin) *cta_begin = plan->cta[which].data();
    if (n_ctas_out) *n_ctas_out = n_ctas(plan, which);
    return JATTN_OK;
}

size_t jattn_fwd_workspace_bytes(const jattn_plan *p) {
    if (p == nullptr) return 0;
    if (p->mode.mxfp8) return mx_copy_bytes(p, p->Tq) + 2 * mx_copy_bytes(p, p->Tk);
    if (!p->staged) return 0;
    return stage_bytes(p, p->Tq) + 2 * stage_bytes(p, p->Tk);
}

size_t jattn_bwd_workspace_bytes(const jattn_plan *p) {
    if (p == nullptr) return 0;
    return bwd_ws_base(p) + mx_bwd_bytes(p) + ds_ws_bytes(p);
}

size_t jattn_bwd_workspace_bytes_min(const jattn_plan *p) { return p == nullptr ? 0 : bwd_ws_min(p); }

void jattn_plan_destroy(jattn_plan *p) {
    if (p == nullptr) return;
    if (p->device >= 0) {
        DeviceGuard g(p->device);
        cudaDeviceSynchronize();
        if (p->d_buf) cudaFree(p->d_buf);
        if (p->d_status) cudaFree(p->d_status);
        for (int k = 0; k < 2; ++k) {
            if (p->h_pin[k]) cudaFreeHost(p->h_pin[k]);
            if (p->ev[k]) cudaEventDestroy(p->ev[k]);
        }
        jattn_plan::HostStep &h = p->hs;
        for (int k = 0; k < 2; ++k) {
            if (h.dev[k]) cudaFree(h.dev[k]);
            if (h.up_done[k]) cudaEventDestroy(h.up_done[k]);
            if (h.comp_done[k]) cudaEventDestroy(h.comp_done[k]);
            if (h.down_done[k]) cudaEventDestroy(h.down_done[k]);
        }
        if (h.ev_start) cudaEventDestroy(h.ev_start);
        if (h.s_up) cudaStreamDestroy(h.s_up);
        if (h.s_comp) cudaStreamDestroy(h.s_comp);
        if (h.s_down) cudaStreamDestroy(h.s_down);
    }
    delete p;
}

jattn_status jattn_fwd(const jattn_plan *p, const void *q, const void *k, const void *v, const float *bias, void *out,
                       float *lse, void *workspace, size_t workspace_bytes, void *stream) {
    return jattn_fwd_rope(p, q, k, v, bias, nullptr, out, lse, workspace, workspace_bytes, stream);
}

jattn_status jattn_fwd_rope(const jattn_plan *p, const void *q, const void *k, const void *v, const float *bias,
                            const jattn_rope *rope, void *out, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream) {
    if (p == nullptr) return JATTN_ERR_INVALID_ARG;
    if (p->device < 0) return JATTN_ERR_NO_DEVICE;
    if (!q || !k || !v || !out) return JATTN_ERR_INVALID_ARG;
    {
        const jattn_status e = check_rope(p, rope);
        if (e != JATTN_OK) return e;
    }
    if ((p->mode.bias_buckets > 0) != (bias != nullptr)) return JATTN_ERR_INVALID_ARG;
    if (lse != nullptr && p->mode.act != JATTN_SOFTMAX) return JATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) || !aligned16(bias))
        return JATTN_ERR_ALIGNMENT;
    const size_t need = jattn_fwd_workspace_bytes(p);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return JATTN_ERR_WORKSPACE;
    if (need > 0 && !aligned16(workspace)) return JATTN_ERR_ALIGNMENT;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_fwd: cudaSetDevice failed");
    (void)cudaGetLastError();  // report only errors of this call
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int f32 = p->mode.dtype == JATTN_FP32;
    const void *qq = q, *kk = k, *vv = v;
    if (p->mode.mxfp8 && p->dev_planned) return JATTN_ERR_UNSUPPORTED;  // the quantisation reads host-planned offsets
    LaunchLog log(p, st);
    if (p->mode.mxfp8) {  // Q, K, V replaced by the values of their MXFP8 quantisation
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        void *qs = ws, *ks = ws + mx_copy_bytes(p, p->Tq), *vs = ws + mx_copy_bytes(p, p->Tq) + mx_copy_bytes(p, p->Tk);
        MxJobs jobs{};
        add_mx_job(jobs, p, JATTN_TILES_Q, q, qs);
        add_mx_job(jobs, p, JATTN_TILES_KV, k, ks);
        add_mx_job(jobs, p, JATTN_TILES_KV, v, vs);
        CUDA_TRY(log.done(launch_mx_quant(jobs, p->H, p->D, st)));
        qq = qs;
        kk = ks;
        vv = vs;
    }
    if (p->staged) {
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        void *qs = ws, *ks = ws + stage_bytes(p, p->Tq), *vs = ws + stage_bytes(p, p->Tq) + stage_bytes(p, p->Tk);
        CUDA_TRY(log.done(launch_stage(q, f32, p->Tq * p->H, p->D, p->Dp, qs, st)));
        CUDA_TRY(log.done(launch_stage(k, f32, p->Tk * p->H, p->D, p->Dp, ks, st)));
        CUDA_TRY(log.done(launch_stage(v, f32, p->Tk * p->H, p->D, p->Dp, vs, st)));
        qq = qs;
        kk = ks;
        vv = vs;
    }
    TmapSet tm;
    if (!make_tmap(&tm.q, qq, q_rows(p), p->H, p->Dp, 128) || !make_tmap(&tm.k, kk, p->Tk, p->H, p->Dp, 128) ||
        !make_tmap(&tm.v, vv, p->Tk, p->H, p->Dp, 128))
        return note_error("jattn_fwd: cuTensorMapEncodeTiled failed");
    tm.dout = tm.q;
    FwdArgs a;
    a.g = make_geom(p, JATTN_TILES_Q);
    a.g.bias = bias;
    a.out = out_desc(p, out);
    a.lse = lse;
    set_rope(a.g, rope);
    const bool act = p->mode.act != JATTN_SOFTMAX;
    return cuda_status(log.done(rope ? launch_fwd_rope(p->Dp, act, tm, a, n_ctas(p, JATTN_TILES_Q), st)
                                     : launch_fwd(p->Dp, act, tm, a, n_ctas(p, JATTN_TILES_Q), st)),
                       "jattn_fwd: forward kernel launch");
}

jattn_status jattn_bwd(const jattn_plan *p, const void *dout, const void *q, const void *k, const void *v,
                       const float *bias, const void *out, const float *lse, void *dq, void *dk, void *dv,
                       float *dbias, void *workspace, size_t workspace_bytes, void *stream) {
    return jattn_bwd_rope(p, dout, q, k, v, bias, nullptr, out, lse, dq, dk, dv, dbias, workspace, workspace_bytes,
                          stream);
}

jattn_status jattn_bwd_rope(const jattn_plan *p, const void *dout, const void *q, const void *k, const void *v,
                            const float *bias, const jattn_rope *rope, const void *out, const float *lse, void *dq,
                            void *dk, void *dv, float *dbias, void *workspace, size_t workspace_bytes, void *stream) {
    if (p == nullptr) return JATTN_ERR_INVALID_ARG;
    if (p->device < 0) return JATTN_ERR_NO_DEVICE;
    if (!dout || !q || !k || !v || !out || !dq || !dk || !dv) return JATTN_ERR_INVALID_ARG;
    {
        const jattn_status e = check_rope(p, rope);
        if (e != JATTN_OK) return e;
    }
    if ((p->mode.bias_buckets > 0) != (bias != nullptr)) return JATTN_ERR_INVALID_ARG;
    if (softmax_full(p) && lse == nullptr) return JATTN_ERR_INVALID_ARG;
    if (dbias != nullptr && bias == nullptr) return JATTN_ERR_INVALID_ARG;
    if (dbias != nullptr && p->mode.block != 0) return JATTN_ERR_UNSUPPORTED;
    if (dbias != nullptr && !aligned16(dbias)) return JATTN_ERR_ALIGNMENT;
    if (!aligned16(dout) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv) || !aligned16(bias) || !aligned16(lse))
        return JATTN_ERR_ALIGNMENT;
    if (p->mode.mxfp8 && p->dev_planned) return JATTN_ERR_UNSUPPORTED;  // the quantisation reads host-planned offsets
    const size_t need = bwd_ws_min(p);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return JATTN_ERR_WORKSPACE;
    if ((need > 0 || workspace != nullptr) && !aligned16(workspace)) return JATTN_ERR_ALIGNMENT;
    // dS chunks when the workspace holds them (and the plan allows them); MXFP8 always
    const size_t base = bwd_ws_base(p), mxb = mx_bwd_bytes(p);
    const size_t ds_need = ds_ws_bytes(p);
    const bool use_ds =
        ds_need > 0 && rope == nullptr && workspace != nullptr && workspace_bytes >= base + mxb + ds_need;
    if (p->mode.mxfp8 && !use_ds) return JATTN_ERR_WORKSPACE;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_bwd: cudaSetDevice failed");
    (void)cudaGetLastError();  // report only errors of this call
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int f32 = p->mode.dtype == JATTN_FP32;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *delta = nullptr;
    if (softmax_full(p)) {
        delta = reinterpret_cast<float *>(ws);
        ws += align_up(static_cast<size_t>(p->H) * p->Tq * 4, kAlign);
    }
    const void *qq = q, *kk = k, *vv = v, *dd = dout;
    LaunchLog log(p, st);
    if (p->staged) {
        void *qs = ws;
        void *ds = ws + stage_bytes(p, p->Tq);
        void *ks = ws + 2 * stage_bytes(p, p->Tq);
        void *vs = ws + 2 * stage_bytes(p, p->Tq) + stage_bytes(p, p->Tk);
        if (log.done(launch_stage(q, f32, p->Tq * p->H, p->D, p->Dp, qs, st)) != cudaSuccess ||
            log.done(launch_stage(dout, f32, p->Tq * p->H, p->D, p->Dp, ds, st)) != cudaSuccess ||
            log.done(launch_stage(k, f32, p->Tk * p->H, p->D, p->Dp, ks, st)) != cudaSuccess ||
            log.done(launch_stage(v, f32, p->Tk * p->H, p->D, p->Dp, vs, st)) != cudaSuccess)
            return JATTN_ERR_CUDA;
        qq = qs;
        dd = ds;
        kk = ks;
        vv = vs;
    }
    float *dq_rows = nullptr;  // broadcast Q: per-sequence float32 dQ rows, after Delta and the staging
    if (p->mode.broadcast_q) dq_rows = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + base - bcast_ws_bytes(p));
    void *ds = use_ds ? static_cast<void *>(static_cast<uint8_t *>(workspace) + base + mxb) : nullptr;
    if (p->mode.mxfp8) {  // Q, dO, K, V replaced by the values of their MXFP8 quantisation
        uint8_t *mx = static_cast<uint8_t *>(workspace) + base;
        void *qs = mx, *ds_ = mx + mx_copy_bytes(p, p->Tq), *ks = mx + 2 * mx_copy_bytes(p, p->Tq);
        void *vs = mx + 2 * mx_copy_bytes(p, p->Tq) + mx_copy_bytes(p, p->Tk);
        MxJobs jobs{};
        add_mx_job(jobs, p, JATTN_TILES_Q, q, qs);
        add_mx_job(jobs, p, JATTN_TILES_Q, dout, ds_);
        add_mx_job(jobs, p, JATTN_TILES_KV, k, ks);
        add_mx_job(jobs, p, JATTN_TILES_KV, v, vs);
        if (log.done(launch_mx_quant(jobs, p->H, p->D, st)) != cudaSuccess)
            return note_error("jattn_bwd: MXFP8 quantisation launch");
        qq = qs;
        dd = ds_;
        kk = ks;
        vv = vs;
    }
    BwdArgs a;
    a.lse = lse;
    a.delta = delta;
    a.dq = out_desc(p, dq);
    if (dq_rows != nullptr) {
        a.dq.ptr = dq_rows;
        a.dq.f32 = 1;
    }
    a.dk = out_desc(p, dk);
    a.dv = out_desc(p, dv);
    a.dbias = dbias;
    TmapSet tm;
    if (p->mode.block != 0) {
        if (!make_tmap(&tm.q, qq, p->Tq, p->H, p->Dp, 128) || !make_tmap(&tm.k, kk, p->Tk, p->H, p->Dp, 128) ||
            !make_tmap(&tm.v, vv, p->Tk, p->H, p->Dp, 128) || !make_tmap(&tm.dout, dd, p->Tq, p->H, p->Dp, 128))
            return note_error("jattn_bwd: cuTensorMapEncodeTiled failed");
        a.g = make_geom(p, JATTN_TILES_Q);
        a.g.bias = bias;
        set_rope(a.g, rope);
        return cuda_status(log.done(launch_bwd_block(p->Dp, tm, a, n_ctas(p, JATTN_TILES_Q), st)),
                           "jattn_bwd: block kernel launch");
    }
    if (delta != nullptr) {
        jattn_status e = cuda_status(log.done(launch_delta(out, dout, f32, p->Tq, p->H, p->D, delta, st)),
                                     "jattn_bwd: delta kernel launch");
        if (e != JATTN_OK) return e;
    }
    const bool act = p->mode.act != JATTN_SOFTMAX;
    if (dbias != nullptr) {  // the pass that sums dS adds every pair's into it
        jattn_status e = cuda_status(
            cudaMemsetAsync(dbias, 0, static_cast<size_t>(p->H) * p->mode.bias_buckets * sizeof(float), st),
            "jattn_bwd: dbias zero fill");
        if (e != JATTN_OK) return e;
    }
    if (use_ds) {
        // pass 1: dK, dV over key-major tiles, writing every block's dS chunk
        if (!make_tmap(&tm.q, qq, q_rows(p), p->H, p->Dp, 64) || !make_tmap(&tm.dout, dd, p->Tq, p->H, p->Dp, 64) ||
            !make_tmap(&tm.k, kk, p->Tk, p->H, p->Dp, 128) || !make_tmap(&tm.v, vv, p->Tk, p->H, p->Dp, 128))
            return note_error("jattn_bwd: cuTensorMapEncodeTiled failed");
        a.g = make_geom(p, JATTN_TILES_KV);
        a.g.bias = bias;
        a.g.ds = ds;
        {
            jattn_status e = cuda_status(log.done(launch_bwd_dkdv(p->Dp, act, tm, a, n_ctas(p, JATTN_TILES_KV), st)),
                                         "jattn_bwd: dK/dV kernel launch");
            if (e != JATTN_OK) return e;
        }
        // pass 2: dQ = scale dS K over query-major tiles (K in 128-row tiles, as above)
        a.g = make_geom(p, JATTN_TILES_Q);
        a.g.bias = bias;
        a.g.ds = ds;
        {
            jattn_status e = cuda_status(log.done(launch_bwd_dq_gemm(p->Dp, act, tm, a, n_ctas(p, JATTN_TILES_Q), st)),
                                         "jattn_bwd: dQ product launch");
            if (e != JATTN_OK) return e;
        }
        if (dq_rows != nullptr)  // the shared queries' gradient: the sum over the sequences
            return cuda_status(
                log.done(launch_bcast_reduce(dq_rows, p->B, p->bcast_n, static_cast<int64_t>(p->H) * p->D, dq, st)),
                "jattn_bwd: dQ reduction launch");
        return JATTN_OK;
    }
    // pass 1: dQ over query-major tiles (128 query rows, keys in blocks of 64)
    if (!make_tmap(&tm.q, qq, q_rows(p), p->H, p->Dp, 128) || !make_tmap(&tm.dout, dd, p->Tq, p->H, p->Dp, 128) ||
        !make_tmap(&tm.k, kk, p->Tk, p->H, p->Dp, 64) || !make_tmap(&tm.v, vv, p->Tk, p->H, p->Dp, 64))
        return note_error("jattn_bwd: cuTensorMapEncodeTiled failed");
    a.g = make_geom(p, JATTN_TILES_Q);
    a.g.bias = bias;
    {
        jattn_status e = cuda_status(log.done(launch_bwd_dq(p->Dp, act, tm, a, n_ctas(p, JATTN_TILES_Q), st)),
                                     "jattn_bwd: dQ kernel launch");
        if (e != JATTN_OK) return e;
    }
    if (dq_rows != nullptr) {  // the shared queries' gradient: the sum over the sequences
        jattn_status e = cuda_status(
            log.done(launch_bcast_reduce(dq_rows, p->B, p->bcast_n, static_cast<int64_t>(p->H) * p->D, dq, st)),
            "jattn_bwd: dQ reduction launch");
        if (e != JATTN_OK) return e;
    }
    // pass 2: dK, dV over key-major tiles (128 key rows, queries in blocks of 64)
    if (!make_tmap(&tm.q, qq, q_rows(p), p->H, p->Dp, 64) || !make_tmap(&tm.dout, dd, p->Tq, p->H, p->Dp, 64) ||
        !make_tmap(&tm.k, kk, p->Tk, p->H, p->Dp, 128) || !make_tmap(&tm.v, vv, p->Tk, p->H, p->Dp, 128))
        return note_error("jattn_bwd: cuTensorMapEncodeTiled failed");
    a.g = make_geom(p, JATTN_TILES_KV);
    a.g.bias = bias;
    return cuda_status(log.done(launch_bwd_dkdv(p->Dp, act, tm, a, n_ctas(p, JATTN_TILES_KV), st)),
                       "jattn_bwd: dK/dV kernel launch");
}

jattn_status jattn_step_host(jattn_plan *p, const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B,
                             const void *q, const void *k, const void *v, const void *dout, const float *bias,
                             void *out, float *lse, void *dq, void *dk, void *dv, void *stream) {
    if (p == nullptr) return JATTN_ERR_INVALID_ARG;
    if (p->mode.broadcast_q) return JATTN_ERR_UNSUPPORTED;
    if (p->device < 0) return JATTN_ERR_NO_DEVICE;
    if (!q || !k || !v || !dout || !out || !dq || !dk || !dv) return JATTN_ERR_INVALID_ARG;
    if ((p->mode.bias_buckets > 0) != (bias != nullptr)) return JATTN_ERR_INVALID_ARG;
    jattn_status st = check_offsets(q_offsets, kv_offsets, B, p->mode.block != 0);
    if (st != JATTN_OK) return st;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_step_host: cudaSetDevice failed");
    (void)cudaGetLastError();
    jattn_plan::HostStep &h = p->hs;
    if (!h.init) {
        CUDA_TRY(cudaStreamCreateWithFlags(&h.s_up, cudaStreamNonBlocking));
        CUDA_TRY(cudaStreamCreateWithFlags(&h.s_comp, cudaStreamNonBlocking));
        CUDA_TRY(cudaStreamCreateWithFlags(&h.s_down, cudaStreamNonBlocking));
        CUDA_TRY(cudaEventCreateWithFlags(&h.ev_start, cudaEventDisableTiming));
        for (int i = 0; i < 2; ++i) {
            CUDA_TRY(cudaEventCreateWithFlags(&h.up_done[i], cudaEventDisableTiming));
            CUDA_TRY(cudaEventCreateWithFlags(&h.comp_done[i], cudaEventDisableTiming));
            CUDA_TRY(cudaEventCreateWithFlags(&h.down_done[i], cudaEventDisableTiming));
        }
        h.init = true;
    }
    const int i = h.next;
    // host side of the re-plan; the tile lists reach the device on the compute
    // stream, after the previous call's kernels
    set_batch(p, q_offsets, kv_offsets, B);

    // staging set i: q, k, v, dout, bias, out, lse, dq, dk, dv, workspaces
    const size_t es = p->mode.dtype == JATTN_FP32 ? 4 : 2;
    const size_t nq = static_cast<size_t>(p->Tq) * p->H * p->D * es;
    const size_t nk = static_cast<size_t>(p->Tk) * p->H * p->D * es;
    const size_t nb = bias ? static_cast<size_t>(p->H) * p->mode.bias_buckets * 4 : 0;
    const size_t nl = p->mode.act == JATTN_SOFTMAX ? static_cast<size_t>(p->H) * p->Tq * 4 : 0;
    const size_t nfw = jattn_fwd_workspace_bytes(p), nbw = jattn_bwd_workspace_bytes(p);
    const size_t sizes[12] = {nq, nk, nk, nq, nb, nq, nl, nq, nk, nk, nfw, nbw};
    size_t offs[12], total = 0;
    for (int j = 0; j < 12; ++j) {
        offs[j] = total;
        total += align_up(sizes[j], kAlign);
    }
    if (total > h.cap[i]) {
        if (h.used[i]) CUDA_TRY(cudaEventSynchronize(h.down_done[i]));  // its last use
        if (h.dev[i]) cudaFree(h.dev[i]);
        h.dev[i] = nullptr;
        h.cap[i] = 0;
        const size_t cap = total + total / 4;
        CUDA_TRY(cudaMalloc(&h.dev[i], cap));
        h.cap[i] = cap;
    }
    uint8_t *d = h.dev[i];
    void *dq_in = d + offs[0], *dk_in = d + offs[1], *dv_in = d + offs[2], *ddo = d + offs[3];
    float *dbias = nb ? reinterpret_cast<float *>(d + offs[4]) : nullptr;
    void *dout_ = d + offs[5];
    float *dlse = nl ? reinterpret_cast<float *>(d + offs[6]) : nullptr;
    void *ddq = d + offs[7], *ddk = d + offs[8], *ddv = d + offs[9];
    void *fws = nfw ? d + offs[10] : nullptr, *bws = nbw ? d + offs[11] : nullptr;

    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaEventRecord(h.ev_start, cs));
    // uploads: after the caller's queued work and after set i's inputs were last read
    CUDA_TRY(cudaStreamWaitEvent(h.s_up, h.ev_start, 0));
    if (h.used[i]) CUDA_TRY(cudaStreamWaitEvent(h.s_up, h.comp_done[i], 0));
    CUDA_TRY(cudaMemcpyAsync(dq_in, q, nq, cudaMemcpyHostToDevice, h.s_up));
    CUDA_TRY(cudaMemcpyAsync(dk_in, k, nk, cudaMemcpyHostToDevice, h.s_up));
    CUDA_TRY(cudaMemcpyAsync(dv_in, v, nk, cudaMemcpyHostToDevice, h.s_up));
    CUDA_TRY(cudaMemcpyAsync(ddo, dout, nq, cudaMemcpyHostToDevice, h.s_up));
    if (nb) CUDA_TRY(cudaMemcpyAsync(dbias, bias, nb, cudaMemcpyHostToDevice, h.s_up));
    CUDA_TRY(cudaEventRecord(h.up_done[i], h.s_up));
    // kernels: after the uploads and after set i's outputs were last read back
    CUDA_TRY(cudaStreamWaitEvent(h.s_comp, h.ev_start, 0));
    CUDA_TRY(cudaStreamWaitEvent(h.s_comp, h.up_done[i], 0));
    if (h.used[i]) CUDA_TRY(cudaStreamWaitEvent(h.s_comp, h.down_done[i], 0));
    st = upload(p, h.s_comp);
    if (st != JATTN_OK) return st;
    st = jattn_fwd(p, dq_in, dk_in, dv_in, dbias, dout_, dlse, fws, nfw, h.s_comp);
    if (st != JATTN_OK) return st;
    st = jattn_bwd(p, ddo, dq_in, dk_in, dv_in, dbias, dout_, dlse, ddq, ddk, ddv, nullptr, bws, nbw, h.s_comp);
    if (st != JATTN_OK) return st;
    CUDA_TRY(cudaEventRecord(h.comp_done[i], h.s_comp));
    // downloads
    CUDA_TRY(cudaStreamWaitEvent(h.s_down, h.comp_done[i], 0));
    CUDA_TRY(cudaMemcpyAsync(out, dout_, nq, cudaMemcpyDeviceToHost, h.s_down));
    if (lse && nl) CUDA_TRY(cudaMemcpyAsync(lse, dlse, nl, cudaMemcpyDeviceToHost, h.s_down));
    CUDA_TRY(cudaMemcpyAsync(dq, ddq, nq, cudaMemcpyDeviceToHost, h.s_down));
    CUDA_TRY(cudaMemcpyAsync(dk, ddk, nk, cudaMemcpyDeviceToHost, h.s_down));
    CUDA_TRY(cudaMemcpyAsync(dv, ddv, nk, cudaMemcpyDeviceToHost, h.s_down));
    CUDA_TRY(cudaEventRecord(h.down_done[i], h.s_down));
    h.used[i] = true;
    h.last = i;
    h.next = i ^ 1;
    return JATTN_OK;
}

jattn_status jattn_step_host_join(jattn_plan *p, void *stream) {
    if (p == nullptr) return JATTN_ERR_INVALID_ARG;
    if (p->device < 0 || p->hs.last < 0) return JATTN_OK;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_step_host_join: cudaSetDevice failed");
    // downloads run in call order on one stream: the last call's event covers all
    CUDA_TRY(cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), p->hs.down_done[p->hs.last], 0));
    return JATTN_OK;
}

jattn_status jattn_plan_set_events(jattn_plan *p, void *const *events, int32_t n_events) {
    if (p == nullptr || n_events < 0 || (n_events > 0 && events == nullptr)) return JATTN_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_events; ++i)
        if (events[i] == nullptr) return JATTN_ERR_INVALID_ARG;
    p->prof_events.clear();
    for (int32_t i = 0; i < n_events; ++i) p->prof_events.push_back(static_cast<cudaEvent_t>(events[i]));
    return JATTN_OK;
}

int64_t jattn_plan_launch_count(const jattn_plan *p) { return p == nullptr ? 0 : p->launches; }

jattn_status jattn_mxfp8_quantize(const jattn_plan *p, const void *x, int32_t which, void *xq, void *stream) {
    if (p == nullptr || x == nullptr || xq == nullptr) return JATTN_ERR_INVALID_ARG;
    if (which != JATTN_TILES_Q && which != JATTN_TILES_KV) return JATTN_ERR_INVALID_ARG;
    if (p->device < 0) return JATTN_ERR_NO_DEVICE;
    if (!p->mode.mxfp8 || p->dev_planned) return JATTN_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(xq)) return JATTN_ERR_ALIGNMENT;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_mxfp8_quantize: cudaSetDevice failed");
    (void)cudaGetLastError();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    MxJobs jobs{};
    add_mx_job(jobs, p, which, x, xq);
    LaunchLog log(p, st);
    return cuda_status(log.done(launch_mx_quant(jobs, p->H, p->D, st)),
                       "jattn_mxfp8_quantize: kernel launch");
}

jattn_status jattn_test_fwd_stall(const jattn_plan *p, const void *q, const void *k, const void *v, void *out,
                                  float *lse, uint64_t wait_ns, void *stream) {
    if (p == nullptr) return JATTN_ERR_INVALID_ARG;
    if (p->device < 0) return JATTN_ERR_NO_DEVICE;
    if (!q || !k || !v || !out || !lse) return JATTN_ERR_INVALID_ARG;
    if (wait_ns < 100000ull || wait_ns > kWaitTimeoutNs) return JATTN_ERR_INVALID_ARG;
    if (p->mode.act != JATTN_SOFTMAX || p->mode.bias_buckets > 0 || p->mode.window > 0 || p->mode.block != 0 ||
        p->mode.broadcast_q || p->staged)
        return JATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return JATTN_ERR_ALIGNMENT;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_test_fwd_stall: cudaSetDevice failed");
    (void)cudaGetLastError();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    TmapSet tm;
    if (!make_tmap(&tm.q, q, q_rows(p), p->H, p->Dp, 128) || !make_tmap(&tm.k, k, p->Tk, p->H, p->Dp, 128) ||
        !make_tmap(&tm.v, v, p->Tk, p->H, p->Dp, 128))
        return note_error("jattn_test_fwd_stall: cuTensorMapEncodeTiled failed");
    tm.dout = tm.q;
    FwdArgs a;
    a.g = make_geom(p, JATTN_TILES_Q);
    a.g.wait_ns = wait_ns;
    a.out = out_desc(p, out);
    a.lse = lse;
    set_rope(a.g, nullptr);
    LaunchLog log(p, st);
    return cuda_status(log.done(launch_fwd_stall(p->Dp, tm, a, n_ctas(p, JATTN_TILES_Q), st)),
                       "jattn_test_fwd_stall: kernel launch");
}

jattn_status jattn_check_device_status(const jattn_plan *p, void *stream) {
    if (p == nullptr) return JATTN_ERR_INVALID_ARG;
    if (p->device < 0) return JATTN_ERR_NO_DEVICE;
    DeviceGuard guard(p->device);
    if (!guard.ok) return note_error("jattn_check_device_status: cudaSetDevice failed");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUDA_TRY(cudaStreamSynchronize(st));
    int code = 0;
    CUDA_TRY(cudaMemcpy(&code, p->d_status, sizeof(int), cudaMemcpyDeviceToHost));
    if (code != 0) CUDA_TRY(cudaMemset(p->d_status, 0, sizeof(int)));
    return static_cast<jattn_status>(code);
}

const char *jattn_last_cuda_error(void) { return g_last_cuda_error; }

jattn_status jattn_shard(const int32_t *q_offsets, const int32_t *kv_offsets, int32_t B, int32_t world,
                         int32_t *rank_of) {
    if (rank_of == nullptr || world < 1) return JATTN_ERR_INVALID_ARG;
    const jattn_status st = check_offsets(q_offsets, kv_offsets, B, false);
    if (st != JATTN_OK) return st;
    std::vector<int64_t> cost(static_cast<size_t>(B));
    for (int32_t b = 0; b < B; ++b) {
        const int64_t lq = q_offsets[b + 1] - q_offsets[b], lk = kv_offsets[b + 1] - kv_offsets[b];
        cost[b] = lq * lk + 64 * (lq + lk);
    }
    std::vector<int32_t> order(static_cast<size_t>(B));
    for (int32_t b = 0; b < B; ++b) order[b] = b;
    std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return cost[x] > cost[y]; });
    using Slot = std::pair<int64_t, int32_t>;  // (load, rank)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int32_t r = 0; r < world; ++r) heap.push({0, r});
    for (int32_t b : order) {
        Slot s = heap.top();
        heap.pop();
        rank_of[b] = s.second;
        heap.push({s.first + cost[b], s.second});
    }
    return JATTN_OK;
}

const char *jattn_status_str(jattn_status s) {
    switch (s) {
        case JATTN_OK: return "ok";
        case JATTN_ERR_INVALID_ARG: return "invalid argument";
        case JATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case JATTN_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
        case JATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case JATTN_ERR_CUDA: return "CUDA runtime error";
        case JATTN_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case JATTN_ERR_DEVICE_CHECK: return "device rejected a tile record";
        case JATTN_ERR_NO_DEVICE: return "plan has no device";
    }
    return "unknown status";
}

}  // extern "C"
