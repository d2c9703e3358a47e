// common.h -- constants and kernel parameter blocks shared by the host glue
// (api.cpp) and the CUDA kernels.  Plain C++ types only.
#pragma once

#include <stdint.h>

namespace jattn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// status codes written to the device status word (same values as jattn_status)
constexpr int kStatusDeviceTimeout = 6;
constexpr int kStatusDeviceCheck = 7;

// a bounded wait gives up after this much wall time (the kernels take the
// limit from Geom::wait_ns, which the library sets to this value; only the
// stall test build of the forward shortens it)
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s

// largest bias table (H * NB floats) the kernels stage in shared memory
constexpr int kMaxBiasFloats = 256;
// largest reflected bias table (H * (2 * (NB + 30) + 1) floats) the softmax kernels stage
constexpr int kMaxBiasExtFloats = 1024;

// online-softmax rescale threshold (log2 units): the running max is only moved,
// and O rescaled, when a row's max grows by more than this, so unnormalised
// probabilities stay below 2^8.
constexpr float kRescaleThreshold = 8.0f;

// Device tile record: the ABI's 24-byte record plus the tile's first query and
// key positions local to its sequence (precomputed by the planner).
struct Tile {
    int32_t b, h, q_start, q_len, kv_start, kv_len, q_loc0, kv_loc0;
};

enum Act : int32_t { kSoftmax = 0, kSilu = 1, kGeluTanh = 2 };

// Geometry and mode shared by every attention kernel.
struct Geom {
    const Tile *tiles;        // scheduled tile list (device)
    const int32_t *cta_begin; // [n_ctas + 1] (device)
    const int32_t *q_off;     // [B + 1] (device)
    const int32_t *kv_off;    // [B + 1] (device)
    int32_t n_tiles;
    int32_t B;
    int32_t H;
    int32_t max_q_len;        // tile validation: largest q_len a record may carry
    int32_t max_kv_len;       // ... and kv_len
    int32_t Tq, Tk;
    int32_t act;
    int32_t block;            // 0 or 64
    int32_t window;           // 0, or W > 0: keys with |i - j| < W only (local positions)
    int32_t nb;               // bias buckets, 0 = none
    float scale;              // score scale
    const float *bias;        // [H, nb] or nullptr
    int *status;              // device status word
    const float *rope_cos;    // rotary embedding: cos [rope_rows, D/2] float32, or nullptr (off)
    const float *rope_sin;    // ... and sin
    int32_t rope_rows;        // table positions 0 .. rope_rows - 1
    int32_t q_bcast;          // 1: every sequence's queries are the rows 0 .. Lq-1 of one shared Q
                              // (Q is read at the local row, O / dO / lse at the sequence's rows)
    unsigned long long wait_ns;  // limit of every bounded wait (kWaitTimeoutNs)
    // backward with dS chunks (full attention): the dK/dV pass writes every block's
    // dS to `ds` and the dQ product reads it back; chunk index of (sequence b,
    // head h, key tile t, 64-query block i) = ds_base[b] + (h * nkt_b + t) * nqb_b + i
    void *ds;                 // chunk workspace (16-byte aligned), or nullptr (off)
    const long long *ds_base; // [B + 1] first chunk of every sequence (device)
    int32_t mxfp8;            // 1: MXFP8 attention (P, and in the backward dS, quantised online)
    int32_t tile_parallel;    // 1: every query tile meets at most one 128-key block (host plans
                              // without a window); the forward may give whole tiles to its groups
};

// one dS chunk: 128 keys x 64 queries of bf16 (activation mode: two of them, hi and lo)
constexpr int kDsChunkBytes = 128 * 64 * 2;

// Where a [T, H, D] result goes: element (t, h, c) at ptr[t*ld + h*cols + c] for c < cols.
struct OutDesc {
    void *ptr;
    int32_t f32;   // 1: float32, 0: bfloat16
    int32_t cols;  // real D (<= padded D)
    int64_t ld;    // row stride in elements (H * cols)
};

struct FwdArgs {
    Geom g;
    OutDesc out;
    float *lse;    // [H, Tq] or nullptr
};

struct BwdArgs {
    Geom g;
    const float *lse;    // [H, Tq] (full softmax)
    const float *delta;  // [H, Tq] (full softmax)
    OutDesc dq, dk, dv;
    float *dbias;        // [H, nb] bias-table gradient (zeroed first, atomically summed) or nullptr
};

}  // namespace jattn
