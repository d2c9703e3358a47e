"""Independent tile enumerator -- TEST INFRASTRUCTURE ONLY.

A plain Python restatement of which work tiles a jagged batch has, used to
check the library's planner record by record.  The pages ("Training GEM at LLM
scale", section "Generalized Dot-Product Attention (GDPA)", software-level tile
scheduling) describe precomputing the valid tiles on the CPU and skipping empty
ones; the tile shape and record layout below are this library's reading:

  record = (b, h, q_start, q_len, kv_start, kv_len), int32, global row indices.

  query-major list (forward and the dQ pass), canonical order b, q-tile, h:
    full attention : one record per 128-row query tile of every sequence with
                     Lq > 0, spanning all of that sequence's keys (kv_len may be 0)
    block attention: one record per 128-row chunk (two 64-token blocks); the key
                     range is the same chunk of rows
  key-major list (the dK/dV pass), canonical order b, kv-tile, h:
    full attention : one record per 128-row key tile of every sequence with
                     Lk > 0, spanning all of that sequence's queries (q_len may be 0)
    block attention: empty (its backward runs on the query-major list)
  sliding window W (section "BlockAttention": off-window tiles are skipped):
    the same records, each one's other range cut to the band |i - j| < W of
    its rows: a query tile [s, s + n) keeps keys [s - W + 1, s + n + W - 1)
    clipped to the sequence, and a key tile keeps queries likewise (the range
    may become empty; the record stays, so its rows are still written)
"""
from __future__ import annotations

import numpy as np

TILE_Q = 128
TILE_KV = 128


def _band(s: int, n: int, L: int, window: int):
    """Positions of the other side within the window of rows [s, s + n)."""
    lo = min(L, max(0, s - window + 1))
    hi = min(L, s + n + window - 1)
    return lo, max(hi, lo)  # empty when nothing is in reach, still inside the sequence


def q_major(q_off, kv_off, H: int, block: int = 0, window: int = 0) -> np.ndarray:
    out = []
    B = len(q_off) - 1
    for b in range(B):
        q0, Lq = int(q_off[b]), int(q_off[b + 1] - q_off[b])
        k0, Lk = int(kv_off[b]), int(kv_off[b + 1] - kv_off[b])
        t = 0
        while t * TILE_Q < Lq:
            ql = min(TILE_Q, Lq - t * TILE_Q)
            for h in range(H):
                if block:
                    out.append((b, h, q0 + t * TILE_Q, ql, k0 + t * TILE_Q, ql))
                elif window:
                    lo, hi = _band(t * TILE_Q, ql, Lk, window)
                    out.append((b, h, q0 + t * TILE_Q, ql, k0 + lo, hi - lo))
                else:
                    out.append((b, h, q0 + t * TILE_Q, ql, k0, Lk))
            t += 1
    return np.array(out, dtype=np.int32).reshape(-1, 6)


def kv_major(q_off, kv_off, H: int, block: int = 0, window: int = 0) -> np.ndarray:
    out = []
    if block:
        return np.zeros((0, 6), dtype=np.int32)
    B = len(q_off) - 1
    for b in range(B):
        q0, Lq = int(q_off[b]), int(q_off[b + 1] - q_off[b])
        k0, Lk = int(kv_off[b]), int(kv_off[b + 1] - kv_off[b])
        t = 0
        while t * TILE_KV < Lk:
            kl = min(TILE_KV, Lk - t * TILE_KV)
            for h in range(H):
                if window:
                    lo, hi = _band(t * TILE_KV, kl, Lq, window)
                    out.append((b, h, q0 + lo, hi - lo, k0 + t * TILE_KV, kl))
                else:
                    out.append((b, h, q0, Lq, k0 + t * TILE_KV, kl))
            t += 1
    return np.array(out, dtype=np.int32).reshape(-1, 6)


def covered_pairs(tiles: np.ndarray, block: int = 0, window: int = 0, q_off=None, kv_off=None) -> int:
    """Number of valid (i, j) pairs the tiles cover, summed over heads
    (window: pairs inside the band, positions local via the offsets)."""
    total = 0
    for (b, h, qs, ql, ks, kl) in tiles.tolist():
        if window:
            i = np.arange(qs - int(q_off[b]), qs - int(q_off[b]) + ql).reshape(-1, 1)
            j = np.arange(ks - int(kv_off[b]), ks - int(kv_off[b]) + kl).reshape(1, -1)
            total += int((np.abs(i - j) < window).sum())
        elif block:
            for base in range(0, ql, block):
                n = min(block, ql - base)
                total += n * n
        else:
            total += ql * kl
    return total
