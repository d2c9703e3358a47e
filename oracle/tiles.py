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
"""
from __future__ import annotations

import numpy as np

TILE_Q = 128
TILE_KV = 128


def q_major(q_off, kv_off, H: int, block: int = 0) -> np.ndarray:
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
                else:
                    out.append((b, h, q0 + t * TILE_Q, ql, k0, Lk))
            t += 1
    return np.array(out, dtype=np.int32).reshape(-1, 6)


def kv_major(q_off, kv_off, H: int, block: int = 0) -> np.ndarray:
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
                out.append((b, h, q0, Lq, k0 + t * TILE_KV, kl))
            t += 1
    return np.array(out, dtype=np.int32).reshape(-1, 6)


def covered_pairs(tiles: np.ndarray, block: int = 0) -> int:
    """Number of valid (i, j) pairs the tiles cover, summed over heads."""
    total = 0
    for (b, h, qs, ql, ks, kl) in tiles.tolist():
        if block:
            for base in range(0, ql, block):
                n = min(block, ql - base)
                total += n * n
        else:
            total += ql * kl
    return total
