"""Rank-local views of a jagged batch for data-parallel runs.

Every (sequence, head) pair of the attention is independent, so ranks split a
batch by whole sequences (the assignment comes from ``jattn_shard`` in the C
library, see :func:`jagged_attention_recommendation_gb300.shard`) and run the
same kernels on their part with no collective on the attention path.  This
module only does the index bookkeeping: which rows of the global Q-side and
K/V-side tensors a rank owns, and its local offsets.
"""
from __future__ import annotations

import numpy as np


def local_rows(q_offsets, kv_offsets, rank_of, rank: int):
    """Sequences of `rank`, in batch order, as a jagged sub-batch.

    Returns ``(seqs, q_off, kv_off, q_rows, kv_rows)``: the global sequence
    indices, the local int32 offsets (length len(seqs) + 1), and the int64 global
    row indices of the local Q-side rows (q, out, dout, dq, lse columns) and
    K/V-side rows (k, v, dk, dv), packed in the local order.
    """
    qo = np.asarray(q_offsets, dtype=np.int64)
    ko = np.asarray(kv_offsets, dtype=np.int64)
    seqs = np.nonzero(np.asarray(rank_of) == rank)[0]
    lq = qo[seqs + 1] - qo[seqs]
    lk = ko[seqs + 1] - ko[seqs]
    q_off = np.zeros(len(seqs) + 1, dtype=np.int64)
    kv_off = np.zeros(len(seqs) + 1, dtype=np.int64)
    np.cumsum(lq, out=q_off[1:])
    np.cumsum(lk, out=kv_off[1:])
    q_rows = np.concatenate([np.arange(qo[s], qo[s + 1]) for s in seqs] or [np.zeros(0, np.int64)])
    kv_rows = np.concatenate([np.arange(ko[s], ko[s + 1]) for s in seqs] or [np.zeros(0, np.int64)])
    return seqs, q_off.astype(np.int32), kv_off.astype(np.int32), q_rows.astype(np.int64), kv_rows.astype(np.int64)
