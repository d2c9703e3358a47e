"""Data-parallel sharding of a jagged batch (host logic, no GPU).

Every (sequence, head) pair of jagged attention is independent, so ranks split a
batch by whole sequences and need no collective on the attention path; only the
gradient of a shared learned input (the bias table) is summed across ranks.
The multi-rank test runs two `gloo` processes on the CPU: each computes its
shard with the CPU oracle, and rank 0 checks that the reassembled outputs equal
the oracle on the whole batch (bit for bit: the per-sequence arithmetic is the
same) and that the all-reduced bias gradient matches.
"""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from oracle import oracle as O


def _cost(lq, lk):
    lq = np.asarray(lq, dtype=np.int64)
    lk = np.asarray(lk, dtype=np.int64)
    return lq * lk + 64 * (lq + lk)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from jagged_attention_recommendation_gb300 import build
    build.build()
    O.build()


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_partitions_and_balances(world):
    lq, lk = W.lengths(2, B=512)
    qo, ko = W.offsets(lq), W.offsets(lk)
    r = J.shard(qo, ko, world)
    assert r.shape == (512,) and r.dtype == np.int32
    assert r.min() >= 0 and r.max() < world
    c = _cost(lq, lk)
    loads = np.array([c[r == k].sum() for k in range(world)])
    # longest-first greedy: no rank exceeds another by more than the largest item
    assert loads.max() - loads.min() <= c.max()
    # same answer on every call (every rank computes it independently)
    assert np.array_equal(r, J.shard(qo, ko, world))


def test_shard_world_one_and_more_ranks_than_sequences():
    qo = np.array([0, 5, 5, 9], dtype=np.int32)
    ko = np.array([0, 3, 7, 7], dtype=np.int32)
    assert np.array_equal(J.shard(qo, ko, 1), np.zeros(3, np.int32))
    r = J.shard(qo, ko, 5)
    assert len(set(r.tolist())) == 3  # each sequence alone on a rank


def test_shard_rejects_bad_input():
    qo = np.array([0, 5, 4], dtype=np.int32)  # decreasing
    ko = np.array([0, 3, 7], dtype=np.int32)
    with pytest.raises(J.JattnError):
        J.shard(qo, ko, 2)
    with pytest.raises(J.JattnError):
        J.shard(np.array([0, 1], np.int32), np.array([0, 1], np.int32), 0)


def test_local_rows_cover_the_batch_once():
    lq = np.array([3, 0, 7, 2, 5])
    lk = np.array([4, 6, 0, 1, 9])
    qo, ko = W.offsets(lq), W.offsets(lk)
    r = J.shard(qo, ko, 2)
    seen_q, seen_k = [], []
    for rank in range(2):
        seqs, lqo, lko, qrows, krows = J.local_rows(qo, ko, r, rank)
        assert np.array_equal(np.diff(lqo), lq[seqs]) and np.array_equal(np.diff(lko), lk[seqs])
        assert len(qrows) == lqo[-1] and len(krows) == lko[-1]
        seen_q += qrows.tolist()
        seen_k += krows.tolist()
    assert sorted(seen_q) == list(range(qo[-1])) and sorted(seen_k) == list(range(ko[-1]))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = {
    "softmax_bias": dict(lq=[37, 5, 130, 0, 64, 17, 90], lk=[37, 5, 130, 9, 64, 17, 90], act=W.SOFTMAX, nb=8,
                         block=0),
    "cross_silu": dict(lq=[12, 40, 3, 77, 25], lk=[50, 0, 31, 8, 66], act=W.SILU, nb=0, block=0),
    "block64": dict(lq=[70, 130, 64, 5], lk=[70, 130, 64, 5], act=W.SOFTMAX, nb=0, block=64),
}


def _dp_worker(rank: int, world: int, port: int, case: str):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = CASES[case]
        b = W.random_batch(7, c["lq"], c["lk"], 2, 16, dtype=torch.float64, bias_buckets=c["nb"])
        qo, ko = b["q_off"], b["kv_off"]
        r = J.shard(qo, ko, world)
        # every rank derived the same assignment on its own
        allr = [None] * world
        dist.all_gather_object(allr, r.tolist())
        assert all(x == allr[0] for x in allr)
        seqs, lqo, lko, qrows, krows = J.local_rows(qo, ko, r, rank)
        qi, ki = torch.from_numpy(qrows), torch.from_numpy(krows)
        q, k, v, do = b["q"][qi], b["k"][ki], b["v"][ki], b["dout"][qi]
        out, lse = O.forward(lqo, lko, q, k, v, b["bias"], act=c["act"], block=c["block"], nthreads=2)
        dq, dk, dv, dt = O.backward(lqo, lko, q, k, v, do, b["bias"], act=c["act"], block=c["block"], nthreads=2)
        # the only exchange: the shared bias table's gradient
        if dt is not None:
            dtt = torch.from_numpy(dt)
            dist.all_reduce(dtt)
            dt = dtt.numpy()
        parts = [None] * world
        dist.all_gather_object(parts, (qrows, krows, out, lse, dq, dk, dv))
        if rank == 0:
            Tq, Tk = int(qo[-1]), int(ko[-1])
            g_out = np.full((Tq, 2, 16), np.nan)
            g_dq = np.full((Tq, 2, 16), np.nan)
            g_dk = np.full((Tk, 2, 16), np.nan)
            g_dv = np.full((Tk, 2, 16), np.nan)
            g_lse = np.full((2, Tq), np.nan)
            for qr, kr, o_, l_, dq_, dk_, dv_ in parts:
                g_out[qr], g_dq[qr], g_dk[kr], g_dv[kr] = o_, dq_, dk_, dv_
                if l_ is not None:
                    g_lse[:, qr] = l_
            f_out, f_lse = O.forward(qo, ko, b["q"], b["k"], b["v"], b["bias"], act=c["act"], block=c["block"],
                                     nthreads=2)
            f_dq, f_dk, f_dv, f_dt = O.backward(qo, ko, b["q"], b["k"], b["v"], b["dout"], b["bias"],
                                                act=c["act"], block=c["block"], nthreads=2)
            assert np.array_equal(g_out, f_out)
            assert np.array_equal(g_dq, f_dq)
            assert np.array_equal(g_dk, f_dk)
            assert np.array_equal(g_dv, f_dv)
            if f_lse is not None:
                assert np.array_equal(g_lse, f_lse)
            if f_dt is not None:
                np.testing.assert_allclose(dt, f_dt, rtol=1e-12, atol=1e-13)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", sorted(CASES))
def test_two_rank_shards_reproduce_the_whole_batch(case):
    mp.spawn(_dp_worker, args=(2, _free_port(), case), nprocs=2, join=True)


def _bcast_worker(rank: int, world: int, port: int):
    """Broadcast Q across data-parallel ranks: each rank sums its shard's
    per-sequence query gradients (what jattn_bwd returns for a broadcast-Q
    plan); one all-reduce of that [n, H, D] sum gives the whole batch's."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n, lk = 8, [50, 3, 31, 80, 66, 9]
        b = W.random_batch(8, [n] * len(lk), lk, 2, 16, dtype=torch.float64)
        shared = b["q"][:n].clone()
        b["q"] = shared.repeat(len(lk), 1, 1)
        qo, ko = b["q_off"], b["kv_off"]
        r = J.shard(qo, ko, world)
        seqs, lqo, lko, qrows, krows = J.local_rows(qo, ko, r, rank)
        qi, ki = torch.from_numpy(qrows), torch.from_numpy(krows)
        dq, _, _, _ = O.backward(lqo, lko, b["q"][qi], b["k"][ki], b["v"][ki], b["dout"][qi], act=W.SILU, nthreads=2)
        local = torch.from_numpy(dq.reshape(len(seqs), n, 2, 16).sum(axis=0) if len(seqs) else np.zeros((n, 2, 16)))
        dist.all_reduce(local)
        f_dq, _, _, _ = O.backward(qo, ko, b["q"], b["k"], b["v"], b["dout"], act=W.SILU, nthreads=2)
        want = f_dq.reshape(len(lk), n, 2, 16).sum(axis=0)
        np.testing.assert_allclose(local.numpy(), want, rtol=1e-12, atol=1e-13)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_broadcast_q_gradient_all_reduce():
    mp.spawn(_bcast_worker, args=(2, _free_port()), nprocs=2, join=True)
