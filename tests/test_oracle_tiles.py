"""Pins of the workload generator and of the independent tile enumerator (CPU only)."""
import json
import os

import numpy as np
import pytest

from jagged_attention_recommendation_gb300 import workloads as W
from oracle import tiles as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "workload_pins.json")


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_workload_lengths_golden(wid):
    g = json.load(open(GOLDEN))[str(wid)]
    lq, lk = W.lengths(wid)
    qo, ko = W.offsets(lq), W.offsets(lk)
    assert int(qo[-1]) == g["Tq"] and int(ko[-1]) == g["Tk"]
    if "pairs" in g:
        assert W.valid_pairs(qo, ko) == g["pairs"]
    if "pairs_block64" in g:
        assert W.valid_pairs(qo, ko, block=64) == g["pairs_block64"]
    if "lengths_q" in g:
        assert lq.tolist() == g["lengths_q"]
    if "max_q" in g:
        assert int(lq.max()) == g["max_q"]
    if "median_q" in g:
        assert float(np.median(lq)) == g["median_q"]


def brute_force_tiles(q_off, kv_off, H, block, which):
    """Per-(b, h) enumeration of every 128-row tile start, collected as a set."""
    recs = set()
    for h in range(H):
        for b in range(len(q_off) - 1):
            q0, q1, k0, k1 = (int(x) for x in (q_off[b], q_off[b + 1], kv_off[b], kv_off[b + 1]))
            if which == "q":
                for r in range(q0, q1):
                    if (r - q0) % 128 == 0:
                        n = min(128, q1 - r)
                        recs.add((b, h, r, n, k0 + (r - q0), n) if block else (b, h, r, n, k0, k1 - k0))
            elif not block:
                for r in range(k0, k1):
                    if (r - k0) % 128 == 0:
                        recs.add((b, h, q0, q1 - q0, r, min(128, k1 - r)))
    return recs


@pytest.mark.parametrize("lens,H,block", [
    (([1, 128, 129, 0, 300], [5, 0, 256, 7, 1]), 3, 0),
    (([64, 65, 200, 1], None), 2, 64),
    ((list(range(0, 700, 37)), list(range(700, 0, -37))), 1, 0),
])
def test_enumerator_matches_brute_force(lens, H, block):
    lq, lk = lens
    lk = lq if lk is None else lk
    qo, ko = W.offsets(np.array(lq)), W.offsets(np.array(lk))
    for which, fn in (("q", T.q_major), ("kv", T.kv_major)):
        tl = fn(qo, ko, H, block)
        assert len(set(map(tuple, tl.tolist()))) == len(tl)
        assert set(map(tuple, tl.tolist())) == brute_force_tiles(qo, ko, H, block, which)


@pytest.mark.parametrize("wid", [2, 3, 5])
def test_total_pair_identity(wid):
    """R10: sum over tiles of covered pairs == sum_b Lq*Lk (block: sum of n^2 over blocks), times H."""
    w = W.WORKLOADS[wid]
    lq, lk = W.lengths(wid)
    qo, ko = W.offsets(lq), W.offsets(lk)
    want = W.valid_pairs(qo, ko, w.block) * w.H
    assert T.covered_pairs(T.q_major(qo, ko, w.H, w.block), w.block) == want
    if not w.block:
        assert T.covered_pairs(T.kv_major(qo, ko, w.H), 0) == want


@pytest.mark.parametrize("window", [1, 50, 200])
def test_window_tiles_cover_exactly_the_band(window):
    """Sliding window: every in-band pair (|i - j| < W) is covered by exactly one
    query-major and one key-major record, and the ranges are tight (the first
    and last key of each query tile's range are inside some row's band)."""
    lq, lk = [1, 128, 129, 300, 0, 700], [5, 130, 129, 300, 9, 40]
    qo, ko = W.offsets(np.array(lq)), W.offsets(np.array(lk))
    want = 0
    for a, b in zip(lq, lk):
        i, j = np.arange(a).reshape(-1, 1), np.arange(b).reshape(1, -1)
        want += int((np.abs(i - j) < window).sum())
    for fn in (T.q_major, T.kv_major):
        tl = fn(qo, ko, 2, 0, window)
        assert T.covered_pairs(tl, 0, window, qo, ko) == 2 * want
        for (b, h, qs, ql, ks, kl) in tl.tolist():  # every range inside its own sequence
            assert qo[b] <= qs and qs + ql <= qo[b + 1] and ko[b] <= ks and ks + kl <= ko[b + 1]
    for (b, h, qs, ql, ks, kl) in T.q_major(qo, ko, 1, 0, window).tolist():
        if kl == 0:
            continue
        i0, j0 = qs - qo[b], ks - ko[b]
        assert i0 - j0 < window and (j0 + kl - 1) - (i0 + ql - 1) < window   # both ends in some row's band
        assert j0 == 0 or i0 - (j0 - 1) >= window                            # one key earlier is out of band
        assert j0 + kl == lk[b] or (j0 + kl) - (i0 + ql - 1) >= window        # one key later is out of band
