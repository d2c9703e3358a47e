"""The device-side planner (jattn_plan_update_device): tile lists built on the
GPU from device offsets, checked bit-exactly against the independent tile
enumerator, a zigzag schedule that covers every tile once with per-CTA counts
within one of each other, results equal to the host-planned path bit for bit,
and bad offsets reported on the device status word."""
import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from oracle import tiles as T
from tests import parity as PT

pytestmark = pytest.mark.gpu

SOFTMAX, SILU = W.SOFTMAX, W.SILU


def canonical(t):
    """Sort records into the enumerator's order: b, then tile start, then h."""
    return t[np.lexsort((t[:, 1], t[:, 2], t[:, 4], t[:, 0]))] if len(t) else t


def _dev(a):
    return torch.from_numpy(np.asarray(a, dtype=np.int32)).to("cuda:0")


def _offsets(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


rng = np.random.default_rng(5)
# (name, q lengths, kv lengths (None: same), H, block, window)
BATCHES = [
    ("self_tails", [1, 127, 128, 129, 300, 0, 1000], None, 3, 0, 0),
    ("cross_empty", [200, 35, 0, 511], [8, 64, 17, 0], 2, 0, 0),
    ("block", [1, 63, 64, 65, 200, 513], None, 2, 64, 0),
    ("window", [45, 700, 129, 0, 3], None, 2, 0, 100),
    ("many_sequences", rng.integers(0, 300, 3000).tolist(), None, 2, 0, 0),
    ("one_sequence", [5000], [70], 4, 0, 0),
]


@pytest.mark.parametrize("batch", BATCHES, ids=[b[0] for b in BATCHES])
def test_device_plan_matches_enumerator(batch):
    _, lq, lk, H, block, window = batch
    qo = _offsets(lq)
    ko = _offsets(lq if lk is None else lk)
    plan = J.Plan(qo, ko, H, 64, block=block, window=window, device=0)
    plan.update_device(_dev(qo), _dev(ko), int(qo[-1]), int(ko[-1]))
    for which, fn in ((J.TILES_Q, T.q_major), (J.TILES_KV, T.kv_major)):
        tiles, cta = plan.tiles(which)
        want = fn(qo, ko, H, block, window) if not (block and which == J.TILES_KV) else np.zeros((0, 6), np.int32)
        assert tiles.shape == want.shape, (which, tiles.shape, want.shape)
        np.testing.assert_array_equal(canonical(tiles), canonical(want))
        counts = np.diff(cta)
        assert cta[0] == 0 and cta[-1] == len(tiles) and np.all(counts >= 0)
        if len(tiles):
            assert counts.max() - counts.min() <= 1  # the zigzag deals the tiles evenly
    assert plan.check_status() == 0
    plan.close()


CASES = [
    ("softmax_bias", [1, 127, 300, 0, 513], None, 2, 128, 16, SOFTMAX, 0, 0),
    ("block", [1, 63, 64, 65, 200, 513], None, 2, 64, 0, SOFTMAX, 64, 0),
    ("window", [45, 700, 129], None, 2, 128, 8, SOFTMAX, 0, 100),
    ("cross_silu", [32, 32, 100], [700, 1500, 129], 2, 128, 0, SILU, 0, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_device_plan_results_equal_host_plan(case):
    """Every tile's result is independent of the CTA that runs it, so the device
    schedule gives the host schedule's outputs bit for bit.  A device plan's
    backward recomputes the scores for dQ (the host does not know the lengths
    the dS chunks need), so the host plan runs that same path here (the
    minimum workspace)."""
    _, lq, lk, H, D, nb, act, block, window = case
    bt = W.random_batch(71, lq, lq if lk is None else lk, H, D, bias_buckets=nb)
    host = PT.run_library(bt, act=act, block=block, window=window, min_workspace=True)
    plan = J.Plan(bt["q_off"], bt["kv_off"], H, D, act=act, block=block, bias_buckets=nb, window=window, device=0)
    # re-plan the same plan on the device (its host lists are replaced)
    plan.update_device(_dev(bt["q_off"]), _dev(bt["kv_off"]), int(bt["q_off"][-1]), int(bt["kv_off"][-1]))
    dev = PT.run_library(bt, act=act, block=block, window=window, plan=plan)
    for n in ("out", "dq", "dk", "dv"):
        np.testing.assert_array_equal(dev[n], host[n], err_msg=n)
    if host["lse"] is not None:
        np.testing.assert_array_equal(dev["lse"], host["lse"])
    plan.close()


@pytest.mark.parametrize("bad", ["decreasing", "wrong_total", "block_unequal"])
def test_device_plan_flags_bad_offsets(bad):
    qo = _offsets([10, 20, 30])
    ko = qo.copy()
    block = 64 if bad == "block_unequal" else 0
    plan = J.Plan(qo, ko, 2, 64, block=block, device=0)
    q, k = qo.copy(), ko.copy()
    Tq, Tk = int(q[-1]), int(k[-1])
    if bad == "decreasing":
        q[2] = 5
    elif bad == "wrong_total":
        Tq += 1
    else:
        k = _offsets([10, 21, 29])
    plan.update_device(_dev(q), _dev(k), Tq, Tk if bad != "block_unequal" else Tq)
    torch.cuda.synchronize()
    assert plan.check_status() == J.ERR_DEVICE_CHECK
    tiles, cta = plan.tiles(J.TILES_Q)
    assert len(tiles) == 0 and np.all(cta == 0)
    plan.close()


def test_device_plan_rejects_too_many_sequences():
    qo = np.arange(8194, dtype=np.int32)
    plan = J.Plan(qo, qo, 1, 64, device=0)
    with pytest.raises(J.JattnError) as e:
        plan.update_device(_dev(qo), _dev(qo), 8193, 8193)
    assert e.value.code == J.ERR_UNSUPPORTED
    plan.close()
