"""Broadcast Q (pooled attention with query rows shared by every sequence):
one shared Q [n, H, D] is read for every sequence, O / lse / dK / dV keep one
row per sequence, and dQ is the sum over the sequences.  Checked against the
oracle on the materialised Q (dQ against the sum of the per-sequence oracle
gradients), against the materialised-Q library path (bitwise for O, lse, dK,
dV), with the device planner, for determinism, and at the full pooled-attention
workload size."""
import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu

SOFTMAX, SILU, GELU = W.SOFTMAX, W.SILU, W.GELU_TANH


def _batch(seed, n, lk, H, D, nb):
    """A jagged batch whose queries are n shared rows repeated per sequence."""
    B = len(lk)
    bt = W.random_batch(seed, [n] * B, lk, H, D, bias_buckets=nb)
    shared = bt["q"][:n].clone()
    bt["q"] = shared.repeat(B, 1, 1)
    return bt, shared


def _run_bcast(bt, shared, act, nb, window=0, device_plan=False, min_ws=False):
    dev = torch.device("cuda", 0)
    H, D = shared.shape[1], shared.shape[2]
    plan = J.Plan(bt["q_off"], bt["kv_off"], H, D, act=act, bias_buckets=nb, window=window, device=0,
                  broadcast_q=True)
    if device_plan:
        qo = torch.from_numpy(np.asarray(bt["q_off"], np.int32)).to(dev)
        ko = torch.from_numpy(np.asarray(bt["kv_off"], np.int32)).to(dev)
        plan.update_device(qo, ko, int(bt["q_off"][-1]), int(bt["kv_off"][-1]))
    q = shared.to(dev)
    k, v, do = (bt[n].to(dev) for n in ("k", "v", "dout"))
    bias = bt["bias"].float().to(dev) if bt["bias"] is not None else None
    out, lse = plan.fwd(q, k, v, bias=bias)
    ws = None
    if min_ws:  # the backward path whose dQ pass recomputes the scores
        ws = torch.empty(max(plan.bwd_workspace_bytes_min, 16), dtype=torch.uint8, device=dev)
    dq, dk, dv = plan.bwd(do, q, k, v, out, lse=lse, bias=bias, workspace=ws)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    plan.close()
    f = lambda t: None if t is None else t.double().cpu().numpy()
    return dict(out=f(out), lse=f(lse), dq=f(dq), dk=f(dk), dv=f(dv))


def _dq_sum(dq_rows, B, n):
    return dq_rows.reshape(B, n, *dq_rows.shape[1:]).sum(axis=0)


CASES = [
    ("softmax_bias", 32, [700, 1500, 129, 1], 2, 128, 8, SOFTMAX, 0),
    ("silu", 32, [700, 1500, 129], 2, 128, 0, SILU, 0),
    ("gelu_d64", 32, [300, 64, 1000], 2, 64, 0, GELU, 0),
    ("softmax_window", 40, [200, 45, 129], 2, 128, 0, SOFTMAX, 16),
    ("n_over_tile", 200, [260, 3], 2, 64, 4, SOFTMAX, 0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_broadcast_q_parity(case):
    _, n, lk, H, D, nb, act, window = case
    bt, shared = _batch(91, n, lk, H, D, nb)
    got = _run_bcast(bt, shared, act, nb, window)
    ref = PT.run_oracle(bt, act=act, window=window)
    for name, tol in (("out", PT.FWD_TOL), ("dk", PT.BWD_TOL), ("dv", PT.BWD_TOL)):
        PT.assert_close(got[name], ref[name], tol, name)
    if ref["lse"] is not None:
        PT.assert_close(got["lse"], ref["lse"], PT.FWD_TOL, "lse")
    assert got["dq"].shape == (n, H, D)
    PT.assert_close(got["dq"], _dq_sum(ref["dq"], len(lk), n), PT.BWD_TOL, "dq (sum over sequences)")


def test_broadcast_q_equals_materialised_path():
    """The shared rows are the values the materialised path reads, so O, lse, dK
    and dV agree bit for bit; dQ is the materialised per-sequence dQ summed."""
    bt, shared = _batch(92, 32, [700, 129, 1500, 64], 2, 128, 16)
    got = _run_bcast(bt, shared, SOFTMAX, 16)
    mat = PT.run_library(bt)
    for name in ("out", "lse", "dk", "dv"):
        np.testing.assert_array_equal(got[name], mat[name], err_msg=name)
    PT.assert_close(got["dq"], _dq_sum(mat["dq"], 4, 32), PT.BWD_TOL, "dq")


def test_broadcast_q_device_plan_and_determinism():
    """A device plan equals a host plan on the same backward path (the one that
    recomputes the scores for dQ, which device plans take) bit for bit; the
    host plan's dS-chunk path is reproducible bit for bit and matches the other
    path within the tolerance."""
    bt, shared = _batch(93, 32, [700, 1500, 129], 2, 128, 0)
    a = _run_bcast(bt, shared, SILU, 0, min_ws=True)
    b = _run_bcast(bt, shared, SILU, 0, device_plan=True)
    c = _run_bcast(bt, shared, SILU, 0)
    d = _run_bcast(bt, shared, SILU, 0)
    for name in ("out", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[name], b[name], err_msg=name)
        np.testing.assert_array_equal(c[name], d[name], err_msg=name)
    for name in ("out", "dk", "dv"):
        np.testing.assert_array_equal(a[name], c[name], err_msg=name)
    PT.assert_close(c["dq"], a["dq"], PT.BWD_TOL, "dq")


def test_broadcast_q_full_size_pooled_workload():
    """The full pooled-attention workload (B=256, 32 shared rows, keys up to 8000,
    SiLU), in the launch configuration the bench times: O, dK and dV equal the
    materialised path bit for bit (that path is checked against the oracle on
    sampled sequences of this workload), and the summed dQ of the shared rows
    is checked element by element against the oracle: its per-sequence
    gradients on the materialised batch, summed over all 256 sequences in
    float64."""
    from oracle import oracle
    b = W.make_batch(4, act=SILU)
    w = b.w
    bt = dict(q_off=b.q_off, kv_off=b.kv_off, q=b.q, k=b.k, v=b.v, bias=b.bias, dout=b.dout, scale=b.scale)
    shared = b.q[:w.q_rows_shared].clone()
    assert torch.equal(b.q, shared.repeat(b.B, 1, 1))
    got = _run_bcast(bt, shared, SILU, 0)
    mat = PT.run_library(bt, act=SILU)
    for name in ("out", "dk", "dv"):
        np.testing.assert_array_equal(got[name], mat[name], err_msg=name)
    ref_dq, _, _, _ = oracle.backward(b.q_off, b.kv_off, b.q, b.k, b.v, b.dout, scale=b.scale, act=SILU)
    PT.assert_close(got["dq"], _dq_sum(ref_dq, b.B, w.q_rows_shared), PT.BWD_TOL, "dq (sum over 256 sequences)")
