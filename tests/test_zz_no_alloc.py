"""jattn_bwd_noalloc: the backward for callers that cannot allocate device
memory, with its scratch in the library's fixed device array.  Checked through
the C ABI against the ordinary jattn_bwd (caller-provided workspace) on two
calls in a row.  Named to run last: a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu


def _dev(bt):
    return {n: (t.to("cuda:0").contiguous() if isinstance(t, torch.Tensor) else t) for n, t in bt.items()}


def _both(plan, d):
    lib = J.load()
    out, lse = plan.fwd(d["q"], d["k"], d["v"], bias=d["bias"])
    ref = plan.bwd(d["dout"], d["q"], d["k"], d["v"], out, lse=lse, bias=d["bias"])
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in ref)
    P = ctypes.c_void_p
    rc = lib.jattn_bwd_noalloc(plan._h, P(d["dout"].data_ptr()), P(d["q"].data_ptr()), P(d["k"].data_ptr()),
                               P(d["v"].data_ptr()), P(d["bias"].data_ptr()) if d["bias"] is not None else None,
                               P(out.data_ptr()), P(lse.data_ptr()), P(dq.data_ptr()), P(dk.data_ptr()),
                               P(dv.data_ptr()), None, P(torch.cuda.current_stream().cuda_stream))
    assert rc == J.OK, J.status_str(rc)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        PT.assert_close(got.double().cpu().numpy(), want.double().cpu().numpy(), PT.BWD_TOL, name)


def test_noalloc_backward_matches_workspace_backward_twice():
    bt1 = _dev(W.random_batch(31, [300, 129, 1, 77], [300, 129, 1, 77], 4, 128, bias_buckets=64))
    plan = J.Plan(bt1["q_off"], bt1["kv_off"], 4, 128, bias_buckets=64, device=0)
    assert plan.bwd_workspace_bytes > 0  # this mode needs scratch (Delta)
    _both(plan, bt1)
    # second call in a row, on a different batch: the array keeps the first call's contents
    bt2 = _dev(W.random_batch(32, [5, 260, 140], [5, 260, 140], 4, 128, bias_buckets=64))
    plan.update(bt2["q_off"], bt2["kv_off"])
    _both(plan, bt2)
    plan.close()


def test_noalloc_rejects_batches_beyond_the_fixed_array():
    lq = np.full(9000, 128)  # H * Tq * 4 bytes of Delta = 4 * 1,152,000 * 4 > 16 MiB
    qo = W.offsets(lq)
    plan = J.Plan(qo, qo, 4, 128, device=0)
    assert plan.bwd_workspace_bytes > (16 << 20)
    rc = J.load().jattn_bwd_noalloc(plan._h, *([None] * 11), None)
    assert rc == J.ERR_WORKSPACE
    plan.close()
