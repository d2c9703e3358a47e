"""jattn_bwd_noalloc: the backward for callers that cannot allocate device
memory, with its scratch in the library's fixed device array.  Checked through
the C ABI against the ordinary jattn_bwd (caller-provided workspace), bit for
bit (both run the same kernels in the same order, and dQ, dK, dV are bitwise
reproducible), on two calls in a row, for every layout the scratch can take:
Delta alone (bf16 softmax), Delta plus staged bf16 copies (float32 data, D = 32),
the broadcast-Q per-sequence float32 dQ rows, the backward's dS chunks (in all
of these, since they fit the array), and no scratch at all (an activation mode
with a sliding window).  Named to run last: a failure here leaves every other test
run.
"""
import ctypes

import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SOFTMAX, SILU, GELU = W.SOFTMAX, W.SILU, W.GELU_TANH


def _dev(bt, dtype=None):
    out = {}
    for n, t in bt.items():
        if isinstance(t, torch.Tensor):
            t = t.to("cuda:0")
            if dtype is not None and n in ("q", "k", "v", "dout"):
                t = t.to(dtype)
            t = t.contiguous()
        out[n] = t
    return out


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _bits(t):
    """The raw bit patterns of a bf16 or float32 tensor (so equal means bitwise equal)."""
    t = t.contiguous()
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


def _both(plan, d):
    """One jattn_bwd with a workspace, then one jattn_bwd_noalloc on NaN-filled
    outputs; the two results must be identical."""
    lib = J.load()
    out, lse = plan.fwd(d["q"], d["k"], d["v"], bias=d["bias"])
    ref = plan.bwd(d["dout"], d["q"], d["k"], d["v"], out, lse=lse, bias=d["bias"])
    dq, dk, dv = (torch.full_like(t, float("nan")) for t in ref)
    rc = lib.jattn_bwd_noalloc(plan._h, _ptr(d["dout"]), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["bias"]),
                               _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), None,
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == J.OK, J.status_str(rc)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        np.testing.assert_array_equal(_bits(got), _bits(want), err_msg=name)


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


def test_noalloc_staged_float32_d32():
    """float32 data with D = 32: the scratch holds Delta and the bf16 staging
    copies of Q, dO, K and V."""
    bt = _dev(W.random_batch(33, [31, 33, 49, 61], [31, 33, 49, 61], 2, 32, dtype=torch.float32))
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, 32, dtype="fp32", device=0)
    assert plan.bwd_workspace_bytes > 2 * 4 * 2 * 174  # more than Delta alone
    _both(plan, bt)
    _both(plan, bt)
    plan.close()


def test_noalloc_broadcast_q_silu():
    """Broadcast Q: the scratch holds the per-sequence float32 dQ rows that the
    library sums into the shared rows' gradient."""
    n, lk = 32, [700, 1500, 129]
    bt = W.random_batch(34, [n] * len(lk), lk, 2, 128)
    shared = bt["q"][:n].clone()
    d = _dev(bt)
    d["q"] = shared.to("cuda:0").contiguous()
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, 128, act=SILU, broadcast_q=True, device=0)
    assert plan.bwd_workspace_bytes >= len(lk) * n * 2 * 128 * 4
    _both(plan, d)
    _both(plan, d)
    plan.close()


def test_noalloc_activation_needs_no_scratch():
    """An activation mode with a sliding window (no dS chunks) on bf16 data
    needs no scratch: the call passes no workspace at all."""
    bt = _dev(W.random_batch(35, [150, 3, 64], [90, 400, 64], 2, 64))
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, act=GELU, window=100, device=0)
    assert plan.bwd_workspace_bytes == 0
    _both(plan, bt)
    _both(plan, bt)
    plan.close()


def test_noalloc_activation_dS_chunks():
    """An activation mode without a window: no scratch is required, but the dS
    chunks (hi and lo parts) fit the array, so the call takes the same path as
    jattn_bwd with the full workspace."""
    bt = _dev(W.random_batch(36, [150, 3, 64], [90, 400, 64], 2, 64))
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, act=GELU, device=0)
    assert plan.bwd_workspace_bytes_min == 0 and 0 < plan.bwd_workspace_bytes <= (16 << 20)
    _both(plan, bt)
    _both(plan, bt)
    plan.close()


def test_noalloc_rejects_batches_beyond_the_fixed_array():
    lq = np.full(9000, 128)  # H * Tq * 4 bytes of Delta = 4 * 1,152,000 * 4 > 16 MiB
    qo = W.offsets(lq)
    plan = J.Plan(qo, qo, 4, 128, device=0)
    assert plan.bwd_workspace_bytes > (16 << 20)
    rc = J.load().jattn_bwd_noalloc(plan._h, *([None] * 11), None)
    assert rc == J.ERR_WORKSPACE
    plan.close()
