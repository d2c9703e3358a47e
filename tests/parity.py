"""Helpers shared by the GPU parity tests: run the library through its C ABI on
seeded inputs, run the oracle on the same host values, compare element-wise.

Tolerances (stated for bf16 inputs with fp32 accumulation):
  forward  : |gpu - ref| <= 1e-2 + 1e-2 |ref|   on O and lse
  backward : |gpu - ref| <= 3e-2 + 3e-2 |ref|   on dQ, dK, dV
"""
import numpy as np
import torch

import jagged_attention_recommendation_gb300 as J
from oracle import oracle

FWD_TOL = (1e-2, 1e-2)
BWD_TOL = (3e-2, 3e-2)


def to_dev(t):
    return None if t is None else t.to("cuda:0").contiguous()


def run_library(bt, act=0, block=0, dtype="bf16", backward=True, plan=None, window=0, rope=None,
                min_workspace=False):
    """Forward (+ backward) of batch dict ``bt`` on cuda:0; returns float64 numpy arrays.
    rope = (cos, sin) host float32 tables: rotary embedding of Q and K.
    min_workspace: the backward gets only jattn_bwd_workspace_bytes_min (the path
    whose dQ pass recomputes the scores) instead of the full workspace."""
    q, k, v, dout = (to_dev(bt[n]) for n in ("q", "k", "v", "dout"))
    bias = to_dev(bt["bias"].float()) if bt.get("bias") is not None else None
    rp = None if rope is None else tuple(to_dev(t.float().contiguous()) for t in rope)
    H, D = q.shape[1], q.shape[2]
    nb = 0 if bias is None else bias.shape[1]
    if plan is None:
        plan = J.Plan(bt["q_off"], bt["kv_off"], H, D, act=act, block=block, bias_buckets=nb, dtype=dtype, device=0,
                      window=window)
    out, lse = plan.fwd(q, k, v, bias=bias, rope=rp)
    res = {"out": out, "lse": lse}
    if backward:
        ws = None
        if min_workspace:
            ws = torch.empty(max(plan.bwd_workspace_bytes_min, 16), dtype=torch.uint8, device="cuda:0")
        dq, dk, dv = plan.bwd(dout, q, k, v, out, lse=lse, bias=bias, rope=rp, workspace=ws)
        res.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    status = plan.check_status()
    assert status == 0, J.status_str(status)
    return {n: (None if t is None else t.double().cpu().numpy()) for n, t in res.items()}


def run_oracle(bt, act=0, block=0, backward=True, window=0, rope=None):
    out, lse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt.get("bias"),
                              scale=bt["scale"], act=act, block=block, window=window, rope=rope)
    res = {"out": out, "lse": lse}
    if backward:
        dq, dk, dv, _ = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"],
                                        bias=bt.get("bias"), scale=bt["scale"], act=act, block=block, window=window,
                                        rope=rope)
        res.update(dq=dq, dk=dk, dv=dv)
    return res


def violations(got, ref, tol):
    atol, rtol = tol
    err = np.abs(got - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))  # NaN counts as a violation
    return int(bad.sum()), float(np.nanmax(err)) if err.size else 0.0


def assert_close(got, ref, tol, name):
    if ref is None:
        return
    assert got is not None, name
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    if ref.size == 0:
        return
    # -inf lse (empty key set) must match exactly
    inf = np.isinf(ref)
    if inf.any():
        assert np.array_equal(got[inf], ref[inf]), name
        got, ref = got[~inf], ref[~inf]
    n, mx = violations(got, ref, tol)
    assert n == 0, "%s: %d of %d elements out of tolerance (max |err| %.4g)" % (name, n, got.size, mx)


def compare(gpu, ref, backward=True):
    assert_close(gpu["out"], ref["out"], FWD_TOL, "out")
    if ref["lse"] is not None and gpu["lse"] is not None:
        assert_close(gpu["lse"], ref["lse"], FWD_TOL, "lse")
    if backward:
        for n in ("dq", "dk", "dv"):
            assert_close(gpu[n], ref[n], BWD_TOL, n)
