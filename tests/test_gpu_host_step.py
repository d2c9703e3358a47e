"""jattn_step_host: a whole training step from host buffers, pipelined over calls.

Consecutive calls alternate between two batches of different sizes (so the
staging sets are re-allocated and the two sets are both in flight), and every
call's downloaded outputs must equal, bit for bit, the device path (jattn_fwd /
jattn_bwd on device tensors) for the same batch: the kernels are deterministic,
so any difference is a copy that overlapped the wrong call. One case is also
checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu


def _batch(seed, lq, lk, H, D, nb):
    return W.random_batch(seed, lq, lk, H, D, dtype=torch.bfloat16, bias_buckets=nb)


def _device_ref(b, H, D, nb, act):
    dev = torch.device("cuda", 0)
    plan = J.Plan(b["q_off"], b["kv_off"], H, D, act=act, bias_buckets=nb, device=0)
    q, k, v, do = (b[n].to(dev) for n in ("q", "k", "v", "dout"))
    bias = b["bias"].float().to(dev) if b["bias"] is not None else None
    out, lse = plan.fwd(q, k, v, bias=bias)
    dq, dk, dv = plan.bwd(do, q, k, v, out, lse=lse, bias=bias)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    res = dict(out=out.cpu(), dq=dq.cpu(), dk=dk.cpu(), dv=dv.cpu(), lse=lse.cpu() if lse is not None else None)
    plan.close()
    return res


def _host_io(b, H, D, act):
    Tq, Tk = int(b["q_off"][-1]), int(b["kv_off"][-1])
    pin = dict(q=b["q"].pin_memory(), k=b["k"].pin_memory(), v=b["v"].pin_memory(), dout=b["dout"].pin_memory(),
               bias=b["bias"].float().contiguous().pin_memory() if b["bias"] is not None else None)
    outs = {n: torch.full((T, H, D), float("nan"), dtype=torch.bfloat16).pin_memory()
            for n, T in (("out", Tq), ("dq", Tq), ("dk", Tk), ("dv", Tk))}
    outs["lse"] = torch.full((H, Tq), float("nan"), dtype=torch.float32).pin_memory() if act == W.SOFTMAX else None
    return pin, outs


@pytest.mark.parametrize("act,nb", [(W.SOFTMAX, 16), (W.SILU, 0)])
def test_step_host_pipelined_matches_device_path(act, nb):
    H, D = 2, 128
    ba = _batch(11, [37, 300, 129, 1], [37, 300, 129, 1], H, D, nb)
    bb = _batch(12, [500, 64, 900, 3, 250], [200, 64, 1000, 3, 250], H, D, nb)
    ref = {"a": _device_ref(ba, H, D, nb, act), "b": _device_ref(bb, H, D, nb, act)}
    plan = J.Plan(ba["q_off"], ba["kv_off"], H, D, act=act, bias_buckets=nb, device=0)
    stream = torch.cuda.current_stream()
    calls = []
    for key in ("a", "b", "a", "b", "b", "a"):
        b = ba if key == "a" else bb
        pin, outs = _host_io(b, H, D, act)
        plan.step_host(b["q_off"], b["kv_off"], pin["q"], pin["k"], pin["v"], pin["dout"], outs["out"], outs["dq"],
                       outs["dk"], outs["dv"], bias=pin["bias"], lse=outs["lse"], stream=stream)
        calls.append((key, pin, outs))  # the host buffers stay alive until the join
    plan.step_host_join(stream)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    for key, _, outs in calls:
        for n in ("out", "dq", "dk", "dv", "lse"):
            if ref[key][n] is None:
                continue
            assert torch.equal(outs[n], ref[key][n]), (key, n)
    plan.close()


def test_step_host_against_oracle():
    H, D, nb = 2, 64, 8
    b = _batch(21, [45, 200, 3], [45, 200, 3], H, D, nb)
    plan = J.Plan(b["q_off"], b["kv_off"], H, D, act=W.SOFTMAX, bias_buckets=nb, device=0)
    pin, outs = _host_io(b, H, D, W.SOFTMAX)
    plan.step_host(b["q_off"], b["kv_off"], pin["q"], pin["k"], pin["v"], pin["dout"], outs["out"], outs["dq"],
                   outs["dk"], outs["dv"], bias=pin["bias"], lse=outs["lse"])
    plan.step_host_join()
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    gpu = dict(out=outs["out"].float().numpy(), lse=outs["lse"].numpy(), dq=outs["dq"].float().numpy(),
               dk=outs["dk"].float().numpy(), dv=outs["dv"].float().numpy())
    ref = PT.run_oracle(b, act=W.SOFTMAX, block=0)
    PT.compare(gpu, ref)
    plan.close()


def test_step_host_rejects_bias_mismatch():
    H, D = 2, 64
    b = _batch(31, [10, 20], [10, 20], H, D, 0)
    plan = J.Plan(b["q_off"], b["kv_off"], H, D, act=W.SOFTMAX, bias_buckets=4, device=0)
    pin, outs = _host_io(b, H, D, W.SOFTMAX)
    with pytest.raises(J.JattnError):
        plan.step_host(b["q_off"], b["kv_off"], pin["q"], pin["k"], pin["v"], pin["dout"], outs["out"],
                       outs["dq"], outs["dk"], outs["dv"], bias=None, lse=outs["lse"])
    plan.close()
