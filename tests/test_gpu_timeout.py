"""The bounded-wait error path on a real launch.  jattn_test_fwd_stall launches
a test build of the forward kernel whose score-issuing thread waits on a
barrier that nothing completes; the wait gives up after a short limit, the
status word reports JATTN_ERR_DEVICE_TIMEOUT, and the kernel returns with its
copies drained and TMEM freed.  Afterwards ordinary calls on the same device
and plan still match the oracle, so the context survived and no TMEM was left
allocated (a leaked allocation would keep later kernels from starting)."""
import ctypes
import time

import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from tests import parity as PT

pytestmark = pytest.mark.gpu


def _stall(plan, d, out, lse, wait_ns):
    P = ctypes.c_void_p
    return J.load().jattn_test_fwd_stall(plan._h, P(d["q"].data_ptr()), P(d["k"].data_ptr()), P(d["v"].data_ptr()),
                                         P(out.data_ptr()), P(lse.data_ptr()), wait_ns,
                                         P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("D", [64, 128])
def test_bounded_wait_runs_out_and_device_recovers(D):
    bt = W.random_batch(41 + D, [200, 70, 129], [200, 70, 129], 2, D)
    d = {n: bt[n].to("cuda:0").contiguous() for n in ("q", "k", "v", "dout")}
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, D, device=0)
    out = torch.empty_like(d["q"])
    lse = torch.empty(2, d["q"].shape[0], dtype=torch.float32, device="cuda:0")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = _stall(plan, d, out, lse, 20_000_000)  # 20 ms limit
    assert rc == J.OK, J.status_str(rc)
    st = plan.check_status()  # synchronises, reads and clears the status word
    elapsed = time.perf_counter() - t0
    assert st == J.ERR_DEVICE_TIMEOUT, J.status_str(st)
    assert elapsed < 1.0, elapsed  # the short limit applied, not the library's 2 s
    assert plan.check_status() == 0  # cleared by the read
    # the same plan and device afterwards: ordinary calls, checked against the oracle
    gpu = PT.run_library(bt, plan=plan)
    PT.compare(gpu, PT.run_oracle(bt))
    # and the stall again, then once more an ordinary call
    assert _stall(plan, d, out, lse, 5_000_000) == J.OK
    assert plan.check_status() == J.ERR_DEVICE_TIMEOUT
    gpu = PT.run_library(bt, plan=plan)
    PT.compare(gpu, PT.run_oracle(bt))
    plan.close()


def test_stall_hook_argument_checks():
    bt = W.random_batch(43, [40, 100], [40, 100], 2, 64, bias_buckets=4)
    d = {n: bt[n].to("cuda:0").contiguous() for n in ("q", "k", "v")}
    out = torch.empty_like(d["q"])
    lse = torch.empty(2, 140, dtype=torch.float32, device="cuda:0")
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, device=0)
    assert _stall(plan, d, out, lse, 10) == J.ERR_INVALID_ARG                 # below 100 us
    assert _stall(plan, d, out, lse, 3_000_000_000) == J.ERR_INVALID_ARG      # above the library's 2 s
    biased = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, bias_buckets=4, device=0)
    assert _stall(biased, d, out, lse, 1_000_000) == J.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert plan.check_status() == 0 and biased.check_status() == 0
    plan.close()
    biased.close()
