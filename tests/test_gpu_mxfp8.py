"""MXFP8 attention ("Training GEM at LLM scale", section "Low Precision Flash
Attention") through the C ABI against the MXFP8 oracle (oracle/mxfp8.py):

* the quantisation of an input tensor, bit for bit (both sides take the same
  E8M0 exponent and E4M3 rounding decisions on the same bf16 values);
* forward and backward element by element, within the stated tolerances plus
  the oracle's flip allowance: the bound on how far a quantised P or dS can
  move when the kernel computes its unquantised value in float32 (zero unless
  that value lies next to a rounding midpoint of its block's grid), carried
  through the products;
* sampled sequences of the full-size self-attention batch (without its bias).
"""
import zlib

import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from oracle import mxfp8 as M
from oracle import oracle
from tests import parity as PT

pytestmark = pytest.mark.gpu

# (name, lq, lk, H, D)
CASES = [
    ("d128_ragged", [1, 31, 33, 128, 129, 300], None, 2, 128),
    ("d64_cross", [200, 35, 129], [64, 300, 1], 2, 64),
    ("d128_long", [700, 90], None, 2, 128),
    ("d64_empty", [10, 0, 140], [0, 5, 30], 2, 64),
]


def _f64(t):
    return t.double().cpu().numpy()


def _within(got, ref, tol, allow, name):
    atol, rtol = tol
    err = np.abs(got - ref)
    bad = ~(err <= atol + rtol * np.abs(ref) + allow)
    assert not bad.any(), "%s: %d of %d out of tolerance + allowance (max excess %.4g)" % (
        name, int(bad.sum()), got.size, float((err - atol - rtol * np.abs(ref) - allow).max()))


def _run(bt, plan):
    dev = torch.device("cuda", 0)
    q, k, v, do = (bt[n].to(dev) for n in ("q", "k", "v", "dout"))
    out, lse = plan.fwd(q, k, v)
    dq, dk, dv = plan.bwd(do, q, k, v, out, lse=lse)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    return {n: _f64(t) for n, t in (("out", out), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}


def test_quantisation_bit_exact():
    bt = W.random_batch(201, [1, 31, 33, 64, 300], [5, 129, 1, 40, 77], 3, 128)
    plan = J.Plan(bt["q_off"], bt["kv_off"], 3, 128, mxfp8=True, device=0)
    dev = torch.device("cuda", 0)
    for name, which, off in (("q", J.TILES_Q, bt["q_off"]), ("k", J.TILES_KV, bt["kv_off"]),
                             ("dout", J.TILES_Q, bt["q_off"])):
        x = bt[name].to(dev)
        got = _f64(plan.mxfp8_quantize(x, which))
        np.testing.assert_array_equal(got, M.qdq_jagged(bt[name].double().numpy(), off), err_msg=name)
    # values spread over many binades, zeros and a block with a single nonzero value
    x = torch.randn(bt["q"].shape, generator=torch.Generator().manual_seed(3)) * \
        torch.exp(4.0 * torch.randn(bt["q"].shape, generator=torch.Generator().manual_seed(4)))
    x[40:60] = 0.0
    x[64, 0, :] = 0.0
    x[64, 0, 5] = 3.0
    xb = x.to(torch.bfloat16)
    got = _f64(plan.mxfp8_quantize(xb.to(dev), J.TILES_Q))
    np.testing.assert_array_equal(got, M.qdq_jagged(xb.double().numpy(), bt["q_off"]))
    assert plan.check_status() == 0
    plan.close()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mxfp8_parity(case):
    name, lq, lk, H, D = case
    lk = lq if lk is None else lk
    bt = W.random_batch(zlib.crc32(name.encode()) % 10000, lq, lk, H, D)
    plan = J.Plan(bt["q_off"], bt["kv_off"], H, D, mxfp8=True, device=0)
    got = _run(bt, plan)
    q, k, v, do = (bt[n].double().numpy() for n in ("q", "k", "v", "dout"))
    out, lse, aout = M.forward(bt["q_off"], bt["kv_off"], q, k, v, with_allowance=True)
    _within(got["out"], out, PT.FWD_TOL, aout, "out")
    PT.assert_close(got["lse"], lse, PT.FWD_TOL, "lse")
    dq, dk, dv, adq, adk, adv = M.backward(bt["q_off"], bt["kv_off"], q, k, v, do, with_allowance=True)
    for n, ref, al in (("dq", dq, adq), ("dk", dk, adk), ("dv", dv, adv)):
        _within(got[n], ref, PT.BWD_TOL, al, n)
    plan.close()


def test_mxfp8_differs_from_bf16_path():
    """The quantisation is really applied: the MXFP8 forward moves away from
    the bf16 path (by about the E4M3 step), which the oracle's plain attention
    matches."""
    bt = W.random_batch(202, [300, 129], [300, 129], 2, 128)
    a = _run(bt, J.Plan(bt["q_off"], bt["kv_off"], 2, 128, mxfp8=True, device=0))
    b = _run(bt, J.Plan(bt["q_off"], bt["kv_off"], 2, 128, device=0))
    assert np.abs(a["out"] - b["out"]).max() > 1e-2
    assert np.abs(a["dq"] - b["dq"]).max() > 1e-2


def test_mxfp8_deterministic():
    bt = W.random_batch(203, [513, 64, 200], [513, 64, 200], 2, 128)
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, 128, mxfp8=True, device=0)
    a, b = _run(bt, plan), _run(bt, plan)
    for n in ("out", "lse", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)
    plan.close()


def test_mxfp8_argument_checks():
    qo = W.offsets(np.array([40, 100]))
    for kw in (dict(act=J.SILU), dict(block=64), dict(window=16), dict(bias_buckets=4), dict(dtype="fp32"),
               dict(broadcast_q=True)):
        off = W.offsets(np.array([40, 40])) if kw.get("broadcast_q") else qo
        with pytest.raises(J.JattnError) as e:
            J.Plan(off, off, 2, 64, mxfp8=True, device=0, **kw)
        assert e.value.code == J.ERR_UNSUPPORTED, kw
    with pytest.raises(J.JattnError) as e:
        J.Plan(qo, qo, 2, 32, mxfp8=True, device=0)
    assert e.value.code == J.ERR_UNSUPPORTED
    plan = J.Plan(qo, qo, 2, 64, mxfp8=True, device=0)
    # the backward has no path without the dS chunks: its minimum is its full size
    assert plan.bwd_workspace_bytes_min == plan.bwd_workspace_bytes > 0
    bt = W.random_batch(204, [40, 100], [40, 100], 2, 64)
    dev = torch.device("cuda", 0)
    q, k, v, do = (bt[n].to(dev) for n in ("q", "k", "v", "dout"))
    out, lse = plan.fwd(q, k, v)
    small = torch.empty(plan.bwd_workspace_bytes - 256, dtype=torch.uint8, device=dev)
    rc = J.load().jattn_bwd(plan._h, *(J._binding._ptr(t) for t in (do, q, k, v)), None, J._binding._ptr(out),
                            J._binding._ptr(lse), *(J._binding._ptr(torch.empty_like(t)) for t in (q, k, v)), None,
                            J._binding._ptr(small), small.numel(), None)
    assert rc == J.ERR_WORKSPACE
    plain = J.Plan(qo, qo, 2, 64, device=0)
    with pytest.raises(J.JattnError) as e:
        plain.mxfp8_quantize(q, J.TILES_Q)
    assert e.value.code == J.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    plan.close()
    plain.close()


def test_mxfp8_full_size_self_attention_sampled():
    """The self-attention workload's batch (B=256, H=4, D=128, lengths up to
    1000; MXFP8 takes no bias), sampled sequences against the oracle."""
    b = W.make_batch(2)
    bt = dict(q_off=b.q_off, kv_off=b.kv_off, q=b.q, k=b.k, v=b.v, bias=None, dout=b.dout, scale=b.scale)
    plan = J.Plan(b.q_off, b.kv_off, b.w.H, b.w.D, mxfp8=True, device=0)
    got = _run(bt, plan)
    for n in ("out", "dq", "dk", "dv"):
        assert np.isfinite(got[n]).all(), n
    lens = np.diff(b.q_off.astype(np.int64))
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 7, 100})
    qo, ko, (q, do), (k, v), qidx, kidx = oracle.sub_batch(b.q_off, b.kv_off, seqs, b.q, b.dout,
                                                           tensors_kv=(b.k, b.v))
    q, k, v, do = (t.double().numpy() for t in (q, k, v, do))
    out, lse, aout = M.forward(qo, ko, q, k, v, with_allowance=True)
    _within(got["out"][qidx], out, PT.FWD_TOL, aout, "out")
    dq, dk, dv, adq, adk, adv = M.backward(qo, ko, q, k, v, do, with_allowance=True)
    _within(got["dq"][qidx], dq, PT.BWD_TOL, adq, "dq")
    _within(got["dk"][kidx], dk, PT.BWD_TOL, adk, "dk")
    _within(got["dv"][kidx], dv, PT.BWD_TOL, adv, "dv")
    # on this representative batch the allowance widens the tolerance of a
    # typical element by well under half
    for al, ref, tol in ((aout, out, PT.FWD_TOL), (adq, dq, PT.BWD_TOL), (adk, dk, PT.BWD_TOL),
                         (adv, dv, PT.BWD_TOL)):
        assert np.median(al / (tol[0] + tol[1] * np.abs(ref))) < 0.5
    plan.close()
