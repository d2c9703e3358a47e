"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
seeded inputs, element by element, within the stated tolerances."""
import zlib

import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from oracle import oracle
from tests import parity as PT

pytestmark = pytest.mark.gpu

SOFTMAX, SILU, GELU = W.SOFTMAX, W.SILU, W.GELU_TANH

# (name, lq, lk, H, D, bias_buckets, act, block, dtype)
CASES = [
    ("self_d128_tails", [1, 127, 128, 129, 300], None, 2, 128, 0, SOFTMAX, 0, torch.bfloat16),
    ("self_d128_bias", [45, 200, 129, 1, 390], None, 4, 128, 64, SOFTMAX, 0, torch.bfloat16),
    ("self_d64", [70, 256, 3, 190], None, 3, 64, 0, SOFTMAX, 0, torch.bfloat16),
    ("self_d64_bias", [70, 256, 3, 190], None, 2, 64, 16, SOFTMAX, 0, torch.bfloat16),
    ("cross_short_kv", [200, 35, 129, 511], [8, 64, 17, 40], 2, 128, 0, SOFTMAX, 0, torch.bfloat16),
    ("short_q_long_kv", [32, 32, 5], [600, 257, 1000], 2, 128, 0, SOFTMAX, 0, torch.bfloat16),
    ("empty_sequences", [10, 0, 140, 7], [0, 5, 30, 0], 2, 128, 0, SOFTMAX, 0, torch.bfloat16),
    ("gdpa_silu", [32, 32, 100], [700, 1500, 129], 2, 128, 0, SILU, 0, torch.bfloat16),
    ("gdpa_gelu", [32, 32, 100], [700, 1500, 129], 2, 128, 0, GELU, 0, torch.bfloat16),
    ("gdpa_silu_d64_bias", [150, 3], [90, 400], 2, 64, 8, SILU, 0, torch.bfloat16),
    ("block64_d64", [1, 63, 64, 65, 200, 513], None, 4, 64, 0, SOFTMAX, 64, torch.bfloat16),
    ("block64_d128_bias", [130, 64, 7, 300], None, 2, 128, 64, SOFTMAX, 64, torch.bfloat16),
    ("block64_silu", [100, 257], None, 2, 64, 0, SILU, 64, torch.bfloat16),
    ("block64_gelu_d128", [100, 257, 64], None, 2, 128, 0, GELU, 64, torch.bfloat16),
    ("fp32_d32", [31, 33, 49, 61], None, 2, 32, 0, SOFTMAX, 0, torch.float32),
    ("bf16_d32", [5, 140, 64], [9, 130, 1], 2, 32, 0, SOFTMAX, 0, torch.bfloat16),
    ("fp32_d128_bias", [40, 130, 257], [300, 20, 129], 2, 128, 16, SOFTMAX, 0, torch.float32),
    ("fp32_d64_block", [70, 130], None, 2, 64, 0, SOFTMAX, 64, torch.float32),
    # every query tile meets at most one 128-key block: the forward's groups take
    # whole tiles (reflected bias table, bias table, empty key sets, exactly 128 keys)
    ("tiles_d128_bias", [1, 64, 100, 128, 77, 260], [1, 64, 100, 128, 77, 100], 4, 128, 64, SOFTMAX, 0,
     torch.bfloat16),
    ("tiles_d64_table", [3, 128, 65, 90], None, 16, 64, 16, SOFTMAX, 0, torch.bfloat16),
    ("tiles_d64_empty", [300, 0, 17, 129], [128, 3, 0, 64], 2, 64, 0, SOFTMAX, 0, torch.bfloat16),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_parity_small(case):
    name, lq, lk, H, D, nb, act, block, dtype = case
    lk = lq if lk is None else lk
    bt = W.random_batch(zlib.crc32(name.encode()) % 10000, lq, lk, H, D, dtype=dtype, bias_buckets=nb)
    gpu = PT.run_library(bt, act=act, block=block, dtype="fp32" if dtype == torch.float32 else "bf16")
    # float32 cases: the oracle takes the unrounded float32 inputs
    ref = PT.run_oracle(bt, act=act, block=block)
    PT.compare(gpu, ref)


# sliding window W (|i - j| < W): (name, lq, lk, H, D, bias_buckets, act, W)
WINDOW_CASES = [
    ("win_self_d128", [1, 127, 128, 129, 300, 700], None, 2, 128, 0, SOFTMAX, 100),
    ("win_self_bias", [45, 200, 129, 390], None, 4, 128, 64, SOFTMAX, 33),
    ("win_one", [5, 130, 257], None, 2, 64, 0, SOFTMAX, 1),
    ("win_cross_empty_rows", [200, 35, 129], [8, 64, 300], 2, 128, 0, SOFTMAX, 20),
    ("win_silu", [300, 40], [500, 40], 2, 128, 0, SILU, 64),
    ("win_gelu_d64_bias", [150, 300], [150, 300], 2, 64, 8, GELU, 128),
    ("win_wider_than_all", [100, 300], None, 2, 128, 0, SOFTMAX, 5000),
]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=[c[0] for c in WINDOW_CASES])
def test_parity_window(case):
    name, lq, lk, H, D, nb, act, win = case
    lk = lq if lk is None else lk
    bt = W.random_batch(zlib.crc32(name.encode()) % 10000, lq, lk, H, D, dtype=torch.bfloat16, bias_buckets=nb)
    gpu = PT.run_library(bt, act=act, window=win)
    ref = PT.run_oracle(bt, act=act, window=win)
    PT.compare(gpu, ref)


def test_tiny_workload_fp32():
    """The tiny fp32 workload, exactly as drawn (B=4, H=2, D=32)."""
    b = W.make_batch(1)
    bt = dict(q_off=b.q_off, kv_off=b.kv_off, q=b.q, k=b.k, v=b.v, bias=None, dout=b.dout, scale=b.scale)
    gpu = PT.run_library(bt, dtype="fp32")
    PT.compare(gpu, PT.run_oracle(bt))


def test_run_to_run_bitwise_deterministic():
    bt = W.random_batch(7, [300, 129, 17], [300, 129, 17], 2, 128, bias_buckets=8)
    a = PT.run_library(bt)
    b = PT.run_library(bt)
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert np.array_equal(a[n], b[n]), n


def _sample_seqs(q_off, kv_off, k=6, seed=0):
    lq = np.diff(q_off.astype(np.int64))
    lk = np.diff(kv_off.astype(np.int64))
    work = lq * np.maximum(lk, 1)
    rng = np.random.default_rng(seed)
    picks = {int(np.argmax(work)), int(np.argmin(work))}
    while len(picks) < min(k, len(lq)):
        picks.add(int(rng.integers(len(lq))))
    return sorted(picks)


@pytest.mark.parametrize("wid,act", [(2, SOFTMAX), (3, SOFTMAX), (4, SILU), (4, GELU), (5, SOFTMAX)])
def test_full_size_workload_sampled(wid, act):
    """Full-size workload on the GPU; sampled sequences checked against the oracle."""
    b = W.make_batch(wid, act=act)
    w = b.w
    bt = dict(q_off=b.q_off, kv_off=b.kv_off, q=b.q, k=b.k, v=b.v, bias=b.bias, dout=b.dout, scale=b.scale)
    gpu = PT.run_library(bt, act=act, block=w.block)
    for n in ("out", "dq", "dk", "dv"):
        assert np.isfinite(gpu[n]).all(), n
    seqs = _sample_seqs(b.q_off, b.kv_off, k=4 if wid == 5 else 6)
    qo, ko, (q, dout), (k, v), qidx, kidx = oracle.sub_batch(b.q_off, b.kv_off, seqs, b.q, b.dout,
                                                             tensors_kv=(b.k, b.v))
    sub = dict(q_off=qo, kv_off=ko, q=q, k=k, v=v, bias=b.bias, dout=dout, scale=b.scale)
    ref = PT.run_oracle(sub, act=act, block=w.block)
    PT.assert_close(gpu["out"][qidx], ref["out"], PT.FWD_TOL, "out")
    if ref["lse"] is not None:
        PT.assert_close(gpu["lse"][:, qidx], ref["lse"], PT.FWD_TOL, "lse")
    PT.assert_close(gpu["dq"][qidx], ref["dq"], PT.BWD_TOL, "dq")
    PT.assert_close(gpu["dk"][kidx], ref["dk"], PT.BWD_TOL, "dk")
    PT.assert_close(gpu["dv"][kidx], ref["dv"], PT.BWD_TOL, "dv")


def test_plan_update_between_batches():
    """One plan re-planned for a second batch gives the same result as a fresh plan."""
    bt1 = W.random_batch(21, [100, 300], [100, 300], 2, 128)
    bt2 = W.random_batch(22, [5, 129, 260, 1], [5, 129, 260, 1], 2, 128)
    plan = J.Plan(bt1["q_off"], bt1["kv_off"], 2, 128, device=0)
    PT.run_library(bt1, plan=plan)
    plan.update(bt2["q_off"], bt2["kv_off"])
    a = PT.run_library(bt2, plan=plan)
    PT.compare(a, PT.run_oracle(bt2))


# bias-table gradient dT[h, n] = sum of dS over head h's pairs with min(|i - j|, NB - 1) = n
DT_CASES = [
    ("dt_self_d128", [45, 200, 129, 1, 390], None, 4, 128, 64, SOFTMAX, 0),
    ("dt_self_d64", [70, 256, 3, 190], None, 2, 64, 16, SOFTMAX, 0),
    ("dt_cross", [200, 35, 129, 511], [8, 64, 17, 40], 2, 128, 8, SOFTMAX, 0),
    ("dt_silu_d64", [150, 3], [90, 400], 2, 64, 8, SILU, 0),
    ("dt_gelu", [60, 300], [300, 60], 2, 128, 32, GELU, 0),
    ("dt_window", [45, 700, 129], None, 2, 128, 64, SOFTMAX, 100),
]


@pytest.mark.parametrize("min_ws", [False, True], ids=["full_workspace", "min_workspace"])
@pytest.mark.parametrize("case", DT_CASES, ids=[c[0] for c in DT_CASES])
def test_bias_gradient(case, min_ws):
    """dT is a sum over up to L^2 pairs whose softmax terms cancel (each row of dS
    sums to zero), so its entries can be far smaller than the terms; the backward
    tolerance is applied per head against the head's largest entry:
    |dT - ref| <= 3e-2 * max|ref_h| + 3e-2 * |ref|."""
    name, lq, lk, H, D, nb, act, win = case
    lk = lq if lk is None else lk
    bt = W.random_batch(zlib.crc32(name.encode()) % 10000, lq, lk, H, D, dtype=torch.bfloat16, bias_buckets=nb)
    dev = torch.device("cuda", 0)
    q, k, v, do = (bt[n].to(dev) for n in ("q", "k", "v", "dout"))
    bias = bt["bias"].float().to(dev)
    plan = J.Plan(bt["q_off"], bt["kv_off"], H, D, act=act, bias_buckets=nb, device=0, window=win)
    out, lse = plan.fwd(q, k, v, bias=bias)
    dbias = torch.full((H, nb), float("nan"), dtype=torch.float32, device=dev)
    # full workspace: the dK/dV pass sums dT (with the dS chunks); minimum: the dQ pass does
    ws = torch.empty(max(plan.bwd_workspace_bytes_min, 16), dtype=torch.uint8, device=dev) if min_ws else None
    plan.bwd(do, q, k, v, out, lse=lse, bias=bias, dbias=dbias, workspace=ws)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    _, _, _, ref = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"],
                                   bias=bt["bias"], scale=bt["scale"], act=act, window=win)
    got = dbias.cpu().double().numpy()
    assert np.isfinite(got).all()
    bound = 3e-2 * np.abs(ref).max(axis=1, keepdims=True) + 3e-2 * np.abs(ref)
    err = np.abs(got - ref)
    assert (err <= bound).all(), (name, float((err / np.maximum(bound, 1e-30)).max()))
    plan.close()


def test_bias_gradient_rejected_in_block_mode():
    bt = W.random_batch(7, [64, 100], [64, 100], 2, 64, dtype=torch.bfloat16, bias_buckets=4)
    dev = torch.device("cuda", 0)
    q, k, v, do = (bt[n].to(dev) for n in ("q", "k", "v", "dout"))
    bias = bt["bias"].float().to(dev)
    plan = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, block=64, bias_buckets=4, device=0)
    out, lse = plan.fwd(q, k, v, bias=bias)
    with pytest.raises(J.JattnError):
        plan.bwd(do, q, k, v, out, lse=lse, bias=bias, dbias=torch.zeros(2, 4, device=dev))
    plan.close()


# (name, lq, lk, H, D, bias_buckets, act)
PATH_CASES = [
    ("paths_self_bias", [1, 127, 129, 300, 64], None, 2, 128, 16, SOFTMAX),
    ("paths_cross", [200, 35, 511], [8, 300, 129], 2, 64, 0, SOFTMAX),
    ("paths_silu", [32, 100, 3], [700, 129, 257], 2, 128, 0, SILU),
    ("paths_gelu_d64", [150, 3], [90, 400], 2, 64, 8, GELU),
]


@pytest.mark.parametrize("case", PATH_CASES, ids=[c[0] for c in PATH_CASES])
def test_backward_paths(case):
    """The backward's two paths: with the full workspace the dK/dV pass writes
    the dS chunks and dQ is a streaming product of them; with the minimum
    workspace a dQ pass recomputes the scores.  Both match the oracle; dK and
    dV are the same kernels' results, bit for bit."""
    name, lq, lk, H, D, nb, act = case
    lk = lq if lk is None else lk
    bt = W.random_batch(zlib.crc32(name.encode()) % 10000, lq, lk, H, D, bias_buckets=nb)
    dev = torch.device("cuda", 0)
    q, k, v, do = (bt[n].to(dev) for n in ("q", "k", "v", "dout"))
    bias = bt["bias"].float().to(dev) if nb else None
    plan = J.Plan(bt["q_off"], bt["kv_off"], H, D, act=act, bias_buckets=nb, device=0)
    assert plan.bwd_workspace_bytes > plan.bwd_workspace_bytes_min
    out, lse = plan.fwd(q, k, v, bias=bias)
    full = plan.bwd(do, q, k, v, out, lse=lse, bias=bias)
    ws = torch.empty(max(plan.bwd_workspace_bytes_min, 16), dtype=torch.uint8, device=dev)
    small = plan.bwd(do, q, k, v, out, lse=lse, bias=bias, workspace=ws)
    torch.cuda.synchronize()
    assert plan.check_status() == 0
    ref = PT.run_oracle(bt, act=act)
    for res in (full, small):
        for t, n_, in zip(res, ("dq", "dk", "dv")):
            PT.assert_close(t.double().cpu().numpy(), ref[n_], PT.BWD_TOL, n_)
    for i in (1, 2):
        assert torch.equal(full[i], small[i])
    plan.close()
