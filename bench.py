"""Benchmark: valid-token jagged attention TFLOP/s, forward + backward, on GB300.

One step = the whole hot path over one synthetic batch: plan (tile lists +
schedule, uploaded), forward, backward.  Inputs are resident in HBM when the
timed region starts; L2 is flushed (a 256 MiB write) between timed steps.  The
planner's host time is measured per step and reported as planner_host_ms; the
device-timed step starts after the plan has been queued.  The forward and the
backward are launched as two CUDA graphs captured once from the library's
calls (the same kernels and arguments, without host launch work between
them); the eager form's step time and the per-kernel times (events recorded by
the library between its kernels) are reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ID] [--impl ours|reference]

With torchrun (N > 1) the batch grows to N x B sequences drawn from the same
length distribution and is split across the ranks by whole sequences, balanced
by cost (jattn_shard): weak scaling with no collective on the attention path.
The reported time is the max over ranks and the value counts the valid-token
work of the whole global batch.  --impl reference times the
fp64 CPU oracle instead (rank 0 only), on a bounded sample of the same batch.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from jagged_attention_recommendation_gb300 import workloads as W  # noqa: E402

METRIC = "valid-token attention TFLOPs fwd+bwd (bf16), % of GB300 dense-BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def workload_config(w: W.Workload, act: int, Bn: int, flush: bool, ws: int = 1, global_B=None) -> dict:
    return {"workload": "%s (B=%d, H=%d, D=%d, %s%s%s)" % (
        w.name, Bn, w.H, w.D, W.ACT_NAMES[act], ", rel-pos bias %d buckets" % w.bias_buckets if w.bias_buckets
        else "", ", block %d" % w.block if w.block else "") + (", sliding window %d" % w.window if w.window else ""),
        "B": Bn, "H": w.H, "D": w.D, "act": W.ACT_NAMES[act], "block": w.block, "bias_buckets": w.bias_buckets,
        "window": w.window,
        "input_dtype": w.dtype, "l2": "flushed between timed steps (256 MiB write)" if flush else "not flushed",
        "parallelism": ("single GPU" if ws == 1 else
                        "dp%d: %d sequences split across ranks by cost (jattn_shard), no collective" % (ws, global_B))}


# ---------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = np.array([num(r[1]) for r in rows])
        mx = np.array([num(r[2]) for r in rows])
        pw = np.array([num(r[3]) for r in rows])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        load = sm[pw >= np.nanmedian(pw)] if np.isfinite(pw).any() else sm
        return {"sm_mhz": float(np.nanmedian(load)), "sm_max_mhz": float(np.nanmax(mx)), "reasons": reasons,
                "samples": len(rows), "power_w_max": float(np.nanmax(pw))}


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def sample_sequences(q_off, kv_off, frac: float, seed: int = 0):
    """Seeded subset of sequences holding about `frac` of the batch's valid pairs."""
    lq = np.diff(q_off.astype(np.int64))
    lk = np.diff(kv_off.astype(np.int64))
    pairs = lq * lk
    order = np.random.default_rng(seed).permutation(len(lq))
    target = frac * pairs.sum()
    picked, acc = [], 0
    for b in order:
        picked.append(int(b))
        acc += pairs[b]
        if acc >= target:
            break
    return sorted(picked)


def variant_keys(args, w: W.Workload) -> dict:
    """Config entries of the optional variants (the same on both arms)."""
    out = {}
    if args.rope:
        out["rope"] = "Q and K rotated in the kernels, standard table (base 10000)"
    if args.broadcast_q:
        out["broadcast_q"] = "%d shared query rows, dQ summed over the sequences" % w.q_rows_shared
    if getattr(args, "mxfp8", False):
        out["mxfp8"] = ("Q, K, V, dO quantised to E4M3 with E8M0 scales per 32 x 32 block, P and dS quantised "
                        "online; products on the bf16 tensor cores (the quantised values are exact in bf16)")
    return out


def rope_tables(batch: W.Batch, w: W.Workload):
    """Standard rotary tables (cos, sin) covering the batch's longest sequence."""
    longest = int(max(np.diff(batch.q_off.astype(np.int64)).max(), np.diff(batch.kv_off.astype(np.int64)).max()))
    return W.rope_table(longest, w.D, "standard")


def time_oracle(batch: W.Batch, frac: float, seed: int = 0, rope=None, mxfp8=False):
    from oracle import oracle
    w = batch.w
    seqs = sample_sequences(batch.q_off, batch.kv_off, frac, seed)
    qo, ko, (q, dout), (k, v), _, _ = oracle.sub_batch(batch.q_off, batch.kv_off, seqs, batch.q, batch.dout,
                                                       tensors_kv=(batch.k, batch.v))
    nthreads = oracle.default_threads()
    t0 = time.perf_counter()
    if mxfp8:  # the MXFP8 oracle (numpy, one thread)
        from oracle import mxfp8 as MX
        nthreads = 1
        qd, kd, vd, dd = (t.double().numpy() for t in (q, k, v, dout))
        MX.forward(qo, ko, qd, kd, vd, scale=batch.scale)
        MX.backward(qo, ko, qd, kd, vd, dd, scale=batch.scale)
    else:
        oracle.forward(qo, ko, q, k, v, bias=batch.bias, scale=batch.scale, act=batch.act, block=w.block,
                       nthreads=nthreads, window=w.window, rope=rope)
        oracle.backward(qo, ko, q, k, v, dout, bias=batch.bias, scale=batch.scale, act=batch.act, block=w.block,
                        nthreads=nthreads, window=w.window, rope=rope)
    dt = time.perf_counter() - t0
    f, b = W.flops(qo, ko, w.H, w.D, w.block, w.window)
    desc = "%d of %d sequences (seeded), %.1f%% of the valid pairs" % (
        len(seqs), batch.B, 100.0 * W.valid_pairs(qo, ko, w.block, w.window) /
        max(W.valid_pairs(batch.q_off, batch.kv_off, w.block, w.window), 1))
    return (f + b) / dt / 1e12, dt, nthreads, desc


def run_reference(args, w, batch):
    rope = rope_tables(batch, w) if args.rope else None
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    for _ in range(args.warmup):
        time_oracle(batch, args.ref_frac, seed=1, rope=rope, mxfp8=args.mxfp8)
    vals, times = [], []
    for s in range(args.steps):
        v, dt, cores, desc = time_oracle(batch, args.ref_frac, seed=2 + s, rope=rope, mxfp8=args.mxfp8)
        vals.append(v)
        times.append(dt)
    value = float(np.mean(vals))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(workload_config(w, batch.act, batch.B, False), **variant_keys(args, w)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: " + desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
# DRAM bytes (read + write) per launch from one ncu capture (the launch list of
# the bench command, profiles/launches_*.md), keyed by (workload, activation,
# MXFP8, kernel), with the hash of the kernel sources the counters were taken
# on; a record whose sources have changed since is reported as null.
KERNEL_FILES = {"fwd": ("fwd.cu", "fwd_kernel.cuh"), "bwd_dkdv": ("bwd_dkdv.cu", "bwd_common.cuh"),
                "bwd_dq_gemm": ("bwd_dqg.cu",), "bwd_dq": ("bwd.cu", "bwd_common.cuh"), "bwd_delta": ("aux.cu",),
                "bwd_block": ("bwd_block.cu",)}
KERNEL_FILES.update({n: ("aux.cu",) for n in ("mx_quant", "bwd_mx_quant")})
NCU_TRAFFIC = {
    (2, "softmax", False, "fwd"): (2.71e+08, "688683d13ce05447"),
    (2, "softmax", False, "bwd_delta"): (1.378e+08, "a8f3db73114ce982"),
    (2, "softmax", False, "bwd_dkdv"): (6.552e+08, "0b28b2c0fd36c3d4"),
    (2, "softmax", False, "bwd_dq_gemm"): (3.689e+08, "d415a547fd8f09fa"),
    (3, "softmax", False, "fwd"): (5.452e+08, "688683d13ce05447"),
    (3, "softmax", False, "bwd_delta"): (4.765e+08, "a8f3db73114ce982"),
    (3, "softmax", False, "bwd_dkdv"): (7.057e+08, "0b28b2c0fd36c3d4"),
    (3, "softmax", False, "bwd_dq_gemm"): (2.959e+08, "d415a547fd8f09fa"),
    (4, "silu", False, "fwd"): (9.357e+08, "688683d13ce05447"),
    (4, "silu", False, "bwd_dkdv"): (1.965e+09, "0b28b2c0fd36c3d4"),
    (4, "silu", False, "bwd_dq_gemm"): (9.018e+08, "d415a547fd8f09fa"),
    (4, "gelu_tanh", False, "fwd"): (9.357e+08, "688683d13ce05447"),
    (4, "gelu_tanh", False, "bwd_dkdv"): (1.966e+09, "0b28b2c0fd36c3d4"),
    (4, "gelu_tanh", False, "bwd_dq_gemm"): (9.019e+08, "d415a547fd8f09fa"),
    (5, "softmax", False, "fwd"): (1.12e+09, "688683d13ce05447"),
    (5, "softmax", False, "bwd_block"): (1.953e+09, "2733bc711320aacd"),
    (2, "softmax", True, "mx_quant"): (3.612e+08, "a8f3db73114ce982"),
    (2, "softmax", True, "fwd"): (2.715e+08, "688683d13ce05447"),
    (2, "softmax", True, "bwd_mx_quant"): (4.996e+08, "a8f3db73114ce982"),
    (2, "softmax", True, "bwd_delta"): (1.379e+08, "a8f3db73114ce982"),
    (2, "softmax", True, "bwd_dkdv"): (6.519e+08, "0b28b2c0fd36c3d4"),
    (2, "softmax", True, "bwd_dq_gemm"): (3.692e+08, "d415a547fd8f09fa"),
}


def kernel_source_hash(files) -> str:
    import hashlib
    m = hashlib.sha256()
    csrc = os.path.join(ROOT, "jagged_attention_recommendation_gb300", "csrc")
    for f in tuple(files) + ("attn.cuh", "device.cuh", "common.h"):
        m.update(open(os.path.join(csrc, f), "rb").read())
    return m.hexdigest()[:16]


def measured_traffic(wid: int, act: int, mxfp8: bool, kernel: str):
    rec = NCU_TRAFFIC.get((wid, W.ACT_NAMES[act], bool(mxfp8), kernel))
    if rec is None or kernel not in KERNEL_FILES or kernel_source_hash(KERNEL_FILES[kernel]) != rec[1]:
        return None
    return rec[0]


KERNELS_FULL = ["fwd", "bwd_delta", "bwd_dq", "bwd_dkdv"]       # backward with the recomputing dQ pass
KERNELS_FULL_DS = ["fwd", "bwd_delta", "bwd_dkdv", "bwd_dq_gemm"]  # backward with dS chunks (full workspace)
KERNELS_BLOCK = ["fwd", "bwd_block"]


def kernel_names(w, act, device_plan=False, broadcast_q=False, mxfp8=False):
    """The kernels one step launches, in order (the library takes the dS-chunk
    backward for full attention on a host plan without a window, given the full
    workspace as the bench does).  MXFP8: the forward first quantises Q, K, V,
    the backward Q, dO, K, V (one launch each)."""
    if w.block:
        return list(KERNELS_BLOCK)
    ds = not w.window and not device_plan
    names = [n for n in (KERNELS_FULL_DS if ds else KERNELS_FULL) if n != "bwd_delta" or act == W.SOFTMAX]
    if broadcast_q:  # the per-sequence dQ rows are summed by one more kernel
        names.insert(names.index("bwd_dq_gemm" if ds else "bwd_dq") + 1, "bwd_dq_reduce")
    if mxfp8:
        names = ["mx_quant"] + names
        names.insert(names.index("fwd") + 1, "bwd_mx_quant")
    return names


def kernel_work(w, batch, name, pk, ds=True):
    """Algorithmic (flops, bytes) of one launch of `name` over the batch (ds:
    the backward writes dS chunks, i.e. full workspace on a host plan)."""
    H, D = w.H, w.D
    p = W.valid_pairs(batch.q_off, batch.kv_off, w.block, w.window)
    Tq, Tk = batch.Tq, batch.Tk
    e = H * D * 2
    if name == "fwd":
        return 4.0 * D * H * p, W.hbm_bytes(batch.q_off, batch.kv_off, H, D, batch.act, w.block)[0]
    if name == "bwd_block":
        return 10.0 * D * H * p, W.hbm_bytes(batch.q_off, batch.kv_off, H, D, batch.act, w.block)[1]
    if name == "bwd_delta":
        return 0.0, 2.0 * Tq * e + 4.0 * H * Tq
    if name == "mx_quant":  # Q, K, V bf16 rows in, their MXFP8 values out (bf16)
        return 0.0, 2.0 * (Tq + 2 * Tk) * e
    if name == "bwd_mx_quant":  # Q, dO, K, V
        return 0.0, 2.0 * (2 * Tq + 2 * Tk) * e
    if name == "bwd_dq_reduce":  # fp32 per-sequence dQ rows in, the shared rows' bf16 sum out
        return 0.0, 4.0 * Tq * H * D + 2.0 * w.q_rows_shared * H * D
    # the dS chunks (bf16 per valid pair and head; activation modes: hi and lo)
    ds_bytes = 2.0 * H * p * (1 if batch.act == W.SOFTMAX else 2)
    if name == "bwd_dq":  # dQ GEMM; its S and dP recompute is not counted
        lse = 8.0 * H * Tq if batch.act == W.SOFTMAX else 0.0
        return 2.0 * D * H * p, 2.0 * Tq * e + 2.0 * Tk * e + Tq * e + lse
    if name == "bwd_dq_gemm":  # dQ = scale dS K: the dS chunks and K in, dQ out
        return 2.0 * D * H * p, ds_bytes + Tk * e + Tq * e
    if name == "bwd_dkdv":  # S, dP, dV, dK (and, on the dS-chunk path, the chunks out)
        lse = 8.0 * H * Tq if batch.act == W.SOFTMAX else 0.0
        ds_out = ds_bytes if (ds and not w.block and not w.window) else 0.0
        return 8.0 * D * H * p, 2.0 * Tq * e + 2.0 * Tk * e + 2.0 * Tk * e + lse + ds_out
    raise KeyError(name)


def run_ours(args, w, batch):
    import torch.distributed as dist

    import jagged_attention_recommendation_gb300 as J
    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    H, D = w.H, w.D
    f32 = w.dtype == "fp32"
    tdt = torch.float32 if f32 else torch.bfloat16

    # resident inputs and outputs
    q, k, v, dout = (t.to(dev) for t in (batch.q, batch.k, batch.v, batch.dout))
    bias = batch.bias.to(dev) if batch.bias is not None else None
    plan = J.Plan(batch.q_off, batch.kv_off, H, D, act=batch.act, block=w.block, bias_buckets=w.bias_buckets,
                  window=w.window,
                  dtype="fp32" if f32 else "bf16", device=local, broadcast_q=args.broadcast_q, mxfp8=args.mxfp8)
    if args.broadcast_q:  # the shared query rows once, not one copy per sequence
        q = q[:w.q_rows_shared].contiguous()
    out = torch.empty(batch.Tq, H, D, dtype=tdt, device=dev)
    lse = torch.empty(H, batch.Tq, dtype=torch.float32, device=dev) if batch.act == W.SOFTMAX else None
    dq = torch.empty(plan.q_rows, H, D, dtype=tdt, device=dev)
    dk = torch.empty(batch.Tk, H, D, dtype=tdt, device=dev)
    dv = torch.empty(batch.Tk, H, D, dtype=tdt, device=dev)
    fws = torch.empty(max(plan.fwd_workspace_bytes, 1), dtype=torch.uint8, device=dev)
    bws = torch.empty(max(plan.bwd_workspace_bytes, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rope = rope_tables(batch, w) if args.rope else None
    rp = None if rope is None else tuple(t.to(dev) for t in rope)
    d_qo = torch.from_numpy(batch.q_off.astype(np.int32)).to(dev)
    d_ko = torch.from_numpy(batch.kv_off.astype(np.int32)).to(dev)

    def replan():
        if args.device_plan:  # tile lists built on the GPU from the device offsets
            plan.update_device(d_qo, d_ko, batch.Tq, batch.Tk, stream)
        else:
            plan.update(batch.q_off, batch.kv_off, stream)

    def step():
        replan()
        plan.fwd(q, k, v, bias=bias, out=out, lse=lse, workspace=fws, stream=stream, rope=rp)
        plan.bwd(dout, q, k, v, out, lse=lse, bias=bias, dq=dq, dk=dk, dv=dv, workspace=bws, stream=stream,
                 rope=rp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = plan.check_status()
    if st != 0:
        raise RuntimeError("device status after warm-up: " + J.status_str(st))

    # planner host time on an idle stream (no wait on earlier uploads)
    plan_host_ms, plan_dev_ms = [], []
    for _ in range(max(args.steps, 5)):
        torch.cuda.synchronize()
        t_p = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        replan()
        plan_host_ms.append((time.perf_counter() - t_p) * 1e3)
        e1.record(stream)
        e1.synchronize()
        plan_dev_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()

    names = kernel_names(w, batch.act, args.device_plan, args.broadcast_q, args.mxfp8)
    n_fwd = names.index("fwd") + 1
    n_bwd = len(names) - n_fwd
    if f32 or D == 32:
        raise SystemExit("bench: staged (fp32 / D=32) workloads are parity cases, not bench lines")
    visible = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    phys = int(visible[local]) if local < len(visible) and visible[local].strip().isdigit() else local

    # The timed step: forward and backward launched as two CUDA graphs (captured
    # once; the same kernels and arguments as the eager calls, without the host's
    # launch work between them), the plan update queued before each step's start
    # event as in the eager form.  --no-graph times the eager calls instead.
    use_graph = not args.no_graph
    if use_graph:
        g_f, g_b = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(g_f, stream=cap):
            plan.fwd(q, k, v, bias=bias, out=out, lse=lse, workspace=fws, stream=cap, rope=rp)
        with torch.cuda.graph(g_b, stream=cap):
            plan.bwd(dout, q, k, v, out, lse=lse, bias=bias, dq=dq, dk=dk, dv=dv, workspace=bws, stream=cap,
                     rope=rp)
        stream.wait_stream(cap)

    def timed_step():
        if use_graph:
            with torch.cuda.stream(stream):
                g_f.replay()
                g_b.replay()
        else:
            plan.fwd(q, k, v, bias=bias, out=out, lse=lse, workspace=fws, stream=stream, rope=rp)
            plan.bwd(dout, q, k, v, out, lse=lse, bias=bias, dq=dq, dk=dk, dv=dv, workspace=bws, stream=stream,
                     rope=rp)

    for _ in range(3):
        replan()
        timed_step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(phys)
    sampler.start()
    # Load soak: the same step, back to back, for --soak seconds right before the
    # timed region, so that the clock sampler (and any outside one) sees the GPU
    # under this load and the timed steps run at its loaded clocks.
    soak_steps = 0
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        for _ in range(16):
            replan()
            timed_step()
        soak_steps += 16
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = plan.launch_count
    t_wall0 = time.perf_counter()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        # the planner's host work (tile lists, schedule, upload enqueue) is reported
        # on its own (planner_host_ms), not inside the device-timed step
        replan()
        starts[s].record(stream)
        timed_step()
        ends[s].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    clocks["window"] = "sampled every 50 ms over a %.1f s load soak (%d steps) and the timed steps" % (
        args.soak, soak_steps)
    # kernels launched in the timed region (graph replays launch the captured ones)
    launches = args.steps * len(names) if use_graph else plan.launch_count - launches0
    st = plan.check_status()
    if st != 0:
        raise RuntimeError("device status after timed region: " + J.status_str(st))
    step_ms = np.array([starts[s].elapsed_time(ends[s]) for s in range(args.steps)])
    ms = float(step_ms.mean())
    if ws > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    # per-kernel device times: the same step from eager calls, CUDA events
    # recorded by the library between its kernels (L2 flushed as above)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        replan()
        es[s].record(stream)
        plan.set_events(kev[s][0:n_fwd + 1])
        plan.fwd(q, k, v, bias=bias, out=out, lse=lse, workspace=fws, stream=stream, rope=rp)
        plan.set_events(kev[s][n_fwd:])
        plan.bwd(dout, q, k, v, out, lse=lse, bias=bias, dq=dq, dk=dk, dv=dv, workspace=bws, stream=stream,
                 rope=rp)
        ee[s].record(stream)
    torch.cuda.synchronize()
    plan.set_events(None)
    st = plan.check_status()
    if st != 0:
        raise RuntimeError("device status after the eager steps: " + J.status_str(st))
    per_kernel = {n: float(np.mean([kev[s][i].elapsed_time(kev[s][i + 1]) for s in range(args.steps)]))
                  for i, n in enumerate(names)}
    eager_ms = float(np.mean([es[s].elapsed_time(ee[s]) for s in range(args.steps)]))
    if ws > 1:
        t = torch.tensor([eager_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        eager_ms = float(t.item())
    if use_graph:
        del g_f, g_b

    f_fwd, f_bwd = W.flops(batch.q_off, batch.kv_off, H, D, w.block, w.window)
    total_flops = args.global_flops if args.global_flops is not None else ws * (f_fwd + f_bwd)
    value = total_flops / (ms * 1e-3) / 1e12
    pk, pk_kind = peaks()

    # roofline of the dominant kernel (largest share of the step's kernel time)
    bf, bb = W.hbm_bytes(batch.q_off, batch.kv_off, H, D, batch.act, w.block)
    intensity = (f_fwd + f_bwd) / (bf + bb)
    roof = roofline_of(w, batch, per_kernel, pk, pk_kind, ds=not args.device_plan, mxfp8=args.mxfp8)
    eager = {"ms_per_step": eager_ms, "value": total_flops / (eager_ms * 1e-3) / 1e12, "unit": UNIT,
             "note": "the same step from eager calls (host launch work between kernels)"}

    # end to end through the public API with host buffers (the host-buffer step
    # has no rotary-embedding form)
    e2e = run_e2e(args, w, batch, plan, dev, stream) if not (args.no_e2e or args.rope or args.broadcast_q) else None
    if ws > 1 and e2e is not None:
        t = torch.tensor([e2e["ms_per_step"]], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e["ms_per_step"] = float(t.item())
        e2e["value"] = total_flops / (e2e["ms_per_step"] * 1e-3) / 1e12

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "launch": "CUDA graphs (forward, backward) replayed per step" if use_graph else "eager calls",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict(workload_config(w, batch.act, batch.B, True, ws, args.global_B), **variant_keys(args, w)),
            "pct_of_bf16_peak": 100.0 * value / ws / pk["bf16_tflops"],
            "pct_of_bf16_peak_sustained": 100.0 * value / ws / pk["bf16_tflops_sustained"],
            "per_kernel_ms": per_kernel, "gpu_launches": int(launches),
            "fwd_ms": float(sum(v_ for k_, v_ in per_kernel.items() if k_ == "fwd")),
            "bwd_ms": float(sum(v_ for k_, v_ in per_kernel.items() if k_ != "fwd")),
            "roofline": roof, "clocks": clocks,
            "workload_intensity_flop_per_byte": intensity,
            "planner_host_ms": float(np.median(plan_host_ms)),
            "planner_stream_ms": float(np.median(plan_dev_ms)),
            "planner": "device (jattn_plan_update_device)" if args.device_plan else "host (jattn_plan_update)",
            "timed_wall_s": t_wall}
    line["eager"] = eager
    if e2e is not None:
        line["e2e"] = {k2: e2e[k2] for k2 in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")}
        line["e2e"]["ms_per_step"] = e2e["ms_per_step"]
    plain = not (args.rope or args.broadcast_q or args.window or args.device_plan or args.act is not None or
                 args.mxfp8)
    if rank == 0 and ws == 1 and w.wid == 2 and plain and not args.no_others:
        # the other workloads' step throughput and dominant-kernel roofline
        # fractions, measured in this run beside the self-attention line
        del q, k, v, dout, out, dq, dk, dv, fws, bws
        torch.cuda.empty_cache()
        others = {}
        for wid, act in OTHER_WORKLOADS:
            key = "%d_%s" % (wid, W.ACT_NAMES[act])
            others[key] = measure_other(wid, act, dev, stream, max(10, min(args.steps, 30)), flush)
            torch.cuda.empty_cache()
        # MXFP8 attention on the self-attention batch (without its bias)
        others["2_mxfp8"] = measure_other(2, W.SOFTMAX, dev, stream, max(10, min(args.steps, 30)), flush,
                                          mxfp8=True)
        torch.cuda.empty_cache()
        line["others"] = others
    if rank == 0 and ws == 1 and not args.no_cpu:
        # the MXFP8 oracle is numpy on one thread: a smaller seeded share of the batch
        v_cpu, dt, cores, desc = time_oracle(batch, min(args.cpu_frac, 0.02) if args.mxfp8 else args.cpu_frac,
                                             seed=0, rope=rope, mxfp8=args.mxfp8)
        line["cpu_baseline"] = {"value": v_cpu, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt}
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# the other workloads measured beside the self-attention line (the tiny fp32
# workload is a parity case only)
OTHER_WORKLOADS = [(3, W.SOFTMAX), (4, W.SILU), (4, W.GELU_TANH), (5, W.SOFTMAX)]


def roofline_of(w, batch, per_kernel, pk, pk_kind, ds=True, mxfp8=False):
    """Roofline record of the kernel with the largest share of the step."""
    dom = max(per_kernel, key=per_kernel.get)
    fl, by = kernel_work(w, batch, dom, pk, ds)
    t_dom = per_kernel[dom] * 1e-3
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if fl > 0 and fl / by >= ridge * 0.5:
        roof = {"bound": "tensor", "achieved": fl / t_dom / 1e12, "peak": pk["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": by / t_dom / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = measured_traffic(w.wid, batch.act, mxfp8, dom)
    roof["traffic_unit"] = "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"
    roof["kernel"] = dom
    roof["peak_source"] = pk_kind + " (burst)"
    roof["algorithmic_flops_per_launch"] = fl
    roof["algorithmic_bytes_per_launch"] = by
    return roof


def measure_other(wid, act, dev, stream, steps, flush, mxfp8=False):
    """One other workload at full size: device-timed steps (plan update queued
    first, L2 flushed between steps), per-kernel times from the library's event
    hook, valid-token TFLOP/s and the dominant kernel's roofline fraction."""
    import jagged_attention_recommendation_gb300 as J
    batch = W.make_batch(wid, act=act)
    if mxfp8:  # MXFP8 takes no bias
        batch.w = dataclasses.replace(batch.w, bias_buckets=0)
        batch.bias = None
    w = batch.w
    H, D = w.H, w.D
    q, k, v, dout = (t.to(dev) for t in (batch.q, batch.k, batch.v, batch.dout))
    bias = batch.bias.to(dev) if batch.bias is not None else None
    plan = J.Plan(batch.q_off, batch.kv_off, H, D, act=batch.act, block=w.block, bias_buckets=w.bias_buckets,
                  device=dev.index, mxfp8=mxfp8)
    out = torch.empty(batch.Tq, H, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(H, batch.Tq, dtype=torch.float32, device=dev) if batch.act == W.SOFTMAX else None
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fws = torch.empty(max(plan.fwd_workspace_bytes, 1), dtype=torch.uint8, device=dev)
    bws = torch.empty(max(plan.bwd_workspace_bytes, 1), dtype=torch.uint8, device=dev)
    names = kernel_names(w, batch.act, mxfp8=mxfp8)
    nf = names.index("fwd") + 1

    def step(evs=None):
        plan.update(batch.q_off, batch.kv_off, stream)
        if evs is not None:
            plan.set_events(evs[0:nf + 1])
        plan.fwd(q, k, v, bias=bias, out=out, lse=lse, workspace=fws, stream=stream)
        if evs is not None:
            plan.set_events(evs[nf:])
        plan.bwd(dout, q, k, v, out, lse=lse, bias=bias, dq=dq, dk=dk, dv=dv, workspace=bws, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(steps)]
    for s_ in range(steps):
        flush.fill_(s_ & 0xFF)
        step(kev[s_])
    torch.cuda.synchronize()
    plan.set_events(None)
    st = plan.check_status()
    if st != 0:
        raise RuntimeError("device status, workload %d: %s" % (wid, J.status_str(st)))
    per_kernel = {n: float(np.mean([kev[s_][i].elapsed_time(kev[s_][i + 1]) for s_ in range(steps)]))
                  for i, n in enumerate(names)}
    ms = float(np.mean([kev[s_][0].elapsed_time(kev[s_][-1]) for s_ in range(steps)]))
    f_fwd, f_bwd = W.flops(batch.q_off, batch.kv_off, H, D, w.block, w.window)
    bf, bb = W.hbm_bytes(batch.q_off, batch.kv_off, H, D, batch.act, w.block)
    pk, pk_kind = peaks()
    roof = roofline_of(w, batch, per_kernel, pk, pk_kind, mxfp8=mxfp8)
    plan.close()
    return {"workload": workload_config(w, batch.act, batch.B, True)["workload"] + (", MXFP8" if mxfp8 else ""),
            "steps": steps,
            "value": (f_fwd + f_bwd) / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "per_kernel_ms": per_kernel,
            "step_hbm_frac": (bf + bb) / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "roofline": roof}


def run_e2e(args, w, batch, plan, dev, stream):
    """Same step through the C ABI with HOST inputs and outputs (jattn_step_host):
    each call re-plans from the host offsets, copies q, k, v, dO (and bias) from
    pinned host memory to the device, runs forward and backward, and copies O,
    dQ, dK, dV back to pinned host memory.  The library pipelines consecutive
    calls (one call's copies run during the neighbouring call's kernels); the
    timed region spans n calls and the wait for the last download."""
    H, D = w.H, w.D
    hq, hk, hv, hdo = (t.contiguous().pin_memory() for t in (batch.q, batch.k, batch.v, batch.dout))
    hbias = batch.bias.float().contiguous().pin_memory() if batch.bias is not None else None
    tdt = hq.dtype
    outs = [tuple(torch.empty(T, H, D, dtype=tdt).pin_memory() for T in (batch.Tq, batch.Tq, batch.Tk, batch.Tk))
            for _ in range(2)]  # one host output set per in-flight call
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo) + ((hbias,) if hbias is not None else ()))
    h2d += 4 * (len(batch.q_off) + len(batch.kv_off))  # offsets (the plan's tile upload is counted too)
    tiles_q, cta_q = plan.tiles(0)
    tiles_k, cta_k = plan.tiles(1)
    h2d += 24 * (len(tiles_q) + len(tiles_k)) + 4 * (len(cta_q) + len(cta_k))
    d2h = sum(t.numel() * t.element_size() for t in outs[0])

    def step(s):
        ho, hdq, hdk, hdv = outs[s & 1]
        plan.step_host(batch.q_off, batch.kv_off, hq, hk, hv, hdo, ho, hdq, hdk, hdv, bias=hbias, stream=stream)

    for s in range(2):
        step(s)
    plan.step_host_join(stream)
    torch.cuda.synchronize()
    n = max(3, args.steps)  # enough calls that filling and draining the pipeline is a small share
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(n):
        step(s)
    plan.step_host_join(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    st = plan.check_status()
    if st != 0:
        raise RuntimeError("device status after the end-to-end steps: " + J.status_str(st))
    ms = e0.elapsed_time(e1) / n
    f_fwd, f_bwd = W.flops(batch.q_off, batch.kv_off, H, D, w.block, w.window)
    return {"value": (f_fwd + f_bwd) / (ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, help="1..5 (default 2: jagged self-attention + bias)")
    ap.add_argument("--act", choices=["softmax", "silu", "gelu_tanh"], default=None)
    ap.add_argument("--cpu-frac", type=float, default=1.0, help="share of the batch's pairs the CPU baseline runs")
    ap.add_argument("--ref-frac", type=float, default=1.0 / 32, help="share of the batch per reference-arm step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager calls instead of CUDA-graph replays of the forward and backward")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--broadcast-q", action="store_true",
                    help="pooled-attention workload: one shared Q read by every sequence, dQ summed (--workload 4)")
    ap.add_argument("--device-plan", action="store_true",
                    help="re-plan every step on the GPU from device offsets (jattn_plan_update_device)")
    ap.add_argument("--rope", action="store_true",
                    help="rotary position embedding of Q and K (standard frequency table; block workload only)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window W (keys with |i - j| < W) on the chosen workload; 0 = off")
    ap.add_argument("--mxfp8", action="store_true",
                    help="MXFP8 attention (jattn_mode.mxfp8) on the chosen softmax workload, without its bias")
    ap.add_argument("--soak", type=float, default=1.5,
                    help="seconds of back-to-back steps right before the timed region (clocks under load)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the other workloads' lines (others) in the self-attention run")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    act = None if args.act is None else {"softmax": 0, "silu": 1, "gelu_tanh": 2}[args.act]
    ws, rank, _ = dist_env()
    args.global_flops = None
    args.global_B = None
    if args.impl == "ours" and ws > 1:
        # weak scaling: a global batch of N x B sequences from the same length
        # distribution, split across the N ranks by cost (jattn_shard); each rank
        # draws only its own sequences' tensors
        import jagged_attention_recommendation_gb300 as J
        w = W.WORKLOADS[args.workload]
        lq, lk = W.lengths(args.workload, B=ws * w.B)
        qo, ko = W.offsets(lq), W.offsets(lk)
        mine = np.nonzero(J.shard(qo, ko, ws) == rank)[0]
        batch = W.make_batch(args.workload, act=act, lens=(lq[mine], lk[mine]))
        args.global_flops = float(sum(W.flops(qo, ko, w.H, w.D, w.block, args.window)))
        args.global_B = int(ws * w.B)
    else:
        batch = W.make_batch(args.workload, act=act)
    if args.broadcast_q and not batch.w.q_rows_shared:
        ap.error("--broadcast-q runs on the pooled-attention workload (--workload 4)")
    if args.rope and not batch.w.block:
        ap.error("--rope runs on the BlockAttention workload (--workload 5)")
    if args.window:
        if batch.w.block:
            ap.error("--window does not combine with the block workload")
        batch.w = dataclasses.replace(batch.w, window=args.window)
    if args.mxfp8:
        if batch.w.block or args.window or args.broadcast_q or batch.act != W.SOFTMAX or batch.w.dtype != "bf16":
            ap.error("--mxfp8 runs softmax full attention on bf16 data (workloads 2, 3)")
        batch.w = dataclasses.replace(batch.w, bias_buckets=0)  # MXFP8 takes no bias
        batch.bias = None
    if args.impl == "reference":
        run_reference(args, batch.w, batch)
    else:
        run_ours(args, batch.w, batch)


if __name__ == "__main__":
    main()
