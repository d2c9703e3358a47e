"""bench.py on the host: the reference arm's JSON line (the oracle timed on the
host cores), flag validation, and the work accounting the roofline uses."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from jagged_attention_recommendation_gb300 import workloads as W  # noqa: E402


def _run(*args, timeout=240):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                          timeout=timeout, cwd=ROOT)


@pytest.mark.parametrize("extra", [[], ["--window", "64"]])
def test_reference_arm_line(extra):
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-frac", "0.002", *extra)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["window"] == (64 if extra else 0)


@pytest.mark.parametrize("args", [["--warmup", "2"], ["--rope"], ["--broadcast-q"], ["--workload", "5", "--window", "64"]])
def test_bench_rejects_bad_flags(args):
    r = _run("--impl", "reference", *args)
    assert r.returncode == 2, (args, r.stderr[-500:])


def test_work_accounting():
    """Roofline numerators: the pages' FLOP convention on valid pairs and one
    HBM crossing per tensor."""
    b = W.make_batch(1)
    w = b.w
    pairs = W.valid_pairs(b.q_off, b.kv_off)
    assert pairs == int(np.sum(np.diff(b.q_off) * np.diff(b.kv_off)))
    fl, by = bench.kernel_work(w, b, "fwd", None)
    assert fl == 4.0 * w.D * w.H * pairs
    assert by == W.hbm_bytes(b.q_off, b.kv_off, w.H, w.D, b.act, w.block)[0]
    fl, _ = bench.kernel_work(w, b, "bwd_dkdv", None)
    assert fl == 8.0 * w.D * w.H * pairs
    fl, _ = bench.kernel_work(w, b, "bwd_dq", None)
    assert fl == 2.0 * w.D * w.H * pairs
    f_fwd, f_bwd = W.flops(b.q_off, b.kv_off, w.H, w.D)
    assert (f_fwd, f_bwd) == (4.0 * w.D * w.H * pairs, 10.0 * w.D * w.H * pairs)


def test_traffic_record_is_keyed_to_the_sources():
    """A recorded ncu traffic figure is reported only while its kernel's sources
    hash to the recorded value; a changed source (a different digest) or an
    unknown key gives null."""
    acts = {v: k for k, v in W.ACT_NAMES.items()}
    for (wid, act, mx, kernel), (value, digest) in bench.NCU_TRAFFIC.items():
        expect = value if bench.kernel_source_hash(bench.KERNEL_FILES[kernel]) == digest else None
        assert bench.measured_traffic(wid, acts[act], mx, kernel) == expect
    assert bench.measured_traffic(99, W.SOFTMAX, False, "fwd") is None
    saved = dict(bench.NCU_TRAFFIC)
    try:
        bench.NCU_TRAFFIC[(2, "softmax", False, "fwd")] = (1.0, "0" * 16)
        assert bench.measured_traffic(2, W.SOFTMAX, False, "fwd") is None
        bench.NCU_TRAFFIC[(2, "softmax", False, "fwd")] = (1.0, bench.kernel_source_hash(bench.KERNEL_FILES["fwd"]))
        assert bench.measured_traffic(2, W.SOFTMAX, False, "fwd") == 1.0
    finally:
        bench.NCU_TRAFFIC.clear()
        bench.NCU_TRAFFIC.update(saved)
