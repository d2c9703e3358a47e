"""Host-side checks of the C ABI (no GPU): exported symbols, planner output
against the independent tile enumerator, schedule validity and error codes."""
import ctypes
import os
import re

import numpy as np
import pytest

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from oracle import tiles as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(J.LIB_PATH):
        from jagged_attention_recommendation_gb300 import build
        build.build()
    return J.load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(jattn_\w+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(J.EXPORTED)


def canonical(t):
    """Sort records into the enumerator's order: b, then tile start, then h."""
    return t[np.lexsort((t[:, 1], t[:, 2], t[:, 4], t[:, 0]))] if len(t) else t


def check_plan(qo, ko, H, D=128, block=0, act=0, window=0):
    p = J.Plan(qo, ko, H, D, act=act, block=block, device=-1, window=window)
    for which, fn in ((J.TILES_Q, T.q_major), (J.TILES_KV, T.kv_major)):
        tiles, cta = p.tiles(which)
        want = fn(qo, ko, H, block, window)
        assert tiles.dtype == np.int32 and tiles.shape == want.shape
        np.testing.assert_array_equal(canonical(tiles), canonical(want))
        # schedule: per-CTA contiguous ranges covering every tile once
        assert cta[0] == 0 and cta[-1] == len(tiles)
        assert np.all(np.diff(cta) >= 1) or len(tiles) == 0
        assert len(cta) - 1 == min(len(tiles), 152)
    p.close()


@pytest.mark.parametrize("lens,H,block", [
    (([1, 128, 129, 0, 300], [5, 0, 256, 7, 1]), 3, 0),
    (([64, 65, 200, 1], None), 2, 64),
    (([17], [4000]), 4, 0),
])
def test_planner_matches_enumerator(lib, lens, H, block):
    lq, lk = lens
    lk = lq if lk is None else lk
    check_plan(W.offsets(np.array(lq)), W.offsets(np.array(lk)), H, block=block)


@pytest.mark.parametrize("window", [1, 64, 257])
def test_planner_matches_enumerator_with_window(lib, window):
    lq, lk = [1, 128, 129, 0, 300, 900], [5, 0, 256, 7, 1, 900]
    check_plan(W.offsets(np.array(lq)), W.offsets(np.array(lk)), 3, window=window)


@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_planner_matches_enumerator_on_workloads(lib, wid):
    w = W.WORKLOADS[wid]
    lq, lk = W.lengths(wid)
    check_plan(W.offsets(lq), W.offsets(lk), w.H, D=w.D, block=w.block, act=w.act)


def test_schedule_balance_reported(lib):
    """LPT over 152 CTAs: report max/mean of the planner's own cost per CTA."""
    lq, lk = W.lengths(2)
    p = J.Plan(W.offsets(lq), W.offsets(lk), 4, 128, device=-1)
    tiles, cta = p.tiles(J.TILES_Q)
    cost = 8 + (tiles[:, 5] + 15) // 16
    loads = np.add.reduceat(cost, cta[:-1])
    ratio = loads.max() / loads.mean()
    assert ratio < 1.1, ratio


def test_plan_update_replans(lib):
    p = J.Plan(W.offsets(np.array([5, 6])), W.offsets(np.array([5, 6])), 2, 64, device=-1)
    qo = W.offsets(np.array([130, 1, 2]))
    p.update(qo, qo)
    tiles, _ = p.tiles(J.TILES_Q)
    np.testing.assert_array_equal(canonical(tiles), canonical(T.q_major(qo, qo, 2)))


def create(lib, qo, ko, H=2, D=64, act=0, block=0, nb=0, dtype=0, scale=0.0, device=-1, window=0):
    qo = np.ascontiguousarray(qo, dtype=np.int32)
    ko = np.ascontiguousarray(ko, dtype=np.int32)
    m = J.Mode(act, block, scale, nb, dtype, window)
    h = ctypes.c_void_p()
    rc = lib.jattn_plan_create(qo.ctypes.data_as(ctypes.c_void_p), ko.ctypes.data_as(ctypes.c_void_p), len(qo) - 1,
                               H, D, ctypes.byref(m), device, ctypes.byref(h))
    if rc == 0:
        lib.jattn_plan_destroy(h)
    return rc


def test_error_codes(lib):
    ok = [0, 3, 7]
    assert create(lib, ok, ok) == J.OK
    assert create(lib, [1, 3, 7], ok) == J.ERR_INVALID_ARG          # offsets[0] != 0
    assert create(lib, [0, 5, 3], ok) == J.ERR_INVALID_ARG          # decreasing
    assert create(lib, ok, ok, D=96) == J.ERR_UNSUPPORTED
    assert create(lib, ok, ok, D=0) == J.ERR_INVALID_ARG
    assert create(lib, ok, ok, H=0) == J.ERR_INVALID_ARG
    assert create(lib, ok, [0, 3, 8], block=64) == J.ERR_INVALID_ARG  # block needs equal lengths
    assert create(lib, ok, ok, block=32) == J.ERR_UNSUPPORTED
    assert create(lib, ok, ok, act=7) == J.ERR_INVALID_ARG
    assert create(lib, ok, ok, dtype=5) == J.ERR_INVALID_ARG
    assert create(lib, ok, ok, nb=-1) == J.ERR_INVALID_ARG
    assert create(lib, ok, ok, H=8, nb=64) == J.ERR_UNSUPPORTED     # bias table larger than staged maximum
    assert create(lib, ok, ok, scale=-1.0) == J.ERR_INVALID_ARG
    assert create(lib, ok, ok, device=-2) == J.ERR_INVALID_ARG
    assert create(lib, ok, ok, window=-1) == J.ERR_INVALID_ARG
    assert create(lib, ok, ok, block=64, window=8) == J.ERR_INVALID_ARG   # window and block exclude each other
    assert create(lib, ok, ok, window=8) == J.OK
    # float32 data: softmax only (their bf16 rounding on entry would exceed the
    # tolerances of the unnormalised activation sums)
    assert create(lib, ok, ok, dtype=1) == J.OK
    assert create(lib, ok, ok, dtype=1, act=1) == J.ERR_UNSUPPORTED
    assert create(lib, ok, ok, dtype=1, act=2) == J.ERR_UNSUPPORTED


def test_host_only_plan_refuses_compute(lib):
    p = J.Plan([0, 3], [0, 3], 1, 64, device=-1)
    rc = lib.jattn_fwd(p._h, None, None, None, None, None, None, None, 0, None)
    assert rc == J.ERR_NO_DEVICE
    rc = lib.jattn_bwd(p._h, None, None, None, None, None, None, None, None, None, None, None, None, 0, None)
    assert rc == J.ERR_NO_DEVICE
    assert lib.jattn_check_device_status(p._h, None) == J.ERR_NO_DEVICE
    assert lib.jattn_fwd(None, None, None, None, None, None, None, None, 0, None) == J.ERR_INVALID_ARG


def test_workspace_sizes(lib):
    qo = W.offsets(np.array([10, 20]))
    chunk = 128 * 64 * 2  # one dS chunk: 128 keys x 64 queries of bf16
    p = J.Plan(qo, qo, 2, 128, device=-1)
    assert p.fwd_workspace_bytes == 0
    assert p.bwd_workspace_bytes_min == 256  # Delta [H, Tq] fp32 = 240 B, 256-byte aligned
    # plus the dS chunks: 2 sequences x 2 heads x 1 key tile x 1 query block
    assert p.bwd_workspace_bytes == 256 + 4 * chunk
    p = J.Plan(qo, qo, 2, 128, act=J.SILU, device=-1)
    assert p.bwd_workspace_bytes_min == 0
    assert p.bwd_workspace_bytes == 4 * 2 * chunk  # hi and lo chunks
    p = J.Plan(qo, qo, 2, 128, act=J.SILU, window=8, device=-1)  # no dS chunks with a window
    assert p.bwd_workspace_bytes == p.bwd_workspace_bytes_min == 0
    lq = np.array([300, 1, 129])  # key tiles 3, 1, 2; query blocks 5, 1, 3
    p = J.Plan(W.offsets(lq), W.offsets(lq), 4, 64, device=-1)
    assert p.bwd_workspace_bytes - p.bwd_workspace_bytes_min == 4 * (3 * 5 + 1 * 1 + 2 * 3) * chunk
    p = J.Plan(qo, qo, 2, 32, dtype="fp32", device=-1)
    # staging of q, k, v to bf16 [T, H, 64]
    assert p.fwd_workspace_bytes == 3 * ((30 * 2 * 64 * 2 + 255) // 256 * 256)


def test_status_strings(lib):
    for code in range(9):
        s = J.status_str(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert J.status_str(99) == "unknown status"


def test_set_events_rejects_null_handles(lib):
    p = J.Plan([0, 3], [0, 3], 1, 64, device=-1)
    arr = (ctypes.c_void_p * 2)(None, None)
    assert lib.jattn_plan_set_events(p._h, arr, 2) == J.ERR_INVALID_ARG
    assert lib.jattn_plan_set_events(p._h, None, 0) == J.OK
    assert lib.jattn_plan_set_events(p._h, None, 3) == J.ERR_INVALID_ARG
    assert lib.jattn_plan_launch_count(p._h) == 0
    assert lib.jattn_last_cuda_error() == b""


def test_broadcast_q_plan_checks():
    """Broadcast Q: every sequence must have the shared rows' count; no block
    mode, fp32 data or D = 32."""
    ko = np.array([0, 50, 60, 200], np.int32)
    qo = np.array([0, 32, 64, 96], np.int32)
    p = J.Plan(qo, ko, 2, 128, device=-1, broadcast_q=True)
    assert p.q_rows == 32
    p.close()
    with pytest.raises(J.JattnError) as e:
        J.Plan(np.array([0, 32, 63, 95], np.int32), ko, 2, 128, device=-1, broadcast_q=True)
    assert e.value.code == J.ERR_INVALID_ARG
    for kw in (dict(block=64), dict(dtype="fp32")):
        with pytest.raises(J.JattnError) as e:
            J.Plan(qo, qo, 2, 128, device=-1, broadcast_q=True, **kw)
        assert e.value.code == J.ERR_UNSUPPORTED
    with pytest.raises(J.JattnError) as e:
        J.Plan(qo, ko, 2, 32, device=-1, broadcast_q=True)
    assert e.value.code == J.ERR_UNSUPPORTED
    p = J.Plan(qo, ko, 2, 128, device=-1, broadcast_q=True)
    with pytest.raises(J.JattnError) as e:  # a re-plan keeps the rule
        p.update(np.array([0, 32, 60, 96], np.int32), ko)
    assert e.value.code == J.ERR_INVALID_ARG
    p.close()


def test_device_update_argument_checks_on_host():
    """jattn_plan_update_device: NULL offsets are an argument error, and a
    host-only plan has no device to plan on (both decided before any pointer is
    read)."""
    import ctypes
    qo = np.array([0, 10, 30], np.int32)
    p = J.Plan(qo, qo, 2, 64, device=-1)
    lib = J.load()
    fake = ctypes.c_void_p(16)  # never dereferenced: the call returns first
    assert lib.jattn_plan_update_device(p._h, None, fake, 2, 30, 30, None) == J.ERR_INVALID_ARG
    assert lib.jattn_plan_update_device(p._h, fake, fake, 2, 30, 30, None) == J.ERR_NO_DEVICE
    assert lib.jattn_plan_update_device(None, fake, fake, 2, 30, 30, None) == J.ERR_INVALID_ARG
    p.close()
