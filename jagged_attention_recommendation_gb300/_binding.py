"""ctypes binding of libjattn.so (include/jattn.h).  Argument marshalling only:
every step of the computation runs in the library's CUDA kernels.  There is no
fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libjattn.so")
_lib = None

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_TIMEOUT, \
    ERR_DEVICE_CHECK, ERR_NO_DEVICE = range(9)
SOFTMAX, SILU, GELU_TANH = 0, 1, 2
BF16, FP32 = 0, 1
TILES_Q, TILES_KV = 0, 1

EXPORTED = ("jattn_plan_create", "jattn_plan_update", "jattn_plan_tiles", "jattn_fwd_workspace_bytes",
            "jattn_bwd_workspace_bytes", "jattn_plan_destroy", "jattn_fwd", "jattn_bwd",
            "jattn_check_device_status", "jattn_status_str", "jattn_plan_set_events", "jattn_plan_launch_count", "jattn_last_cuda_error", "jattn_bwd_noalloc",
            "jattn_shard", "jattn_step_host", "jattn_step_host_join", "jattn_fwd_rope", "jattn_bwd_rope",
            "jattn_plan_update_device", "jattn_test_fwd_stall", "jattn_bwd_workspace_bytes_min",
            "jattn_mxfp8_quantize")


class JattnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        detail = ""
        if code == ERR_CUDA:
            detail = " [%s]" % load().jattn_last_cuda_error().decode()
        super().__init__("%s failed: %s (status %d)%s" % (what, status_str(code), code, detail))


class Mode(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int32), ("block", ctypes.c_int32), ("scale", ctypes.c_float),
                ("bias_buckets", ctypes.c_int32), ("dtype", ctypes.c_int32), ("window", ctypes.c_int32),
                ("broadcast_q", ctypes.c_int32), ("mxfp8", ctypes.c_int32)]


class Rope(ctypes.Structure):
    _fields_ = [("cos", ctypes.c_void_p), ("sin", ctypes.c_void_p), ("rows", ctypes.c_int32)]


def _rope(rope):
    """(cos, sin) float32 device tensors [P, D/2] -> a jattn_rope (kept alive by
    the caller's tensors for the call), or None."""
    if rope is None:
        return None
    cos, sin = rope
    if cos.shape != sin.shape or cos.dim() != 2:
        raise ValueError("rope tables: cos and sin must both be [P, D/2]")
    if cos.dtype != torch.float32 or sin.dtype != torch.float32 or not cos.is_contiguous() or not sin.is_contiguous():
        raise ValueError("rope tables: contiguous float32 tensors expected")
    return Rope(cos.data_ptr(), sin.data_ptr(), int(cos.shape[0]))


class TileRec(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("b", "h", "q_start", "q_len", "kv_start", "kv_len")]


def load():
    """Load libjattn.so (built in-tree by build.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libjattn.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.jattn_plan_create.argtypes = [P, P, i32, i32, i32, ctypes.POINTER(Mode), i32, ctypes.POINTER(P)]
    lib.jattn_plan_update.argtypes = [P, P, P, i32, P]
    lib.jattn_plan_tiles.argtypes = [P, i32, ctypes.POINTER(ctypes.POINTER(TileRec)), ctypes.POINTER(i64),
                                     ctypes.POINTER(ctypes.POINTER(i32)), ctypes.POINTER(i32)]
    lib.jattn_fwd_workspace_bytes.argtypes = [P]
    lib.jattn_fwd_workspace_bytes.restype = sz
    lib.jattn_bwd_workspace_bytes.argtypes = [P]
    lib.jattn_bwd_workspace_bytes.restype = sz
    lib.jattn_bwd_workspace_bytes_min.argtypes = [P]
    lib.jattn_bwd_workspace_bytes_min.restype = sz
    lib.jattn_plan_destroy.argtypes = [P]
    lib.jattn_plan_destroy.restype = None
    lib.jattn_fwd.argtypes = [P, P, P, P, P, P, P, P, sz, P]
    lib.jattn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.jattn_plan_update_device.argtypes = [P, P, P, i32, i64, i64, P]
    lib.jattn_plan_update_device.restype = i32
    lib.jattn_fwd_rope.argtypes = [P, P, P, P, P, ctypes.POINTER(Rope), P, P, P, sz, P]
    lib.jattn_fwd_rope.restype = i32
    lib.jattn_bwd_rope.argtypes = [P, P, P, P, P, P, ctypes.POINTER(Rope), P, P, P, P, P, P, P, sz, P]
    lib.jattn_bwd_rope.restype = i32
    lib.jattn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.jattn_bwd_noalloc.restype = i32
    lib.jattn_mxfp8_quantize.argtypes = [P, P, i32, P, P]
    lib.jattn_mxfp8_quantize.restype = i32
    lib.jattn_test_fwd_stall.argtypes = [P, P, P, P, P, P, ctypes.c_uint64, P]
    lib.jattn_test_fwd_stall.restype = i32
    lib.jattn_step_host.argtypes = [P, P, P, i32, P, P, P, P, P, P, P, P, P, P, P]
    lib.jattn_step_host.restype = i32
    lib.jattn_step_host_join.argtypes = [P, P]
    lib.jattn_step_host_join.restype = i32
    lib.jattn_check_device_status.argtypes = [P, P]
    lib.jattn_plan_set_events.argtypes = [P, P, i32]
    lib.jattn_plan_set_events.restype = i32
    lib.jattn_plan_launch_count.argtypes = [P]
    lib.jattn_plan_launch_count.restype = i64
    lib.jattn_last_cuda_error.argtypes = []
    lib.jattn_last_cuda_error.restype = ctypes.c_char_p
    lib.jattn_shard.argtypes = [P, P, i32, i32, P]
    lib.jattn_shard.restype = i32
    lib.jattn_status_str.argtypes = [i32]
    lib.jattn_status_str.restype = ctypes.c_char_p
    for f in ("jattn_plan_create", "jattn_plan_update", "jattn_plan_tiles", "jattn_fwd", "jattn_bwd",
              "jattn_check_device_status"):
        getattr(lib, f).restype = i32
    _lib = lib
    return lib


def shard(q_offsets, kv_offsets, world: int) -> np.ndarray:
    """Rank of every sequence (int32 [B]) for `world` data-parallel ranks (jattn_shard)."""
    qo, ko = _i32(q_offsets), _i32(kv_offsets)
    B = len(qo) - 1
    out = np.zeros(max(B, 0), dtype=np.int32)
    _check(load().jattn_shard(qo.ctypes.data_as(ctypes.c_void_p), ko.ctypes.data_as(ctypes.c_void_p), B, int(world),
                              out.ctypes.data_as(ctypes.c_void_p)), "jattn_shard")
    return out


def status_str(code: int) -> str:
    return load().jattn_status_str(int(code)).decode()


def _check(code: int, what: str):
    if code != OK:
        raise JattnError(code, what)


def _i32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Plan:
    """A planned jagged batch (tile lists + schedule) for one (H, D, mode)."""

    def __init__(self, q_off, kv_off, H: int, D: int, act: int = SOFTMAX, block: int = 0, scale: float = 0.0,
                 bias_buckets: int = 0, dtype: str = "bf16", device: int = 0, window: int = 0,
                 broadcast_q: bool = False, mxfp8: bool = False):
        """broadcast_q: every sequence's queries are the rows of one shared Q
        [n, H, D] (n = each sequence's Lq); bwd then returns dq [n, H, D], the
        sum over the sequences.  mxfp8: MXFP8 attention (jattn_mode.mxfp8)."""
        lib = load()
        qo, ko = _i32(q_off), _i32(kv_off)
        self.H, self.D, self.act, self.block, self.bias_buckets = H, D, act, block, bias_buckets
        self.window = window
        self.dtype = dtype
        self.device = device
        self.broadcast_q = bool(broadcast_q)
        self.mxfp8 = bool(mxfp8)
        self.mode = Mode(act, block, float(scale), bias_buckets, FP32 if dtype == "fp32" else BF16, window,
                         1 if broadcast_q else 0, 1 if mxfp8 else 0)
        self._h = ctypes.c_void_p()
        _check(lib.jattn_plan_create(qo.ctypes.data_as(ctypes.c_void_p), ko.ctypes.data_as(ctypes.c_void_p),
                                     len(qo) - 1, H, D, ctypes.byref(self.mode), device, ctypes.byref(self._h)),
               "jattn_plan_create")
        self.Tq, self.Tk = int(qo[-1]), int(ko[-1])
        self.q_rows = int(qo[1] - qo[0]) if broadcast_q else self.Tq

    def update(self, q_off, kv_off, stream=None):
        qo, ko = _i32(q_off), _i32(kv_off)
        st = _stream(stream) if self.device >= 0 else None
        _check(load().jattn_plan_update(self._h, qo.ctypes.data_as(ctypes.c_void_p),
                                        ko.ctypes.data_as(ctypes.c_void_p), len(qo) - 1, st), "jattn_plan_update")
        self.Tq, self.Tk = int(qo[-1]), int(ko[-1])
        self.q_rows = int(qo[1] - qo[0]) if self.broadcast_q else self.Tq

    def update_device(self, q_off, kv_off, Tq: int, Tk: int, stream=None):
        """Re-plan on the device (jattn_plan_update_device): q_off, kv_off are
        int32 CUDA tensors [B+1]; Tq, Tk their last entries."""
        if q_off.dtype != torch.int32 or kv_off.dtype != torch.int32 or not q_off.is_cuda or not kv_off.is_cuda:
            raise ValueError("update_device: int32 CUDA offset tensors expected")
        if q_off.numel() != kv_off.numel():
            raise ValueError("update_device: offsets of different lengths")
        _check(load().jattn_plan_update_device(self._h, q_off.data_ptr(), kv_off.data_ptr(), q_off.numel() - 1,
                                               int(Tq), int(Tk), _stream(stream)), "jattn_plan_update_device")
        self.Tq, self.Tk = int(Tq), int(Tk)
        self.q_rows = self.Tq // (q_off.numel() - 1) if self.broadcast_q else self.Tq

    def tiles(self, which: int = TILES_Q):
        """(tiles int32 [n, 6] in schedule order, cta_begin int32 [n_ctas + 1])."""
        tp = ctypes.POINTER(TileRec)()
        n = ctypes.c_int64()
        cp = ctypes.POINTER(ctypes.c_int32)()
        nc = ctypes.c_int32()
        _check(load().jattn_plan_tiles(self._h, which, ctypes.byref(tp), ctypes.byref(n), ctypes.byref(cp),
                                       ctypes.byref(nc)), "jattn_plan_tiles")
        if n.value:
            arr = np.ctypeslib.as_array(ctypes.cast(tp, ctypes.POINTER(ctypes.c_int32)), shape=(n.value * 6,))
            tiles = arr.reshape(-1, 6).copy()
        else:
            tiles = np.zeros((0, 6), np.int32)
        cta = np.ctypeslib.as_array(cp, shape=(nc.value + 1,)).copy()
        return tiles, cta

    @property
    def fwd_workspace_bytes(self) -> int:
        return int(load().jattn_fwd_workspace_bytes(self._h))

    @property
    def bwd_workspace_bytes(self) -> int:
        return int(load().jattn_bwd_workspace_bytes(self._h))

    @property
    def bwd_workspace_bytes_min(self) -> int:
        return int(load().jattn_bwd_workspace_bytes_min(self._h))

    def _tdtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def _ws(self, nbytes, ws):
        if nbytes == 0:
            return None
        if ws is None or ws.numel() * ws.element_size() < nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda:%d" % self.device)
        return ws

    def fwd(self, q, k, v, bias=None, out=None, lse=None, want_lse=True, workspace=None, stream=None, rope=None):
        """Forward.  Returns (out, lse or None).  rope = (cos, sin): rotary
        position embedding of Q and K (jattn_fwd_rope)."""
        if out is None:
            out = torch.empty(self.Tq, self.H, self.D, dtype=self._tdtype(), device=q.device)
        if lse is None and want_lse and self.act == SOFTMAX:
            lse = torch.empty(self.H, self.Tq, dtype=torch.float32, device=q.device)
        ws = self._ws(self.fwd_workspace_bytes, workspace)
        nbytes = 0 if ws is None else ws.numel() * ws.element_size()
        if rope is not None:
            r = _rope(rope)
            _check(load().jattn_fwd_rope(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(bias), ctypes.byref(r), _ptr(out),
                                         _ptr(lse), _ptr(ws), nbytes, _stream(stream)), "jattn_fwd_rope")
            return out, lse
        _check(load().jattn_fwd(self._h, _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(out), _ptr(lse), _ptr(ws),
                                nbytes, _stream(stream)), "jattn_fwd")
        return out, lse

    def bwd(self, dout, q, k, v, out, lse=None, bias=None, dq=None, dk=None, dv=None, dbias=None, workspace=None,
            stream=None, rope=None):
        """Backward.  Returns (dq, dk, dv).  rope = (cos, sin) as in fwd: dq and
        dk are then the gradients of the unrotated Q and K (jattn_bwd_rope)."""
        dt = self._tdtype()
        dq = torch.empty(self.q_rows, self.H, self.D, dtype=dt, device=q.device) if dq is None else dq
        dk = torch.empty(self.Tk, self.H, self.D, dtype=dt, device=q.device) if dk is None else dk
        dv = torch.empty(self.Tk, self.H, self.D, dtype=dt, device=q.device) if dv is None else dv
        # a given workspace of at least the minimum is passed as it is (the library
        # takes its fastest path that fits); otherwise the full size is allocated
        if workspace is not None and workspace.numel() * workspace.element_size() >= self.bwd_workspace_bytes_min:
            ws = workspace
        else:
            ws = self._ws(self.bwd_workspace_bytes, None)
        nbytes = 0 if ws is None else ws.numel() * ws.element_size()
        if rope is not None:
            r = _rope(rope)
            _check(load().jattn_bwd_rope(self._h, _ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), ctypes.byref(r),
                                         _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias), _ptr(ws),
                                         nbytes, _stream(stream)), "jattn_bwd_rope")
            return dq, dk, dv
        _check(load().jattn_bwd(self._h, _ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(out), _ptr(lse),
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias), _ptr(ws), nbytes, _stream(stream)),
               "jattn_bwd")
        return dq, dk, dv

    def mxfp8_quantize(self, x, which: int = TILES_Q, out=None, stream=None):
        """x [T, H, D] bf16 (device) -> the values of its MXFP8 quantisation, as
        bf16 [T, H, D] (jattn_mxfp8_quantize; which: TILES_Q = query offsets,
        TILES_KV = key offsets)."""
        out = torch.empty_like(x) if out is None else out
        _check(load().jattn_mxfp8_quantize(self._h, _ptr(x), which, _ptr(out), _stream(stream)),
               "jattn_mxfp8_quantize")
        return out

    def bwd_noalloc(self, dout, q, k, v, out, lse=None, bias=None, dq=None, dk=None, dv=None, dbias=None,
                    stream=None):
        """Backward with the library's fixed device scratch instead of a workspace.
        Returns (dq, dk, dv); the output tensors are allocated here unless given."""
        dt = self._tdtype()
        dq = torch.empty(self.q_rows, self.H, self.D, dtype=dt, device=q.device) if dq is None else dq
        dk = torch.empty(self.Tk, self.H, self.D, dtype=dt, device=q.device) if dk is None else dk
        dv = torch.empty(self.Tk, self.H, self.D, dtype=dt, device=q.device) if dv is None else dv
        _check(load().jattn_bwd_noalloc(self._h, _ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(out),
                                        _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias), _stream(stream)),
               "jattn_bwd_noalloc")
        return dq, dk, dv

    def step_host(self, q_off, kv_off, q, k, v, dout, out, dq, dk, dv, bias=None, lse=None, stream=None):
        """One training step on host tensors (pinned memory overlaps the copies): re-plan
        for the batch, upload q, k, v, dout (bias), forward, backward, download into
        out, dq, dk, dv (lse).  Asynchronous and pipelined with the previous call; the
        host tensors must stay untouched until step_host_join's wait has passed."""
        qo, ko = _i32(q_off), _i32(kv_off)
        Tq, Tk = int(qo[-1]), int(ko[-1])
        nq, nk = Tq * self.H * self.D, Tk * self.H * self.D
        for name, t, n in (("q", q, nq), ("k", k, nk), ("v", v, nk), ("dout", dout, nq), ("out", out, nq),
                           ("dq", dq, nq), ("dk", dk, nk), ("dv", dv, nk)):
            if t.is_cuda or not t.is_contiguous() or t.numel() != n or t.dtype != self._tdtype():
                raise ValueError("step_host: %s must be a contiguous %s host tensor of %d elements"
                                 % (name, self._tdtype(), n))
        for name, t, n in (("bias", bias, self.H * self.bias_buckets), ("lse", lse, self.H * Tq)):
            if t is not None and (t.is_cuda or not t.is_contiguous() or t.numel() != n or t.dtype != torch.float32):
                raise ValueError("step_host: %s must be a contiguous float32 host tensor of %d elements" % (name, n))
        _check(load().jattn_step_host(self._h, qo.ctypes.data_as(ctypes.c_void_p), ko.ctypes.data_as(ctypes.c_void_p),
                                      len(qo) - 1, _ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(bias), _ptr(out),
                                      _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)), "jattn_step_host")
        self.Tq, self.Tk = Tq, Tk

    def step_host_join(self, stream=None):
        """Makes `stream` wait for every step_host call issued so far."""
        _check(load().jattn_step_host_join(self._h, _stream(stream)), "jattn_step_host_join")

    def set_events(self, events):
        """Record torch.cuda.Event objects around each kernel of later fwd / bwd calls (None: off)."""
        if not events:
            _check(load().jattn_plan_set_events(self._h, None, 0), "jattn_plan_set_events")
            self._events = None
            return
        self._events = list(events)  # keep the handles alive
        for e in self._events:
            if not e.cuda_event:  # torch creates the CUDA event on its first record
                e.record()
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in self._events])
        _check(load().jattn_plan_set_events(self._h, arr, len(events)), "jattn_plan_set_events")

    @property
    def launch_count(self) -> int:
        return int(load().jattn_plan_launch_count(self._h))

    def check_status(self, stream=None) -> int:
        return int(load().jattn_check_device_status(self._h, _stream(stream)))

    def close(self):
        if self._h:
            load().jattn_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
