"""Python front end of the fp64 CPU oracle -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It compiles ``jattn_oracle.c`` with gcc
(no CUDA, nothing shared with the library) and calls it through ctypes.

Inputs are the exact values handed to the library: bf16 tensors are widened to
float64 bit-exactly, float32 tensors are widened unrounded.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "jattn_oracle.c")
_LIB = os.path.join(_HERE, "libjattn_oracle.so")
_lib = None

SOFTMAX, SILU, GELU_TANH = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source (plain gcc, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", _SRC,
                               "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i, d = ctypes.c_int, ctypes.c_double
        lib.jattn_oracle_fwd.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, i, d, P, P, i]
        lib.jattn_oracle_fwd.restype = i
        lib.jattn_oracle_bwd.argtypes = [i, i, i, i, i, i, P, P, P, P, P, P, i, d, P, P, P, P, P, i]
        lib.jattn_oracle_bwd.restype = i
        lib.jattn_oracle_act.argtypes = [i, d]
        lib.jattn_oracle_act.restype = d
        lib.jattn_oracle_act_grad.argtypes = [i, d]
        lib.jattn_oracle_act_grad.restype = d
        _lib = lib
    return _lib


def default_threads() -> int:
    return os.cpu_count() or 1


def _f64(t) -> np.ndarray:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        t = t.detach().to("cpu")
        return np.ascontiguousarray(t.to(torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def rope_rotate(x, offsets, cos, sin, transpose=False) -> np.ndarray:
    """Rotary position embedding of a jagged [T, H, D] tensor, in float64.

    "Training GEM at LLM scale", section "BlockAttention": RoPE is applied to
    the queries and keys before the attention, and its backward is fused into
    the attention's epilogue.  The pages give no formula; this is the standard
    rotary embedding with the half-split pairing.  Row t of sequence b sits at
    local position p = t - offsets[b].  Each feature pair (d, d + D/2), d < D/2,
    is turned by the angle whose cosine and sine are cos[p, d] and sin[p, d]:
        y[d]       = x[d] cos - x[d + D/2] sin
        y[d + D/2] = x[d + D/2] cos + x[d] sin
    transpose=True applies the transposed rotation.  That maps a gradient with
    respect to the rotated rows back to the unrotated ones.
    """
    x = _f64(x)
    cos, sin = _f64(cos), _f64(sin)
    off = np.asarray(offsets, dtype=np.int64)
    T, _, D = x.shape
    half = D // 2
    pos = np.zeros(T, dtype=np.int64)
    for b in range(len(off) - 1):
        pos[off[b]:off[b + 1]] = np.arange(off[b + 1] - off[b])
    c = cos[pos][:, None, :]  # [T, 1, D/2]
    s = sin[pos][:, None, :]
    if transpose:
        s = -s
    a, b_ = x[..., :half], x[..., half:]
    y = np.concatenate([a * c - b_ * s, b_ * c + a * s], axis=-1)
    return y


def forward(q_off, kv_off, q, k, v, bias=None, scale=None, act=SOFTMAX, block=0, nthreads=None, window=0,
            rope=None):
    """Returns (out [Tq,H,D] float64, lse [H,Tq] float64 or None).
    window W > 0: row i attends only keys with |i - j| < W (sliding window).
    rope = (cos, sin), tables [P, D/2]: Q and K are rotated first (rope_rotate),
    exactly, in float64."""
    lib = _load()
    qo, ko = _i32(q_off), _i32(kv_off)
    q, k, v, bias = _f64(q), _f64(k), _f64(v), _f64(bias)
    if rope is not None:
        q = rope_rotate(q, qo, rope[0], rope[1])
        k = rope_rotate(k, ko, rope[0], rope[1])
    Tq, H, D = q.shape
    B = len(qo) - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((Tq, H, D), dtype=np.float64)
    lse = np.zeros((H, Tq), dtype=np.float64) if act == SOFTMAX else None
    nb = 0 if bias is None else bias.shape[1]
    rc = lib.jattn_oracle_fwd(act, block, int(window), B, H, D, _ptr(qo), _ptr(ko), _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                              nb, float(scale), _ptr(out), _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle forward rejected its input (code %d)" % rc)
    return out, lse


def backward(q_off, kv_off, q, k, v, dout, bias=None, scale=None, act=SOFTMAX, block=0, nthreads=None, window=0,
             rope=None):
    """Returns (dq, dk, dv, dbias or None), all float64 (window and rope as in
    forward; with rope, dq and dk are the gradients of the unrotated Q and K)."""
    lib = _load()
    qo, ko = _i32(q_off), _i32(kv_off)
    q, k, v, dout, bias = _f64(q), _f64(k), _f64(v), _f64(dout), _f64(bias)
    if rope is not None:
        q = rope_rotate(q, qo, rope[0], rope[1])
        k = rope_rotate(k, ko, rope[0], rope[1])
    Tq, H, D = q.shape
    Tk = k.shape[0]
    B = len(qo) - 1
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.zeros((Tq, H, D), dtype=np.float64)
    dk = np.zeros((Tk, H, D), dtype=np.float64)
    dv = np.zeros((Tk, H, D), dtype=np.float64)
    nb = 0 if bias is None else bias.shape[1]
    dbias = np.zeros((H, nb), dtype=np.float64) if bias is not None else None
    rc = lib.jattn_oracle_bwd(act, block, int(window), B, H, D, _ptr(qo), _ptr(ko), _ptr(q), _ptr(k), _ptr(v), _ptr(bias),
                              nb, float(scale), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias),
                              nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle backward rejected its input (code %d)" % rc)
    if rope is not None:
        dq = rope_rotate(dq, qo, rope[0], rope[1], transpose=True)
        dk = rope_rotate(dk, ko, rope[0], rope[1], transpose=True)
    return dq, dk, dv, dbias


def act(kind: int, x: float) -> float:
    return _load().jattn_oracle_act(kind, float(x))


def act_grad(kind: int, x: float) -> float:
    return _load().jattn_oracle_act_grad(kind, float(x))


def sub_batch(q_off, kv_off, seqs, *tensors_q, tensors_kv=()):
    """Cut sequences ``seqs`` out of a jagged batch (for sampled checks).

    Returns (q_off', kv_off', [q-side tensors...], [kv-side tensors...]) with the
    chosen sequences packed in the given order.  Pure indexing, no arithmetic.
    """
    qo = np.asarray(q_off, dtype=np.int64)
    ko = np.asarray(kv_off, dtype=np.int64)
    qidx = np.concatenate([np.arange(qo[s], qo[s + 1]) for s in seqs] or [np.zeros(0, np.int64)])
    kidx = np.concatenate([np.arange(ko[s], ko[s + 1]) for s in seqs] or [np.zeros(0, np.int64)])
    nqo = np.zeros(len(seqs) + 1, np.int64)
    nko = np.zeros(len(seqs) + 1, np.int64)
    nqo[1:] = np.cumsum([qo[s + 1] - qo[s] for s in seqs])
    nko[1:] = np.cumsum([ko[s + 1] - ko[s] for s in seqs])
    qi = torch.from_numpy(qidx)
    ki = torch.from_numpy(kidx)
    return (nqo.astype(np.int32), nko.astype(np.int32), [t[qi] for t in tensors_q],
            [t[ki] for t in tensors_kv], qidx, kidx)
