"""Seeded synthetic jagged-attention workloads.

This module only draws numbers: sequence lengths, offsets and i.i.d. Gaussian
tensors.  It holds none of the attention arithmetic, so both the CUDA path and
the CPU oracle can take their inputs from it without sharing any computation.

The five workloads stand in for the private GEM production traffic described in
"Training GEM at LLM scale" (Meta engineering post, section "Jagged Sequence
Flash Attention"): long jagged self-attention over user history, cross-attention
with long queries and short keys/values, pooled multi-head attention (GDPA) with
short queries and long keys/values, and 64-token BlockAttention over very long
histories.

Recipe (fixed so every run sees the same batch):
  * lengths: ``numpy.random.default_rng(workload_id)``; lognormal lengths are
    ``clip(rint(lognormal(mu, sigma, B)), lo, hi)``; uniform lengths are
    ``integers(lo, hi + 1, B)``; the cross-attention workload draws Q lengths
    first and K/V lengths second from the same generator.
  * tensors: ``torch.Generator().manual_seed(100 + workload_id)`` on the CPU,
    ``randn`` in float32 in the order q, k, v, bias table, dO, then cast to
    bfloat16 (the tiny workload stays float32).  The bias table is N(0, 0.1)
    (standard deviation 0.1).  The pooled-attention workload draws its 32 query
    rows once and repeats them for every sample.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# activation codes shared with the C ABI (jattn_act)
SOFTMAX, SILU, GELU_TANH = 0, 1, 2
ACT_NAMES = {SOFTMAX: "softmax", SILU: "silu", GELU_TANH: "gelu_tanh"}


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int                 # 1..5
    name: str
    B: int
    H: int
    D: int
    dtype: str               # "fp32" or "bf16"
    act: int                 # SOFTMAX / SILU / GELU_TANH
    block: int               # 0 = full attention, 64 = BlockAttention
    bias_buckets: int        # 0 = no bias, else the table width (64)
    q_rows_shared: int = 0   # >0: that many query rows shared by every sample
    window: int = 0          # >0: sliding window, keys with |i - j| < window only


WORKLOADS = {
    1: Workload(1, "tiny_self_fp32", B=4, H=2, D=32, dtype="fp32", act=SOFTMAX, block=0, bias_buckets=0),
    2: Workload(2, "self_relpos_bias", B=256, H=4, D=128, dtype="bf16", act=SOFTMAX, block=0, bias_buckets=64),
    3: Workload(3, "cross_longq_shortkv", B=512, H=4, D=128, dtype="bf16", act=SOFTMAX, block=0, bias_buckets=0),
    4: Workload(4, "gdpa_pma_silu", B=256, H=4, D=128, dtype="bf16", act=SILU, block=0, bias_buckets=0,
                q_rows_shared=32),
    5: Workload(5, "block64_long_history", B=64, H=8, D=64, dtype="bf16", act=SOFTMAX, block=64, bias_buckets=0),
}


def lengths(wid: int, B: Optional[int] = None) -> tuple[np.ndarray, np.ndarray]:
    """Per-sample (Lq, Lk) for workload ``wid`` (int64 arrays)."""
    w = WORKLOADS[wid]
    B = w.B if B is None else B
    rng = np.random.default_rng(wid)

    def lognormal(median, sigma, lo, hi):
        return np.clip(np.rint(rng.lognormal(math.log(median), sigma, B)), lo, hi).astype(np.int64)

    if wid == 1:
        lq = rng.integers(1, 65, B).astype(np.int64)
        return lq, lq.copy()
    if wid == 2:
        lq = lognormal(200, 0.8, 16, 1000)
        return lq, lq.copy()
    if wid == 3:
        lq = lognormal(300, 0.9, 32, 2000)
        lk = rng.integers(8, 65, B).astype(np.int64)
        return lq, lk
    if wid == 4:
        lk = lognormal(1000, 1.0, 200, 8000)
        return np.full(B, 32, dtype=np.int64), lk
    if wid == 5:
        lq = lognormal(4000, 0.7, 512, 16384)
        return lq, lq.copy()
    raise KeyError(wid)


def offsets(lens: np.ndarray) -> np.ndarray:
    """Exclusive prefix sum, int32, length B+1."""
    off = np.zeros(len(lens) + 1, dtype=np.int64)
    np.cumsum(lens, out=off[1:])
    assert off[-1] < 2**31
    return off.astype(np.int32)


@dataclasses.dataclass
class Batch:
    w: Workload
    act: int
    q_off: np.ndarray        # int32 [B+1]
    kv_off: np.ndarray       # int32 [B+1]
    q: torch.Tensor          # [Tq, H, D] (CPU), float32 or bfloat16
    k: torch.Tensor          # [Tk, H, D]
    v: torch.Tensor          # [Tk, H, D]
    bias: Optional[torch.Tensor]  # [H, NB] float32 or None
    dout: torch.Tensor       # [Tq, H, D]
    scale: float

    @property
    def B(self):
        return len(self.q_off) - 1

    @property
    def Tq(self):
        return int(self.q_off[-1])

    @property
    def Tk(self):
        return int(self.kv_off[-1])


def make_batch(wid: int, act: Optional[int] = None, B: Optional[int] = None,
               lens: Optional[tuple[np.ndarray, np.ndarray]] = None) -> Batch:
    """Draw the full synthetic batch of workload ``wid`` on the CPU.

    ``act`` overrides the score activation (the pooled-attention workload is
    run once with SiLU and once with tanh-GELU).  ``B`` truncates the batch to
    its first ``B`` samples (same seeds); ``lens`` replaces the drawn lengths
    with explicit (Lq, Lk) arrays, which tests use for edge cases.
    """
    w = WORKLOADS[wid]
    if lens is None:
        lq, lk = lengths(wid)
        if B is not None:
            lq, lk = lq[:B], lk[:B]
    else:
        lq, lk = (np.asarray(x, dtype=np.int64) for x in lens)
    qo, ko = offsets(lq), offsets(lk)
    Tq, Tk = int(qo[-1]), int(ko[-1])
    H, D = w.H, w.D
    g = torch.Generator().manual_seed(100 + wid)
    if w.q_rows_shared:
        assert np.all(lq == w.q_rows_shared)
        q_rows = torch.randn(w.q_rows_shared, H, D, generator=g)
        q = q_rows.repeat(len(lq), 1, 1)
    else:
        q = torch.randn(Tq, H, D, generator=g)
    k = torch.randn(Tk, H, D, generator=g)
    v = torch.randn(Tk, H, D, generator=g)
    bias = None
    if w.bias_buckets:
        bias = 0.1 * torch.randn(H, w.bias_buckets, generator=g)
    dout = torch.randn(Tq, H, D, generator=g)
    if w.dtype == "bf16":
        q, k, v, dout = (t.to(torch.bfloat16) for t in (q, k, v, dout))
    return Batch(w=w, act=w.act if act is None else act, q_off=qo, kv_off=ko, q=q, k=k, v=v,
                 bias=bias, dout=dout, scale=1.0 / math.sqrt(D))


def random_batch(seed: int, lq, lk, H: int, D: int, dtype=torch.bfloat16, bias_buckets: int = 0,
                 std: float = 1.0) -> dict:
    """Small seeded batch with explicit lengths (edge cases and tiny tests)."""
    lq = np.asarray(lq, dtype=np.int64)
    lk = np.asarray(lk, dtype=np.int64)
    qo, ko = offsets(lq), offsets(lk)
    g = torch.Generator().manual_seed(seed)
    Tq, Tk = int(qo[-1]), int(ko[-1])
    q = std * torch.randn(Tq, H, D, generator=g)
    k = std * torch.randn(Tk, H, D, generator=g)
    v = torch.randn(Tk, H, D, generator=g)
    bias = 0.1 * torch.randn(H, bias_buckets, generator=g) if bias_buckets else None
    dout = torch.randn(Tq, H, D, generator=g)
    if dtype != torch.float32:
        q, k, v, dout = (t.to(dtype) for t in (q, k, v, dout))
    return dict(q_off=qo, kv_off=ko, q=q, k=k, v=v, bias=bias, dout=dout, scale=1.0 / math.sqrt(D))


def rope_table(P: int, D: int, kind: str = "standard", base: float = 10000.0, seed: int = 0):
    """Rotary-embedding tables (cos, sin), float32 [P, D/2], for positions 0..P-1.

    kind "standard": angle p * base^(-2d/D) for feature pair d (the usual
    frequency ladder); "random": seeded uniform angles in [-pi, pi), so that no
    structure of the ladder can hide an indexing slip; "identity": angle 0.
    """
    half = D // 2
    if kind == "standard":
        inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / D)
        phi = np.arange(P, dtype=np.float64)[:, None] * inv[None, :]
    elif kind == "random":
        phi = np.random.default_rng(seed).uniform(-np.pi, np.pi, size=(P, half))
    elif kind == "identity":
        phi = np.zeros((P, half))
    else:
        raise ValueError(kind)
    return (torch.from_numpy(np.cos(phi).astype(np.float32)), torch.from_numpy(np.sin(phi).astype(np.float32)))


# ---------------------------------------------------------------------------
# Work accounting (valid tokens only; padding and recompute are not counted)
# ---------------------------------------------------------------------------

def valid_pairs(q_off: np.ndarray, kv_off: np.ndarray, block: int = 0, window: int = 0) -> int:
    lq = np.diff(np.asarray(q_off).astype(np.int64))
    lk = np.diff(np.asarray(kv_off).astype(np.int64))
    if window:
        total = 0
        for a, b in zip(lq.tolist(), lk.tolist()):
            i = np.arange(a, dtype=np.int64)
            total += int(np.clip(np.minimum(b, i + window) - np.maximum(0, i - window + 1), 0, None).sum())
        return total
    if block:
        full, rem = lq // block, lq % block
        return int((full * block * block + rem * rem).sum())
    return int((lq * lk).sum())


def flops(q_off, kv_off, H: int, D: int, block: int = 0, window: int = 0) -> tuple[float, float]:
    """(forward, backward) FLOPs: 4*D*H*pairs and 10*D*H*pairs."""
    p = valid_pairs(q_off, kv_off, block, window)
    return 4.0 * D * H * p, 10.0 * D * H * p


def hbm_bytes(q_off, kv_off, H: int, D: int, act: int, block: int, elem_bytes: int = 2) -> tuple[float, float]:
    """(forward, backward) algorithmic HBM bytes: each tensor crosses HBM once."""
    Tq, Tk = int(q_off[-1]), int(kv_off[-1])
    e = H * D * elem_bytes
    if block:
        return 4.0 * Tq * e, 8.0 * Tq * e
    if act == SOFTMAX:
        return (2 * Tq + 2 * Tk) * e + 4.0 * H * Tq, (4 * Tq + 4 * Tk) * e + 4.0 * H * Tq
    return (2 * Tq + 2 * Tk) * e, (3 * Tq + 4 * Tk) * e
