"""MXFP8 attention reference (forward and backward) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` may import this module.  Plain numpy in float64; nothing is
shared with the CUDA path.

"Training GEM at LLM scale", section "Low Precision Flash Attention": attention
with block-scaled MXFP8 tensor-core products in the forward and backward passes.
Q, K and V are quantised with one scale per 32 x 32 block, so a tensor and its
transpose have the same quantised values.  The softmax output P is quantised
online in the softmax warps, with the scale derived from bits, not from
log2 / round / clamp.

The pages do not give the element format or the scale rule.  The format read
here is the one MXFP8 names, the microscaling (MX) format.  Each block of
values shares one power-of-two scale 2^e (an 8-bit exponent, E8M0), and each
element is an FP8 E4M3 number, defined as follows:
  - 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
  - normals are (1 + m/8) * 2^(E-7) for E = 1..15;
  - subnormals are (m/8) * 2^-6;
  - there is no infinity; S.1111.111 is NaN, so the largest finite value is
    1.75 * 2^8 = 448.
The shared exponent of a block is floor(log2(amax)) - 8, where 8 is the
exponent of E4M3's largest normal, clamped to the E8M0 range [-127, 127].
Each element x / 2^e is then rounded to the nearest E4M3 value, ties to even,
and values beyond 448 are saturated to +-448.

The readings of the pages taken here:
  * Q, K, V: blocks of 32 local rows of one sequence x 32 features of one head.
    Blocks start at the sequence's first row; the last block of a sequence is
    partial.
  * P: quantised per query row in groups of 32 keys (the K dimension of the
    P V product), after exp(s - m) with the row max m.
  * The row sum l is accumulated from the unquantised P, as the softmax warps
    hold it in float32 before the conversion.
  * O = (P_q V_q) / l, with lse = m + ln l.
  * Backward: dO is quantised like Q (32 x 32 blocks).  P and dS each feed
    two products with different K dimensions (P: dV = P^T dO; dS: dQ = dS K
    and dK = dS^T Q), so in the backward they are quantised in 32 x 32 blocks,
    which serve a matrix and its transpose alike.  The backward P is exp(s - lse)
    (normalised), and Delta_i = <dO_i, O_i> uses the unquantised dO and O (the
    Delta pre-pass).  dS = P (dP - Delta) uses the unquantised P and
    dP = dO_q V_q^T; then dV = P_q^T dO_q, dQ = scale dS_q K_q,
    dK = scale dS_q^T Q_q.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal, 448 = 1.75 * 2^8
E8M0_MIN, E8M0_MAX = -127, 127


def e4m3_values() -> np.ndarray:
    """All finite E4M3 values, ascending, decoded from the 256 bit patterns."""
    vals = set()
    for code in range(256):
        s = (code >> 7) & 1
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:  # NaN
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals.add(-mag if s else mag)
    return np.array(sorted(vals), dtype=np.float64)


_GRID = e4m3_values()
_POS = _GRID[_GRID >= 0.0]  # 0 and the positive values, ascending


def quantize_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value, ties to the even code (mantissa LSB 0); saturating."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    i = np.searchsorted(_POS, a, side="left")  # first grid value >= a
    i = np.clip(i, 1, len(_POS) - 1)
    lo, hi = _POS[i - 1], _POS[i]
    take_hi = (a - lo) > (hi - a)
    tie = (a - lo) == (hi - a)
    # on a tie the even code wins: consecutive positive values have consecutive
    # codes, so the even one is the one at an even index of _POS (code = index)
    take_hi = np.where(tie, (i % 2) == 0, take_hi)
    q = np.where(take_hi, hi, lo)
    q = np.where(a == lo, lo, q)
    return np.where(x < 0, -q, q)


def block_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared E8M0 exponent of a block with largest magnitude amax."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - E4M3_EMAX
    e = np.where(amax > 0, e, E8M0_MIN)
    return np.clip(e, E8M0_MIN, E8M0_MAX)


def qdq_block(x: np.ndarray) -> np.ndarray:
    """Quantise one block (any shape) to MXFP8 and return the values it stands for."""
    x = np.asarray(x, dtype=np.float64)
    scale = 2.0 ** block_exponent(np.max(np.abs(x)) if x.size else 0.0)
    return quantize_e4m3(x / scale) * scale


def qdq_rows_cols(x: np.ndarray, rb: int, cb: int) -> np.ndarray:
    """Quantise a 2-D array in blocks of rb rows x cb columns (partial blocks at the ends)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    R, Cn = x.shape
    for r in range(0, R, rb):
        for c in range(0, Cn, cb):
            out[r:r + rb, c:c + cb] = qdq_block(x[r:r + rb, c:c + cb])
    return out


def qdq_jagged(x, offsets) -> np.ndarray:
    """[T, H, D]: per sequence and head, 32 local rows x 32 features per block."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    off = np.asarray(offsets, dtype=np.int64)
    for b in range(len(off) - 1):
        r0, r1 = off[b], off[b + 1]
        for h in range(x.shape[1]):
            out[r0:r1, h] = qdq_rows_cols(x[r0:r1, h], 32, 32)
    return out


def forward(q_off, kv_off, q, k, v, scale=None):
    """MXFP8 softmax attention forward: returns (out [Tq,H,D], lse [H,Tq]) in float64."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    Tq, H, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    qq, kq, vq = qdq_jagged(q, q_off), qdq_jagged(k, kv_off), qdq_jagged(v, kv_off)
    out = np.zeros((Tq, H, D))
    lse = np.full((H, Tq), -np.inf)
    qo = np.asarray(q_off, dtype=np.int64)
    ko = np.asarray(kv_off, dtype=np.int64)
    for b in range(len(qo) - 1):
        q0, q1, k0, k1 = qo[b], qo[b + 1], ko[b], ko[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            s = scale * qq[q0:q1, h] @ kq[k0:k1, h].T
            m = s.max(axis=1, keepdims=True)
            p = np.exp(s - m)
            l = p.sum(axis=1, keepdims=True)
            pq = qdq_rows_cols(p, 1, 32)
            out[q0:q1, h] = (pq @ vq[k0:k1, h]) / l
            lse[h, q0:q1] = (m + np.log(l))[:, 0]
    return out, lse


def backward(q_off, kv_off, q, k, v, dout, scale=None):
    """MXFP8 softmax attention backward: returns (dq, dk, dv) in float64."""
    q, k, v, dout = (np.asarray(t, dtype=np.float64) for t in (q, k, v, dout))
    Tq, H, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out, lse = forward(q_off, kv_off, q, k, v, scale)
    qq, kq, vq = qdq_jagged(q, q_off), qdq_jagged(k, kv_off), qdq_jagged(v, kv_off)
    dq_ = qdq_jagged(dout, q_off)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    qo = np.asarray(q_off, dtype=np.int64)
    ko = np.asarray(kv_off, dtype=np.int64)
    for b in range(len(qo) - 1):
        q0, q1, k0, k1 = qo[b], qo[b + 1], ko[b], ko[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            s = scale * qq[q0:q1, h] @ kq[k0:k1, h].T
            p = np.exp(s - lse[h, q0:q1, None])
            delta = np.sum(dout[q0:q1, h] * out[q0:q1, h], axis=1, keepdims=True)
            dp = dq_[q0:q1, h] @ vq[k0:k1, h].T
            ds = p * (dp - delta)
            pq, dsq = qdq_rows_cols(p, 32, 32), qdq_rows_cols(ds, 32, 32)
            dv[k0:k1, h] = pq.T @ dq_[q0:q1, h]
            dq[q0:q1, h] = scale * dsq @ kq[k0:k1, h]
            dk[k0:k1, h] = scale * dsq.T @ qq[q0:q1, h]
    return dq, dk, dv
