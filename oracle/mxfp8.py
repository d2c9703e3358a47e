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
    P V product).  "Online" in the softmax warps means against a running row
    max; read here as a max kept as an integer M in log2 units (an integer no
    smaller than any score of the row in log2 units): P = 2^(s log2 e - M).
    Every rescale of an online softmax is then a power of two, and a
    power-of-two factor moves the block exponent and leaves the quantised
    mantissas as they are, so the result does not depend on the order of the
    key blocks or on when the max was raised; M = ceil(max_j s_ij log2 e)
    gives it in one step here.
  * The row sum l is accumulated from the unquantised P, as the softmax warps
    hold it in float32 before the conversion.
  * O = (P_q V_q) / l; lse = ln sum_j exp(s_ij) (the max cancels).
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


def qdq_allowance(x: np.ndarray, rb: int, cb: int, err: np.ndarray) -> np.ndarray:
    """Per element, how far the quantised value of x could move if x itself
    moved by up to err (elementwise, >= 0): one grid step where x lies within
    err of a rounding midpoint of its block's grid, and a quarter of |x| plus a
    step of the next coarser grid for every element of a block whose largest
    magnitude lies within err of a power of two (its exponent could differ).
    Zero elsewhere: there the rounding decision cannot change.  This bounds the
    effect of computing x in another floating-point precision (float32 instead
    of float64) on the quantised result."""
    x = np.asarray(x, dtype=np.float64)
    err = np.broadcast_to(np.asarray(err, dtype=np.float64), x.shape)
    out = np.zeros_like(x)
    R, Cn = x.shape
    for r in range(0, R, rb):
        for c in range(0, Cn, cb):
            xb, eb = np.abs(x[r:r + rb, c:c + cb]), err[r:r + rb, c:c + cb]
            amax = xb.max() if xb.size else 0.0
            e = block_exponent(amax)
            sc = 2.0 ** e
            # the block's largest magnitude lies in [max(|x| - err), max(|x| + err)]
            lo_e = block_exponent(max((xb - eb).max(), 0.0) if xb.size else 0.0)
            hi_e = block_exponent((xb + eb).max() if xb.size else 0.0)
            if lo_e != e or hi_e != e:
                out[r:r + rb, c:c + cb] = 0.25 * xb + 2.0 ** (max(e, hi_e) + 1 - 9)
                continue
            v = np.minimum(xb / sc, E4M3_MAX)
            i = np.clip(np.searchsorted(_POS, v, side="left"), 1, len(_POS) - 1)
            lo, hi = _POS[i - 1], _POS[i]
            near = np.abs(v - 0.5 * (lo + hi)) <= eb / sc
            out[r:r + rb, c:c + cb] = np.where(near, (hi - lo) * sc, 0.0)
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


LOG2E = 1.0 / np.log(2.0)
# relative size of the float32 rounding of an unquantised P or dS value that
# flip allowances assume (generous: the kernels' float32 scores and exponentials
# are far closer)
FP32_REL = 1e-4


def forward(q_off, kv_off, q, k, v, scale=None, with_allowance=False):
    """MXFP8 softmax attention forward: returns (out [Tq,H,D], lse [H,Tq]) in
    float64, and with with_allowance also allow [Tq,H,D]: how far out could move
    if P were computed in float32 (qdq_allowance of P with a relative error of
    FP32_REL, carried through P V / l)."""
    q, k, v = (np.asarray(t, dtype=np.float64) for t in (q, k, v))
    Tq, H, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    qq, kq, vq = qdq_jagged(q, q_off), qdq_jagged(k, kv_off), qdq_jagged(v, kv_off)
    out = np.zeros((Tq, H, D))
    allow = np.zeros((Tq, H, D))
    lse = np.full((H, Tq), -np.inf)
    qo = np.asarray(q_off, dtype=np.int64)
    ko = np.asarray(kv_off, dtype=np.int64)
    for b in range(len(qo) - 1):
        q0, q1, k0, k1 = qo[b], qo[b + 1], ko[b], ko[b + 1]
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            s = scale * qq[q0:q1, h] @ kq[k0:k1, h].T
            t = s * LOG2E
            M = np.ceil(t.max(axis=1, keepdims=True))  # integer max, log2 units
            p = 2.0 ** (t - M)
            l = p.sum(axis=1, keepdims=True)
            pq = qdq_rows_cols(p, 1, 32)
            out[q0:q1, h] = (pq @ vq[k0:k1, h]) / l
            m = s.max(axis=1, keepdims=True)
            lse[h, q0:q1] = (m + np.log(np.exp(s - m).sum(axis=1, keepdims=True)))[:, 0]
            if with_allowance:
                a = qdq_allowance(p, 1, 32, FP32_REL * p)
                allow[q0:q1, h] = (a @ np.abs(vq[k0:k1, h])) / l
    if with_allowance:
        return out, lse, allow
    return out, lse


def backward(q_off, kv_off, q, k, v, dout, scale=None, with_allowance=False):
    """MXFP8 softmax attention backward: returns (dq, dk, dv) in float64, and
    with with_allowance also (allow_dq, allow_dk, allow_dv): how far they could
    move through flipped quantisation decisions of P and dS if those were
    computed in float32 from a forward output rounded to bf16 and a forward
    that is itself within its own allowance (qdq_allowance with a relative
    error of FP32_REL on P; on dS the same on P and dP, plus, for Delta, the
    bf16 rounding of O, 2^-9 sum_d |dO O|, and sum_d |dO| times the forward
    allowance)."""
    q, k, v, dout = (np.asarray(t, dtype=np.float64) for t in (q, k, v, dout))
    Tq, H, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out, lse, fallow = forward(q_off, kv_off, q, k, v, scale, with_allowance=True)
    qq, kq, vq = qdq_jagged(q, q_off), qdq_jagged(k, kv_off), qdq_jagged(v, kv_off)
    dq_ = qdq_jagged(dout, q_off)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    adq, adk, adv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
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
            if with_allowance:
                do_h, o_h = dout[q0:q1, h], out[q0:q1, h]
                d_err = 2.0 ** -9 * np.sum(np.abs(do_h * o_h), axis=1, keepdims=True) + \
                    np.abs(do_h) @ np.ones((D, 1)) * fallow[q0:q1, h].max(axis=1, keepdims=True)
                ap = qdq_allowance(p, 32, 32, FP32_REL * p)
                e_ds = FP32_REL * np.abs(ds) + p * (FP32_REL * (np.abs(dp) + np.abs(delta)) + d_err)
                ads = qdq_allowance(ds, 32, 32, e_ds)
                adv[k0:k1, h] = ap.T @ np.abs(dq_[q0:q1, h])
                adq[q0:q1, h] = scale * ads @ np.abs(kq[k0:k1, h])
                adk[k0:k1, h] = scale * ads.T @ np.abs(qq[q0:q1, h])
    if with_allowance:
        return dq, dk, dv, adq, adk, adv
    return dq, dk, dv
