"""Dense per-sequence torch float64 computations used to pin the oracle.

These go through library routines (scaled_dot_product_attention, softmax,
silu, gelu, autograd) on padded/masked dense matrices, which is a different
computation from the oracle's per-row loops.
"""
import numpy as np
import torch
import torch.nn.functional as F

SOFTMAX, SILU, GELU_TANH = 0, 1, 2


def bias_matrix(table_h, Lq, Lk):
    i = torch.arange(Lq).view(-1, 1)
    j = torch.arange(Lk).view(1, -1)
    idx = (i - j).abs().clamp(max=table_h.shape[0] - 1)
    return table_h[idx]


def block_mask(L, block):
    i = torch.arange(L).view(-1, 1) // block
    j = torch.arange(L).view(1, -1) // block
    return i == j


def band_mask(Lq, Lk, window):
    """True where |i - j| < window (sliding-window attention)."""
    i = torch.arange(Lq).view(-1, 1)
    j = torch.arange(Lk).view(1, -1)
    return (i - j).abs() < window


def sdpa_forward(q_off, kv_off, q, k, v, bias=None, scale=None, block=0, window=0):
    """Softmax attention per sequence with torch SDPA in float64."""
    q, k, v = (t.to(torch.float64) for t in (q, k, v))
    Tq, H, D = q.shape
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = torch.zeros(Tq, H, D, dtype=torch.float64)
    for b in range(len(q_off) - 1):
        q0, q1, k0, k1 = int(q_off[b]), int(q_off[b + 1]), int(kv_off[b]), int(kv_off[b + 1])
        if q1 == q0 or k1 == k0:
            continue
        qb = q[q0:q1].permute(1, 0, 2)  # [H, Lq, D]
        kb = k[k0:k1].permute(1, 0, 2)
        vb = v[k0:k1].permute(1, 0, 2)
        mask = torch.zeros(H, q1 - q0, k1 - k0, dtype=torch.float64)
        if bias is not None:
            for h in range(H):
                mask[h] = bias_matrix(bias[h].to(torch.float64), q1 - q0, k1 - k0)
        if block:
            mask = mask.masked_fill(~block_mask(q1 - q0, block), float("-inf"))
        if window:
            mask = mask.masked_fill(~band_mask(q1 - q0, k1 - k0, window), float("-inf"))
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=scale)
        out[q0:q1] = o.permute(1, 0, 2)
    return out


def rotate_complex(x, phi):
    """Rotary embedding as complex multiplication: the feature pair
    (x[d], x[d + D/2]) is the complex number x[d] + i x[d + D/2], multiplied by
    e^(i phi[p, d]) at padded position p (the row index of dimension -2)."""
    half = x.shape[-1] // 2
    z = torch.complex(x[..., :half], x[..., half:])
    w = torch.polar(torch.ones_like(phi), phi)[: x.shape[-2]]
    y = z * w
    return torch.cat([y.real, y.imag], dim=-1)


def padded_dense(q_off, kv_off, q, k, v, dout=None, bias=None, scale=None, act=SOFTMAX, block=0, window=0,
                 rope_phi=None):
    """Pad the jagged batch to [B, H, Lmax, D], mask, and run attention densely.

    Softmax rows are masked with -inf; activation mode multiplies by a 0/1 mask
    (a -inf score would give NaN through SiLU).  rope_phi [P, D/2] (float64
    angles): the padded Q and K are rotated by ``rotate_complex`` first, inside
    the autograd graph.  If ``dout`` is given the gradients come from torch
    autograd.  Returns (out, lse, dq, dk, dv, dbias) in the jagged layout,
    float64.
    """
    B = len(q_off) - 1
    Tq, H, D = q.shape
    Tk = k.shape[0]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    lq = np.diff(np.asarray(q_off, dtype=np.int64))
    lk = np.diff(np.asarray(kv_off, dtype=np.int64))
    Mq, Mk = max(int(lq.max(initial=0)), 1), max(int(lk.max(initial=0)), 1)
    qd = torch.zeros(B, H, Mq, D, dtype=torch.float64)
    kd = torch.zeros(B, H, Mk, D, dtype=torch.float64)
    vd = torch.zeros(B, H, Mk, D, dtype=torch.float64)
    valid = torch.zeros(B, 1, Mq, Mk, dtype=torch.bool)
    for b in range(B):
        q0, k0 = int(q_off[b]), int(kv_off[b])
        qd[b, :, :lq[b]] = q[q0:q0 + lq[b]].to(torch.float64).permute(1, 0, 2)
        kd[b, :, :lk[b]] = k[k0:k0 + lk[b]].to(torch.float64).permute(1, 0, 2)
        vd[b, :, :lk[b]] = v[k0:k0 + lk[b]].to(torch.float64).permute(1, 0, 2)
        m = torch.zeros(Mq, Mk, dtype=torch.bool)
        m[:lq[b], :lk[b]] = True
        if block:
            m[:lq[b], :lk[b]] &= block_mask(max(lq[b], lk[b]), block)[:lq[b], :lk[b]]
        if window:
            m[:lq[b], :lk[b]] &= band_mask(int(lq[b]), int(lk[b]), window)
        valid[b, 0] = m
    tbl = None
    if bias is not None:
        tbl = bias.to(torch.float64).clone().requires_grad_(dout is not None)
    for t in (qd, kd, vd):
        t.requires_grad_(dout is not None)
    qa, ka = qd, kd
    if rope_phi is not None:
        qa = rotate_complex(qd, rope_phi.to(torch.float64))
        ka = rotate_complex(kd, rope_phi.to(torch.float64))
    s = scale * qa @ ka.transpose(-1, -2)
    if tbl is not None:
        i = torch.arange(Mq).view(-1, 1)
        j = torch.arange(Mk).view(1, -1)
        idx = (i - j).abs().clamp(max=tbl.shape[1] - 1)
        s = s + tbl[:, idx].unsqueeze(0)
    lse = None
    if act == SOFTMAX:
        sm = s.masked_fill(~valid, float("-inf"))
        lse_d = torch.logsumexp(sm, dim=-1)
        p = torch.softmax(sm, dim=-1)
        p = torch.nan_to_num(p, nan=0.0)  # rows with no keys
        lse = torch.full((H, Tq), float("-inf"), dtype=torch.float64)
    else:
        a = F.silu(s) if act == SILU else F.gelu(s, approximate="tanh")
        p = a * valid
    o = p @ vd
    out = torch.zeros(Tq, H, D, dtype=torch.float64)
    for b in range(B):
        q0 = int(q_off[b])
        out[q0:q0 + lq[b]] = o[b, :, :lq[b]].detach().permute(1, 0, 2)
        if lse is not None and lk[b] > 0:
            lse[:, q0:q0 + lq[b]] = lse_d[b, :, :lq[b]].detach()
    if dout is None:
        return out, lse, None, None, None, None
    dd = torch.zeros(B, H, Mq, D, dtype=torch.float64)
    for b in range(B):
        q0 = int(q_off[b])
        dd[b, :, :lq[b]] = dout[q0:q0 + lq[b]].to(torch.float64).permute(1, 0, 2)
    (o * dd).sum().backward()
    dq = torch.zeros(Tq, H, D, dtype=torch.float64)
    dk = torch.zeros(Tk, H, D, dtype=torch.float64)
    dv = torch.zeros(Tk, H, D, dtype=torch.float64)
    for b in range(B):
        q0, k0 = int(q_off[b]), int(kv_off[b])
        dq[q0:q0 + lq[b]] = qd.grad[b, :, :lq[b]].permute(1, 0, 2)
        dk[k0:k0 + lk[b]] = kd.grad[b, :, :lk[b]].permute(1, 0, 2)
        dv[k0:k0 + lk[b]] = vd.grad[b, :, :lk[b]].permute(1, 0, 2)
    dbias = tbl.grad if tbl is not None else None
    return out, lse, dq, dk, dv, dbias
