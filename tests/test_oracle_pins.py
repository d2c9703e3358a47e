"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test names what it pins: torch SDPA (a library routine, the "padded SDPA"
special case the pages compare against), padded-and-masked dense attention with
torch autograd, closed forms, invariants, central finite differences and the
identity between 64-token BlockAttention and full attention over 64-token
sub-sequences.  A plausible slip in the oracle (a dropped bias term, a wrong
sign, a transposed operand, a missing scale, a wrong block boundary) fails at
least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle
from oracle.oracle import GELU_TANH, SILU, SOFTMAX
from jagged_attention_recommendation_gb300 import workloads as W
from tests import dense_ref

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def batch(seed, lq, lk, H=2, D=8, nb=0, dtype=torch.float64, std=1.0):
    bt = W.random_batch(seed, lq, lk, H, D, dtype=dtype, bias_buckets=nb, std=std)
    if bt["bias"] is not None:
        bt["bias"] = bt["bias"].to(dtype)
    return bt


# --- pointwise activations -------------------------------------------------

@pytest.mark.parametrize("kind,fn", [(SILU, F.silu), (GELU_TANH, lambda x: F.gelu(x, approximate="tanh"))])
def test_activation_matches_torch(kind, fn):
    """act and act' equal torch's silu / tanh-gelu and their autograd derivative."""
    xs = torch.linspace(-12, 12, 241, dtype=torch.float64, requires_grad=True)
    y = fn(xs)
    (g,) = torch.autograd.grad(y.sum(), xs)
    for x, yy, gg in zip(xs.tolist(), y.tolist(), g.tolist()):
        assert abs(oracle.act(kind, x) - yy) <= 1e-14 * max(1.0, abs(yy))
        assert abs(oracle.act_grad(kind, x) - gg) <= 1e-13 * max(1.0, abs(gg))


def test_activation_identities():
    """SiLU(-x) = SiLU(x) - x and GELU(x) - GELU(-x) = x (tanh is odd)."""
    for x in np.linspace(-7, 7, 57):
        assert abs(oracle.act(SILU, -x) - (oracle.act(SILU, x) - x)) < 1e-13
        assert abs(oracle.act(GELU_TANH, x) - oracle.act(GELU_TANH, -x) - x) < 1e-13
    assert oracle.act(SILU, 0.0) == 0.0 and oracle.act(GELU_TANH, 0.0) == 0.0
    assert abs(oracle.act_grad(SILU, 0.0) - 0.5) < 1e-15
    assert abs(oracle.act_grad(GELU_TANH, 0.0) - 0.5) < 1e-15


# --- forward ----------------------------------------------------------------

@pytest.mark.parametrize("lq,lk,nb", [
    ([5, 1, 17, 9], [5, 1, 17, 9], 0),        # self-attention
    ([5, 1, 17, 9], [5, 1, 17, 9], 8),        # with relative-position bias
    ([23, 7, 40], [3, 12, 1], 6),             # cross-attention, asymmetric lengths
    ([2, 4], [30, 19], 0),                    # short Q, long K/V
])
def test_softmax_forward_matches_sdpa(lq, lk, nb):
    """R2: per-sequence torch SDPA in float64 with the bias as an additive float mask."""
    bt = batch(1, lq, lk, nb=nb)
    out, lse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"])
    ref = dense_ref.sdpa_forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"])
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU_TANH])
@pytest.mark.parametrize("nb", [0, 5])
def test_forward_matches_padded_dense(act, nb):
    """R1: padded-and-masked dense attention (torch float64), incl. lse."""
    bt = batch(2, [9, 3, 14, 1], [6, 11, 2, 8], nb=nb)
    out, lse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], act=act)
    ref, rlse, *_ = dense_ref.padded_dense(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"],
                                           bias=bt["bias"], act=act)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    if act == SOFTMAX:
        np.testing.assert_allclose(lse, rlse.numpy(), rtol=1e-12, atol=1e-12)
    else:
        assert lse is None


def test_softmax_rows_sum_to_one():
    """R3: with V = 1 every softmax output entry is sum_j P_ij = 1."""
    bt = batch(3, [7, 20, 3], [9, 4, 30], nb=4)
    v = torch.ones_like(bt["v"])
    out, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], v, bias=bt["bias"])
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU_TANH])
def test_single_key(act):
    """R4: one key per sequence -> softmax O_i = v_0 exactly; activation O_i = act(s_i0) v_0."""
    bt = batch(4, [6, 3], [1, 1], nb=3)
    out, lse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], act=act)
    for b in range(2):
        q0, q1, k0 = int(bt["q_off"][b]), int(bt["q_off"][b + 1]), int(bt["kv_off"][b])
        v0 = bt["v"][k0].numpy()
        for i in range(q1 - q0):
            if act == SOFTMAX:
                np.testing.assert_array_equal(out[q0 + i], v0)
            else:
                for h in range(2):
                    s = bt["scale"] * float(bt["q"][q0 + i, h] @ bt["k"][k0, h])
                    s += float(bt["bias"][h, min(i, 2)])
                    np.testing.assert_allclose(out[q0 + i, h], oracle.act(act, s) * v0[h], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("act", [SOFTMAX, GELU_TANH])
def test_batch_order_invariance(act):
    """R5: permuting the sequences of the batch permutes the outputs identically."""
    lq, lk = [5, 12, 1, 8], [7, 3, 10, 8]
    bt = batch(5, lq, lk, nb=4)
    out, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], act=act)
    perm = [2, 0, 3, 1]
    qo, ko, (qp,), (kp, vp), qidx, _ = oracle.sub_batch(bt["q_off"], bt["kv_off"], perm, bt["q"],
                                                         tensors_kv=(bt["k"], bt["v"]))
    outp, _ = oracle.forward(qo, ko, qp, kp, vp, bias=bt["bias"], act=act)
    np.testing.assert_array_equal(outp, out[qidx])


def test_bias_shift_and_identical_keys():
    """R8: a constant added to the whole table leaves softmax unchanged; equal keys give mean(V)."""
    bt = batch(6, [8, 5], [6, 9], nb=6)
    out, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"])
    out2, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"] + 3.25)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-13)
    k = bt["k"].clone()
    for b in range(2):
        k0, k1 = int(bt["kv_off"][b]), int(bt["kv_off"][b + 1])
        k[k0:k1] = k[k0]
    out3, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], k, bt["v"])
    for b in range(2):
        q0, q1 = int(bt["q_off"][b]), int(bt["q_off"][b + 1])
        k0, k1 = int(bt["kv_off"][b]), int(bt["kv_off"][b + 1])
        mean = bt["v"][k0:k1].mean(0).numpy()
        np.testing.assert_allclose(out3[q0:q1], np.broadcast_to(mean, out3[q0:q1].shape), rtol=1e-12, atol=1e-13)


def test_empty_sequences():
    """Reading for an empty key set: O = 0, lse = -inf; empty query sets produce nothing."""
    bt = batch(7, [4, 0, 3], [0, 5, 6], nb=0)
    out, lse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"])
    assert np.all(out[0:4] == 0.0) and np.all(np.isneginf(lse[:, 0:4]))
    ref = dense_ref.sdpa_forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"])
    np.testing.assert_allclose(out[4:], ref.numpy()[4:], rtol=1e-12, atol=1e-12)


# --- BlockAttention ---------------------------------------------------------

def _recut(off, block):
    """Offsets that cut every sequence into consecutive ``block``-token sub-sequences."""
    cuts = [0]
    for b in range(len(off) - 1):
        L = int(off[b + 1] - off[b])
        base = int(off[b])
        for s in range(0, L, block):
            cuts.append(base + min(s + block, L))
    return np.array(cuts, dtype=np.int32)


@pytest.mark.parametrize("act", [SOFTMAX, SILU])
def test_block_equals_full_on_subsequences(act):
    """R7: 64-token BlockAttention == full attention with every sequence cut at multiples of 64."""
    lens = [130, 64, 17, 200]
    bt = batch(8, lens, lens, D=4, nb=7)
    out, lse = oracle.forward(bt["q_off"], bt["q_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], act=act,
                              block=64)
    cut = _recut(bt["q_off"], 64)
    out2, lse2 = oracle.forward(cut, cut, bt["q"], bt["k"], bt["v"], bias=bt["bias"], act=act)
    np.testing.assert_allclose(out, out2, rtol=1e-13, atol=1e-14)
    dq, dk, dv, db = oracle.backward(bt["q_off"], bt["q_off"], bt["q"], bt["k"], bt["v"], bt["dout"],
                                     bias=bt["bias"], act=act, block=64)
    dq2, dk2, dv2, db2 = oracle.backward(cut, cut, bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"], act=act)
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2), (db, db2)):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_block_short_sequences_equal_full():
    """R7: sequences no longer than one block are unchanged by the block restriction."""
    lens = [64, 5, 33]
    bt = batch(9, lens, lens, D=8)
    a, _ = oracle.forward(bt["q_off"], bt["q_off"], bt["q"], bt["k"], bt["v"], block=64)
    b, _ = oracle.forward(bt["q_off"], bt["q_off"], bt["q"], bt["k"], bt["v"])
    np.testing.assert_array_equal(a, b)


def test_block_matches_sdpa_with_block_mask():
    """R7 + R2: block mode equals SDPA with a block-diagonal -inf mask."""
    lens = [150, 70]
    bt = batch(10, lens, lens, D=8, nb=5)
    out, _ = oracle.forward(bt["q_off"], bt["q_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], block=64)
    ref = dense_ref.sdpa_forward(bt["q_off"], bt["q_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], block=64)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


# --- backward ---------------------------------------------------------------

@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU_TANH])
@pytest.mark.parametrize("block", [0, 64])
def test_backward_matches_autograd(act, block):
    """Gradients equal torch autograd through the padded dense computation."""
    if block:
        lq = lk = [70, 9, 130]
    else:
        lq, lk = [9, 3, 14, 1], [6, 11, 2, 8]
    bt = batch(11, lq, lk, nb=6)
    dq, dk, dv, db = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"],
                                     bias=bt["bias"], act=act, block=block)
    _, _, rdq, rdk, rdv, rdb = dense_ref.padded_dense(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"],
                                                      dout=bt["dout"], bias=bt["bias"], act=act, block=block)
    for a, r in ((dq, rdq), (dk, rdk), (dv, rdv), (db, rdb)):
        np.testing.assert_allclose(a, r.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU_TANH])
def test_backward_finite_differences(act):
    """R6: central differences (h = 1e-6) of L = sum(O * dO) through the oracle's own forward."""
    bt = batch(12, [3, 2], [2, 4], H=1, D=3, nb=3)
    args = dict(bias=bt["bias"], act=act)
    dq, dk, dv, db = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], **args)
    dout = bt["dout"].numpy()
    base = {n: bt[n].clone() for n in ("q", "k", "v", "bias")}

    def loss(**over):
        t = dict(base)
        t.update(over)
        out, _ = oracle.forward(bt["q_off"], bt["kv_off"], t["q"], t["k"], t["v"], bias=t["bias"], act=act)
        return float((out * dout).sum())

    h = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv), ("bias", db)):
        x = base[name]
        num = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.clone(), x.clone()
            xp[idx] += h
            xm[idx] -= h
            num[idx] = (loss(**{name: xp}) - loss(**{name: xm})) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-8)


@pytest.mark.parametrize("act", [SILU, GELU_TANH])
def test_gdpa_zero_queries_closed_form(act):
    """R9: Q = 0, no bias -> s = 0 -> O = 0, dV = 0, dQ_i = scale * 1/2 * sum_j <dO_i, v_j> k_j."""
    bt = batch(13, [4, 6], [5, 3], D=6)
    q = torch.zeros_like(bt["q"])
    out, _ = oracle.forward(bt["q_off"], bt["kv_off"], q, bt["k"], bt["v"], act=act)
    assert np.all(out == 0.0)
    dq, dk, dv, _ = oracle.backward(bt["q_off"], bt["kv_off"], q, bt["k"], bt["v"], bt["dout"], act=act)
    assert np.all(dv == 0.0) and np.all(dk == 0.0)
    for b in range(2):
        q0, q1 = int(bt["q_off"][b]), int(bt["q_off"][b + 1])
        k0, k1 = int(bt["kv_off"][b]), int(bt["kv_off"][b + 1])
        for h in range(2):
            Kb = bt["k"][k0:k1, h].numpy()
            Vb = bt["v"][k0:k1, h].numpy()
            dO = bt["dout"][q0:q1, h].numpy()
            ref = bt["scale"] * 0.5 * (dO @ Vb.T) @ Kb
            np.testing.assert_allclose(dq[q0:q1, h], ref, rtol=1e-12, atol=1e-13)


def test_softmax_gradient_of_bias_rows_sum_zero():
    """Softmax rows of dS sum to zero, so with a single bias bucket dT = 0."""
    bt = batch(14, [5, 8], [7, 3], nb=1)
    _, _, _, db = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"])
    np.testing.assert_allclose(db, 0.0, atol=1e-12)


def test_thread_count_does_not_change_result():
    bt = batch(15, [40, 17, 3, 60], [40, 17, 3, 60], nb=4)
    a = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"],
                        nthreads=1)
    b = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"],
                        nthreads=7)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_planted_mistakes_are_caught():
    """A dropped bias term or a missing scale in the oracle's inputs is visible to the SDPA pin."""
    bt = batch(16, [6, 9], [6, 9], nb=4)
    ref = dense_ref.sdpa_forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"]).numpy()
    no_bias, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"])
    assert np.abs(no_bias - ref).max() > 1e-3
    wrong_scale, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], scale=1.0)
    assert np.abs(wrong_scale - ref).max() > 1e-3


# --- sliding window (|i - j| < W) ------------------------------------------

def test_window_matches_sdpa_with_band_mask():
    """Window W: SDPA with -inf outside the band |i - j| < W, bias included."""
    bt = batch(41, [9, 30, 1, 17], [9, 30, 1, 17], nb=6)
    for w in (1, 3, 8):
        out, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], window=w)
        ref = dense_ref.sdpa_forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"],
                                     window=w).numpy()
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU_TANH])
def test_window_forward_backward_match_autograd(act):
    """Window with cross-attention lengths (some rows see no key at all): forward,
    lse and every gradient against masked dense attention under torch autograd."""
    bt = batch(42, [12, 3, 25, 0], [5, 9, 30, 4], nb=5)
    w = 4
    out, lse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], act=act,
                              window=w)
    dq, dk, dv, dt = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"],
                                     bias=bt["bias"], act=act, window=w)
    r_out, r_lse, r_dq, r_dk, r_dv, r_dt = dense_ref.padded_dense(bt["q_off"], bt["kv_off"], bt["q"], bt["k"],
                                                                  bt["v"], dout=bt["dout"], bias=bt["bias"],
                                                                  act=act, window=w)
    np.testing.assert_allclose(out, r_out.numpy(), rtol=1e-11, atol=1e-11)
    if act == SOFTMAX:
        np.testing.assert_allclose(lse, r_lse.numpy(), rtol=1e-11, atol=1e-11)
    for got, ref in ((dq, r_dq), (dk, r_dk), (dv, r_dv), (dt, r_dt)):
        np.testing.assert_allclose(got, ref.detach().numpy(), rtol=1e-10, atol=1e-10)


def test_window_one_is_the_diagonal():
    """W = 1 keeps only j = i: O = V and lse = s_ii exactly; then P = 1, so
    dS = dP - Delta = 0 gives dQ = dK = 0 and dV = dO."""
    bt = batch(43, [7, 20, 1], [7, 20, 1], nb=0)
    out, lse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], window=1)
    q, k, v, do = (bt[n].numpy() for n in ("q", "k", "v", "dout"))
    assert np.array_equal(out, v)
    D = q.shape[2]
    np.testing.assert_allclose(lse, (np.einsum("thd,thd->ht", q, k) / math.sqrt(D)), rtol=1e-13, atol=1e-13)
    dq, dk, dv, _ = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], window=1)
    assert np.array_equal(dq, np.zeros_like(dq)) and np.array_equal(dk, np.zeros_like(dk))
    assert np.array_equal(dv, do)


def test_window_wider_than_every_sequence_is_full_attention():
    bt = batch(44, [13, 40, 2], [13, 40, 2], nb=4)
    full, flse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"])
    win, wlse = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], window=40)
    assert np.array_equal(full, win) and np.array_equal(flse, wlse)


def test_window_band_is_symmetric_and_rejects_block():
    """An off-by-one band (|i - j| <= W, or one-sided) changes row 0 against the
    SDPA pin above; here: the W = 2 output of row i uses exactly keys i-1, i, i+1."""
    bt = batch(45, [6], [6], nb=0)
    out, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], window=2)
    q, k, v = (bt[n].numpy()[:, 0] for n in ("q", "k", "v"))
    D = q.shape[1]
    for i in range(6):
        js = [j for j in (i - 1, i, i + 1) if 0 <= j < 6]
        s = np.array([q[i] @ k[j] / math.sqrt(D) for j in js])
        p = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
        np.testing.assert_allclose(out[i, 0], p @ v[js], rtol=1e-12, atol=1e-12)
    with pytest.raises(ValueError):
        oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], block=64, window=2)


# --- rotary position embedding (RoPE, then attention) -----------------------

def test_rope_hand_rotation():
    """Half-split pairing, sign and local position, worked by hand.

    D = 4; the row under test is local position 1 of the second sequence (global
    row 4).  Table row 1: cos = (0.6, 0), sin = (0.8, 1); x = (1, 2, 3, 4):
      pair (0, 2): 1*0.6 - 3*0.8 = -1.8,  3*0.6 + 1*0.8 = 2.6
      pair (1, 3): 2*0   - 4*1   = -4,    4*0   + 2*1   = 2
    so y = (-1.8, -4, 2.6, 2).  Local position 0 (global row 3) takes table row
    0, the identity.  Rows 3 and 4 of the table hold other angles, so global
    indexing would give other values.
    """
    off = [0, 3, 5]
    x = np.zeros((5, 1, 4))
    x[3, 0] = x[4, 0] = [1.0, 2.0, 3.0, 4.0]
    cos = np.array([[1.0, 1.0], [0.6, 0.0], [0.0, 0.0], [0.0, 1.0], [-1.0, 0.0]])
    sin = np.array([[0.0, 0.0], [0.8, 1.0], [1.0, 1.0], [1.0, 0.0], [0.0, -1.0]])
    y = oracle.rope_rotate(x, off, cos, sin)
    np.testing.assert_allclose(y[4, 0], [-1.8, -4.0, 2.6, 2.0], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(y[3, 0], [1.0, 2.0, 3.0, 4.0])
    # cos^2 + sin^2 = 1 in both pairs: the transposed rotation undoes it
    back = oracle.rope_rotate(y, off, cos, sin, transpose=True)
    np.testing.assert_allclose(back[4, 0], [1.0, 2.0, 3.0, 4.0], rtol=0, atol=1e-15)


def _phi(P, D, seed):
    return torch.from_numpy(np.random.default_rng(seed).uniform(-np.pi, np.pi, size=(P, D // 2)))


@pytest.mark.parametrize("act", [SOFTMAX, SILU])
@pytest.mark.parametrize("block", [0, 64])
def test_rope_matches_autograd_complex(act, block):
    """Rotate-then-attend equals torch autograd through padded dense attention
    whose Q and K are rotated by complex multiplication (x[d] + i x[d+D/2]) e^(i phi):
    outputs and the gradients of the unrotated Q, K, V and the bias table."""
    if block:
        lq = lk = [70, 9, 130]
    else:
        lq, lk = [9, 3, 14, 1], [6, 11, 2, 8]
    bt = batch(51, lq, lk, nb=6)
    phi = _phi(140, 8, 52)
    rope = (np.cos(phi.numpy()), np.sin(phi.numpy()))
    out, _ = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], act=act,
                            block=block, rope=rope)
    dq, dk, dv, db = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"],
                                     bias=bt["bias"], act=act, block=block, rope=rope)
    rout, _, rdq, rdk, rdv, rdb = dense_ref.padded_dense(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"],
                                                         dout=bt["dout"], bias=bt["bias"], act=act, block=block,
                                                         rope_phi=phi)
    np.testing.assert_allclose(out, rout.numpy(), rtol=1e-11, atol=1e-12)
    for a, r in ((dq, rdq), (dk, rdk), (dv, rdv), (db, rdb)):
        np.testing.assert_allclose(a, r.numpy(), rtol=1e-11, atol=1e-12)


def test_rope_identity_table_is_no_rope():
    """Angle 0 everywhere: outputs and gradients equal the unrotated oracle exactly."""
    bt = batch(53, [70, 9, 130], [70, 9, 130], nb=4)
    cos, sin = W.rope_table(130, 8, "identity")
    for block in (0, 64):
        a = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], block=block,
                           rope=(cos, sin))[0]
        b = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], block=block)[0]
        np.testing.assert_array_equal(a, b)
        ga = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"],
                             block=block, rope=(cos, sin))
        gb = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"],
                             block=block)
        for x, y in zip(ga[:3], gb[:3]):
            np.testing.assert_array_equal(x, y)


def _ladder(P, D, shift=0):
    inv = 10000.0 ** (-2.0 * np.arange(D // 2) / D)
    phi = (np.arange(P)[:, None] + shift) * inv[None, :]
    return np.cos(phi), np.sin(phi)


@pytest.mark.parametrize("block", [0, 64])
def test_rope_scores_depend_on_offset_only(block):
    """With angles linear in the position, <R_i q, R_j k> depends on i - j only:
    starting every sequence at position 37 instead of 0 leaves O (and dV)
    unchanged.  Rotating K the wrong way (angle -phi) breaks this."""
    bt = batch(54, [70, 9, 130], [70, 9, 130], nb=4)
    r0, r37 = _ladder(130, 8), _ladder(130, 8, shift=37)
    o0 = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], block=block, rope=r0)[0]
    o37 = oracle.forward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bias=bt["bias"], block=block,
                         rope=r37)[0]
    np.testing.assert_allclose(o0, o37, rtol=1e-11, atol=1e-12)
    g0 = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"],
                         block=block, rope=r0)
    g37 = oracle.backward(bt["q_off"], bt["kv_off"], bt["q"], bt["k"], bt["v"], bt["dout"], bias=bt["bias"],
                          block=block, rope=r37)
    np.testing.assert_allclose(g0[2], g37[2], rtol=1e-11, atol=1e-12)

    def planted(rope):  # a slip planted on the CPU: K rotated by -phi
        q = oracle.rope_rotate(bt["q"], bt["q_off"], rope[0], rope[1])
        k = oracle.rope_rotate(bt["k"], bt["kv_off"], rope[0], rope[1], transpose=True)
        return oracle.forward(bt["q_off"], bt["kv_off"], q, k, bt["v"], bias=bt["bias"], block=block)[0]

    assert np.abs(planted(r0) - planted(r37)).max() > 1e-3


def test_rope_preserves_norms_and_transpose_inverts():
    bt = batch(55, [40, 17], [40, 17], D=16)
    cos, sin = _ladder(40, 16)
    y = oracle.rope_rotate(bt["q"], bt["q_off"], cos, sin)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(bt["q"].numpy(), axis=-1), rtol=1e-13)
    np.testing.assert_allclose(oracle.rope_rotate(y, bt["q_off"], cos, sin, transpose=True), bt["q"].numpy(),
                               rtol=0, atol=1e-13)
