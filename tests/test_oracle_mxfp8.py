"""Pins of the MXFP8 attention reference (oracle/mxfp8.py) against things other
than itself: torch's float8_e4m3fn decoding and rounding, the round-to-even and
saturation rules of the format, the block-exponent rule, the transpose
invariance of 32 x 32 blocks that the pages state, closed forms, and the fp64
oracle's plain attention on the quantised inputs (with the P-quantisation error
bound)."""
import numpy as np
import pytest
import torch

from oracle import mxfp8 as M
from oracle import oracle
from jagged_attention_recommendation_gb300 import workloads as W

f8 = getattr(torch, "float8_e4m3fn", None)


def test_e4m3_grid_decoding():
    g = M.e4m3_values()
    assert len(g) == 253  # 254 finite codes, +0 and -0 equal
    assert g.max() == 448.0 and g.min() == -448.0
    pos = g[g > 0]
    assert pos.min() == 2.0 ** -9          # smallest subnormal
    assert 2.0 ** -6 in pos and 1.0 in pos and 1.125 in pos and 1.0625 not in pos
    np.testing.assert_array_equal(g, -g[::-1])


@pytest.mark.skipif(f8 is None, reason="torch without float8_e4m3fn")
def test_e4m3_grid_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8).view(f8).to(torch.float64).numpy()
    finite = np.unique(codes[np.isfinite(codes)])
    np.testing.assert_array_equal(finite, M.e4m3_values())


@pytest.mark.skipif(f8 is None, reason="torch without float8_e4m3fn")
def test_e4m3_rounding_matches_torch_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000), rng.normal(0, 0.01, 5000),
                        (M.e4m3_values()[1:] + M.e4m3_values()[:-1]) / 2])  # every midpoint
    ref = torch.from_numpy(x).to(f8).to(torch.float64).numpy()
    np.testing.assert_array_equal(M.quantize_e4m3(x), ref)


def test_e4m3_ties_to_even_and_saturation():
    q = M.quantize_e4m3(np.array([1.0625, 1.1875, -1.0625, 500.0, -1e9, 448.0, 0.0, 2.0 ** -10, 3 * 2.0 ** -10]))
    # 1.0625: between 1.0 (code 0x38) and 1.125 (0x39) -> 1.0; 1.1875 -> 1.25 (0x3A);
    # beyond 448 -> 448; 2^-10 is half the smallest subnormal -> 0 (even); 3*2^-10 -> 2^-8 (code 2)
    np.testing.assert_array_equal(q, [1.0, 1.25, -1.0, 448.0, -448.0, 448.0, 0.0, 0.0, 2.0 ** -8])


def test_block_exponent_rule():
    np.testing.assert_array_equal(M.block_exponent(np.array([448.0, 256.0, 511.9, 1.0, 0.75, 2.0 ** -130, 0.0])),
                                  [0, 0, 0, -8, -9, -127, -127])
    # amax / 2^e lies in [256, 512): the largest element lands at the top of E4M3's range
    rng = np.random.default_rng(1)
    a = np.exp(rng.uniform(-20, 20, 1000))
    r = a / 2.0 ** M.block_exponent(a)
    assert np.all((r >= 256) & (r < 512))


def test_qdq_error_bound_and_fixed_points():
    rng = np.random.default_rng(2)
    for s in (1e-3, 1.0, 37.0):
        x = rng.normal(0, s, (64, 96))
        y = M.qdq_rows_cols(x, 32, 32)
        for r in range(0, 64, 32):
            for c in range(0, 96, 32):
                xb, yb = x[r:r + 32, c:c + 32], y[r:r + 32, c:c + 32]
                sc = 2.0 ** M.block_exponent(np.abs(xb).max())
                sat = np.abs(xb) > 448 * sc
                bound = np.maximum(2.0 ** -4 * np.abs(xb), 2.0 ** -10 * sc)
                assert np.all(np.abs(xb - yb)[~sat] <= bound[~sat])
                assert np.all(np.abs(yb[sat]) == 448 * sc)
                np.testing.assert_array_equal(M.qdq_rows_cols(yb, 32, 32), yb)  # already representable


def test_square_blocks_are_transpose_invariant():
    """The pages' reason for 32 x 32 blocks: quantising X^T gives (quantised X)^T."""
    x = np.random.default_rng(3).normal(0, 1, (100, 70))
    np.testing.assert_array_equal(M.qdq_rows_cols(x, 32, 32).T, M.qdq_rows_cols(x.T, 32, 32))
    # row blocks of 1 x 32 (how P is quantised) are not
    assert not np.array_equal(M.qdq_rows_cols(x, 1, 32).T, M.qdq_rows_cols(x.T, 1, 32))


def test_jagged_blocks_start_at_each_sequence():
    """Blocks restart at every sequence's first row: a batch quantises like its
    sequences quantised alone."""
    bt = W.random_batch(4, [40, 7, 70], [40, 7, 70], 2, 64, dtype=torch.float64)
    whole = M.qdq_jagged(bt["q"].numpy(), bt["q_off"])
    off = bt["q_off"]
    for b in range(3):
        alone = M.qdq_jagged(bt["q"][off[b]:off[b + 1]].numpy(), [0, off[b + 1] - off[b]])
        np.testing.assert_array_equal(whole[off[b]:off[b + 1]], alone)


def test_single_key_closed_form():
    """One key: with the integer running max M = ceil(t), t = s log2 e, the row's
    one P value is p = 2^(t - M) in (1/2, 1]; its block exponent is -9 (or -8
    for p = 1), so P_q = E4M3(p 2^9) 2^-9 and O = (P_q / p) v_q (the row sum is
    the unquantised p).  lse is s itself."""
    bt = W.random_batch(5, [3, 40], [1, 1], 2, 64, dtype=torch.float64)
    q, k, v = (bt[n].numpy() for n in ("q", "k", "v"))
    out, lse = M.forward(bt["q_off"], bt["kv_off"], q, k, v)
    qq, kq = M.qdq_jagged(q, bt["q_off"]), M.qdq_jagged(k, bt["kv_off"])
    vq = M.qdq_jagged(v, bt["kv_off"])
    ratios = []
    for b, (q0, q1) in enumerate(((0, 3), (3, 43))):
        for h in range(2):
            s_ = (qq[q0:q1, h] @ kq[b, h]) / 8.0
            t = s_ / np.log(2.0)
            p = 2.0 ** (t - np.ceil(t))
            assert np.all((p > 0.5) & (p <= 1.0))
            e = np.where(p < 1.0, -9.0, -8.0)
            pq = M.quantize_e4m3(p * 2.0 ** -e) * 2.0 ** e
            np.testing.assert_allclose(out[q0:q1, h], (pq / p)[:, None] * vq[b, h][None, :], rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(lse[h, q0:q1], s_, rtol=1e-12, atol=1e-12)
            ratios.append(pq / p)
    # half a grid step (1/16) below 448, saturation at 448 of values up to 512 above
    r = np.concatenate(ratios)
    assert np.all((r >= 448.0 / 512.0 - 1e-12) & (r <= 1.0 + 1.0 / 16 + 1e-12)) and np.any(r != 1.0)


def test_power_of_two_factor_commutes_with_quantisation():
    """The property the integer running max rests on: a power-of-two factor 2^k
    moves every block exponent by k and leaves the E4M3 mantissas alone, so
    qdq(2^k x) = 2^k qdq(x) (blocks of 1 x 32 and 32 x 32, k in -20..20)."""
    rng = np.random.default_rng(12)
    x = np.exp(rng.normal(0.0, 2.0, (64, 96))) * rng.choice([-1.0, 1.0], (64, 96))
    for rb, cb in ((1, 32), (32, 32)):
        base = M.qdq_rows_cols(x, rb, cb)
        for k in (-20, -7, -1, 1, 3, 20):
            np.testing.assert_array_equal(M.qdq_rows_cols(x * 2.0 ** k, rb, cb), base * 2.0 ** k)
    # a factor that is not a power of two changes rounding decisions
    assert not np.array_equal(M.qdq_rows_cols(x * 1.3, 1, 32), M.qdq_rows_cols(x, 1, 32) * 1.3)


def test_flip_allowance():
    """qdq_allowance: zero where a perturbation within err cannot change the
    rounding, one grid step next to a midpoint, and a bound that holds for
    values actually perturbed by up to err."""
    rng = np.random.default_rng(13)
    x = rng.uniform(0.0, 1.0, (32, 64))
    err = 1e-4 * x
    a = M.qdq_allowance(x, 32, 32, err)
    base = M.qdq_rows_cols(x, 32, 32)
    for trial in range(20):
        xp = x + rng.uniform(-1.0, 1.0, x.shape) * err
        assert np.all(np.abs(M.qdq_rows_cols(xp, 32, 32) - base) <= a + 1e-15)
    assert 0 < np.count_nonzero(a) < a.size // 10  # only values next to a midpoint
    # a value exactly at a midpoint (272 = (256 + 288) / 2 in a block scaled by 2^0)
    y = np.full((1, 32), 300.0)
    y[0, 0] = 272.0
    ay = M.qdq_allowance(y, 1, 32, 1e-9 * np.ones_like(y))
    assert ay[0, 0] == 32.0 and np.all(ay[0, 1:] == 0.0)


def test_against_plain_attention_on_quantised_inputs():
    """On the quantised Q, K, V the fp64 oracle's plain softmax attention gives
    the same lse exactly (up to fp64 rounding) and an O that differs only by the
    quantisation of P: |O_mx - O| <= sum_j |P_j - Pq_j| |v_j| / l, with
    |P - Pq| <= max(2^-4 P, 2^-10 * block scale) per element."""
    bt = W.random_batch(6, [45, 200, 3], [130, 64, 300], 2, 64, dtype=torch.float64)
    q, k, v = (bt[n].numpy() for n in ("q", "k", "v"))
    out, lse = M.forward(bt["q_off"], bt["kv_off"], q, k, v)
    qq, kq, vq = (M.qdq_jagged(t, o) for t, o in ((q, bt["q_off"]), (k, bt["kv_off"]), (v, bt["kv_off"])))
    ref, ref_lse = oracle.forward(bt["q_off"], bt["kv_off"], qq, kq, vq)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    # element-wise bound, computed per row from the unquantised P
    scale = 1.0 / np.sqrt(64)
    for b in range(3):
        q0, q1 = bt["q_off"][b], bt["q_off"][b + 1]
        k0, k1 = bt["kv_off"][b], bt["kv_off"][b + 1]
        for h in range(2):
            s = scale * qq[q0:q1, h] @ kq[k0:k1, h].T
            # P against the integer running max (log2 units), as the oracle reads it
            t = s / np.log(2.0)
            p = 2.0 ** (t - np.ceil(t.max(axis=1, keepdims=True)))
            l = p.sum(axis=1, keepdims=True)
            blk_amax = np.maximum.reduceat(p, np.arange(0, p.shape[1], 32), axis=1)
            sc = 2.0 ** M.block_exponent(blk_amax)
            sc = np.repeat(sc, 32, axis=1)[:, :p.shape[1]]
            dp = np.maximum(2.0 ** -4 * p, 2.0 ** -10 * sc)
            bound = (dp @ np.abs(vq[k0:k1, h])) / l
            err = np.abs(out[q0:q1, h] - ref[q0:q1, h])
            assert np.all(err <= bound + 1e-12)
            assert err.max() > 0  # P's quantisation is visible


def test_backward_against_plain_gradients_on_quantised_inputs():
    """Backward vs the fp64 oracle's plain gradients on the quantised Q, K, V, dO:
    they differ only by the quantisation of P (in dV) and dS (in dQ, dK), within
    the bounds that per-element errors of max(2^-4 |x|, 2^-10 * block scale)
    give; with P and dS exactly representable they would agree."""
    bt = W.random_batch(7, [45, 70], [130, 33], 2, 64, dtype=torch.float64)
    q, k, v, do = (bt[n].numpy() for n in ("q", "k", "v", "dout"))
    dq, dk, dv = M.backward(bt["q_off"], bt["kv_off"], q, k, v, do)
    qq, kq, vq, dq_ = (M.qdq_jagged(t, o) for t, o in ((q, bt["q_off"]), (k, bt["kv_off"]), (v, bt["kv_off"]),
                                                      (do, bt["q_off"])))
    out_mx, _ = M.forward(bt["q_off"], bt["kv_off"], q, k, v)
    scale = 1.0 / np.sqrt(64)

    def err_bound(x):  # per element, 32 x 32 blocks
        out = np.empty_like(x)
        for r in range(0, x.shape[0], 32):
            for c in range(0, x.shape[1], 32):
                xb = x[r:r + 32, c:c + 32]
                sc = 2.0 ** M.block_exponent(np.abs(xb).max())
                out[r:r + 32, c:c + 32] = np.maximum(2.0 ** -4 * np.abs(xb), 2.0 ** -10 * sc)
        return out

    for b in range(2):
        q0, q1 = bt["q_off"][b], bt["q_off"][b + 1]
        k0, k1 = bt["kv_off"][b], bt["kv_off"][b + 1]
        for h in range(2):
            s = scale * qq[q0:q1, h] @ kq[k0:k1, h].T
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            delta = np.sum(do[q0:q1, h] * out_mx[q0:q1, h], axis=1, keepdims=True)
            ds = p * (dq_[q0:q1, h] @ vq[k0:k1, h].T - delta)
            # plain products of the unquantised P and dS
            dv_p = p.T @ dq_[q0:q1, h]
            dq_p = scale * ds @ kq[k0:k1, h]
            dk_p = scale * ds.T @ qq[q0:q1, h]
            ep, eds = err_bound(p), err_bound(ds)
            assert np.all(np.abs(dv[k0:k1, h] - dv_p) <= ep.T @ np.abs(dq_[q0:q1, h]) + 1e-12)
            assert np.all(np.abs(dq[q0:q1, h] - dq_p) <= scale * eds @ np.abs(kq[k0:k1, h]) + 1e-12)
            assert np.all(np.abs(dk[k0:k1, h] - dk_p) <= scale * eds.T @ np.abs(qq[q0:q1, h]) + 1e-12)


def _single_key_ratio(qq_rows, kq_row, scale):
    """The forward's one-key factor P_q / p (see test_single_key_closed_form)."""
    t = (qq_rows @ kq_row) * scale / np.log(2.0)
    p = 2.0 ** (t - np.ceil(t))
    e = np.where(p < 1.0, -9.0, -8.0)
    return M.quantize_e4m3(p * 2.0 ** -e) * 2.0 ** e / p


def test_backward_single_key_closed_form():
    """One key: the backward P = exp(s - lse) = 1 exactly, so dV is the sum of
    the quantised dO rows.  The forward's O is r v_q with r = P_q / p (the
    one-key factor of the forward), so dS_i = dP_i - Delta_i =
    dO_q,i . v_q - r_i dO_i . v_q; dQ_i = scale * dS_q,i k_q and
    dK = scale * sum_i dS_q,i q_q,i with dS quantised in 32 x 32 blocks (here
    32 x 1)."""
    bt = W.random_batch(8, [5, 40], [1, 1], 2, 64, dtype=torch.float64)
    q, k, v, do = (bt[n].numpy() for n in ("q", "k", "v", "dout"))
    dq, dk, dv = M.backward(bt["q_off"], bt["kv_off"], q, k, v, do)
    qq = M.qdq_jagged(q, bt["q_off"])
    kq, vq = M.qdq_jagged(k, bt["kv_off"]), M.qdq_jagged(v, bt["kv_off"])
    doq = M.qdq_jagged(do, bt["q_off"])
    scale = 1.0 / 8.0
    for b, (q0, q1) in enumerate(((0, 5), (5, 45))):
        for h in range(2):
            r = _single_key_ratio(qq[q0:q1, h], kq[b, h], scale)
            ds = doq[q0:q1, h] @ vq[b, h] - r * (do[q0:q1, h] @ vq[b, h])  # [Lq]
            dsq = M.qdq_rows_cols(ds[:, None], 32, 32)[:, 0]
            np.testing.assert_allclose(dv[b, h], doq[q0:q1, h].sum(axis=0), rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(dq[q0:q1, h], scale * dsq[:, None] * kq[b, h][None, :], rtol=1e-12,
                                       atol=1e-15)
            np.testing.assert_allclose(dk[b, h], scale * dsq @ qq[q0:q1, h], rtol=1e-12, atol=1e-15)
            assert np.abs(ds).max() > 0 and np.abs(ds).max() < 0.2 * np.abs(doq[q0:q1, h] @ vq[b, h]).max()
