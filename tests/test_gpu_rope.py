"""GPU parity of the rotary-embedding path (softmax BlockAttention with RoPE of
Q and K, "Training GEM at LLM scale", section "BlockAttention"): the CUDA path
through jattn_fwd_rope / jattn_bwd_rope against the fp64 oracle's exact
rotate-then-attend, element by element; the identity table against the plain
path bit for bit; run-to-run determinism; the argument checks (activation
mode is refused); and sampled rows of the full-size BlockAttention workload
with a standard frequency table, against the exact rotation."""
import zlib

import numpy as np
import pytest
import torch

import jagged_attention_recommendation_gb300 as J
from jagged_attention_recommendation_gb300 import workloads as W
from oracle import oracle
from tests import parity as PT

pytestmark = pytest.mark.gpu

SOFTMAX, SILU, GELU = W.SOFTMAX, W.SILU, W.GELU_TANH

# (name, lengths, H, D, bias_buckets, act, table kind, extra table rows)
CASES = [
    ("d64_random", [1, 63, 64, 65, 200, 513], 4, 64, 0, SOFTMAX, "random", 5),
    ("d64_bias_exact_rows", [130, 64, 7, 300], 2, 64, 16, SOFTMAX, "random", 0),
    ("d128_standard_bias", [130, 64, 7, 300], 2, 128, 64, SOFTMAX, "standard", 3),
    ("d128_random", [1, 127, 128, 129, 250], 2, 128, 0, SOFTMAX, "random", 0),
    ("d64_short_bias", [100, 257, 33], 2, 64, 8, SOFTMAX, "random", 1),
    ("d128_ragged", [90, 200, 1], 2, 128, 0, SOFTMAX, "random", 2),
    ("d64_long", [1000, 333, 2], 2, 64, 0, SOFTMAX, "standard", 0),
]


def _case(case):
    name, lens, H, D, nb, act, kind, extra = case
    bt = W.random_batch(zlib.crc32(name.encode()) % 10000, lens, lens, H, D, bias_buckets=nb)
    rope = W.rope_table(max(lens) + extra, D, kind, seed=7)
    return bt, act, rope


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rope_parity(case):
    """Against the oracle's exact float64 rotation, then attention."""
    bt, act, rope = _case(case)
    gpu = PT.run_library(bt, act=act, block=64, rope=rope)
    PT.compare(gpu, PT.run_oracle(bt, act=act, block=64, rope=rope))


def test_rope_identity_table_is_plain_path():
    """Angle 0: the rotation maps every bf16 value to itself, so outputs and
    gradients equal the plain BlockAttention path bit for bit."""
    bt = W.random_batch(61, [70, 9, 130, 300], [70, 9, 130, 300], 2, 64, bias_buckets=8)
    rope = W.rope_table(300, 64, "identity")
    a = PT.run_library(bt, block=64, rope=rope)
    b = PT.run_library(bt, block=64)
    for n in ("out", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


def test_rope_differs_from_plain_path():
    """A non-trivial table changes the result (the rotation is really applied)."""
    bt = W.random_batch(62, [70, 130], [70, 130], 2, 64)
    a = PT.run_library(bt, block=64, rope=W.rope_table(130, 64, "random", seed=3))
    b = PT.run_library(bt, block=64)
    assert np.abs(a["out"] - b["out"]).max() > 1e-2
    assert np.abs(a["dq"] - b["dq"]).max() > 1e-2


def test_rope_deterministic():
    bt = W.random_batch(63, [513, 64, 200], [513, 64, 200], 4, 128, bias_buckets=16)
    rope = W.rope_table(513, 128, "random", seed=4)
    a = PT.run_library(bt, block=64, rope=rope)
    b = PT.run_library(bt, block=64, rope=rope)
    for n in ("out", "dq", "dk", "dv"):
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)


def _dev(t):
    return t.to("cuda:0")


def test_rope_argument_checks():
    bt = W.random_batch(64, [40, 100], [40, 100], 2, 64)
    q, k, v = (_dev(bt[n]) for n in ("q", "k", "v"))
    cos, sin = (_dev(t) for t in W.rope_table(100, 64))
    full = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, device=0)
    with pytest.raises(J.JattnError) as e:
        full.fwd(q, k, v, rope=(cos, sin))
    assert e.value.code == J.ERR_UNSUPPORTED
    blk = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, block=64, device=0)
    short = (cos[:99].contiguous(), sin[:99].contiguous())
    with pytest.raises(J.JattnError) as e:
        blk.fwd(q, k, v, rope=short)
    assert e.value.code == J.ERR_INVALID_ARG
    out, lse = blk.fwd(q, k, v, rope=(cos, sin))
    with pytest.raises(J.JattnError) as e:
        blk.bwd(_dev(bt["dout"]), q, k, v, out, lse=lse, rope=short)
    assert e.value.code == J.ERR_INVALID_ARG
    flat_c = torch.zeros(100 * 32 + 1, device="cuda:0")
    with pytest.raises(J.JattnError) as e:  # a table starting 4 bytes off a 16-byte boundary
        blk.fwd(q, k, v, rope=(flat_c[1:].view(100, 32), sin))
    assert e.value.code == J.ERR_ALIGNMENT
    f32 = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, block=64, dtype="fp32", device=0)
    with pytest.raises(J.JattnError) as e:
        f32.fwd(q.float(), k.float(), v.float(), rope=(cos, sin))
    assert e.value.code == J.ERR_UNSUPPORTED
    # activation mode: the rotation is offered with softmax only
    silu = J.Plan(bt["q_off"], bt["kv_off"], 2, 64, act=SILU, block=64, device=0)
    with pytest.raises(J.JattnError) as e:
        silu.fwd(q, k, v, rope=(cos, sin))
    assert e.value.code == J.ERR_UNSUPPORTED
    o_act, _ = silu.fwd(q, k, v)
    with pytest.raises(J.JattnError) as e:
        silu.bwd(_dev(bt["dout"]), q, k, v, o_act, rope=(cos, sin))
    assert e.value.code == J.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    for p in (full, blk, f32, silu):
        assert p.check_status() == 0
        p.close()


def test_rope_full_size_block_workload_sampled():
    """The full-size BlockAttention workload (B=64, H=8, D=64, lengths up to
    16384) with a standard table, in the launch configuration the bench times;
    sampled sequences checked against the oracle."""
    b = W.make_batch(5)
    w = b.w
    lens = np.diff(b.q_off.astype(np.int64))
    rope = W.rope_table(int(lens.max()), w.D, "standard")
    bt = dict(q_off=b.q_off, kv_off=b.kv_off, q=b.q, k=b.k, v=b.v, bias=b.bias, dout=b.dout, scale=b.scale)
    gpu = PT.run_library(bt, block=w.block, rope=rope)
    for n in ("out", "dq", "dk", "dv"):
        assert np.isfinite(gpu[n]).all(), n
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 7, 33})
    qo, ko, (q, dout), (k, v), qidx, kidx = oracle.sub_batch(b.q_off, b.kv_off, seqs, b.q, b.dout,
                                                             tensors_kv=(b.k, b.v))
    sub = dict(q_off=qo, kv_off=ko, q=q, k=k, v=v, bias=b.bias, dout=dout, scale=b.scale)
    ref = PT.run_oracle(sub, block=w.block, rope=rope)
    PT.assert_close(gpu["out"][qidx], ref["out"], PT.FWD_TOL, "out")
    PT.assert_close(gpu["dq"][qidx], ref["dq"], PT.BWD_TOL, "dq")
    PT.assert_close(gpu["dk"][kidx], ref["dk"], PT.BWD_TOL, "dk")
    PT.assert_close(gpu["dv"][kidx], ref["dv"], PT.BWD_TOL, "dv")
