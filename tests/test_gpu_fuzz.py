"""GPU parity on seeded random shapes: both entry points against the float64
oracle, with the shape, the program, the B layout, the reduction axis, the
row-statistics exchange and the key split drawn at random (fixed seeds, so
every run checks the same cases).  Each case stays small enough for the
oracle to finish in well under a second."""
import math

import numpy as np
import pytest
import torch

from oracle import cf_oracle as O
from back_gemm_fusion_gb300 import inputs as I
from tests.parity import assert_rows_close
from tests.test_gpu_b2b import _abs_bound, b2b_gate

pytestmark = pytest.mark.gpu

PROGRAMS = [
    [],
    [("bias",)],
    [("scale", 0.37)],
    [("bias",), ("relu",)],
    [("bias",), ("gelu_tanh",)],
    [("bias",), ("layernorm", 1e-5)],
    [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
    [("scale", 0.125), ("softmax",)],
    [("bias",), ("residual",), ("layernorm", 1e-5)],
    [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)],
    [("rmsnorm", 1e-6), ("scale", 1.5), ("softmax",)],
]


@pytest.fixture(scope="module")
def cf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from back_gemm_fusion_gb300 import build
    build.build()
    import back_gemm_fusion_gb300 as cf
    return cf


def _draw_gemm_case(i):
    rng = np.random.default_rng(1000 + i)
    ops = PROGRAMS[int(rng.integers(len(PROGRAMS)))]
    rowops = [o for o in ops if o[0] in ("layernorm", "rmsnorm", "softmax")]
    axis = "col" if rowops and len(rowops) == 1 and rng.random() < 0.45 else "row"
    M = int(rng.integers(1, 700))
    N = int(8 * rng.integers(1, 326))  # 16-byte row pitch of B and of the output
    K = int(8 * rng.integers(8, 97))   # 64 .. 768, a multiple of 8
    b_trans = True if axis == "col" else bool(rng.random() < 0.5)
    red_len = M if axis == "col" else N
    exchanges = ["auto", "global"]
    if len(rowops) == 1 and red_len <= 4096:
        exchanges.append("cluster")
    if len(rowops) == 1 and axis == "row":
        exchanges.append("global_dynamic")
    exchange = exchanges[int(rng.integers(len(exchanges)))]
    return ops, axis, M, N, K, b_trans, exchange


@pytest.mark.parametrize("i", range(24))
def test_gemm_epilogue_random_shapes(cf, i):
    ops, axis, M, N, K, b_trans, exchange = _draw_gemm_case(i)
    case = I.gemm_epilogue_case("fuzz", M, N, K, ops, seed=2000 + i, need_bias=True, need_gamma=True,
                                need_beta=True)
    rng = np.random.default_rng(3000 + i)
    R = None
    if any(o[0] == "residual" for o in ops):
        R = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32))
    B = case.B.t().contiguous() if b_trans else case.B
    out = cf.cf_gemm_epilogue(case.A.cuda(), B.cuda(), case.ops, case.bias.cuda(), case.gamma.cuda(),
                              case.beta.cuda(), b_trans=b_trans, exchange=exchange, axis=axis,
                              residual=None if R is None else R.cuda())
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), residual=I.to_f64(R), axis=axis)
    got = out.cpu().numpy()
    what = f"case {i}: {ops} {axis} {M}x{N}x{K} b_trans={b_trans} {exchange}"
    if axis == "col":
        assert_rows_close(np.ascontiguousarray(got.T), np.ascontiguousarray(ref.T), what=what)
    else:
        assert_rows_close(got, ref, what=what)


def _t(a):
    return torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("i", range(10))
def test_attention_random_shapes(cf, i):
    rng = np.random.default_rng(4000 + i)
    batch = int(rng.integers(1, 4))
    Lq = int(rng.integers(1, 400))
    N1 = int(rng.integers(1, 1500))
    dk = int(8 * rng.integers(4, 17))   # 32 .. 128
    dv = int(8 * rng.integers(1, 17))   # 8 .. 128
    op = "scale_softmax" if rng.random() < 0.7 else "scale_relu"
    key_split = int(rng.choice([0, 1, 2, 3]))
    scale = 1.0 / math.sqrt(dk)
    Q, K, V = _t(rng.standard_normal((batch, Lq, dk))), _t(rng.standard_normal((batch, N1, dk))), \
        _t(rng.standard_normal((batch, N1, dv)))
    out = cf.cf_b2bgemm(Q.cuda(), K.cuda(), V.cuda(), op, scale, w1_trans=True, key_split=key_split)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    got = out.cpu().numpy()
    for b in range(batch):
        q, k, v = (I.to_f64(x[b]) for x in (Q, K, V))
        ref = O.b2bgemm(q, k.T, v, op, scale)
        b2b_gate(got[b], ref, _abs_bound(q, k, v, op, scale),
                 f"case {i}: {op} batch {b} {Lq}x{N1} d={dk}/{dv} key_split={key_split}")


@pytest.mark.parametrize("i", range(8))
def test_mlp_random_shapes(cf, i):
    rng = np.random.default_rng(5000 + i)
    M = int(rng.integers(1, 700))
    K = int(8 * rng.integers(8, 65))    # 64 .. 512
    N1 = int(8 * rng.integers(1, 163))  # 16-byte row pitch of W1 (K x N1)
    N2 = int(8 * rng.integers(1, 129))  # 16-byte row pitch of W2 and of the output
    op, scale = ("relu", 1.0) if rng.random() < 0.5 else ("scale_relu", 0.6)
    w1_trans = bool(rng.random() < 0.5)
    X = _t(rng.standard_normal((M, K)))
    W1 = _t(rng.standard_normal((K, N1)) / math.sqrt(K))
    W2 = _t(rng.standard_normal((N1, N2)) / math.sqrt(N1))
    W1d = W1.t().contiguous() if w1_trans else W1
    out = cf.cf_b2bgemm(X.cuda(), W1d.cuda(), W2.cuda(), op, scale, w1_trans=w1_trans)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    x, w1, w2 = (I.to_f64(t) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, op, scale)
    bound = np.abs(O.mid_op(x @ w1, op, scale)) @ np.abs(w2)
    b2b_gate(out.cpu().numpy(), ref, bound, f"case {i}: mlp {op} {M}x{K}x{N1}x{N2} trans={w1_trans}")
