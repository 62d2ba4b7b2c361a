"""GPU parity of the unfused comparison path (cuBLASLt GEMM -> HBM
intermediate -> separate epilogue / mid-op kernel), so the fused-vs-unfused
numbers compare two correct implementations."""

import numpy as np
import pytest
import torch

from oracle import cf_oracle as O
from back_gemm_fusion_gb300 import inputs as I
from tests.parity import assert_rows_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from back_gemm_fusion_gb300 import build
    build.build()
    import back_gemm_fusion_gb300 as cf
    return cf


@pytest.mark.parametrize("N", [256, 1024, 4096])
@pytest.mark.parametrize("rowop", ["layernorm", "rmsnorm", "softmax"])
def test_unfused_gemm_epilogue(cf, N, rowop):
    ops = {"layernorm": [("bias",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 1 / 16), ("softmax",)]}[rowop]
    case = I.gemm_epilogue_case(rowop, 256, N, 256, ops, seed=N, need_bias=True, need_gamma=True, need_beta=True)
    vec = [None if t is None else t.cuda() for t in (case.bias, case.gamma, case.beta)]
    out = cf.cf_unfused_gemm_epilogue(case.A.cuda(), case.B.cuda(), case.ops, *vec)
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta))
    assert_rows_close(out.cpu().numpy(), ref, what=f"unfused {rowop} N={N}")


@pytest.mark.parametrize("res_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N", [512, 4096])
def test_unfused_residual(cf, N, res_dtype):
    ops = [("bias",), ("residual",), ("layernorm", 1e-5)]
    case = I.gemm_epilogue_case("res", 256, N, 256, ops, seed=N + 1, need_bias=True, need_gamma=True, need_beta=True)
    R = torch.from_numpy(np.random.default_rng(N).standard_normal((256, N)).astype(np.float32)).to(res_dtype)
    vec = [t.cuda() for t in (case.bias, case.gamma, case.beta)]
    out = cf.cf_unfused_gemm_epilogue(case.A.cuda(), case.B.cuda(), case.ops, *vec, residual=R.cuda())
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), residual=I.to_f64(R))
    assert_rows_close(out.cpu().numpy(), ref, what=f"unfused residual N={N} {res_dtype}")


@pytest.mark.parametrize("op", ["scale_softmax", "scale_relu"])
def test_unfused_attention(cf, op):
    case = I.attention_b2b(batch=2, heads=2, L=1024, op=op)
    out = cf.cf_unfused_b2bgemm(case.A.cuda(), case.W1.cuda(), case.W2.cuda(), op, case.scale, w1_trans=True)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for h in range(case.batch):
        q, k, v = (I.to_f64(t[h]) for t in (case.A, case.W1, case.W2))
        ref = O.b2bgemm(q, k.T, v, op, case.scale)
        err = np.abs(got[h] - ref)
        bound = 2.0 ** -7 * (np.abs(O.mid_op(q @ k.T, op, case.scale)) @ np.abs(v)) + 1e-6
        assert np.all(err <= bound), f"unfused attention {op} head {h}: {(err / bound).max():.3g}x"


def test_unfused_mlp(cf):
    case = I.mlp_b2b(M=256, K=256, N1=2048, N2=512)
    out = cf.cf_unfused_b2bgemm(case.A[0].cuda(), case.W1[0].cuda(), case.W2[0].cuda(), "relu")
    torch.cuda.synchronize()
    x, w1, w2 = I.to_f64(case.A[0]), I.to_f64(case.W1[0]), I.to_f64(case.W2[0])
    ref = O.b2bgemm(x, w1, w2, "relu")
    bound = 2.0 ** -7 * (np.abs(np.maximum(x @ w1, 0)) @ np.abs(w2)) + 1e-6
    assert np.all(np.abs(out.cpu().numpy() - ref) <= bound)


def test_unfused_mlp_bf16_output(cf):
    # bf16 output from the second cuBLASLt GEMM (fp32 accumulation, one
    # rounding to nearest even at the store).
    case = I.mlp_b2b(M=256, K=256, N1=1024, N2=512)
    out = torch.empty((256, 512), dtype=torch.bfloat16, device="cuda")
    cf.cf_unfused_b2bgemm(case.A[0].cuda(), case.W1[0].cuda(), case.W2[0].cuda(), "relu", out=out)
    torch.cuda.synchronize()
    x, w1, w2 = I.to_f64(case.A[0]), I.to_f64(case.W1[0]), I.to_f64(case.W2[0])
    ref = O.b2bgemm(x, w1, w2, "relu")
    bound = 2.0 ** -7 * (np.abs(np.maximum(x @ w1, 0)) @ np.abs(w2)) + 2.0 ** -8 * np.abs(ref) * 1.01 + 1e-6
    assert np.all(np.abs(out.float().cpu().numpy() - ref) <= bound)


@pytest.mark.parametrize("N", [264, 1000])
def test_unfused_ragged_n(cf, N):
    ops = [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)]
    case = I.gemm_epilogue_case("ragged", 256, N, 128, ops, seed=N, need_bias=True, need_gamma=True)
    vec = [None if t is None else t.cuda() for t in (case.bias, case.gamma, case.beta)]
    out = cf.cf_unfused_gemm_epilogue(case.A.cuda(), case.B.cuda(), case.ops, *vec)
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          None)
    assert_rows_close(out.cpu().numpy(), ref, what=f"unfused ragged N={N}")


def test_unfused_attention_ragged_keys(cf):
    rng = np.random.default_rng(5)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    Q, K, V = t(rng.standard_normal((2, 256, 64))), t(rng.standard_normal((2, 200, 64))), \
        t(rng.standard_normal((2, 200, 64)))
    out = cf.cf_unfused_b2bgemm(Q.cuda(), K.cuda(), V.cuda(), "scale_softmax", 0.125, w1_trans=True)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for h in range(2):
        q, k, v = (I.to_f64(x[h]) for x in (Q, K, V))
        ref = O.b2bgemm(q, k.T, v, "scale_softmax", 0.125)
        bound = 2.0 ** -7 * (np.abs(O.mid_op(q @ k.T, "scale_softmax", 0.125)) @ np.abs(v)) + 1e-6
        assert np.all(np.abs(got[h] - ref) <= bound)


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("M,N", [(512, 256), (1000, 200), (4104, 64)])
@pytest.mark.parametrize("prog", ["layernorm", "rmsnorm", "softmax", "chained"])
def test_unfused_column_reductions(cf, prog, M, N, b_trans):
    # The unfused column path: cuBLASLt GEMM, then one CTA per 32 columns
    # (ragged N, long columns, either B layout, chained stages).
    ops = {"layernorm": [("bias",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("residual",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 0.5), ("softmax",)],
           "chained": [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)]}[prog]
    case = I.gemm_epilogue_case("col_unfused", M, N, 128, ops, seed=M + N, need_bias=True, need_gamma=True,
                                need_beta=True)
    rng = np.random.default_rng(M)
    R = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    g0 = torch.from_numpy((1 + 0.3 * rng.standard_normal(N)).astype(np.float32))
    b0 = torch.from_numpy((0.3 * rng.standard_normal(N)).astype(np.float32))
    B = case.B.t().contiguous() if b_trans else case.B
    vec = [None if t is None else t.cuda() for t in (case.bias, case.gamma, case.beta)]
    kw = {"stage0_gamma": g0.cuda(), "stage0_beta": b0.cuda()} if prog == "chained" else {}
    out = cf.cf_unfused_gemm_epilogue(case.A.cuda(), B.cuda(), case.ops, *vec, b_trans=b_trans, axis="col",
                                      residual=R.cuda() if prog == "rmsnorm" else None, **kw)
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), residual=I.to_f64(R) if prog == "rmsnorm" else None,
                          stage0_gamma=I.to_f64(g0) if prog == "chained" else None,
                          stage0_beta=I.to_f64(b0) if prog == "chained" else None, axis="col")
    assert_rows_close(np.ascontiguousarray(out.cpu().numpy().T), np.ascontiguousarray(ref.T),
                      what=f"unfused columns {prog} {M}x{N}")
