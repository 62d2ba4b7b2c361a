"""cf_gemm_epilogue_noalloc: the fused GEMM + epilogue for callers that cannot
allocate device memory (latency-bound code, plugins without an allocator,
steady-state loops that must not allocate).  It takes the scratch for
partial row statistics from the library's own static device array instead
of a caller workspace.  This file is collected last on purpose.

Each GPU case runs the call twice in a row (the array keeps the previous
call's contents) and checks both results against the float64 oracle and
against the workspace entry point, which runs the same kernel with the same
launch decisions and must give the same bits."""
import ctypes

import numpy as np
import pytest
import torch

from back_gemm_fusion_gb300 import inputs as I
from oracle import cf_oracle as O
from tests.parity import assert_rows_close, sample_rows

LIMIT = 4 << 20  # CF_NOALLOC_WORKSPACE_BYTES


def _lib():
    from back_gemm_fusion_gb300 import build
    build.build()
    from back_gemm_fusion_gb300 import binding
    return binding


def test_noalloc_rejects_problems_beyond_the_static_array():
    b = _lib()
    lib = b.load_library()
    # Softmax over 8192 x 32768: its scratch (8 MiB + counters) exceeds the 4 MiB array.
    A = b.cf_matrix(0x10000, b.CF_BF16, 0, 8192, 256, 256)
    B = b.cf_matrix(0x20000, b.CF_BF16, 0, 256, 32768, 32768)
    O_ = b.cf_matrix(0x30000, b.CF_FP32, 0, 8192, 32768, 32768)
    d = b.epi_desc([("softmax",)])
    assert lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B), ctypes.byref(d)) > LIMIT
    st = lib.cf_gemm_epilogue_noalloc(ctypes.byref(A), ctypes.byref(B), None, None, None, ctypes.byref(d),
                                      ctypes.byref(O_), None)
    assert st == 7  # CF_ERR_WORKSPACE, before anything touches the device
    # Two chained reductions need one statistics region each, so the limit
    # halves: 8192 x 8192 fits with one stage but not with two.
    B2 = b.cf_matrix(0x20000, b.CF_BF16, 0, 256, 8192, 8192)
    O2 = b.cf_matrix(0x30000, b.CF_FP32, 0, 8192, 8192, 8192)
    one = b.epi_desc([("softmax",)])
    two = b.epi_desc([("layernorm", 1e-5), ("softmax",)])
    assert lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B2), ctypes.byref(one)) <= LIMIT
    assert lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B2), ctypes.byref(two)) > LIMIT
    st = lib.cf_gemm_epilogue_noalloc(ctypes.byref(A), ctypes.byref(B2), None, None, None, ctypes.byref(two),
                                      ctypes.byref(O2), None)
    assert st == 7


@pytest.mark.gpu
@pytest.mark.parametrize("N,exchange,ops", [
    (4352, "auto", [("scale", 0.25), ("softmax",)]),             # 17 tiles: wider than a cluster
    (1024, "global", [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)]),
    (2048, "global", [("bias",), ("layernorm", 1e-5)]),
])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(N, exchange, ops):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b = _lib()
    case = I.gemm_epilogue_case("noalloc", 256, N, 192, ops, seed=N, need_bias=True, need_gamma=True,
                                need_beta=True)
    A, B = case.A.cuda(), case.B.cuda()
    vec = [None if t is None else t.cuda() for t in (case.bias, case.gamma, case.beta)]
    ws_out = b.cf_gemm_epilogue(A, B, case.ops, *vec, exchange=exchange)
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta))
    out = torch.empty((256, N), dtype=torch.float32, device="cuda")
    for call in range(2):  # the array keeps the previous call's contents
        out.fill_(float("nan"))
        b.cf_gemm_epilogue_noalloc(A, B, case.ops, *vec, out=out, exchange=exchange)
        torch.cuda.synchronize()
        assert b.cf_last_device_status() == 0
        assert_rows_close(out.cpu().numpy(), ref, what=f"noalloc call {call} vs oracle")
        assert torch.equal(out, ws_out), f"noalloc call {call} differs from the workspace entry point"


@pytest.mark.gpu
def test_noalloc_chained_reductions_twice():
    # Two reduction stages: the second statistics region starts right after
    # the first inside the static array.
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b = _lib()
    M, N = 384, 2048
    ops = [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)]
    case = I.gemm_epilogue_case("noalloc_chain", M, N, 128, ops, seed=21, need_bias=True, need_gamma=True)
    rng = np.random.default_rng(22)
    g0 = torch.from_numpy((1 + 0.3 * rng.standard_normal(N)).astype(np.float32)).cuda()
    b0 = torch.from_numpy((0.3 * rng.standard_normal(N)).astype(np.float32)).cuda()
    A, B, bias, gamma = case.A.cuda(), case.B.cuda(), case.bias.cuda(), case.gamma.cuda()
    ws_out = b.cf_gemm_epilogue(A, B, case.ops, bias, gamma, None, stage0_gamma=g0, stage0_beta=b0)
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          None, stage0_gamma=I.to_f64(g0.cpu()), stage0_beta=I.to_f64(b0.cpu()))
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for call in range(2):
        out.fill_(float("nan"))
        b.cf_gemm_epilogue_noalloc(A, B, case.ops, bias, gamma, None, out=out, stage0_gamma=g0, stage0_beta=b0)
        torch.cuda.synchronize()
        assert b.cf_last_device_status() == 0
        assert_rows_close(out.cpu().numpy(), ref, what=f"noalloc chained call {call}")
        assert torch.equal(out, ws_out), f"noalloc chained call {call} differs from the workspace entry point"


@pytest.mark.gpu
def test_noalloc_column_reduction_twice():
    # LayerNorm down the columns over M = 4104 rows (17 tiles down each
    # column: the workspace exchange on P^T), B given as N x K.
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b = _lib()
    M, N, K = 4104, 256, 64
    ops = [("bias",), ("layernorm", 1e-5)]
    case = I.gemm_epilogue_case("noalloc_col", M, N, K, ops, seed=23, need_bias=True, need_gamma=True,
                                need_beta=True)
    A, Bt = case.A.cuda(), case.B.t().contiguous().cuda()
    vec = [t.cuda() for t in (case.bias, case.gamma, case.beta)]
    ws_out = b.cf_gemm_epilogue(A, Bt, case.ops, *vec, b_trans=True, axis="col")
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), axis="col")
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for call in range(2):
        out.fill_(float("nan"))
        b.cf_gemm_epilogue_noalloc(A, Bt, case.ops, *vec, out=out, b_trans=True, axis="col")
        torch.cuda.synchronize()
        assert b.cf_last_device_status() == 0
        got = out.cpu().numpy()
        assert_rows_close(np.ascontiguousarray(got.T), np.ascontiguousarray(ref.T),
                          what=f"noalloc columns call {call}")
        assert torch.equal(out, ws_out), f"noalloc column call {call} differs from the workspace entry point"


@pytest.mark.gpu
def test_noalloc_near_the_limit_twice():
    # Scratch just under the 4 MiB array: softmax over 8192 x 16128 (63 tiles
    # per row, 64 strips), so the counters sit at the array's far end.
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b = _lib()
    M, N, K = 8192, 16128, 64
    ops = [("scale", 0.5), ("softmax",)]
    case = I.gemm_epilogue_case("noalloc_limit", M, N, K, ops, seed=24)
    A, B = case.A.cuda(), case.B.cuda()
    need = b.cf_workspace_size(A, B, case.ops)
    assert 0.95 * LIMIT < need <= LIMIT
    ws_out = b.cf_gemm_epilogue(A, B, case.ops)
    torch.cuda.synchronize()
    rows = sample_rows(M, 64, seed=24)
    ref = O.gemm_epilogue(I.to_f64(case.A)[rows], I.to_f64(case.B), case.ops)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for call in range(2):
        out.fill_(float("nan"))
        b.cf_gemm_epilogue_noalloc(A, B, case.ops, out=out)
        torch.cuda.synchronize()
        assert b.cf_last_device_status() == 0
        assert_rows_close(out[rows].cpu().numpy(), ref, what=f"noalloc near the limit, call {call}")
        assert torch.equal(out, ws_out), f"noalloc near-limit call {call} differs from the workspace entry point"
