"""cf_gemm_epilogue_noalloc: the fused GEMM + epilogue for callers that cannot
allocate device memory (latency-bound code, plugins without an allocator,
steady-state loops that must not allocate).  It takes the scratch for
partial row statistics from the library's own static device array instead
of a caller workspace.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from back_gemm_fusion_gb300 import inputs as I
from tests.parity import assert_rows_close

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
    O = b.cf_matrix(0x30000, b.CF_FP32, 0, 8192, 32768, 32768)
    d = b.epi_desc([("softmax",)])
    assert lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B), ctypes.byref(d)) > LIMIT
    st = lib.cf_gemm_epilogue_noalloc(ctypes.byref(A), ctypes.byref(B), None, None, None, ctypes.byref(d),
                                      ctypes.byref(O), None)
    assert st == 7  # CF_ERR_WORKSPACE, before anything touches the device


@pytest.mark.gpu
@pytest.mark.parametrize("N,exchange,ops", [
    (4352, "auto", [("scale", 0.25), ("softmax",)]),             # 17 tiles: wider than a cluster
    (1024, "global", [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)]),
    (2048, "global", [("bias",), ("layernorm", 1e-5)]),
])
def test_noalloc_matches_workspace_entry_point_twice(N, exchange, ops):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    b = _lib()
    case = I.gemm_epilogue_case("noalloc", 256, N, 192, ops, seed=N, need_bias=True, need_gamma=True,
                                need_beta=True)
    A, B = case.A.cuda(), case.B.cuda()
    vec = [None if t is None else t.cuda() for t in (case.bias, case.gamma, case.beta)]
    ref = b.cf_gemm_epilogue(A, B, case.ops, *vec, exchange=exchange)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    out = torch.empty((256, N), dtype=torch.float32, device="cuda")
    for call in range(2):  # the array keeps the previous call's contents
        out.fill_(float("nan"))
        b.cf_gemm_epilogue_noalloc(A, B, case.ops, *vec, out=out, exchange=exchange)
        torch.cuda.synchronize()
        assert b.cf_last_device_status() == 0
        got = out.cpu().numpy()
        assert_rows_close(got, ref, what=f"noalloc call {call} vs workspace entry point")
