"""The workspace exchange's two schedules.

Static (the default): a CTA takes fixed tiles in strip-major order.  Tickets
(CF_XCHG_GLOBAL_DYNAMIC, and rows wider than the CTAs): tiles are claimed
from a counter by the CTAs that run, so a launch whose grid cannot all be
resident (another kernel holds some SMs) still finishes its strips with the
running CTAs.  A long attention call on a second stream holds 40 SMs (one
CTA per query block, about 16 ms); the GEMM epilogue runs on a third stream
with a wait budget of about 2 ms.  Items owned in advance by CTAs that
cannot start until the attention call ends would leave their strip-mates
waiting past that budget; with tickets the running CTAs take every item and
the late ones find none left."""
import math

import numpy as np
import pytest
import torch

from back_gemm_fusion_gb300 import inputs as I
from oracle import cf_oracle as O
from tests.parity import assert_rows_close, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from back_gemm_fusion_gb300 import build
    build.build()
    import back_gemm_fusion_gb300 as cf
    return cf


@pytest.mark.parametrize("M,N,K,ops", [
    (2048, 4096, 1024, [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)]),   # CTA pairs, 16 tiles per strip pair
    (1920, 8192, 512, [("scale", 0.125), ("softmax",)]),                   # 15 strips: one CTA per tile
])
def test_workspace_exchange_with_sms_held_elsewhere(cf, monkeypatch, M, N, K, ops):
    rng = np.random.default_rng(M + N)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()
    # The other kernel: 40 query blocks over 2^21 keys shared by all of them
    # (batch stride 0 for K and V), one CTA per block.
    heads, keys = 40, 1 << 21
    Qa = t(rng.standard_normal((heads, 128, 128)))
    Ka = t(rng.standard_normal((1, keys, 128))).expand(heads, keys, 128)
    Va = t(rng.standard_normal((1, keys, 128))).expand(heads, keys, 128)
    Oa = torch.empty((heads, 128, 128), dtype=torch.float32, device="cuda")
    case = I.gemm_epilogue_case("tickets", M, N, K, ops, seed=M, need_bias=True, need_gamma=True, need_beta=True)
    A, B = case.A.cuda(), case.B.cuda()
    vec = [t_.cuda() for t_ in (case.bias, case.gamma, case.beta)]
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    need = cf.cf_workspace_size(A, B, case.ops, exchange="global_dynamic")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    s_other, s_fused = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s_other):
        cf.cf_b2bgemm(Qa, Ka, Va, "scale_softmax", 1 / math.sqrt(128), w1_trans=True, out=Oa, key_split=1)
    monkeypatch.setenv("CF_WAIT_TIMEOUT_CYCLES", "4000000")  # about 2 ms at 2 GHz
    try:
        with torch.cuda.stream(s_fused):
            cf.cf_gemm_epilogue(A, B, case.ops, *vec, out=out, workspace=ws, exchange="global_dynamic")
    finally:
        monkeypatch.delenv("CF_WAIT_TIMEOUT_CYCLES")
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    rows = sample_rows(M, 64, seed=1)
    ref = O.gemm_epilogue(I.to_f64(case.A)[rows], I.to_f64(case.B), case.ops, I.to_f64(case.bias),
                          I.to_f64(case.gamma), I.to_f64(case.beta))
    assert_rows_close(out[rows].cpu().numpy(), ref, what=f"workspace exchange beside another kernel {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,exchange", [
    (8192, 4096, 1024, "global_dynamic"),  # tickets, CTA pairs, about 7 items per pair
    (8192, 4096, 1024, "global"),          # the static order on the same shape
    (256, 25600, 128, "global"),           # one strip pair of 100 tiles over 76 pairs: tickets
    (384, 51200, 64, "global"),            # three strips of 200 tiles over 152 one-CTA workers: tickets
])
def test_workers_holding_two_tiles_of_a_strip(cf, M, N, K, exchange):
    # With tickets a worker may hold two tiles of the same strip; it
    # publishes the second tile's statistics while the first waits for its
    # strip.  Rows wider than the workers take tickets under the plain
    # workspace exchange too.  The call must finish (no bounded wait gives
    # up) and match the oracle, on every one of several back-to-back calls.
    ops = [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)] if N <= 4096 else [("scale", 0.25), ("softmax",)]
    case = I.gemm_epilogue_case("two_tiles", M, N, K, ops, seed=N, need_bias=True, need_gamma=True)
    A, B = case.A.cuda(), case.B.cuda()
    vec = [None if t_ is None else t_.cuda() for t_ in (case.bias, case.gamma, case.beta)]
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    for _ in range(4):
        cf.cf_gemm_epilogue(A, B, case.ops, *vec, out=out, exchange=exchange)
        torch.cuda.synchronize()
        assert cf.cf_last_device_status() == 0
    rows = sample_rows(M, 48, seed=2)
    ref = O.gemm_epilogue(I.to_f64(case.A)[rows], I.to_f64(case.B), case.ops, I.to_f64(case.bias),
                          I.to_f64(case.gamma), I.to_f64(case.beta))
    assert_rows_close(out[rows].cpu().numpy(), ref, what=f"two tiles of a strip per worker {M}x{N}x{K}")


@pytest.mark.parametrize("M,N", [(256, 8192), (512, 12288)])
def test_chained_static_order_wide_rows(cf, M, N):
    # Chained programs keep the static order: a strip's tiles must not
    # outnumber the workers (32 and 48 tiles per strip pair on 76 pairs).
    ops = [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)]
    case = I.gemm_epilogue_case("chain_wide", M, N, 128, ops, seed=N, need_bias=True, need_gamma=True)
    A, B = case.A.cuda(), case.B.cuda()
    out = cf.cf_gemm_epilogue(A, B, case.ops, case.bias.cuda(), case.gamma.cuda(), None)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    rows = sample_rows(M, 48, seed=3)
    ref = O.gemm_epilogue(I.to_f64(case.A)[rows], I.to_f64(case.B), case.ops, I.to_f64(case.bias),
                          I.to_f64(case.gamma), None)
    assert_rows_close(out[rows].cpu().numpy(), ref, what=f"chained wide rows {M}x{N}")


def test_row_width_limit(cf):
    # The widest rows the workspace exchange accepts: 304 tiles per strip on
    # one-CTA workers (one strip, an odd count), twice the 152 workers of a
    # 152-SM GB300: N = 77,824 runs (claimed items, two tiles of the strip per
    # worker) and matches the oracle; one tile more is refused on the host.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, K = 128, 64
    N = 2 * sms * 256
    ops = [("scale", 0.125), ("softmax",)]
    case = I.gemm_epilogue_case("widest", M, N, K, ops, seed=5)
    A, B = case.A.cuda(), case.B.cuda()
    out = cf.cf_gemm_epilogue(A, B, case.ops)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    rows = sample_rows(M, 24, seed=4)
    ref = O.gemm_epilogue(I.to_f64(case.A)[rows], I.to_f64(case.B), case.ops, None, None, None)
    assert_rows_close(out[rows].cpu().numpy(), ref, what=f"softmax over {N} columns")
    wider = I.gemm_epilogue_case("too_wide", M, N + 256, K, ops, seed=6)
    with pytest.raises(cf.CFError):
        cf.cf_gemm_epilogue(wider.A.cuda(), wider.B.cuda(), wider.ops)
