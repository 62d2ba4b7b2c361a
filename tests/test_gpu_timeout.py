"""Bounded waits that run out: with a wait budget of one clock cycle
(CF_WAIT_TIMEOUT_CYCLES, read by the library at every call) the first wait
that is not already satisfied gives up, the kernel records the timeout in
the device status word and every role leaves its loop.  The MMAs and TMA
loads already in flight are drained (with a budget of their own) before
TMEM is freed and the CTA exits.  The host then reads CF_ERR_TIMEOUT from
cf_last_device_status, and the next call on the same context, with the
default budget, must match the oracle.

No wait is made endless and nothing faults on purpose: a timeout is the
bounded wait's ordinary error status.  The configurations: one CTA per
tile and the attention and MLP kernels, whose CTAs wait for their own
in-flight loads exactly, and CTA pairs, whose loads complete on the pair
leader's barrier (both CTAs settle after the cluster barrier)."""
import math

import numpy as np
import pytest
import torch

from back_gemm_fusion_gb300 import inputs as I
from oracle import cf_oracle as O
from tests.parity import assert_rows_close
from tests.test_gpu_b2b import _abs_bound, b2b_gate

pytestmark = pytest.mark.gpu

CF_ERR_TIMEOUT = 6


@pytest.fixture(scope="module")
def cf():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from back_gemm_fusion_gb300 import build
    build.build()
    import back_gemm_fusion_gb300 as cf
    return cf


def _timed_out(cf, monkeypatch, call):
    """Run `call` with a one-cycle wait budget; return the device status."""
    assert cf.cf_last_device_status() == 0  # nothing pending from earlier calls
    monkeypatch.setenv("CF_WAIT_TIMEOUT_CYCLES", "1")
    try:
        call()
        torch.cuda.synchronize()
    finally:
        monkeypatch.delenv("CF_WAIT_TIMEOUT_CYCLES")
    return cf.cf_last_device_status()


@pytest.mark.parametrize("M,N,exchange", [(384, 2048, "global"), (384, 256, "auto"), (512, 2048, "global"),
                                          (512, 256, "auto")])
def test_gemm_epilogue_timeout_then_parity(cf, monkeypatch, M, N, exchange):
    # Three row strips (an odd count): one CTA per tile, with the workspace
    # exchange across 8 tiles per row, or a single tile per row.  Four strips:
    # CTA pairs, likewise.
    case = I.gemm_epilogue_case("timeout", M, N, 1024, [("bias",), ("layernorm", 1e-5)], seed=N,
                                need_bias=True, need_gamma=True, need_beta=True)
    A, B = case.A.cuda(), case.B.cuda()
    vec = [t.cuda() for t in (case.bias, case.gamma, case.beta)]
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = _timed_out(cf, monkeypatch, lambda: cf.cf_gemm_epilogue(A, B, case.ops, *vec, out=out, exchange=exchange))
    assert st == CF_ERR_TIMEOUT
    cf.cf_gemm_epilogue(A, B, case.ops, *vec, out=out, exchange=exchange)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta))
    assert_rows_close(out.cpu().numpy(), ref, what=f"after a timeout, {M}x{N} {exchange}")


@pytest.mark.parametrize("key_split", [1, 4])
def test_attention_timeout_then_parity(cf, monkeypatch, key_split):
    rng = np.random.default_rng(12)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()
    Q, K, V = t(rng.standard_normal((2, 256, 128))), t(rng.standard_normal((2, 2048, 128))), \
        t(rng.standard_normal((2, 2048, 128)))
    scale = 1 / math.sqrt(128)
    out = torch.empty((2, 256, 128), dtype=torch.float32, device="cuda")
    run = lambda: cf.cf_b2bgemm(Q, K, V, "scale_softmax", scale, w1_trans=True, out=out, key_split=key_split)
    assert _timed_out(cf, monkeypatch, run) == CF_ERR_TIMEOUT
    run()
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    got = out.cpu().numpy()
    q, k, v = (I.to_f64(x.cpu()) for x in (Q, K, V))
    for b in range(2):
        ref = O.b2bgemm(q[b], k[b].T, v[b], "scale_softmax", scale)
        b2b_gate(got[b], ref, _abs_bound(q[b], k[b], v[b], "scale_softmax", scale),
                 f"attention after a timeout, key split {key_split}, b={b}")


def test_mlp_timeout_then_parity(cf, monkeypatch):
    # N2 = 256: one CTA per cluster (no S' copies between CTAs).
    rng = np.random.default_rng(13)
    t = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()
    X = t(rng.standard_normal((384, 512)))
    W1 = t(rng.standard_normal((512, 1024)) / math.sqrt(512))
    W2 = t(rng.standard_normal((1024, 256)) / math.sqrt(1024))
    out = torch.empty((384, 256), dtype=torch.float32, device="cuda")
    run = lambda: cf.cf_b2bgemm(X, W1, W2, "relu", out=out)
    assert _timed_out(cf, monkeypatch, run) == CF_ERR_TIMEOUT
    run()
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    x, w1, w2 = (I.to_f64(t.cpu()) for t in (X, W1, W2))
    ref = O.b2bgemm(x, w1, w2, "relu")
    b2b_gate(out.cpu().numpy(), ref, np.abs(O.mid_op(x @ w1, "relu")) @ np.abs(w2), "mlp after a timeout")
