"""The host-only cost model (cf_cost_gemm_epilogue / cf_cost_b2bgemm): CPU
tests of its decisions, its calibration against fused and unfused times
measured with bench.py on one GB300 (CUDA-graph replay, L2 flushed, the
unfused launches timed on the device alone), and its basic monotonicity.  The model is a heuristic: the bands are wide."""
import pytest

from back_gemm_fusion_gb300 import binding as B

GELU_RMS = [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)]
SOFTMAX = [("scale", 1 / 64), ("softmax",)]
LN = [("bias",), ("layernorm", 1e-5)]

# (measured fused us, measured unfused us) on one GB300 at 2.07 GHz.
MEASURED = {
    "gelu_rmsnorm": (171.6, 195.8),
    "scaled_softmax": (381.2, 426.7),
    "layernorm_256": (15.7, 12.4),
    "mlp_b2b": (348.3, 219.4),
    "attention_softmax": (788.9, 4203.2),
    "column_layernorm": (209.2, 319.3),
    "chained_ln_gelu_rms": (219.4, 214.1),
}


@pytest.fixture(scope="module")
def lib():
    from back_gemm_fusion_gb300 import build
    build.build()
    return B.load_library()


def _within(pred, meas, tol):
    return abs(pred - meas) <= tol * meas


def test_gemm_epilogue_calibration_and_decisions(lib):
    c2 = B.cf_cost_gemm_epilogue(8192, 4096, 4096, GELU_RMS)
    c3 = B.cf_cost_gemm_epilogue(4096, 16384, 4096, SOFTMAX)
    c1 = B.cf_cost_gemm_epilogue(256, 256, 256, LN)
    for c, key in ((c2, "gelu_rmsnorm"), (c3, "scaled_softmax"), (c1, "layernorm_256")):
        fm, um = MEASURED[key]
        assert _within(c["fused_us"], fm, 0.25), (key, c["fused_us"], fm)
        assert _within(c["unfused_us"], um, 0.25), (key, c["unfused_us"], um)
    assert c2["fused_preferred"] == 1 and c3["fused_preferred"] == 1
    assert c1["fused_preferred"] == 0            # a latency case: one tile per CTA, nothing to hide the epilogue
    assert c2["epilogue_hidden"] == 1 and c1["epilogue_hidden"] == 0
    assert c2["flops"] == 2.0 * 8192 * 4096 * 4096
    assert c2["unfused_bytes"] - c2["fused_bytes"] == 8.0 * 8192 * 4096  # the intermediate written and read back


def test_chained_program_prefers_unfused(lib):
    # Two strip-wide exchanges per tile: measured slower fused than unfused.
    c = B.cf_cost_gemm_epilogue(8192, 4096, 4096, [("bias",), ("layernorm", 1e-5), ("gelu_tanh",),
                                                   ("rmsnorm", 1e-6)])
    fm, um = MEASURED["chained_ln_gelu_rms"]
    assert _within(c["fused_us"], fm, 0.25) and _within(c["unfused_us"], um, 0.25)
    assert c["fused_preferred"] == 0


def test_column_reductions(lib):
    c = B.cf_cost_gemm_epilogue(8192, 4096, 4096, LN, b_trans=True, axis="col")
    fm, um = MEASURED["column_layernorm"]
    assert _within(c["fused_us"], fm, 0.25) and _within(c["unfused_us"], um, 0.25)
    assert c["fused_preferred"] == 1
    with pytest.raises(B.CFError):               # B must be given as N x K for columns
        B.cf_cost_gemm_epilogue(8192, 4096, 4096, LN, axis="col")


def test_b2b_calibration_and_decisions(lib):
    mlp = B.cf_cost_b2bgemm(16384, 1024, 4096, 1024, "relu")
    att = B.cf_cost_b2bgemm(2048, 128, 2048, 128, "scale_softmax", 128 ** -0.5, batch=512, w1_trans=True)
    fm, um = MEASURED["mlp_b2b"]
    assert _within(mlp["fused_us"], fm, 0.25) and _within(mlp["unfused_us"], um, 0.25)
    assert mlp["fused_preferred"] == 0           # the fused MLP kernel is slower than cuBLASLt + mid op + cuBLASLt
    fm, um = MEASURED["attention_softmax"]
    assert _within(att["fused_us"], fm, 0.25) and _within(att["unfused_us"], um, 0.25)
    assert att["fused_preferred"] == 1           # S would be 4.3 GB in HBM
    with pytest.raises(B.CFError):               # softmax on the MLP shape: no fused kernel
        B.cf_cost_b2bgemm(1024, 256, 512, 256, "scale_softmax", 0.5)


def test_monotonic_and_device_overrides(lib):
    ks = [64, 256, 1024, 4096, 16384]
    t = [B.cf_cost_gemm_epilogue(4096, 4096, k, GELU_RMS)["fused_us"] for k in ks]
    assert all(a < b for a, b in zip(t, t[1:]))
    # The GEMM hides the epilogue once K is large enough, and not for a tiny K.
    assert B.cf_cost_gemm_epilogue(4096, 4096, 64, GELU_RMS)["epilogue_hidden"] == 0
    assert B.cf_cost_gemm_epilogue(4096, 4096, 4096, GELU_RMS)["epilogue_hidden"] == 1
    base = B.cf_cost_gemm_epilogue(8192, 4096, 4096, GELU_RMS)
    fast = B.cf_cost_gemm_epilogue(8192, 4096, 4096, GELU_RMS, device={"tensor_tflops": 2 * 1908.0})
    assert fast["mainloop_us"] == pytest.approx(base["mainloop_us"] / 2, rel=1e-12)
    assert fast["fused_us"] < base["fused_us"]
    # K below one 64-wide block costs that block's main loop; K % 8 != 0 is refused.
    assert B.cf_cost_gemm_epilogue(256, 256, 16, LN)["mainloop_us"] == \
        pytest.approx(B.cf_cost_gemm_epilogue(256, 256, 64, LN)["mainloop_us"], rel=1e-12)
    with pytest.raises(B.CFError):
        B.cf_cost_gemm_epilogue(256, 256, 60, LN)
    # Rows up to twice the resident CTAs in tiles (304 x 256 = 77,824) are
    # accepted, wider ones refused like the fused call refuses them.
    assert B.cf_cost_gemm_epilogue(1024, 77824, 256, SOFTMAX)["fused_us"] > 0
    with pytest.raises(B.CFError):
        B.cf_cost_gemm_epilogue(1024, 77824 + 256, 256, SOFTMAX)
