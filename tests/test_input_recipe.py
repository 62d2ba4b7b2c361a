"""The seeded synthetic input recipe (CPU): determinism, the documented draw
order and distributions (N(0, v) names the variance v), and bf16 rounding of
the matrix operands."""
import math

import numpy as np
import torch

from back_gemm_fusion_gb300 import inputs as I


def test_deterministic_and_seed_dependent():
    a = I.gemm_epilogue_case("x", 64, 256, 128, [("bias",), ("layernorm", 1e-5)], seed=3, need_bias=True,
                             need_gamma=True, need_beta=True)
    b = I.gemm_epilogue_case("x", 64, 256, 128, [("bias",), ("layernorm", 1e-5)], seed=3, need_bias=True,
                             need_gamma=True, need_beta=True)
    c = I.gemm_epilogue_case("x", 64, 256, 128, [("bias",), ("layernorm", 1e-5)], seed=4, need_bias=True,
                             need_gamma=True, need_beta=True)
    for k in ("A", "B", "bias", "gamma", "beta"):
        assert torch.equal(getattr(a, k), getattr(b, k))
        assert not torch.equal(getattr(a, k), getattr(c, k))


def test_draw_order_and_rounding():
    # A first, then B, then bias, gamma, beta, each standard_normal * sigma
    # from one PCG64 stream; matrices rounded to bf16, vectors to fp32.
    M, N, K = 32, 256, 64
    c = I.gemm_epilogue_case("x", M, N, K, [], seed=11, need_bias=True, need_gamma=True, need_beta=True)
    rng = np.random.default_rng(11)
    A = rng.standard_normal((M, K)) / math.sqrt(K)
    B = rng.standard_normal((K, N)) / math.sqrt(K)
    bias = rng.standard_normal(N) * math.sqrt(0.1)
    gamma = 1.0 + rng.standard_normal(N) * math.sqrt(0.1)
    beta = rng.standard_normal(N) * math.sqrt(0.1)
    assert c.A.dtype == torch.bfloat16 and c.bias.dtype == torch.float32
    assert torch.equal(c.A, torch.from_numpy(A.astype(np.float32)).to(torch.bfloat16))
    assert torch.equal(c.B, torch.from_numpy(B.astype(np.float32)).to(torch.bfloat16))
    assert torch.equal(c.bias, torch.from_numpy(bias.astype(np.float32)))
    assert torch.equal(c.gamma, torch.from_numpy(gamma.astype(np.float32)))
    assert torch.equal(c.beta, torch.from_numpy(beta.astype(np.float32)))


def test_documented_distributions():
    # Variances, not standard deviations: A, B ~ N(0, 1/K), bias ~ N(0, 0.1).
    c = I.gemm_epilogue_case("x", 512, 1024, 256, [], seed=0, need_bias=True, need_gamma=True)
    assert abs(c.A.float().std().item() - 1 / math.sqrt(256)) < 0.002
    assert abs(c.bias.std().item() - math.sqrt(0.1)) < 0.03
    assert abs(c.gamma.mean().item() - 1.0) < 0.05
    mlp = I.mlp_b2b(M=256, K=512, N1=256, N2=256)
    assert abs(mlp.A.float().std().item() - 1.0) < 0.02                    # X ~ N(0, 1)
    assert abs(mlp.W1.float().std().item() - 1 / math.sqrt(512)) < 0.002   # weights ~ N(0, 1/fan_in)
    att = I.target_attention(batch=2)
    assert att.M == 512 and att.N1 == 200 and att.K == 128 and att.w1_k_major
    assert abs(att.scale - 1 / math.sqrt(128)) < 1e-15
