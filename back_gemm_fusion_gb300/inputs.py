"""Seeded synthetic inputs for the fused GEMM-epilogue and B2BGEMM workloads.

This module only draws random numbers and converts dtypes: it holds none of
the fused method's arithmetic.  The same bytes go to the CUDA path and to the
float64 oracle (which receives them as numpy arrays).

Recipe (one ``numpy.random.default_rng(seed)`` PCG64 stream per workload,
draws in a fixed order): the first matrix operand (A, X or Q), then the second
(B, W1 or K), then the third (W2 or V), then bias, gamma, beta.  Each draw is
``standard_normal(shape) * sigma`` in float64; matrix operands are converted
to bfloat16 (round to nearest even), vectors to float32.  ``N(0, v)`` in a
workload's text names the *variance* v, so sigma = sqrt(v); gamma is
``1 + N(0, 0.1)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


@dataclass
class GemmEpilogueCase:
    """One GEMM + epilogue problem: A (M x K) bf16, B (K x N) bf16 row-major."""

    name: str
    M: int
    N: int
    K: int
    ops: List[Tuple]  # ("bias",), ("gelu_tanh",), ("rmsnorm", eps) ...
    A: torch.Tensor = None
    B: torch.Tensor = None
    bias: Optional[torch.Tensor] = None
    gamma: Optional[torch.Tensor] = None
    beta: Optional[torch.Tensor] = None
    residual: Optional[torch.Tensor] = None  # M x N, read by the ("residual",) op
    stage0_gamma: Optional[torch.Tensor] = None  # affine vectors of the first of two row reductions
    stage0_beta: Optional[torch.Tensor] = None
    meta: Dict = field(default_factory=dict)


def gemm_epilogue_case(name: str, M: int, N: int, K: int, ops: List[Tuple], seed: int = 0,
                       a_var: Optional[float] = None, b_var: Optional[float] = None,
                       vec_var: float = 0.1, need_bias: bool = False,
                       need_gamma: bool = False, need_beta: bool = False) -> GemmEpilogueCase:
    """Draw A, B ~ N(0, 1/K) (unless given) and the epilogue vectors."""
    rng = np.random.default_rng(seed)
    a_sd = math.sqrt(a_var if a_var is not None else 1.0 / K)
    b_sd = math.sqrt(b_var if b_var is not None else 1.0 / K)
    v_sd = math.sqrt(vec_var)
    A = _bf16(rng.standard_normal((M, K)) * a_sd)
    B = _bf16(rng.standard_normal((K, N)) * b_sd)
    bias = _f32(rng.standard_normal(N) * v_sd) if need_bias else None
    gamma = _f32(1.0 + rng.standard_normal(N) * v_sd) if need_gamma else None
    beta = _f32(rng.standard_normal(N) * v_sd) if need_beta else None
    return GemmEpilogueCase(name, M, N, K, list(ops), A, B, bias, gamma, beta)


# The three GEMM + epilogue workloads, by what they are.
def postnorm_layernorm(seed: int = 0, M: int = 8192, N: int = 4096, K: int = 4096) -> GemmEpilogueCase:
    """Post-norm block: GEMM + bias + residual add + row LayerNorm (eps 1e-5),
    fp32 out; the residual stream R ~ N(0, 1) is bf16 and drawn after the
    vectors."""
    c = gemm_epilogue_case("gemm_bias_residual_layernorm", M, N, K,
                           [("bias",), ("residual",), ("layernorm", 1e-5)], seed,
                           need_bias=True, need_gamma=True, need_beta=True)
    rng = np.random.default_rng([seed, 1])
    c.residual = _bf16(rng.standard_normal((M, N)))
    return c


def column_layernorm(seed: int = 0, M: int = 8192, N: int = 4096, K: int = 4096) -> GemmEpilogueCase:
    """Column reductions: GEMM + bias + LayerNorm down each column (over the
    M = 8192 rows, a batch normalisation of every output feature, eps 1e-5),
    fp32 out; same draws as the GELU + RMSNorm workload's shapes."""
    c = gemm_epilogue_case("gemm_bias_column_layernorm", M, N, K, [("bias",), ("layernorm", 1e-5)], seed,
                           need_bias=True, need_gamma=True, need_beta=True)
    c.meta["axis"] = "col"
    return c


def chained_ln_gelu_rms(seed: int = 0, M: int = 8192, N: int = 4096, K: int = 4096) -> GemmEpilogueCase:
    """Two reduction stages in one epilogue: GEMM + bias + LayerNorm (its own
    gamma0/beta0) + tanh-GELU + RMSNorm (gamma), fp32 out; the first stage's
    vectors are drawn after the others, like the bias/gamma/beta."""
    c = gemm_epilogue_case("gemm_bias_layernorm_gelu_rmsnorm", M, N, K,
                           [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)], seed,
                           need_bias=True, need_gamma=True)
    rng = np.random.default_rng([seed, 2])
    c.stage0_gamma = _f32(1.0 + rng.standard_normal(N) * math.sqrt(0.1))
    c.stage0_beta = _f32(rng.standard_normal(N) * math.sqrt(0.1))
    return c


def layernorm_256(seed: int = 0, M: int = 256, N: int = 256, K: int = 256) -> GemmEpilogueCase:
    """GEMM + bias + row LayerNorm (eps 1e-5), fp32 out; 256^3 by default."""
    return gemm_epilogue_case("gemm_bias_layernorm", M, N, K,
                              [("bias",), ("layernorm", 1e-5)], seed,
                              need_bias=True, need_gamma=True, need_beta=True)


def gelu_rmsnorm(seed: int = 0, M: int = 8192, N: int = 4096, K: int = 4096) -> GemmEpilogueCase:
    """GEMM + bias + tanh-GELU + row RMSNorm (eps 1e-6), fp32 out."""
    return gemm_epilogue_case("gemm_bias_gelu_rmsnorm", M, N, K,
                              [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)], seed,
                              need_bias=True, need_gamma=True)


def scaled_softmax(seed: int = 0, M: int = 4096, N: int = 16384, K: int = 4096) -> GemmEpilogueCase:
    """GEMM + scale 1/sqrt(K) + row softmax (a logit head), fp32 out."""
    return gemm_epilogue_case("gemm_scaled_softmax", M, N, K,
                              [("scale", 1.0 / math.sqrt(K)), ("softmax",)], seed)


@dataclass
class B2BCase:
    """O = F(A . W1) . W2 per batch entry; A: [b, M, K], W1: [b, K, N1] or its
    transpose (``w1_k_major``: W1 stored as [b, N1, K]), W2: [b, N1, N2]."""

    name: str
    batch: int
    M: int
    K: int
    N1: int
    N2: int
    op: str
    scale: float
    w1_k_major: bool
    A: torch.Tensor = None
    W1: torch.Tensor = None
    W2: torch.Tensor = None


def mlp_b2b(seed: int = 0, M: int = 16384, K: int = 1024, N1: int = 4096, N2: int = 1024) -> B2BCase:
    """X (M x K) ~ N(0,1); W1 (K x N1) ~ N(0, 1/K); W2 (N1 x N2) ~ N(0, 1/N1); ReLU."""
    rng = np.random.default_rng(seed)
    X = _bf16(rng.standard_normal((1, M, K)))
    W1 = _bf16(rng.standard_normal((1, K, N1)) / math.sqrt(K))
    W2 = _bf16(rng.standard_normal((1, N1, N2)) / math.sqrt(N1))
    return B2BCase("b2b_mlp_relu", 1, M, K, N1, N2, "relu", 1.0, False, X, W1, W2)


def mlp_bottom(seed: int = 0, rows: int = 64, K: int = 512, N1: int = 128, N2: int = 256) -> B2BCase:
    """The small-batch bottom-MLP regime of the B2BGEMM evaluation: feature
    dims 512 -> 128 -> 256 (in the order the evaluation lists them), ReLU,
    ``rows`` = batch in 1..64; same draws as mlp_b2b."""
    c = mlp_b2b(seed, M=rows, K=K, N1=N1, N2=N2)
    c.name = "b2b_mlp_bottom_relu"
    return c


def attention_b2b(seed: int = 0, batch: int = 32, heads: int = 16, L: int = 2048, d: int = 128,
                  op: str = "scale_softmax") -> B2BCase:
    """Q, K, V [batch*heads, L, d] ~ N(0, 1); S = Q K^T / sqrt(d); F = softmax or ReLU."""
    rng = np.random.default_rng(seed)
    bh = batch * heads
    Q = _bf16(rng.standard_normal((bh, L, d)))
    Kt = _bf16(rng.standard_normal((bh, L, d)))
    V = _bf16(rng.standard_normal((bh, L, d)))
    return B2BCase(f"b2b_attention_{op}", bh, L, d, L, d, op, 1.0 / math.sqrt(d), True, Q, Kt, V)


def target_attention(seed: int = 0, batch: int = 64, targets: int = 512, behaviours: int = 200, d: int = 128,
                     op: str = "scale_softmax") -> B2BCase:
    """Target-attention-like short key sequences: per batch entry, ``targets``
    query rows attend over ``behaviours`` keys/values (a short behaviour
    sequence, not a multiple of 128); Q, K, V ~ N(0, 1), scale 1/sqrt(d)."""
    rng = np.random.default_rng(seed)
    Q = _bf16(rng.standard_normal((batch, targets, d)))
    Kt = _bf16(rng.standard_normal((batch, behaviours, d)))
    V = _bf16(rng.standard_normal((batch, behaviours, d)))
    return B2BCase(f"b2b_target_attention_{op}", batch, targets, d, behaviours, d, op, 1.0 / math.sqrt(d), True,
                   Q, Kt, V)


def attention_long_keys(seed: int = 0, heads: int = 8, queries: int = 128, keys: int = 16384, d: int = 128,
                        op: str = "scale_softmax") -> B2BCase:
    """Few query rows over a long key sequence (one 128-query block per head,
    a prefill chunk or decode batch against a long context): Q, K, V ~ N(0, 1),
    scale 1/sqrt(d).  With fewer query blocks than SMs this is the shape the
    key-range split across a cluster is for."""
    rng = np.random.default_rng(seed)
    Q = _bf16(rng.standard_normal((heads, queries, d)))
    Kt = _bf16(rng.standard_normal((heads, keys, d)))
    V = _bf16(rng.standard_normal((heads, keys, d)))
    return B2BCase(f"b2b_attention_long_keys_{op}", heads, queries, d, keys, d, op, 1.0 / math.sqrt(d), True,
                   Q, Kt, V)


def to_f64(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Exact float64 copy of a bf16/fp32 CPU tensor (for the oracle)."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
