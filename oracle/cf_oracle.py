"""Oracle for the fused GEMM-epilogue and back-to-back GEMM hot path.

TEST INFRASTRUCTURE ONLY.  This module is a plain, slow, obviously correct
CPU restatement in float64 of what the fused kernels compute.  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it.  It shares no code with the CUDA path and imports nothing from
the product package: inputs arrive as numpy arrays.

Source of the method: the Pith review of "ComFuse: Fusing Complex
Memory-Intensive Subgraphs with Compute-Intensive Kernels For Modern GPU
Architectures" (arXiv 2608.03537).

* "What carries the argument": the GEMM output P is streamed tile by tile
  through elementwise nodes, and each reduction is a stage boundary that
  aggregates along one logical dimension only.
* Referee report, major comment 1 [Sec. III, Eq. (1)]: the reduction runs
  along the second (column) dimension of P, so each output row depends only on
  its own row strip.
* "If this is right", first bullet: the epilogues named are LayerNorm,
  RMSNorm and softmax.
* "What carries the argument" and major comment 2 [Sec. IV-A, Eqs. (3)-(5)]:
  B2BGEMM computes GEMM1, applies an elementwise/reduction op F to the
  intermediate S and feeds the result to GEMM2 without materialising it.

The fused method reaches exactly the plain definition (only the rounding order
of the float arithmetic differs), so every function below is that definition
written out:

1. P = A . B, summed exactly enough in float64 (no bf16 rounding of P: the
   kernels accumulate in fp32 and never round P).
2. Elementwise ops in descriptor order (bias, scale, ReLU, tanh-GELU, and
   the residual add x + R[m, n] of the "post-norm" MatMul + Add + norm
   subgraphs the evaluation fuses).
3. Row reductions (LayerNorm, RMSNorm, softmax), each a stage boundary: a
   program is elementwise nodes, a reduction, and optionally more elementwise
   nodes and a second reduction that ends it (the Stage-Stream model's chain
   of stages; the kernels support up to two).  The same reductions down the
   columns of P (along its first dimension, the complementary strip of major
   comment 1) are the ``col_*`` functions.
4. For B2BGEMM the single rounding point is the intermediate S' = F(S), which
   is rounded to bfloat16 round-to-nearest-even before the second GEMM.

Readings where the pages are silent (each is listed in the design notes):
LayerNorm uses the biased (1/N) variance with eps inside the square root;
RMSNorm has no mean subtraction and no beta; tanh-GELU is the usual
0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))); the attention softmax rounds
the *normalised* probabilities to bf16.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
closed forms, invariants, exact rational brute force, and library routines in
special cases.  Nothing here is "parity unpinned".
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np

__all__ = [
    "BF16_MAX",
    "bf16_round",
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "matmul",
    "elementwise",
    "row_layernorm",
    "row_rmsnorm",
    "row_softmax",
    "col_layernorm",
    "col_rmsnorm",
    "col_softmax",
    "gemm_epilogue",
    "mid_op",
    "b2bgemm",
    "attention",
]

# Largest finite bfloat16: (2 - 2^-7) * 2^127.
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
# Smallest positive (subnormal) bfloat16: 2^-133 (8-bit exponent like fp32,
# 7 stored mantissa bits, so the subnormal quantum is 2^(-126-7)).
_BF16_MIN_SUB = 2.0 ** -133


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16, ties to even.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the fp32
    exponent range.  A normal value x = m * 2^e with 0.5 <= |m| < 1 therefore
    has quantum q = 2^(e-8); below 2^-126 the quantum is fixed at 2^-133.
    x / q is rounded to the nearest integer, halves to the even integer
    (numpy's rint), and scaled back.  Results beyond the largest finite
    bfloat16 after rounding become +-inf; NaN stays NaN; -0 stays -0.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    _, e = np.frexp(xf)  # xf = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)  # 2^-126 = 0.5 * 2^-125: below it the quantum is fixed
    q = np.ldexp(1.0, e - 8)
    r = np.rint(xf / q) * q  # exact: xf / q and the product are exact in fp64
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, xf), r)
    out[finite] = r
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode IEEE bfloat16 bit patterns (uint16) to float64, exactly.

    Layout: bit 15 sign, bits 14..7 biased exponent (bias 127), bits 6..0
    mantissa.  Exponent 0 is zero/subnormal, exponent 255 is inf/NaN.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    ex = (b >> 7) & 0xFF
    man = (b & 0x7F).astype(np.float64)
    normal = sign * np.ldexp(1.0 + man / 128.0, (ex - 127).astype(np.int64))
    sub = sign * np.ldexp(man / 128.0, -126)
    special = np.where(man == 0, sign * np.inf, np.nan)
    return np.where(ex == 0, sub, np.where(ex == 255, special, normal))


def f64_to_bf16_bits(x) -> np.ndarray:
    """Encode float64 values as bfloat16 bit patterns after RNE rounding."""
    r = bf16_round(x)
    out = np.zeros(r.shape, dtype=np.uint16)
    flat_r = r.reshape(-1)
    flat_o = out.reshape(-1)
    for i, v in enumerate(flat_r):
        if math.isnan(v):
            flat_o[i] = 0x7FC0
            continue
        s = 0x8000 if math.copysign(1.0, v) < 0 else 0
        a = abs(v)
        if a == math.inf:
            flat_o[i] = s | 0x7F80
        elif a == 0.0:
            flat_o[i] = s
        elif a < 2.0 ** -126:
            flat_o[i] = s | int(round(a / _BF16_MIN_SUB))
        else:
            m, e = math.frexp(a)  # a = m 2^e, m in [0.5, 1)
            ex = e - 1 + 127
            man = int(round((m * 2.0 - 1.0) * 128.0))
            flat_o[i] = s | (ex << 7) | man
    return out


def matmul(A, B) -> np.ndarray:
    """P[m, n] = sum_k A[m, k] B[k, n] in float64 (a library primitive).

    The inputs are bf16 values (exact in float64); products are exact in
    float64 and only the float64 summation rounds.
    """
    return np.asarray(A, dtype=np.float64) @ np.asarray(B, dtype=np.float64)


def _gelu_tanh(x: np.ndarray) -> np.ndarray:
    c = math.sqrt(2.0 / math.pi)
    return 0.5 * x * (1.0 + np.tanh(c * (x + 0.044715 * x ** 3)))


def elementwise(x: np.ndarray, op: str, scalar: float = 0.0, bias=None, residual=None) -> np.ndarray:
    """One elementwise epilogue node, applied per element of a row strip.

    ``bias`` adds bias[n] along the column index; ``residual`` adds the
    matrix R[m, n] of the same shape (the residual stream of a post-norm
    block); ``scale`` multiplies by the scalar; ``relu`` is max(x, 0);
    ``gelu_tanh`` is the tanh approximation of GELU.
    """
    if op == "bias":
        return x + np.asarray(bias, dtype=np.float64)[None, :]
    if op == "residual":
        r = np.asarray(residual, dtype=np.float64)
        if r.shape != x.shape:
            raise ValueError("the residual must have the shape of the GEMM output")
        return x + r
    if op == "scale":
        return x * float(scalar)
    if op == "relu":
        return np.maximum(x, 0.0)
    if op == "gelu_tanh":
        return _gelu_tanh(x)
    raise ValueError(f"unknown elementwise op {op!r}")


def row_layernorm(x, gamma, beta, eps: float) -> np.ndarray:
    """LayerNorm along each row: mean, then the biased variance of x - mean.

    y[m, n] = gamma[n] (x[m, n] - mu_m) / sqrt(var_m + eps) + beta[n].
    """
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    g = np.asarray(gamma, dtype=np.float64)[None, :]
    b = np.asarray(beta, dtype=np.float64)[None, :]
    return g * (x - mu) / np.sqrt(var + eps) + b


def row_rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """RMSNorm along each row: y = gamma[n] x / sqrt(mean(x^2) + eps)."""
    x = np.asarray(x, dtype=np.float64)
    ms = (x * x).mean(axis=1, keepdims=True)
    return np.asarray(gamma, dtype=np.float64)[None, :] * x / np.sqrt(ms + eps)


def row_softmax(x) -> np.ndarray:
    """Softmax along each row: exp(x - max) / sum(exp(x - max))."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def col_layernorm(x, gamma, beta, eps: float) -> np.ndarray:
    """LayerNorm down each column: the reduction along the first dimension of
    P (referee report, major comment 1 [Sec. III, Eq. (1)]: such reductions
    need the complementary strip, the column of tiles T_{m,n} over m).  Mean
    and biased variance over m; the affine vectors stay indexed by the column
    (a per-feature scale and shift, as for a batch normalisation):

    y[m, n] = gamma[n] (x[m, n] - mu_n) / sqrt(var_n + eps) + beta[n].
    """
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=0, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=0, keepdims=True)
    g = np.asarray(gamma, dtype=np.float64)[None, :]
    b = np.asarray(beta, dtype=np.float64)[None, :]
    return g * (x - mu) / np.sqrt(var + eps) + b


def col_rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """RMSNorm down each column: y = gamma[n] x / sqrt(mean_m(x^2) + eps)."""
    x = np.asarray(x, dtype=np.float64)
    ms = (x * x).mean(axis=0, keepdims=True)
    return np.asarray(gamma, dtype=np.float64)[None, :] * x / np.sqrt(ms + eps)


def col_softmax(x) -> np.ndarray:
    """Softmax down each column: exp(x - max_m) / sum_m exp(x - max_m)."""
    x = np.asarray(x, dtype=np.float64)
    e = np.exp(x - x.max(axis=0, keepdims=True))
    return e / e.sum(axis=0, keepdims=True)


_ROW_OPS = ("layernorm", "rmsnorm", "softmax")


def _apply_program(x, ops: Sequence[tuple], bias, gamma, beta, residual=None, stage0_gamma=None,
                   stage0_beta=None, axis: str = "row") -> np.ndarray:
    """Run an epilogue program: elementwise nodes and reductions in order.

    ``ops`` is a sequence of ``(name,)`` or ``(name, scalar)`` tuples; the
    scalar is the scale for ``scale`` and eps for the norms.  At most two
    reductions, and if there is one the program ends with a reduction.  The
    last reduction uses ``gamma`` / ``beta``; an earlier one uses
    ``stage0_gamma`` / ``stage0_beta`` (None: 1 and 0, no affine transform).
    ``axis="row"`` reduces along each row, ``axis="col"`` down each column
    (every vector is indexed by the column in both cases).
    """
    if axis not in ("row", "col"):
        raise ValueError("axis is 'row' or 'col'")
    norms = {"row": (row_layernorm, row_rmsnorm, row_softmax), "col": (col_layernorm, col_rmsnorm, col_softmax)}
    layernorm, rmsnorm, softmax = norms[axis]
    names = [o[0] for o in ops]
    row_at = [i for i, n in enumerate(names) if n in _ROW_OPS]
    if len(row_at) > 2 or (row_at and row_at[-1] != len(names) - 1):
        raise ValueError("at most two row reductions, the last one ending the program")
    N = x.shape[1]
    for i, op in enumerate(ops):
        name = op[0]
        scalar = op[1] if len(op) > 1 else 0.0
        if name in _ROW_OPS:
            last = i == len(names) - 1
            g = gamma if last else (np.ones(N) if stage0_gamma is None else stage0_gamma)
            b = beta if last else (np.zeros(N) if stage0_beta is None else stage0_beta)
            if name == "layernorm":
                x = layernorm(x, g, b, scalar)
            elif name == "rmsnorm":
                x = rmsnorm(x, g, scalar)
            else:
                x = softmax(x)
        else:
            x = elementwise(x, name, scalar, bias, residual)
    return x


def gemm_epilogue(A, B, ops: Iterable[tuple], bias=None, gamma=None, beta=None, residual=None,
                  stage0_gamma=None, stage0_beta=None, axis: str = "row") -> np.ndarray:
    """GEMM followed by an epilogue program, all in float64.

    A: M x K, B: K x N (row-major, bf16 values as float64); ``residual``
    (M x N) is read by the ``residual`` op; ``stage0_gamma`` / ``stage0_beta``
    are the affine vectors of the first of two reductions; ``axis`` picks
    row reductions (over n) or column reductions (over m).  Returns M x N.
    """
    return _apply_program(matmul(A, B), list(ops), bias, gamma, beta, residual, stage0_gamma, stage0_beta, axis)


def mid_op(S, op: str, scale: float = 1.0) -> np.ndarray:
    """The op F between the two GEMMs of a B2BGEMM.

    ``relu``: max(S, 0) (no scale).  ``scale_relu``: max(scale S, 0).
    ``scale_softmax``: row softmax of scale S.
    """
    S = np.asarray(S, dtype=np.float64)
    if op == "relu":
        return np.maximum(S, 0.0)
    if op == "scale_relu":
        return np.maximum(scale * S, 0.0)
    if op == "scale_softmax":
        return row_softmax(scale * S)
    raise ValueError(f"unknown mid op {op!r}")


def b2bgemm(A, W1, W2, op: str, scale: float = 1.0, round_intermediate: bool = True) -> np.ndarray:
    """O = bf16(F(A . W1)) . W2 with A: M x K, W1: K x N1, W2: N1 x N2.

    The intermediate F(S) is rounded to bf16 (RNE) exactly once, which is the
    precision policy of the fused kernel (bf16 operands for the second GEMM,
    fp32 accumulation).  ``round_intermediate=False`` gives the unrounded
    product, used only by pins that compare with library routines.
    """
    Sp = mid_op(matmul(A, W1), op, scale)
    if round_intermediate:
        Sp = bf16_round(Sp)
    return matmul(Sp, W2)


def attention(Q, K, V, op: str, scale: float, round_intermediate: bool = True) -> np.ndarray:
    """Attention-shaped B2BGEMM per (batch, head): O = bf16(F(Q K^T)) V.

    Q, K: [..., L, d], V: [..., L, dv].  F is ``scale_softmax`` or
    ``scale_relu``; there is no mask.  Leading axes are independent problems.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    lead = Q.shape[:-2]
    out = np.empty(lead + (Q.shape[-2], V.shape[-1]), dtype=np.float64)
    for idx in np.ndindex(*lead):
        out[idx] = b2bgemm(Q[idx], K[idx].T, V[idx], op, scale, round_intermediate)
    return out
