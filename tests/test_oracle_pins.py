"""Pins for the float64 oracle: closed forms, invariants, exact brute force and
library routines in special cases.  CPU only (``-m "not gpu"``).

Every part of the oracle is pinned by something other than itself, chosen so a
plausible mistake (a dropped term, a wrong sign or index, a transposed operand,
the unbiased variance, eps outside the root, a wrong GELU constant, the wrong
bf16 tie rule) fails at least one test here; ``test_oracle_mutations`` plants
such mistakes in the oracle and checks that they are caught.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import cf_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- hand example
def _hand():
    with open(os.path.join(GOLDEN, "hand_2x3x4.json")) as f:
        return json.load(f)


def test_hand_example_gemm_exact():
    h = _hand()
    P = O.matmul(np.array(h["A"], float), np.array(h["B"], float))
    assert P.tolist() == h["P"]


def test_hand_example_epilogues():
    h = _hand()
    A = np.array(h["A"], float)
    B = np.array(h["B"], float)
    for key, ops in (("layernorm_eps0", [("layernorm", 0.0)]),
                     ("rmsnorm_eps0", [("rmsnorm", 0.0)]),
                     ("softmax", [("softmax",)]),
                     ("gelu_tanh", [("gelu_tanh",)])):
        exp = np.array([[_closed(v) for v in row] for row in h[key]], float)
        got = O.gemm_epilogue(A, B, ops, gamma=np.ones(4), beta=np.zeros(4))
        np.testing.assert_allclose(got[: exp.shape[0]], exp, rtol=0, atol=1e-12, err_msg=key)


def test_hand_example_bias_and_scale():
    # Bias along the column index and a non-power-of-two scale: exact dyadic
    # values written by hand.  The square 4 x 4 product makes a bias indexed
    # by the row broadcast silently instead of failing, so it must fail here.
    h = _hand()
    A = np.array(h["A"], float)
    B = np.array(h["B"], float)
    bias = np.array(h["bias"], float)
    assert O.gemm_epilogue(A, B, [("bias",)], bias=bias).tolist() == h["P_plus_bias"]
    A_sq = np.array(h["A_sq"], float)
    assert O.matmul(A_sq, B).tolist() == h["P_sq"]
    assert O.gemm_epilogue(A_sq, B, [("bias",)], bias=bias).tolist() == h["P_sq_plus_bias"]
    assert O.gemm_epilogue(A, B, [("scale", h["scale"])]).tolist() == h["P_times_scale"]
    # Bias then LayerNorm, scale then softmax: closed forms in the golden file.
    for key, ops in (("bias_layernorm_eps0", [("bias",), ("layernorm", 0.0)]),
                     ("scale_softmax", [("scale", h["scale"]), ("softmax",)])):
        exp = np.array([[_closed(v) for v in row] for row in h[key]], float)
        got = O.gemm_epilogue(A, B, ops, bias=bias, gamma=np.ones(4), beta=np.zeros(4))
        np.testing.assert_allclose(got, exp, rtol=0, atol=1e-12, err_msg=key)


def test_bias_scale_brute_force_fraction():
    # Exact rational evaluation of (P + bias[n]) * s on a small non-square
    # shape with dyadic inputs: every value is exact in float64.
    rng = np.random.default_rng(11)
    M, K, N = 5, 4, 6
    A = rng.integers(-9, 10, (M, K)) / 4.0
    B = rng.integers(-9, 10, (K, N)) / 8.0
    bias = rng.integers(-9, 10, N) / 2.0
    s = Fraction(3, 8)
    P = _frac_matmul(A.tolist(), B.tolist())
    exact = [[(P[m][n] + Fraction(bias[n])) * s for n in range(N)] for m in range(M)]
    got = O.gemm_epilogue(A, B, [("bias",), ("scale", float(s))], bias=bias)
    assert got.tolist() == [[float(v) for v in row] for row in exact]
    # Node order matters: scaling first leaves the bias unscaled.
    exact2 = [[P[m][n] * s + Fraction(bias[n]) for n in range(N)] for m in range(M)]
    got2 = O.gemm_epilogue(A, B, [("scale", float(s)), ("bias",)], bias=bias)
    assert got2.tolist() == [[float(v) for v in row] for row in exact2]


def test_hand_example_b2b_relu_exact():
    h = _hand()
    O_ = O.b2bgemm(np.array(h["A"], float), np.array(h["B"], float),
                   np.array(h["W2"], float), "relu")
    assert O_.tolist() == h["b2b_relu_out"]


def test_hand_example_residual():
    # Residual add: exact integer sums (R is not symmetric, so a transposed
    # or misindexed residual fails), then RMSNorm of the sum.
    h = _hand()
    A = np.array(h["A"], float)
    B = np.array(h["B"], float)
    R = np.array(h["R"], float)
    assert O.gemm_epilogue(A, B, [("residual",)], residual=R).tolist() == h["P_plus_R"]
    exp = np.array([[_closed(v) for v in row] for row in h["residual_rmsnorm_eps0"]], float)
    got = O.gemm_epilogue(A, B, [("residual",), ("rmsnorm", 0.0)], gamma=np.ones(4), residual=R)
    np.testing.assert_allclose(got, exp, rtol=0, atol=1e-12)


def test_residual_order_in_program():
    # With R = -P - 1, residual-then-ReLU is all zeros, while ReLU-then-residual
    # is relu(P) - P - 1: the node order of the program is respected.
    h = _hand()
    A = np.array(h["A"], float)
    B = np.array(h["B"], float)
    P = np.array(h["P"], float)
    R = -P - 1.0
    assert np.all(O.gemm_epilogue(A, B, [("residual",), ("relu",)], residual=R) == 0.0)
    got = O.gemm_epilogue(A, B, [("relu",), ("residual",)], residual=R)
    assert got.tolist() == (np.maximum(P, 0.0) - P - 1.0).tolist()
    with pytest.raises(ValueError):
        O.gemm_epilogue(A, B, [("residual",)], residual=R.T)


def test_chained_reductions_hand_example():
    h = _hand()
    A = np.array(h["A"], float)
    B = np.array(h["B"], float)
    ln = np.array([[_closed(v) for v in row] for row in h["layernorm_eps0"]], float)
    ones, zeros = np.ones(4), np.zeros(4)
    # LayerNorm rows have mean 0 and mean square 1, so RMSNorm leaves them unchanged.
    got = O.gemm_epilogue(A, B, [("layernorm", 0.0), ("rmsnorm", 0.0)], gamma=ones, beta=zeros)
    np.testing.assert_allclose(got, ln, rtol=0, atol=1e-12)
    # Softmax of the LayerNorm rows (closed form in the golden file).
    exp = np.array([[_closed(v) for v in row] for row in h["layernorm_then_softmax"]], float)
    got = O.gemm_epilogue(A, B, [("layernorm", 0.0), ("softmax",)], gamma=ones, beta=zeros)
    np.testing.assert_allclose(got, exp, rtol=0, atol=1e-12)
    # The first reduction's own affine vectors: z = 2 LN + 1 has mean square 5,
    # and the last reduction's gamma (3) scales the result.
    got = O.gemm_epilogue(A, B, [("layernorm", 0.0), ("rmsnorm", 0.0)], gamma=3 * ones, beta=zeros,
                          stage0_gamma=2 * ones, stage0_beta=ones)
    np.testing.assert_allclose(got, 3 * (2 * ln + 1) / math.sqrt(5.0), rtol=0, atol=1e-12)


def test_chained_reductions_rules():
    h = _hand()
    A = np.array(h["A"], float)
    B = np.array(h["B"], float)
    with pytest.raises(ValueError):  # three reductions
        O.gemm_epilogue(A, B, [("layernorm", 0.0), ("rmsnorm", 0.0), ("softmax",)], gamma=np.ones(4),
                        beta=np.zeros(4))
    with pytest.raises(ValueError):  # a reduction that does not end the program
        O.gemm_epilogue(A, B, [("layernorm", 0.0), ("rmsnorm", 0.0), ("relu",)], gamma=np.ones(4),
                        beta=np.zeros(4))


def test_hand_example_column_reductions():
    # Reductions down the columns of P (two rows per column): closed forms
    # from the golden file, including per-column affine vectors.
    h = _hand()
    A = np.array(h["A"], float)
    B = np.array(h["B"], float)
    ones, zeros = np.ones(4), np.zeros(4)
    for key, ops, g, b in (("col_layernorm_eps0", [("layernorm", 0.0)], ones, zeros),
                           ("col_layernorm_affine", [("layernorm", 0.0)], np.array(h["col_layernorm_affine_gamma"]),
                            np.array(h["col_layernorm_affine_beta"])),
                           ("col_rmsnorm_eps0", [("rmsnorm", 0.0)], ones, zeros),
                           ("col_softmax", [("softmax",)], ones, zeros)):
        exp = np.array([[_closed(str(v)) for v in row] for row in h[key]], float)
        got = O.gemm_epilogue(A, B, ops, gamma=g, beta=b, axis="col")
        np.testing.assert_allclose(got, exp, rtol=0, atol=1e-12, err_msg=key)


def test_column_reductions_invariants_and_library():
    rng = np.random.default_rng(77)
    x = rng.standard_normal((37, 9)) * 3 + 1
    np.testing.assert_allclose(O.col_softmax(x).sum(axis=0), np.ones(9), rtol=0, atol=1e-14)
    y = O.col_layernorm(x, np.ones(9), np.zeros(9), 0.0)
    np.testing.assert_allclose(y.mean(axis=0), np.zeros(9), atol=1e-13)
    np.testing.assert_allclose((y ** 2).mean(axis=0), np.ones(9), atol=1e-12)
    r = O.col_rmsnorm(x, np.ones(9), 0.0)
    np.testing.assert_allclose((r ** 2).mean(axis=0), np.ones(9), atol=1e-12)
    # A single row: softmax down a column of one element is 1.
    np.testing.assert_array_equal(O.col_softmax(x[:1]), np.ones((1, 9)))
    # Library routines in float64: softmax along dim 0, and layer_norm of the
    # transposed matrix followed by the per-column affine vectors.
    g, b = rng.standard_normal(9), rng.standard_normal(9)
    t = torch.from_numpy(x)
    np.testing.assert_allclose(O.col_softmax(x), torch.softmax(t, dim=0).numpy(), rtol=1e-13, atol=1e-15)
    ln = torch.nn.functional.layer_norm(t.T, (37,), eps=1e-5).T.numpy() * g[None] + b[None]
    np.testing.assert_allclose(O.col_layernorm(x, g, b, 1e-5), ln, rtol=1e-10, atol=1e-12)
    ms = (t * t).mean(dim=0, keepdim=True)
    np.testing.assert_allclose(O.col_rmsnorm(x, g, 1e-6), (torch.from_numpy(g)[None] * t / torch.sqrt(ms + 1e-6)).numpy(),
                               rtol=1e-13, atol=1e-14)
    with pytest.raises(ValueError):
        O.gemm_epilogue(x[:, :3], np.eye(3), [("softmax",)], axis="diagonal")


def _closed(expr: str) -> float:
    """Evaluate a closed form written in the golden file (sqrt, exp, tanh only)."""
    return float(eval(expr, {"__builtins__": {}},
                      {"sqrt": math.sqrt, "exp": math.exp, "tanh": math.tanh, "pi": math.pi}))


# ------------------------------------------------------------------ invariants
RNG = np.random.default_rng(1234)


def test_softmax_rows_sum_to_one():
    x = RNG.standard_normal((37, 300)) * 5
    y = O.row_softmax(x)
    assert np.all(y > 0)
    assert np.max(np.abs(y.sum(1) - 1.0)) <= 1e-12


def test_softmax_shift_invariance_and_constant_row():
    x = RNG.standard_normal((9, 64))
    c = RNG.standard_normal((9, 1)) * 100
    np.testing.assert_allclose(O.row_softmax(x + c), O.row_softmax(x), rtol=1e-12, atol=1e-15)
    y = O.row_softmax(np.full((3, 40), 7.25))
    assert np.all(y == 1.0 / 40)


def test_softmax_large_logits_do_not_overflow():
    y = O.row_softmax(np.array([[1000.0, 1000.0, 0.0]]))
    np.testing.assert_allclose(y, [[0.5, 0.5, 0.0]], atol=1e-300)


def test_layernorm_mean_zero_var_one_eps0():
    x = RNG.standard_normal((25, 513)) * 3 + 11
    y = O.row_layernorm(x, np.ones(513), np.zeros(513), 0.0)
    assert np.max(np.abs(y.mean(1))) <= 1e-9
    assert np.max(np.abs((y ** 2).mean(1) - 1.0)) <= 1e-9


def test_layernorm_eps_inside_root_closed_form():
    # With gamma=1, beta=0 the normalised variance is var / (var + eps).
    x = RNG.standard_normal((8, 256)) * 0.01
    eps = 1e-5
    y = O.row_layernorm(x, np.ones(256), np.zeros(256), eps)
    var = x.var(axis=1)
    np.testing.assert_allclose((y ** 2).mean(1), var / (var + eps), rtol=1e-10)


def test_layernorm_constant_row_gives_beta():
    beta = RNG.standard_normal(16)
    y = O.row_layernorm(np.full((2, 16), -3.5), RNG.standard_normal(16), beta, 1e-5)
    np.testing.assert_allclose(y, np.broadcast_to(beta, (2, 16)), atol=0)


def test_rmsnorm_mean_square_one_and_scale_invariance():
    x = RNG.standard_normal((12, 777)) + 0.5
    y = O.row_rmsnorm(x, np.ones(777), 0.0)
    assert np.max(np.abs((y ** 2).mean(1) - 1.0)) <= 1e-12
    np.testing.assert_allclose(O.row_rmsnorm(3.7 * x, np.ones(777), 0.0), y, rtol=1e-12)
    # No mean subtraction: a constant positive row maps to all ones.
    np.testing.assert_allclose(O.row_rmsnorm(np.full((1, 5), 2.0), np.ones(5), 0.0), np.ones((1, 5)))


def test_gelu_special_values():
    x = np.array([0.0, 40.0, -40.0])
    y = O.elementwise(x, "gelu_tanh")
    assert y[0] == 0.0 and y[1] == 40.0 and abs(y[2]) < 1e-300
    # Odd part: gelu(x) - gelu(-x) = x.
    z = RNG.standard_normal(100) * 3
    np.testing.assert_allclose(O.elementwise(z, "gelu_tanh") - O.elementwise(-z, "gelu_tanh"), z, atol=1e-14)


# ------------------------------------------------------- library special cases
def test_epilogues_match_torch_float64():
    x = RNG.standard_normal((31, 200)) * 2
    g = 1 + RNG.standard_normal(200) * 0.3
    b = RNG.standard_normal(200) * 0.3
    tx = torch.from_numpy(x)
    tg, tb = torch.from_numpy(g), torch.from_numpy(b)
    F = torch.nn.functional
    np.testing.assert_allclose(O.row_layernorm(x, g, b, 1e-5),
                               F.layer_norm(tx, (200,), tg, tb, 1e-5).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.row_rmsnorm(x, g, 1e-6),
                               F.rms_norm(tx, (200,), tg, 1e-6).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(O.row_softmax(x), torch.softmax(tx, 1).numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(O.elementwise(x, "gelu_tanh"),
                               F.gelu(tx, approximate="tanh").numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(O.elementwise(x, "relu"), F.relu(tx).numpy(), atol=0)
    # Bias along the last (column) dimension, as torch broadcasts a vector;
    # a scale by a non-power-of-two multiplies.
    np.testing.assert_allclose(O.elementwise(x, "bias", bias=b), torch.add(tx, tb).numpy(), rtol=0, atol=0)
    np.testing.assert_allclose(O.elementwise(x, "scale", 0.3), torch.mul(tx, 0.3).numpy(), rtol=0, atol=0)
    sq = x[:, :31]
    np.testing.assert_allclose(O.elementwise(sq, "bias", bias=b[:31]), torch.add(tx[:, :31], tb[:31]).numpy(),
                               rtol=0, atol=0)


def test_attention_unrounded_matches_sdpa():
    q = RNG.standard_normal((3, 64, 16))
    k = RNG.standard_normal((3, 64, 16))
    v = RNG.standard_normal((3, 64, 8))
    got = O.attention(q, k, v, "scale_softmax", 0.25, round_intermediate=False)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=0.25).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_attention_rounding_is_within_bf16_half_ulp_of_unrounded():
    q = RNG.standard_normal((2, 32, 16))
    k = RNG.standard_normal((2, 32, 16))
    v = np.abs(RNG.standard_normal((2, 32, 8)))  # non-negative: bound is sum p|v| 2^-9
    a = O.attention(q, k, v, "scale_softmax", 0.25)
    b = O.attention(q, k, v, "scale_softmax", 0.25, round_intermediate=False)
    assert np.all(np.abs(a - b) <= 2.0 ** -9 * b + 1e-15)
    assert not np.array_equal(a, b)


def test_attention_zero_keys_gives_column_mean_of_v():
    # Q K^T == 0, so P = 1/L = 2^-11 exactly (exact in bf16) and O = mean_j V[j].
    L = 2048
    q = RNG.standard_normal((1, L, 4))
    k = np.zeros((1, L, 4))
    v = RNG.standard_normal((1, L, 3))
    got = O.attention(q, k, v, "scale_softmax", 1 / math.sqrt(128))
    np.testing.assert_allclose(got[0], np.broadcast_to(v[0].mean(0), (L, 3)), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------- brute force exact
def _frac_matmul(A, B):
    M, K = len(A), len(A[0])
    N = len(B[0])
    return [[sum(Fraction(A[m][k]) * Fraction(B[k][n]) for k in range(K)) for n in range(N)]
            for m in range(M)]


@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 2), (8, 8, 8), (7, 3, 6)])
def test_matmul_brute_force_fraction(shape):
    M, K, N = shape
    rng = np.random.default_rng(M * 100 + K * 10 + N)
    A = O.bf16_round(rng.standard_normal((M, K)))
    B = O.bf16_round(rng.standard_normal((K, N)))
    exact = _frac_matmul(A.tolist(), B.tolist())
    got = O.matmul(A, B)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(got[m, n]) - exact[m][n]) <= Fraction(1, 2 ** 50) * (1 + abs(exact[m][n]))
    # Orientation: P[m, n] uses row m of A and column n of B.
    assert got.shape == (M, N)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_b2b_relu_brute_force_with_library_rounding(seed):
    # Dyadic inputs keep S exact in fp32, so torch's fp32->bf16 conversion (RNE,
    # a library routine) rounds the exact S; GEMM2 is then exact in fractions.
    rng = np.random.default_rng(seed)
    M, K, N1, N2 = 5, 7, 6, 4
    A = rng.integers(-40, 41, (M, K)) / 8.0
    W1 = rng.integers(-40, 41, (K, N1)) / 4.0
    W2 = rng.integers(-9, 10, (N1, N2)) / 2.0
    S = _frac_matmul(A.tolist(), W1.tolist())
    relu = [[max(s, Fraction(0)) for s in row] for row in S]
    relu_f32 = torch.tensor([[float(s) for s in row] for row in relu], dtype=torch.float32)
    assert all(Fraction(float(s)) == s for row in relu for s in row)  # exact in fp32
    rounded = relu_f32.to(torch.bfloat16).to(torch.float64).numpy()
    exact = _frac_matmul(rounded.tolist(), W2.tolist())
    got = O.b2bgemm(A, W1, W2, "relu")
    assert got.tolist() == [[float(x) for x in row] for row in exact]
    # Some of these S values need more than 8 significant bits, so the rounding is exercised.
    assert not np.array_equal(rounded, relu_f32.double().numpy())


def test_b2b_scale_relu_brute_force():
    rng = np.random.default_rng(7)
    A = rng.integers(-8, 9, (4, 3)) / 4.0
    W1 = rng.integers(-8, 9, (3, 5)) / 2.0
    W2 = rng.integers(-8, 9, (5, 2)) / 1.0
    S = _frac_matmul(A.tolist(), W1.tolist())
    sc = Fraction(1, 4)
    P = [[max(sc * s, Fraction(0)) for s in row] for row in S]
    # All P here have at most 8 significant bits -> bf16 rounding is exact.
    exact = _frac_matmul([[float(p) for p in row] for row in P], W2.tolist())
    got = O.b2bgemm(A, W1, W2, "scale_relu", 0.25)
    assert got.tolist() == [[float(x) for x in row] for row in exact]


def test_norms_brute_force_math_module():
    x = RNG.standard_normal((4, 9))
    g = RNG.standard_normal(9)
    b = RNG.standard_normal(9)
    for r in range(4):
        row = list(x[r])
        mu = math.fsum(row) / 9
        var = math.fsum((v - mu) ** 2 for v in row) / 9
        ln = [g[n] * (row[n] - mu) / math.sqrt(var + 1e-5) + b[n] for n in range(9)]
        ms = math.fsum(v * v for v in row) / 9
        rms = [g[n] * row[n] / math.sqrt(ms + 1e-6) for n in range(9)]
        mx = max(row)
        den = math.fsum(math.exp(v - mx) for v in row)
        sm = [math.exp(v - mx) / den for v in row]
        np.testing.assert_allclose(O.row_layernorm(x, g, b, 1e-5)[r], ln, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(O.row_rmsnorm(x, g, 1e-6)[r], rms, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(O.row_softmax(x)[r], sm, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- bf16 rounding
@pytest.mark.parametrize("x,expect_bits", [
    (1.0 + 2 ** -8, 0x3F80),            # tie -> even (1.0)
    (1.0 + 3 * 2 ** -8, 0x3F82),        # tie -> even (1 + 2^-6)
    (1.0 + 2 ** -8 + 2 ** -30, 0x3F81),  # just above the tie -> up
    (-0.0, 0x8000),
    (0.0, 0x0000),
    (2.0 ** -133, 0x0001),              # smallest subnormal
    (2.0 ** -134, 0x0000),              # half the smallest subnormal: tie -> 0 (even)
    (3 * 2.0 ** -134, 0x0002),          # 1.5 quanta: tie -> 2 quanta (even)
    (2.0 ** -126, 0x0080),              # smallest normal
    (O.BF16_MAX, 0x7F7F),
    ((2 - 2 ** -8) * 2.0 ** 127, 0x7F80),  # overflow threshold: tie to even -> inf
    (-1e39, 0xFF80),
    (math.inf, 0x7F80),
    (3.140625, 0x4049),
])
def test_bf16_rne_bit_patterns(x, expect_bits):
    assert int(O.f64_to_bf16_bits(np.array([x]))[0]) == expect_bits
    back = O.bf16_bits_to_f64(np.array([expect_bits], np.uint16))[0]
    r = O.bf16_round(np.array([x]))[0]
    assert (back == r) and (math.copysign(1, back) == math.copysign(1, r))


def test_bf16_nan():
    assert np.isnan(O.bf16_round(np.array([np.nan]))[0])
    assert np.isnan(O.bf16_bits_to_f64(np.array([0x7FC0], np.uint16))[0])


def test_bf16_round_matches_torch_on_float32_values():
    # For inputs already in fp32, torch's fp32 -> bf16 conversion is a single
    # RNE rounding, so it must agree bit for bit with the oracle.
    rng = np.random.default_rng(99)
    parts = [rng.standard_normal(50000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 50000).astype(np.float32),
             (rng.standard_normal(2000) * 2.0 ** -128).astype(np.float32),
             np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3e38, -3.3e38], np.float32)]
    x32 = np.concatenate(parts).astype(np.float32)
    x32 = x32[np.isfinite(x32)]
    t = torch.from_numpy(x32).to(torch.bfloat16)
    tb = t.view(torch.int16).numpy().astype(np.uint16)
    ob = O.f64_to_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(tb, ob)
    np.testing.assert_array_equal(O.bf16_bits_to_f64(tb), t.to(torch.float64).numpy())


# ------------------------------------------------------------- planted mistakes
_ORIG_ELEMENTWISE = O.elementwise


def _wrap_elementwise(which, bad):
    """The oracle's elementwise node with one op replaced by a planted mistake."""
    def f(x, op, scalar=0.0, bias=None, residual=None):
        if op == which:
            return bad(np.asarray(x, float), scalar, bias)
        return _ORIG_ELEMENTWISE(x, op, scalar, bias, residual)
    return f


def test_oracle_mutations_are_caught(monkeypatch):
    """Plant plausible mistakes in the oracle and check that a pin fails."""
    mutations = {
        "unbiased_variance": ("row_layernorm", lambda x, g, b, eps: (
            np.asarray(g)[None] * (x - x.mean(1, keepdims=True)) /
            np.sqrt(x.var(1, ddof=1, keepdims=True) + eps) + np.asarray(b)[None])),
        "eps_outside_root": ("row_layernorm", lambda x, g, b, eps: (
            np.asarray(g)[None] * (x - x.mean(1, keepdims=True)) /
            (np.sqrt(x.var(1, keepdims=True)) + eps) + np.asarray(b)[None])),
        "rms_subtracts_mean": ("row_rmsnorm", lambda x, g, eps: (
            np.asarray(g)[None] * (x - x.mean(1, keepdims=True)) /
            np.sqrt(((x - x.mean(1, keepdims=True)) ** 2).mean(1, keepdims=True) + eps))),
        "softmax_column_axis": ("row_softmax", lambda x: np.exp(x) / np.exp(x).sum(0, keepdims=True)),
        "matmul_transposed_B": ("matmul", lambda A, B: np.asarray(A, float) @ np.asarray(B, float).T
                                if np.asarray(B).shape[0] == np.asarray(B).shape[1] else
                                np.asarray(A, float) @ np.asarray(B, float) * 1.0000001),
        "bf16_truncation": ("bf16_round", lambda x: np.trunc(np.asarray(x, float) * 128) / 128),
        "col_softmax_row_axis": ("col_softmax", lambda x: np.exp(x) / np.exp(x).sum(1, keepdims=True)),
        "col_layernorm_gamma_by_row": ("col_layernorm", lambda x, g, b, eps: (
            (x - x.mean(0, keepdims=True)) / np.sqrt(x.var(0, keepdims=True) + eps) * np.resize(g, (x.shape[0], 1))
            + np.resize(b, (x.shape[0], 1)))),
        "col_rmsnorm_unbiased": ("col_rmsnorm", lambda x, g, eps: (
            np.asarray(g)[None] * x / np.sqrt((x * x).sum(0, keepdims=True) / (x.shape[0] - 1) + eps))),
        "bias_by_row": ("elementwise", _wrap_elementwise(
            "bias", lambda x, scalar, bias: x + np.resize(np.asarray(bias, float), (x.shape[0], 1)))),
        "scale_divides": ("elementwise", _wrap_elementwise("scale", lambda x, scalar, bias: x / float(scalar))),
        "bias_dropped": ("elementwise", _wrap_elementwise("bias", lambda x, scalar, bias: x)),
    }
    checks = [test_hand_example_epilogues, test_layernorm_eps_inside_root_closed_form,
              test_rmsnorm_mean_square_one_and_scale_invariance, test_epilogues_match_torch_float64,
              test_softmax_rows_sum_to_one, test_hand_example_gemm_exact,
              test_matmul_brute_force_fraction, test_b2b_relu_brute_force_with_library_rounding,
              test_bf16_round_matches_torch_on_float32_values, test_hand_example_column_reductions,
              test_hand_example_bias_and_scale]
    for name, (attr, bad) in mutations.items():
        with monkeypatch.context() as mp:
            mp.setattr(O, attr, bad)
            caught = False
            for chk in checks:
                try:
                    if chk is test_matmul_brute_force_fraction:
                        chk((8, 8, 8))
                    elif chk is test_b2b_relu_brute_force_with_library_rounding:
                        chk(0)
                    else:
                        chk()
                except (AssertionError, ValueError, TypeError):
                    caught = True
                    break
            assert caught, f"planted mistake {name} was not caught by any pin"
