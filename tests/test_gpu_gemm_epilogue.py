"""GPU parity: fused GEMM + epilogue (cf_gemm_epilogue through the C ABI)
against the float64 oracle on the same seeded bf16/fp32 inputs."""

import numpy as np
import pytest
import torch

from oracle import cf_oracle as O
from back_gemm_fusion_gb300 import inputs as I
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


def _dev(t):
    return None if t is None else t.cuda()


def _run(cf, case, b_trans=False, exchange="auto"):
    A = case.A.cuda()
    B = case.B.cuda()
    if b_trans:
        B = B.t().contiguous()  # stored N x K
    out = cf.cf_gemm_epilogue(A, B, case.ops, _dev(case.bias), _dev(case.gamma), _dev(case.beta),
                              b_trans=b_trans, exchange=exchange)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    return out.cpu().numpy()


def _oracle(case, rows=None):
    A = I.to_f64(case.A)
    if rows is not None:
        A = A[rows]
    return O.gemm_epilogue(A, I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                           I.to_f64(case.beta))


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (128, 256, 128), (256, 512, 320), (384, 768, 1024)])
def test_plain_gemm(cf, M, N, K, b_trans):
    case = I.gemm_epilogue_case("gemm", M, N, K, [], seed=M + N + K)
    assert_rows_close(_run(cf, case, b_trans), _oracle(case), strict=1e-4, what=f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("b_trans", [False, True])
def test_layernorm_256(cf, b_trans):
    case = I.layernorm_256()
    assert_rows_close(_run(cf, case, b_trans), _oracle(case), what="gemm+bias+layernorm 256^3")


@pytest.mark.parametrize("b_trans", [False, True])
def test_layernorm_pairs_wide(cf, b_trans):
    # 32 tiles per row with an even number of strips: CTA pairs run 256 x 256
    # tiles, each CTA of a pair loading its own half of the B tile
    # (cta_group::2 MMAs read both halves).
    case = I.gemm_epilogue_case("ln_wide", 256, 8192, 128, [("bias",), ("layernorm", 1e-5)], seed=9,
                                need_bias=True, need_gamma=True, need_beta=True)
    assert_rows_close(_run(cf, case, b_trans), _oracle(case), what="layernorm 32 tiles, pairs")


@pytest.mark.parametrize("ops", [[("bias",)], [("bias",), ("relu",)], [("scale", 0.5), ("gelu_tanh",)],
                                 [("bias",), ("gelu_tanh",), ("scale", -2.0)]])
def test_elementwise_programs(cf, ops):
    case = I.gemm_epilogue_case("ew", 256, 512, 192, ops, seed=3, need_bias=True)
    assert_rows_close(_run(cf, case), _oracle(case), strict=1e-4, what=str(ops))


@pytest.mark.parametrize("exchange", ["cluster", "global"])
@pytest.mark.parametrize("rowop", ["layernorm", "rmsnorm", "softmax"])
@pytest.mark.parametrize("N", [512, 2048])
def test_row_ops_multi_tile(cf, rowop, exchange, N):
    ops = {"layernorm": [("bias",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 1 / 16), ("softmax",)]}[rowop]
    case = I.gemm_epilogue_case(rowop, 384, N, 256, ops, seed=N, need_bias=True, need_gamma=True,
                                need_beta=True)
    assert_rows_close(_run(cf, case, exchange=exchange), _oracle(case), what=f"{rowop} N={N} {exchange}")


@pytest.mark.parametrize("M", [1, 77, 200, 333, 640])
@pytest.mark.parametrize("rowop", ["none", "layernorm", "rmsnorm", "softmax"])
def test_ragged_m(cf, M, rowop):
    # The last 128-row strip is partial: zero-filled loads, clipped stores.
    ops = {"none": [("bias",), ("gelu_tanh",)], "layernorm": [("bias",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 0.125), ("softmax",)]}[rowop]
    case = I.gemm_epilogue_case("ragged", M, 1024, 128, ops, seed=M, need_bias=True, need_gamma=True,
                                need_beta=True)
    assert_rows_close(_run(cf, case), _oracle(case), strict=1e-4 if rowop == "none" else 2e-3,
                      what=f"ragged M={M} {rowop}")


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("M,K,rowop", [(128, 72, "none"), (256, 200, "layernorm"), (384, 1000, "rmsnorm"),
                                       (333, 136, "softmax")])
def test_ragged_k(cf, M, K, rowop, b_trans):
    # K not a multiple of the 64-wide K block: the last block reads zeros.
    ops = {"none": [("bias",), ("relu",)], "layernorm": [("bias",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 0.125), ("softmax",)]}[rowop]
    case = I.gemm_epilogue_case("ragged_k", M, 512, K, ops, seed=M + K, need_bias=True, need_gamma=True,
                                need_beta=True)
    assert_rows_close(_run(cf, case, b_trans), _oracle(case), strict=1e-4 if rowop == "none" else 2e-3,
                      what=f"ragged K={K} M={M} {rowop} b_trans={b_trans}")


@pytest.mark.parametrize("M,N,K,rowop,b_trans,exchange", [
    (128, 512, 8, "none", False, "auto"), (300, 512, 16, "layernorm", True, "auto"),
    (256, 1024, 24, "rmsnorm", False, "cluster"), (200, 768, 56, "softmax", True, "auto"),
    (384, 4096, 16, "layernorm", False, "global"), (129, 2056, 40, "softmax", False, "global_dynamic")])
def test_short_k(cf, M, N, K, rowop, b_trans, exchange):
    # K below one 64-wide block (e.g. a first layer over 13 dense features
    # padded to 16): the only K block reads zeros past K.
    ops = {"none": [("bias",), ("relu",)], "layernorm": [("bias",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 0.125), ("softmax",)]}[rowop]
    case = I.gemm_epilogue_case("short_k", M, N, K, ops, seed=M + N + K, need_bias=True, need_gamma=True,
                                need_beta=True)
    assert_rows_close(_run(cf, case, b_trans, exchange=exchange), _oracle(case),
                      strict=1e-4 if rowop == "none" else 2e-3,
                      what=f"short K={K} {M}x{N} {rowop} b_trans={b_trans} {exchange}")


@pytest.mark.parametrize("res_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,N,K,prog", [(256, 512, 128, "layernorm"), (333, 1024, 256, "rmsnorm"),
                                        (256, 4352, 128, "softmax"), (200, 256, 64, "none"),
                                        (512, 2048, 256, "layernorm")])
def test_residual_postnorm(cf, M, N, K, prog, res_dtype):
    # Post-norm blocks: the residual stream is added in the epilogue before the
    # row reduction (fp32 or bf16 residual; ragged M; cluster and workspace
    # exchanges; 1-CTA and CTA-pair tiles).
    ops = {"layernorm": [("bias",), ("residual",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("residual",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 0.25), ("residual",), ("softmax",)],
           "none": [("residual",), ("relu",), ("residual",)]}[prog]
    case = I.gemm_epilogue_case("residual", M, N, K, ops, seed=M + N, need_bias=True, need_gamma=True,
                                need_beta=True)
    R = torch.from_numpy(np.random.default_rng(M * 3 + N).standard_normal((M, N)).astype(np.float32)).to(res_dtype)
    out = cf.cf_gemm_epilogue(case.A.cuda(), case.B.cuda(), case.ops, _dev(case.bias), _dev(case.gamma),
                              _dev(case.beta), residual=R.cuda())
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), residual=I.to_f64(R))
    assert_rows_close(out.cpu().numpy(), ref, strict=1e-4 if prog == "none" else 2e-3,
                      what=f"residual {prog} {M}x{N}x{K} {res_dtype}")


CHAINS = {
    "ln_gelu_rms": [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)],
    "rms_ln": [("rmsnorm", 1e-6), ("layernorm", 1e-5)],
    "ln_scale_softmax": [("bias",), ("layernorm", 1e-5), ("scale", 2.0), ("softmax",)],
    "res_rms_relu_rms": [("residual",), ("rmsnorm", 1e-6), ("relu",), ("rmsnorm", 1e-6)],
}


@pytest.mark.parametrize("affine0", [False, True])
@pytest.mark.parametrize("M,N", [(256, 256), (384, 1024), (200, 4352), (512, 2048)])
@pytest.mark.parametrize("chain", sorted(CHAINS))
def test_chained_reductions(cf, chain, M, N, affine0):
    # Two reduction stages in one epilogue: per-tile (N = 256) and workspace
    # exchanges, 1-CTA (odd strip count) and CTA-pair tiles, ragged M.
    ops = CHAINS[chain]
    case = I.gemm_epilogue_case("chain", M, N, 128, ops, seed=M + N, need_bias=True, need_gamma=True,
                                need_beta=True)
    rng = np.random.default_rng(N)
    g0 = b0 = R = None
    if affine0:
        g0 = torch.from_numpy((1.0 + 0.3 * rng.standard_normal(N)).astype(np.float32))
        b0 = torch.from_numpy((0.3 * rng.standard_normal(N)).astype(np.float32))
    if any(o[0] == "residual" for o in ops):
        R = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32))
    out = cf.cf_gemm_epilogue(case.A.cuda(), case.B.cuda(), case.ops, _dev(case.bias), _dev(case.gamma),
                              _dev(case.beta), residual=_dev(R), stage0_gamma=_dev(g0), stage0_beta=_dev(b0))
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), residual=I.to_f64(R), stage0_gamma=I.to_f64(g0),
                          stage0_beta=I.to_f64(b0))
    assert_rows_close(out.cpu().numpy(), ref, what=f"chain {chain} {M}x{N} affine0={affine0}")


@pytest.mark.parametrize("N", [2048, 1000])
@pytest.mark.parametrize("chain", sorted(CHAINS))
def test_chained_reductions_unfused(cf, chain, N):
    # The unfused comparison path: register-resident rows (N a multiple of
    # 1024) or the shared-memory kernel (other N), first-stage affine vectors.
    ops = CHAINS[chain]
    case = I.gemm_epilogue_case("chain_unfused", 256, N, 128, ops, seed=7, need_bias=True, need_gamma=True,
                                need_beta=True)
    rng = np.random.default_rng(3)
    g0 = torch.from_numpy((1.0 + 0.3 * rng.standard_normal(N)).astype(np.float32))
    b0 = torch.from_numpy((0.3 * rng.standard_normal(N)).astype(np.float32))
    R = torch.from_numpy(rng.standard_normal((256, N)).astype(np.float32)).to(torch.bfloat16)
    out = cf.cf_unfused_gemm_epilogue(case.A.cuda(), case.B.cuda(), case.ops, _dev(case.bias), _dev(case.gamma),
                                      _dev(case.beta), stage0_gamma=g0.cuda(), stage0_beta=b0.cuda(),
                                      residual=R.cuda())
    torch.cuda.synchronize()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), residual=I.to_f64(R), stage0_gamma=I.to_f64(g0),
                          stage0_beta=I.to_f64(b0))
    assert_rows_close(out.cpu().numpy(), ref, what=f"unfused chain {chain} N={N}")


@pytest.mark.parametrize("N", [4096, 4352, 8192])
def test_softmax_wide_rows(cf, N):
    # AUTO picks the workspace exchange at all three widths on a 152-SM GB300:
    # 16 tiles (only 7 clusters of 16 CTAs are resident, too few to fill the
    # GPU), 17 tiles (wider than a cluster), 32 tiles (CTA pairs).  The forced
    # 16-CTA cluster exchange is tested below.
    case = I.gemm_epilogue_case("sm", 256, N, 128, [("scale", 0.25), ("softmax",)], seed=5)
    assert_rows_close(_run(cf, case), _oracle(case), what=f"softmax N={N}")


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("rowop", ["layernorm", "rmsnorm", "softmax"])
def test_cluster_exchange_16_ctas(cf, rowop, b_trans):
    # N = 4096 with the DSMEM exchange forced: 16 tiles per row, one
    # non-portable 16-CTA cluster per row strip (AUTO does not pick it on a
    # 152-SM GB300, where only 7 such clusters are resident at once).  Three
    # strips: the persistent clusters take more than one strip when fewer
    # are resident.
    ops = {"layernorm": [("bias",), ("layernorm", 1e-5)],
           "rmsnorm": [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
           "softmax": [("scale", 0.25), ("softmax",)]}[rowop]
    case = I.gemm_epilogue_case("cluster16", 384, 4096, 128, ops, seed=16, need_bias=True, need_gamma=True,
                                need_beta=True)
    assert_rows_close(_run(cf, case, b_trans, exchange="cluster"), _oracle(case),
                      what=f"{rowop} N=4096 16-CTA cluster b_trans={b_trans}")


@pytest.mark.parametrize("exchange", ["auto", "cluster"])
def test_gelu_rmsnorm_full_size_sampled(cf, exchange):
    # The GELU + RMSNorm workload at full size with AUTO (workspace exchange,
    # CTA pairs) and with the 16-CTA DSMEM exchange forced (64 strips over the
    # resident 16-CTA clusters).
    case = I.gelu_rmsnorm()
    gpu = _run(cf, case, exchange=exchange)
    rows = sample_rows(case.M)
    assert_rows_close(gpu[rows], _oracle(case, rows), what=f"gemm+bias+gelu+rmsnorm 8192x4096x4096 {exchange}")


def test_scaled_softmax_full_size_sampled(cf):
    case = I.scaled_softmax()
    gpu = _run(cf, case)
    rows = sample_rows(case.M)
    ref = _oracle(case, rows)
    assert_rows_close(gpu[rows], ref, what="gemm+scaled softmax 4096x16384x4096")
    # Every row of a softmax sums to one (all rows, not only the sample).
    assert np.max(np.abs(gpu.sum(1, dtype=np.float64) - 1.0)) < 1e-3


def bf16_out_gate(gpu, ref, strict, what):
    """bf16 output: the kernel's fp32 value f (within strict * rms of the
    oracle row) is rounded once to nearest even (8-bit significand, unit
    roundoff 2^-8), |g - f| <= 2^-8 |f|, so
    |g - ref| <= 2^-8 |ref| + (1 + 2^-8) strict * rms per element.  The fp32
    contract gate is taken on the fp32 output of the same program."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    bound = 2.0 ** -8 * np.abs(ref) + (1 + 2.0 ** -8) * strict * rms + 1e-30
    worst = (err / bound).max()
    assert worst <= 1.0, f"{what}: bf16-output bound exceeded ({worst:.3g} x)"


BF16_PROGRAMS = {
    "gelu": ([("bias",), ("gelu_tanh",)], 1e-4),
    "layernorm": ([("bias",), ("layernorm", 1e-5)], 2e-3),
    "rmsnorm": ([("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)], 2e-3),
    "softmax": ([("scale", 0.125), ("softmax",)], 2e-3),
    "chained": ([("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)], 2e-3),
}


@pytest.mark.parametrize("exchange", ["auto", "global"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (333, 2048, 200), (128, 4352, 64)])
@pytest.mark.parametrize("prog", sorted(BF16_PROGRAMS))
def test_bf16_output(cf, prog, M, N, K, exchange):
    # bf16 output tiles: rounded in the epilogue, stored by TMA from an
    # unswizzled staging buffer (ragged M and K, cluster and workspace
    # exchanges, 1-CTA and CTA-pair tiles).
    ops, strict = BF16_PROGRAMS[prog]
    if prog == "chained" and exchange == "auto":
        exchange = "global"  # chained programs take the workspace exchange in any case
    case = I.gemm_epilogue_case("bf16_out", M, N, K, ops, seed=M + N + K, need_bias=True, need_gamma=True,
                                need_beta=True)
    A, B = case.A.cuda(), case.B.cuda()
    args = (A, B, case.ops, _dev(case.bias), _dev(case.gamma), _dev(case.beta))
    g = cf.cf_gemm_epilogue(*args, exchange=exchange, out_dtype=torch.bfloat16)
    f = cf.cf_gemm_epilogue(*args, exchange=exchange)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    assert g.dtype == torch.bfloat16
    ref = _oracle(case)
    assert_rows_close(f.cpu().numpy(), ref, strict=strict, what=f"fp32 out {prog} {M}x{N}x{K} {exchange}")
    bf16_out_gate(g.float().cpu().numpy(), ref, strict, f"bf16 out {prog} {M}x{N}x{K} {exchange}")
    # The same epilogue value is rounded: the bf16 tile is the fp32 tile
    # rounded to nearest even, element for element.
    assert torch.equal(g.cpu(), f.cpu().to(torch.bfloat16)), f"bf16 out {prog}: differs from rounded fp32 out"


def test_bf16_output_strided_noalloc(cf):
    # A bf16 output view with a padded leading dimension, written through the
    # no-allocation entry point; the padding columns stay untouched.
    case = I.gemm_epilogue_case("bf16_ld", 200, 1024, 128, [("bias",), ("rmsnorm", 1e-6)], seed=5, need_bias=True,
                                need_gamma=True)
    buf = torch.full((200, 1024 + 40), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:, :1024]
    cf.cf_gemm_epilogue_noalloc(case.A.cuda(), case.B.cuda(), case.ops, _dev(case.bias), _dev(case.gamma), None,
                                out=out)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    bf16_out_gate(out.float().cpu().numpy(), _oracle(case), 2e-3, "bf16 out, padded ld")
    assert torch.all(buf[:, 1024:] == 7.0)


RAGGED_N_PROGRAMS = {
    "none": ([("bias",), ("gelu_tanh",)], 1e-4),
    "layernorm": ([("bias",), ("layernorm", 1e-5)], 2e-3),
    "rmsnorm": ([("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)], 2e-3),
    "softmax": ([("scale", 0.125), ("softmax",)], 2e-3),
}


@pytest.mark.parametrize("b_trans", [False, True])
@pytest.mark.parametrize("N", [8, 40, 264, 1000, 2056, 4104])
@pytest.mark.parametrize("prog", sorted(RAGGED_N_PROGRAMS))
def test_ragged_n(cf, prog, N, b_trans):
    # N not a multiple of the 256-column tile: the last tile of each row holds
    # N % 256 valid columns (one partial 32-column chunk, or a few whole
    # ones); its B columns past N load as zeros, the row statistics skip
    # them, the vectors are never read past N, and the stores clip them.
    # 2056 takes the cluster exchange (9 tiles), 4104 the workspace (17).
    ops, strict = RAGGED_N_PROGRAMS[prog]
    case = I.gemm_epilogue_case("ragged_n", 200, N, 136, ops, seed=N, need_bias=True, need_gamma=True,
                                need_beta=True)
    assert_rows_close(_run(cf, case, b_trans), _oracle(case), strict=strict,
                      what=f"ragged N={N} {prog} b_trans={b_trans}")


@pytest.mark.parametrize("exchange", ["cluster", "global"])
@pytest.mark.parametrize("rowop", ["layernorm", "softmax"])
def test_ragged_n_exchanges(cf, rowop, exchange):
    # Same row, both exchanges: tile counts 3 (the last with 8 columns).
    ops = [("bias",), ("layernorm", 1e-5)] if rowop == "layernorm" else [("scale", 0.5), ("softmax",)]
    case = I.gemm_epilogue_case("ragged_n_x", 384, 520, 64, ops, seed=7, need_bias=True, need_gamma=True,
                                need_beta=True)
    assert_rows_close(_run(cf, case, exchange=exchange), _oracle(case), what=f"ragged N=520 {rowop} {exchange}")


def test_ragged_n_padded_rows(cf):
    # N = 300 (not a multiple of 8) inside 304-element rows: B, out and the
    # residual are views of padded buffers; out's padding is never written.
    M, N, K = 130, 300, 128
    ops = [("bias",), ("residual",), ("rmsnorm", 1e-6)]
    case = I.gemm_epilogue_case("ragged_n_ld", M, N, K, ops, seed=300, need_bias=True, need_gamma=True)
    R = torch.from_numpy(np.random.default_rng(301).standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16)
    Bp = torch.zeros((K, 304), dtype=torch.bfloat16, device="cuda")
    Bp[:, :N] = case.B.cuda()
    Rp = torch.zeros((M, 304), dtype=torch.bfloat16, device="cuda")
    Rp[:, :N] = R.cuda()
    Op = torch.full((M, 304), 5.0, dtype=torch.float32, device="cuda")
    cf.cf_gemm_epilogue(case.A.cuda(), Bp[:, :N], case.ops, _dev(case.bias), _dev(case.gamma), None,
                        out=Op[:, :N], residual=Rp[:, :N])
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          None, residual=I.to_f64(R))
    assert_rows_close(Op[:, :N].cpu().numpy(), ref, what="ragged N=300, padded rows")
    assert torch.all(Op[:, N:] == 5.0)


@pytest.mark.parametrize("N", [264, 1000, 4104])
def test_ragged_n_chained(cf, N):
    # Two reduction stages over a ragged row: both stages' statistics skip the
    # columns past N (the first stage's affine output there is not zero).
    ops = [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)]
    case = I.gemm_epilogue_case("ragged_n_chain", 256, N, 64, ops, seed=N + 5, need_bias=True, need_gamma=True)
    rng = np.random.default_rng(N)
    g0 = torch.from_numpy((1 + 0.3 * rng.standard_normal(N)).astype(np.float32))
    b0 = torch.from_numpy((0.3 * rng.standard_normal(N)).astype(np.float32))
    out = cf.cf_gemm_epilogue(case.A.cuda(), case.B.cuda(), case.ops, _dev(case.bias), _dev(case.gamma), None,
                              stage0_gamma=g0.cuda(), stage0_beta=b0.cuda())
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          None, stage0_gamma=I.to_f64(g0), stage0_beta=I.to_f64(b0))
    assert_rows_close(out.cpu().numpy(), ref, what=f"ragged N={N} chained")


def test_ragged_n_bf16_output(cf):
    ops, strict = BF16_PROGRAMS["layernorm"]
    case = I.gemm_epilogue_case("ragged_n_bf16", 256, 1000, 128, ops, seed=11, need_bias=True, need_gamma=True,
                                need_beta=True)
    args = (case.A.cuda(), case.B.cuda(), case.ops, _dev(case.bias), _dev(case.gamma), _dev(case.beta))
    g = cf.cf_gemm_epilogue(*args, out_dtype=torch.bfloat16)
    f = cf.cf_gemm_epilogue(*args)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    assert torch.equal(g.cpu(), f.cpu().to(torch.bfloat16))
    bf16_out_gate(g.float().cpu().numpy(), _oracle(case), strict, "ragged N=1000 bf16 out")


COL_PROGRAMS = {
    "layernorm": [("bias",), ("layernorm", 1e-5)],
    "rmsnorm": [("bias",), ("gelu_tanh",), ("rmsnorm", 1e-6)],
    "softmax": [("scale", 0.5), ("softmax",)],
}


def _run_col(cf, case, exchange="auto", out_dtype=torch.float32, residual=None, stage0=None):
    Bt = case.B.t().contiguous().cuda()  # stored N x K
    kw = {}
    if stage0 is not None:
        kw = {"stage0_gamma": stage0[0].cuda(), "stage0_beta": stage0[1].cuda()}
    out = cf.cf_gemm_epilogue(case.A.cuda(), Bt, case.ops, _dev(case.bias), _dev(case.gamma), _dev(case.beta),
                              b_trans=True, exchange=exchange, out_dtype=out_dtype, axis="col",
                              residual=None if residual is None else residual.cuda(), **kw)
    torch.cuda.synchronize()
    assert cf.cf_last_device_status() == 0
    return out


def _col_gate(gpu, ref, strict, what):
    # The per-row gate applied to the columns (the reduction's own axis).
    assert_rows_close(np.ascontiguousarray(gpu.T), np.ascontiguousarray(ref.T), strict=strict, what=what)


@pytest.mark.parametrize("M,N,K", [(256, 256, 64), (512, 384, 128), (1000, 520, 72), (4104, 256, 64),
                                   (77, 136, 64)])
@pytest.mark.parametrize("prog", sorted(COL_PROGRAMS))
def test_column_reductions(cf, prog, M, N, K):
    # Reductions down the columns of P (over m): the kernel runs on P^T with
    # the strip machinery (cluster or workspace exchange across the M tiles),
    # per-column vectors as per-row scalars, and transposed output tiles.
    # Shapes: one tile; 2 tiles down a column with an odd strip count; ragged
    # in both dims; 17 tiles (workspace exchange); a single partial tile.
    case = I.gemm_epilogue_case("col", M, N, K, COL_PROGRAMS[prog], seed=M + N, need_bias=True, need_gamma=True,
                                need_beta=True)
    got = _run_col(cf, case).cpu().numpy()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), axis="col")
    _col_gate(got, ref, 2e-3, f"columns {prog} {M}x{N}x{K}")


@pytest.mark.parametrize("exchange", ["cluster", "global"])
def test_column_reductions_exchanges(cf, exchange):
    case = I.gemm_epilogue_case("col_x", 768, 256, 64, COL_PROGRAMS["layernorm"], seed=3, need_bias=True,
                                need_gamma=True, need_beta=True)
    got = _run_col(cf, case, exchange=exchange).cpu().numpy()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          I.to_f64(case.beta), axis="col")
    _col_gate(got, ref, 2e-3, f"columns layernorm {exchange}")


@pytest.mark.parametrize("res_dtype", [torch.float32, torch.bfloat16])
def test_column_residual_and_bf16_output(cf, res_dtype):
    ops = [("bias",), ("residual",), ("rmsnorm", 1e-6)]
    case = I.gemm_epilogue_case("col_res", 600, 264, 128, ops, seed=9, need_bias=True, need_gamma=True)
    R = torch.from_numpy(np.random.default_rng(10).standard_normal((600, 264)).astype(np.float32)).to(res_dtype)
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          None, residual=I.to_f64(R), axis="col")
    f = _run_col(cf, case, residual=R)
    g = _run_col(cf, case, residual=R, out_dtype=torch.bfloat16)
    _col_gate(f.cpu().numpy(), ref, 2e-3, f"columns residual {res_dtype}")
    assert torch.equal(g.cpu(), f.cpu().to(torch.bfloat16))


def test_column_chained(cf):
    ops = [("bias",), ("layernorm", 1e-5), ("gelu_tanh",), ("rmsnorm", 1e-6)]
    case = I.gemm_epilogue_case("col_chain", 520, 256, 64, ops, seed=13, need_bias=True, need_gamma=True)
    rng = np.random.default_rng(14)
    g0 = torch.from_numpy((1 + 0.3 * rng.standard_normal(256)).astype(np.float32))
    b0 = torch.from_numpy((0.3 * rng.standard_normal(256)).astype(np.float32))
    got = _run_col(cf, case, stage0=(g0, b0)).cpu().numpy()
    ref = O.gemm_epilogue(I.to_f64(case.A), I.to_f64(case.B), case.ops, I.to_f64(case.bias), I.to_f64(case.gamma),
                          None, stage0_gamma=I.to_f64(g0), stage0_beta=I.to_f64(b0), axis="col")
    _col_gate(got, ref, 2e-3, "columns chained")


def test_column_layernorm_full_size_sampled(cf):
    # The column-reduction bench workload at full size (M = 8192 rows reduced
    # per column, 32 tiles down each column: workspace exchange); 64 sampled
    # columns against the oracle, each over all rows.
    case = I.column_layernorm()
    got = _run_col(cf, case).cpu().numpy()
    cols = sample_rows(case.N, 64, seed=5)
    B = I.to_f64(case.B)[:, cols]
    ref = O.gemm_epilogue(I.to_f64(case.A), B, case.ops, I.to_f64(case.bias)[cols], I.to_f64(case.gamma)[cols],
                          I.to_f64(case.beta)[cols], axis="col")
    _col_gate(got[:, cols], ref, 2e-3, "column layernorm 8192x4096x4096")
