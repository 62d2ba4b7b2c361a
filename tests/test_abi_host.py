"""Host-side tests of the C ABI (no GPU needed): the library builds, loads
and exports every symbol include/cf.h declares; argument validation returns
the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from back_gemm_fusion_gb300 import build
    build.build()
    from back_gemm_fusion_gb300 import binding
    return binding.load_library()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "cf.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"CF_API\s+[\w\s\*]+?\b(cf_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    syms = _declared_symbols()
    for s in ["cf_gemm_epilogue", "cf_b2bgemm", "cf_workspace_size", "cf_status_string",
              "cf_last_device_status", "cf_unfused_gemm_epilogue", "cf_unfused_b2bgemm", "cf_abi_version"]:
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    for s in _declared_symbols():
        assert hasattr(lib, s), f"{s} declared in include/cf.h but not exported"


def test_abi_version_and_status_strings(lib):
    assert lib.cf_abi_version() == 1
    from back_gemm_fusion_gb300.binding import STATUS_NAMES
    for code, name in STATUS_NAMES.items():
        assert lib.cf_status_string(code).decode() == name


def _mats(M=256, N=256, K=256, a_ptr=0x10000, b_ptr=0x20000, o_ptr=0x30000):
    from back_gemm_fusion_gb300.binding import cf_matrix, CF_BF16, CF_FP32
    A = cf_matrix(a_ptr, CF_BF16, 0, M, K, K)
    B = cf_matrix(b_ptr, CF_BF16, 0, K, N, N)
    O = cf_matrix(o_ptr, CF_FP32, 0, M, N, N)
    return A, B, O


def _call(lib, A, B, O, ops, bias=0x40000, gamma=0x50000, beta=0x60000, exchange="auto", ws=None, ws_bytes=0):
    from back_gemm_fusion_gb300.binding import epi_desc
    d = epi_desc(ops, exchange)
    return lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), bias, gamma, beta, ctypes.byref(d),
                                ctypes.byref(O), ws, ws_bytes, None)


LN = [("bias",), ("layernorm", 1e-5)]


def test_validation_errors(lib):
    A, B, O = _mats()
    assert _call(lib, A, B, O, LN, bias=None) == 1          # missing bias
    assert _call(lib, A, B, O, LN, beta=None) == 1          # LayerNorm needs beta
    assert _call(lib, A, B, O, [("softmax",), ("bias",)]) == 1  # reduction must be last
    assert _call(lib, A, B, O, [("layernorm", -1.0)]) == 1  # negative eps
    A2, B2, O2 = _mats(K=256)
    B2.rows = 128
    assert _call(lib, A2, B2, O2, LN) == 1                  # inconsistent K
    A3, B3, O3 = _mats(M=200)
    assert _call(lib, A3, B3, O3, LN) in (0, 4, 8)          # ragged M is supported (device check follows)
    A4, B4, O4 = _mats(N=384)
    assert _call(lib, A4, B4, O4, LN) in (0, 4, 8)          # ragged last N tile is supported
    A4, B4, O4 = _mats(N=300)
    assert _call(lib, A4, B4, O4, LN) == 3                  # N = ld = 300: rows not 16-byte aligned
    B4.ld, O4.ld = 304, 304
    assert _call(lib, A4, B4, O4, LN) in (0, 4, 8)          # N = 300 in padded rows
    A4, B4, O4 = _mats(N=256 * 16 + 8)
    assert _call(lib, A4, B4, O4, LN, exchange="cluster") == 2  # 17 tiles (last one ragged) > 16-CTA cluster
    A5, B5, O5 = _mats(K=96)
    assert _call(lib, A5, B5, O5, LN) in (0, 4, 8)          # ragged K (K % 8 == 0) is supported
    A6, B6, O6 = _mats(K=56)
    assert _call(lib, A6, B6, O6, LN) in (0, 4, 8)          # K below 64: one zero-filled block
    A6, B6, O6 = _mats(K=8)
    assert _call(lib, A6, B6, O6, LN) in (0, 4, 8)
    A6, B6, O6 = _mats(K=0)
    A6.ld = 8
    assert _call(lib, A6, B6, O6, LN) == 2                  # no K at all
    A6, B6, O6 = _mats(K=60)
    A6.ld, B6.cols, O6.cols = 64, 256, 256
    assert _call(lib, A6, B6, O6, LN) == 2                  # K % 8 != 0
    A6, B6, O6 = _mats(a_ptr=0x10008)
    assert _call(lib, A6, B6, O6, LN) == 3                  # misaligned pointer
    A7, B7, O7 = _mats()
    A7.ld = 260
    assert _call(lib, A7, B7, O7, LN) == 3                  # ld*2 not a multiple of 16
    A8, B8, O8 = _mats()
    assert _call(lib, A8, B8, O8, LN, bias=0x40004) == 3    # misaligned vector
    A9, B9, O9 = _mats(N=256 * 17)
    assert _call(lib, A9, B9, O9, LN, exchange="cluster") == 2  # 17 tiles > 16-CTA cluster
    A10, B10, O10 = _mats(N=256 * 17)
    assert _call(lib, A10, B10, O10, LN) == 7               # wide rows need a workspace
    A11, B11, O11 = _mats(M=0)
    assert _call(lib, A11, B11, O11, LN) == 0               # empty problem: nothing to do


def test_valid_call_without_gpu_reports_device(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    A, B, O = _mats()
    assert _call(lib, A, B, O, LN) in (4, 8)  # unsupported device / no device: never a CPU fallback


def test_workspace_size(lib):
    from back_gemm_fusion_gb300.binding import epi_desc
    A, B, O = _mats(M=4096, N=16384, K=4096)
    d = epi_desc([("scale", 1 / 64), ("softmax",)])
    n = lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B), ctypes.byref(d))
    assert n >= 4096 // 128 * 64 * 128 * 8 + 4096 // 128 * 16
    assert n < 3 * 2 ** 20
    d2 = epi_desc([("bias",)])
    assert lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B), ctypes.byref(d2)) == 0


def test_residual_validation(lib):
    from back_gemm_fusion_gb300.binding import cf_matrix, epi_desc, CF_FP32, CF_BF16
    A, B, O = _mats()
    POST = [("bias",), ("residual",), ("layernorm", 1e-5)]

    def call(residual, version=2):
        d = epi_desc(POST)
        d.version = version
        if residual is not None:
            d.residual = residual
        return lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000, ctypes.byref(d),
                                    ctypes.byref(O), None, 0, None)

    assert call(None) == 1                                              # residual op without a residual
    assert call(cf_matrix(0x70000, CF_FP32, 0, 256, 128, 256)) == 1     # wrong shape
    assert call(cf_matrix(0x70000, CF_FP32, 1, 256, 256, 256)) == 1     # transposed view
    assert call(cf_matrix(0x70008, CF_FP32, 0, 256, 256, 256)) == 3     # misaligned pointer
    assert call(cf_matrix(0x70000, CF_BF16, 0, 256, 256, 260)) == 3     # leading dim not 16-byte aligned
    assert call(cf_matrix(0x70000, CF_FP32, 0, 256, 256, 256), version=1) == 1  # version 1 has no residual
    assert call(cf_matrix(0x70000, CF_BF16, 0, 256, 256, 256)) in (0, 4, 8)    # valid: device check follows
    d = epi_desc(LN)
    d.version = 1                                                       # version-1 descriptors still accepted
    assert lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000, ctypes.byref(d),
                                ctypes.byref(O), None, 0, None) in (0, 4, 8)


def test_chained_reduction_rules(lib):
    from back_gemm_fusion_gb300.binding import epi_desc
    A, B, O = _mats(N=1024)

    def call(ops, version=2, exchange="auto"):
        d = epi_desc(ops, exchange)
        d.version = version
        return lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000, ctypes.byref(d),
                                    ctypes.byref(O), None, 0, None)

    LN_RMS = [("layernorm", 1e-5), ("rmsnorm", 1e-6)]
    assert call(LN_RMS, version=1) == 1                                  # chaining needs version 2
    assert call([("softmax",), ("rmsnorm", 1e-6)]) == 1                  # the first stage must be a norm
    assert call([("layernorm", 1e-5), ("rmsnorm", 1e-6), ("softmax",)]) == 1  # at most two reductions
    assert call(LN_RMS, exchange="cluster") == 2                        # chained stages: no DSMEM exchange
    assert call(LN_RMS) == 7                                             # workspace exchange needs a workspace
    from back_gemm_fusion_gb300.binding import cf_matrix, CF_BF16
    d = epi_desc(LN_RMS)
    one = lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B), ctypes.byref(epi_desc([("rmsnorm", 1e-6)])))
    two = lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(B), ctypes.byref(d))
    assert one > 0 and two == 2 * one                                    # one statistics region per stage


def test_output_dtype_rules(lib):
    # out may be fp32 or bf16; its dtype must match the descriptor's, and a
    # bf16 leading dimension must keep 16-byte row alignment (8 elements).
    from back_gemm_fusion_gb300.binding import cf_matrix, epi_desc, CF_FP32, CF_BF16
    A, B, _ = _mats()

    def call(out, out_dtype):
        d = epi_desc(LN, out_dtype=out_dtype)
        return lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000, ctypes.byref(d),
                                    ctypes.byref(out), None, 0, None)

    assert call(cf_matrix(0x30000, CF_BF16, 0, 256, 256, 256), CF_FP32) == 1   # dtype differs from the descriptor
    assert call(cf_matrix(0x30000, CF_FP32, 0, 256, 256, 256), CF_BF16) == 1
    assert call(cf_matrix(0x30000, CF_BF16, 0, 256, 256, 256), 7) == 1         # unknown dtype
    assert call(cf_matrix(0x30000, CF_BF16, 0, 256, 256, 260), CF_BF16) == 3   # 520-byte rows
    assert call(cf_matrix(0x30008, CF_BF16, 0, 256, 256, 256), CF_BF16) == 3   # misaligned pointer
    assert call(cf_matrix(0x30000, CF_BF16, 0, 256, 256, 264), CF_BF16) in (0, 4, 8)  # valid: device check follows
    assert call(cf_matrix(0x30000, CF_FP32, 0, 256, 256, 260), CF_FP32) in (0, 4, 8)


def test_b2b_validation(lib):
    from back_gemm_fusion_gb300.binding import cf_matrix, b2b_desc, CF_FP32, CF_BF16
    Q = cf_matrix(0x10000, CF_BF16, 0, 256, 128, 128)
    K = cf_matrix(0x20000, CF_BF16, 1, 128, 512, 128)   # stored 512 x 128, used transposed
    V = cf_matrix(0x30000, CF_BF16, 0, 512, 128, 128)

    def call(out, out_dtype=CF_FP32, op="scale_softmax", W1=K, A=Q, batch=1):
        d = b2b_desc(op, 0.125, batch, out_dtype=out_dtype)
        return lib.cf_b2bgemm(ctypes.byref(A), ctypes.byref(W1), ctypes.byref(V), ctypes.byref(d),
                              ctypes.byref(out), None)

    O32 = cf_matrix(0x40000, CF_FP32, 0, 256, 128, 128)
    O16 = cf_matrix(0x40000, CF_BF16, 0, 256, 128, 128)
    assert call(O32) in (0, 4, 8)                                       # attention shape, fp32 out
    assert call(O16, CF_BF16) in (0, 4, 8)                              # attention shape, bf16 out
    assert call(O16, CF_FP32) == 1                                      # out dtype differs from the descriptor
    assert call(cf_matrix(0x40000, CF_BF16, 0, 256, 128, 132), CF_BF16) == 3  # 264-byte rows
    assert call(O32, batch=0) == 1                                      # no problems
    assert call(cf_matrix(0x40000, CF_FP32, 0, 256, 64, 128)) == 1      # out shape differs
    assert call(O32, W1=cf_matrix(0x20000, CF_BF16, 0, 128, 512, 512)) == 2  # softmax needs the attention shape
    X = cf_matrix(0x10000, CF_BF16, 0, 256, 128, 128)
    W1 = cf_matrix(0x20000, CF_BF16, 0, 128, 512, 512)
    W2 = cf_matrix(0x30000, CF_BF16, 0, 512, 256, 256)

    def mlp(out, out_dtype=CF_FP32, op="relu"):
        d = b2b_desc(op, 1.0, 1, out_dtype=out_dtype)
        return lib.cf_b2bgemm(ctypes.byref(X), ctypes.byref(W1), ctypes.byref(W2), ctypes.byref(d),
                              ctypes.byref(out), None)

    assert mlp(cf_matrix(0x40000, CF_BF16, 0, 256, 256, 256), CF_BF16) in (0, 4, 8)  # MLP shape, bf16 out
    assert mlp(cf_matrix(0x40000, CF_FP32, 0, 256, 256, 256), op="scale_softmax") == 2  # MLP: elementwise F only


def test_b2b_shape_rules(lib):
    # Attention shape: any N1 >= 1, head dims K, N2 <= 128; MLP shape: any
    # N1, N2 <= 1024; the softmax needs a positive scale.
    from back_gemm_fusion_gb300.binding import cf_matrix, b2b_desc, CF_FP32, CF_BF16

    def call(M, K, N1, N2, op="scale_softmax", scale=0.125, trans=True):
        A = cf_matrix(0x10000, CF_BF16, 0, M, K, K + (-K) % 8)
        W1 = cf_matrix(0x20000, CF_BF16, 1, K, N1, K + (-K) % 8) if trans else \
            cf_matrix(0x20000, CF_BF16, 0, K, N1, N1 + (-N1) % 8)
        W2 = cf_matrix(0x30000, CF_BF16, 0, N1, N2, N2 + (-N2) % 8)
        O = cf_matrix(0x40000, CF_FP32, 0, M, N2, N2 + (-N2) % 4)
        d = b2b_desc(op, scale, 1)
        return lib.cf_b2bgemm(ctypes.byref(A), ctypes.byref(W1), ctypes.byref(W2), ctypes.byref(d),
                              ctypes.byref(O), None)

    ok = (0, 4, 8)
    assert call(256, 128, 100, 128) in ok                 # ragged keys
    assert call(256, 128, 1, 128) in ok                   # a single key
    assert call(256, 64, 200, 64) in ok                   # head dim 64
    assert call(77, 96, 300, 32) in ok                    # head dims 96 / 32
    assert call(256, 136, 256, 128) == 2                  # head dim above 128
    assert call(256, 60, 256, 128) == 2                   # K % 8 != 0
    assert call(256, 128, 0, 128) == 2                    # no keys
    assert call(256, 128, 256, 128, scale=0.0) == 1       # softmax scale must be positive
    assert call(256, 128, 256, 128, scale=-0.5) == 1
    assert call(256, 128, 256, 128, op="scale_relu", scale=-0.5) in ok  # ReLU takes any finite scale
    assert call(256, 256, 200, 300, op="relu", trans=False) in ok       # MLP, ragged N1 and N2
    assert call(256, 256, 512, 1000, op="relu", trans=False) in ok      # MLP, C = 4, last block ragged
    assert call(256, 256, 512, 1100, op="relu", trans=False) == 2       # MLP, C = 5 > 4
    assert call(256, 16, 512, 256, op="relu", trans=False) in ok        # MLP, K below one 64-wide block
    assert call(256, 8, 512, 256, op="relu", trans=True) in ok


def test_dynamic_exchange_rules(lib):
    # CF_XCHG_GLOBAL_DYNAMIC (3) is accepted for single-stage programs and
    # refused for chained ones; larger values are argument errors.
    from back_gemm_fusion_gb300.binding import epi_desc
    A, B, O = _mats()
    ok = (0, 4, 8)

    def call(ops, exchange):
        d = epi_desc(ops)
        d.exchange = exchange
        return lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000, ctypes.byref(d),
                                    ctypes.byref(O), 0x80000, 1 << 24, None)

    assert call([("bias",), ("layernorm", 1e-5)], 3) in ok
    assert call([("bias",), ("layernorm", 1e-5), ("rmsnorm", 1e-6)], 3) == 2
    assert call([("bias",), ("layernorm", 1e-5)], 4) == 1


def test_b2b_key_split_rules(lib):
    # Descriptor version 2 carries key_split (0 auto, 1 off, 2..8 CTAs per
    # query block); out-of-range values are argument errors found on the
    # host; version-1 descriptors (no key_split field) are still accepted.
    from back_gemm_fusion_gb300.binding import cf_matrix, b2b_desc, CF_BF16, CF_FP32
    Q = cf_matrix(0x10000, CF_BF16, 0, 128, 128, 128)
    K = cf_matrix(0x20000, CF_BF16, 1, 128, 2048, 128)
    V = cf_matrix(0x30000, CF_BF16, 0, 2048, 128, 128)
    O = cf_matrix(0x40000, CF_FP32, 0, 128, 128, 128)

    def call(ks, version=2):
        d = b2b_desc("scale_softmax", 0.125, 1, key_split=ks)
        d.version = version
        return lib.cf_b2bgemm(ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V), ctypes.byref(d), ctypes.byref(O),
                              None)

    ok = (0, 4, 8)
    for ks in (0, 1, 2, 3, 8):
        assert call(ks) in ok
    assert call(-1) == 1
    assert call(9) == 1
    assert call(9, version=1) in ok      # version 1 never reads the field
    assert call(0, version=3) == 1       # unknown version


def test_column_axis_rules(lib):
    # Column reductions: descriptor version 3, B given as N x K, the kernel
    # runs on P^T (so the workspace follows the swapped shape).
    from back_gemm_fusion_gb300.binding import cf_matrix, epi_desc, CF_BF16, CF_FP32
    M, N, K = 4096, 512, 256
    A = cf_matrix(0x10000, CF_BF16, 0, M, K, K)
    Bt = cf_matrix(0x20000, CF_BF16, 1, K, N, K)     # stored N x K
    Bn = cf_matrix(0x20000, CF_BF16, 0, K, N, N)     # stored K x N
    O = cf_matrix(0x30000, CF_FP32, 0, M, N, N)

    def call(B, ops, axis="col", exchange="auto", ws=0x80000, ws_bytes=1 << 24):
        d = epi_desc(ops, exchange, axis=axis)
        return lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000, ctypes.byref(d),
                                    ctypes.byref(O), ws, ws_bytes, None)

    assert call(Bt, LN) in (0, 4, 8)                          # B as N x K: supported
    assert call(Bn, LN) == 2                                  # B as K x N: the kernel needs it K-major
    assert call(Bn, [("bias",), ("relu",)]) in (0, 4, 8)      # no reduction: the axis is ignored
    assert call(Bt, LN, exchange="cluster") in (0, 4, 8)      # the reduced dim M = 4096: 16 tiles fit a cluster
    A17 = cf_matrix(0x10000, CF_BF16, 0, 4352, K, K)
    O17 = cf_matrix(0x30000, CF_FP32, 0, 4352, N, N)
    d17 = epi_desc(LN, "cluster", axis="col")
    assert lib.cf_gemm_epilogue(ctypes.byref(A17), ctypes.byref(Bt), 0x40000, 0x50000, 0x60000, ctypes.byref(d17),
                                ctypes.byref(O17), 0x80000, 1 << 24, None) == 2  # 17 tiles down a column
    d = epi_desc(LN, axis="col")
    d.axis = 2
    assert lib.cf_gemm_epilogue(ctypes.byref(A), ctypes.byref(Bt), 0x40000, 0x50000, 0x60000, ctypes.byref(d),
                                ctypes.byref(O), 0x80000, 1 << 24, None) == 1  # unknown axis
    # Workspace: strips of P^T (N / 128 = 4) x tiles along M (4096 / 256 = 16).
    ws_col = lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(Bt), ctypes.byref(epi_desc(LN, axis="col")))
    ws_row = lib.cf_workspace_size(ctypes.byref(A), ctypes.byref(Bt), ctypes.byref(epi_desc(LN, axis="row")))
    # Statistics (strips x tiles x 128 rows x 8 bytes) then 16 bytes of
    # counters per strip and a 4-byte ticket counter, each region padded to
    # 256 bytes.
    assert ws_col == 4 * 16 * 128 * 8 + 256      # 4 strips of P^T, 16 tiles along M
    assert ws_row == 32 * 2 * 128 * 8 + 768      # 32 strips of P, 2 tiles along N (516 -> 768)
    # An unknown axis is rejected by the unfused path too.
    dd = epi_desc(LN, axis="col")
    dd.axis = 5
    assert lib.cf_unfused_gemm_epilogue(ctypes.byref(A), ctypes.byref(Bt), 0x40000, 0x50000, 0x60000,
                                        ctypes.byref(dd), ctypes.byref(O), 0x90000, None) == 1


def test_b2b_batch_output_must_not_overlap(lib):
    from back_gemm_fusion_gb300.binding import cf_matrix, b2b_desc, CF_FP32, CF_BF16
    Q = cf_matrix(0x10000, CF_BF16, 0, 256, 128, 128)
    K = cf_matrix(0x20000, CF_BF16, 1, 128, 512, 128)
    V = cf_matrix(0x30000, CF_BF16, 0, 512, 128, 128)
    O = cf_matrix(0x40000, CF_FP32, 0, 256, 128, 128)

    def call(stride_out, stride_in=256 * 128):
        d = b2b_desc("scale_softmax", 0.125, 4, strides=(stride_in, 512 * 128, 512 * 128, stride_out))
        return lib.cf_b2bgemm(ctypes.byref(Q), ctypes.byref(K), ctypes.byref(V), ctypes.byref(d),
                              ctypes.byref(O), None)

    assert call(256 * 128) in (0, 4, 8)          # contiguous batch of outputs
    assert call(0) == 1                           # every entry writes the same output
    assert call(255 * 128) == 1                   # entries overlap by one row
    assert call(256 * 128, stride_in=0) in (0, 4, 8)  # a broadcast input is fine


def test_unfused_residual_alignment(lib):
    # The unfused row kernels read the residual with vector loads: the same
    # alignment rule as the fused call, checked before anything is enqueued.
    from back_gemm_fusion_gb300.binding import cf_matrix, epi_desc, CF_FP32, CF_BF16
    A, B, O = _mats()
    d = epi_desc([("bias",), ("residual",), ("layernorm", 1e-5)])
    d.residual = cf_matrix(0x70008, CF_FP32, 0, 256, 256, 256)      # misaligned pointer
    assert lib.cf_unfused_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000,
                                        ctypes.byref(d), ctypes.byref(O), 0x90000, None) == 3
    d.residual = cf_matrix(0x70000, CF_BF16, 0, 256, 256, 260)      # 520-byte rows
    assert lib.cf_unfused_gemm_epilogue(ctypes.byref(A), ctypes.byref(B), 0x40000, 0x50000, 0x60000,
                                        ctypes.byref(d), ctypes.byref(O), 0x90000, None) == 3
