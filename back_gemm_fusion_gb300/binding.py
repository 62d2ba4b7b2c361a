"""ctypes binding of ``libcf_gb300.so`` (argument marshalling only).

Every function here has the name of the C entry point it wraps and does no
arithmetic of its own: it builds the ``cf_matrix`` / descriptor structs from
torch CUDA tensors (pointer, strides) and the caller's current CUDA stream,
calls the library, and raises ``CFError`` on a non-OK status.  There is no
CPU fallback: if the library is missing the import of this module's loader
fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libcf_gb300.so")

# ------------------------------------------------------------------- C types
CF_OK = 0
STATUS_NAMES = {0: "CF_OK", 1: "CF_ERR_INVALID_ARG", 2: "CF_ERR_UNSUPPORTED_SHAPE", 3: "CF_ERR_MISALIGNED",
                4: "CF_ERR_UNSUPPORTED_DEVICE", 5: "CF_ERR_CUDA", 6: "CF_ERR_TIMEOUT", 7: "CF_ERR_WORKSPACE",
                8: "CF_ERR_NO_DEVICE"}
CF_BF16, CF_FP32 = 0, 1
OP_CODES = {"bias": 1, "scale": 2, "relu": 3, "gelu_tanh": 4, "residual": 5, "layernorm": 16, "rmsnorm": 17,
            "softmax": 18}
MID_CODES = {"relu": 1, "scale_relu": 2, "scale_softmax": 3}
EXCHANGE_CODES = {"auto": 0, "cluster": 1, "global": 2, "global_dynamic": 3}
EPI_MAX_OPS = 8


class cf_matrix(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("trans", ctypes.c_int32),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld", ctypes.c_int64)]


class cf_op(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("scalar", ctypes.c_float)]


class cf_epi_desc(ctypes.Structure):
    _fields_ = [("version", ctypes.c_uint32), ("n_ops", ctypes.c_uint32), ("ops", cf_op * EPI_MAX_OPS),
                ("out_dtype", ctypes.c_int32), ("exchange", ctypes.c_int32), ("residual", cf_matrix),
                ("stage0_gamma", ctypes.c_void_p), ("stage0_beta", ctypes.c_void_p), ("axis", ctypes.c_int32)]


class cf_device_model(ctypes.Structure):
    _fields_ = [("tensor_tflops", ctypes.c_double), ("hbm_gbs", ctypes.c_double), ("sms", ctypes.c_int32),
                ("clock_ghz", ctypes.c_double), ("launch_us", ctypes.c_double)]


class cf_cost(ctypes.Structure):
    _fields_ = [("flops", ctypes.c_double), ("fused_bytes", ctypes.c_double), ("unfused_bytes", ctypes.c_double),
                ("mainloop_us", ctypes.c_double), ("epilogue_us", ctypes.c_double), ("fused_us", ctypes.c_double),
                ("unfused_us", ctypes.c_double), ("fused_preferred", ctypes.c_int32),
                ("epilogue_hidden", ctypes.c_int32)]


class cf_b2b_desc(ctypes.Structure):
    _fields_ = [("version", ctypes.c_uint32), ("mid_op", ctypes.c_int32), ("mid_scale", ctypes.c_float),
                ("out_dtype", ctypes.c_int32), ("batch", ctypes.c_int64), ("strideA", ctypes.c_int64),
                ("strideW1", ctypes.c_int64), ("strideW2", ctypes.c_int64), ("strideOut", ctypes.c_int64),
                ("key_split", ctypes.c_int32)]


class CFError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


_P = ctypes.POINTER
_SIGNATURES = {
    "cf_gemm_epilogue": (ctypes.c_int, [_P(cf_matrix), _P(cf_matrix), ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, _P(cf_epi_desc), _P(cf_matrix), ctypes.c_void_p,
                                        ctypes.c_size_t, ctypes.c_void_p]),
    "cf_workspace_size": (ctypes.c_size_t, [_P(cf_matrix), _P(cf_matrix), _P(cf_epi_desc)]),
    "cf_gemm_epilogue_noalloc": (ctypes.c_int, [_P(cf_matrix), _P(cf_matrix), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, _P(cf_epi_desc), _P(cf_matrix), ctypes.c_void_p]),
    "cf_b2bgemm": (ctypes.c_int, [_P(cf_matrix), _P(cf_matrix), _P(cf_matrix), _P(cf_b2b_desc),
                                  _P(cf_matrix), ctypes.c_void_p]),
    "cf_unfused_gemm_epilogue": (ctypes.c_int, [_P(cf_matrix), _P(cf_matrix), ctypes.c_void_p, ctypes.c_void_p,
                                                ctypes.c_void_p, _P(cf_epi_desc), _P(cf_matrix), ctypes.c_void_p,
                                                ctypes.c_void_p]),
    "cf_unfused_b2bgemm": (ctypes.c_int, [_P(cf_matrix), _P(cf_matrix), _P(cf_matrix), _P(cf_b2b_desc),
                                          _P(cf_matrix), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "cf_cost_gemm_epilogue": (ctypes.c_int, [_P(cf_matrix), _P(cf_matrix), _P(cf_epi_desc), _P(cf_device_model),
                                             _P(cf_cost)]),
    "cf_cost_b2bgemm": (ctypes.c_int, [_P(cf_matrix), _P(cf_matrix), _P(cf_matrix), _P(cf_b2b_desc),
                                       _P(cf_device_model), _P(cf_cost)]),
    "cf_last_device_status": (ctypes.c_int, [ctypes.c_void_p]),
    "cf_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "cf_abi_version": (ctypes.c_int, []),
}

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) the C-ABI library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libcf_gb300.so not found at {path}: run back_gemm_fusion_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


# ------------------------------------------------------------- marshalling
def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CF_BF16
    if t.dtype == torch.float32:
        return CF_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def matrix(t: torch.Tensor, trans: bool = False) -> cf_matrix:
    """cf_matrix view of a 2-D tensor with unit column stride.

    ``trans=True`` describes the logical transpose of ``t`` (the stored matrix
    is ``t``, the operand is ``t.T``)."""
    if t.dim() != 2:
        raise ValueError("expected a 2-D tensor")
    if t.stride(1) != 1:
        raise ValueError("the innermost dimension must be contiguous")
    rows, cols = t.shape
    if trans:
        rows, cols = cols, rows
    return cf_matrix(t.data_ptr(), _dtype_code(t), 1 if trans else 0, rows, cols, max(t.stride(0), 1))


AXIS_CODES = {"row": 0, "col": 1}


def epi_desc(ops: Sequence[Tuple], exchange: str = "auto", residual: Optional[torch.Tensor] = None,
             stage0_gamma: Optional[torch.Tensor] = None, stage0_beta: Optional[torch.Tensor] = None,
             out_dtype: int = CF_FP32, axis: str = "row") -> cf_epi_desc:
    """Descriptor (version 3); ``residual`` is the M x N matrix read by the
    ``residual`` op, ``stage0_gamma`` / ``stage0_beta`` the affine vectors of
    the first of two reductions, ``out_dtype`` CF_FP32 or CF_BF16, ``axis``
    "row" (reductions along rows) or "col" (down columns)."""
    d = cf_epi_desc()
    d.version = 3
    d.axis = AXIS_CODES[axis]
    d.n_ops = len(ops)
    if len(ops) > EPI_MAX_OPS:
        raise ValueError("too many epilogue ops")
    for i, op in enumerate(ops):
        d.ops[i].kind = OP_CODES[op[0]]
        d.ops[i].scalar = float(op[1]) if len(op) > 1 else 0.0
    d.out_dtype = out_dtype
    d.exchange = EXCHANGE_CODES[exchange]
    if residual is not None:
        d.residual = matrix(residual)
    d.stage0_gamma = None if stage0_gamma is None else stage0_gamma.data_ptr()
    d.stage0_beta = None if stage0_beta is None else stage0_beta.data_ptr()
    return d


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != CF_OK:
        raise CFError(status, where)


# ----------------------------------------------------------------- wrappers
def cf_workspace_size(A: torch.Tensor, B: torch.Tensor, ops: Sequence[Tuple], b_trans: bool = False,
                      exchange: str = "auto", axis: str = "row") -> int:
    lib = load_library()
    a, b, d = matrix(A), matrix(B, b_trans), epi_desc(ops, exchange, axis=axis)
    return int(lib.cf_workspace_size(ctypes.byref(a), ctypes.byref(b), ctypes.byref(d)))


def cf_gemm_epilogue(A: torch.Tensor, B: torch.Tensor, ops: Sequence[Tuple], bias=None, gamma=None, beta=None,
                     out: Optional[torch.Tensor] = None, b_trans: bool = False, exchange: str = "auto",
                     workspace: Optional[torch.Tensor] = None, stream=None,
                     residual: Optional[torch.Tensor] = None, stage0_gamma: Optional[torch.Tensor] = None,
                     stage0_beta: Optional[torch.Tensor] = None,
                     out_dtype: torch.dtype = torch.float32, axis: str = "row") -> torch.Tensor:
    """out = epilogue(A @ B) in one fused kernel.  ``B`` is K x N, or N x K
    with ``b_trans=True``; ``residual`` (M x N, fp32 or bf16) feeds the
    ``residual`` op.  ``out`` is fp32 or bf16 (``out_dtype`` when it is
    allocated here).  ``axis="col"`` reduces down the columns (needs
    ``b_trans=True``).  A workspace is allocated if needed and not given."""
    lib = load_library()
    M = A.shape[0]
    N = B.shape[0] if b_trans else B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    a, b, o, d = (matrix(A), matrix(B, b_trans), matrix(out),
                  epi_desc(ops, exchange, residual, stage0_gamma, stage0_beta, _dtype_code(out), axis))
    need = int(lib.cf_workspace_size(ctypes.byref(a), ctypes.byref(b), ctypes.byref(d)))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    ws_ptr = _ptr(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.cf_gemm_epilogue(ctypes.byref(a), ctypes.byref(b), _ptr(bias), _ptr(gamma), _ptr(beta),
                              ctypes.byref(d), ctypes.byref(o), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "cf_gemm_epilogue")
    return out


def cf_gemm_epilogue_noalloc(A: torch.Tensor, B: torch.Tensor, ops: Sequence[Tuple], bias=None, gamma=None,
                             beta=None, out: Optional[torch.Tensor] = None, b_trans: bool = False,
                             exchange: str = "auto", stream=None,
                             residual: Optional[torch.Tensor] = None, stage0_gamma: Optional[torch.Tensor] = None,
                             stage0_beta: Optional[torch.Tensor] = None,
                             out_dtype: torch.dtype = torch.float32, axis: str = "row") -> torch.Tensor:
    """Same as cf_gemm_epilogue, but the library takes any scratch it needs
    from its own static device array: nothing is allocated by this call
    (``out`` must be given by callers that cannot allocate)."""
    lib = load_library()
    if out is None:
        M = A.shape[0]
        N = B.shape[0] if b_trans else B.shape[1]
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    a, b, o, d = (matrix(A), matrix(B, b_trans), matrix(out),
                  epi_desc(ops, exchange, residual, stage0_gamma, stage0_beta, _dtype_code(out), axis))
    st = lib.cf_gemm_epilogue_noalloc(ctypes.byref(a), ctypes.byref(b), _ptr(bias), _ptr(gamma), _ptr(beta),
                                      ctypes.byref(d), ctypes.byref(o), _stream(stream))
    _check(st, "cf_gemm_epilogue_noalloc")
    return out


def b2b_desc(op: str, scale: float, batch: int, strides=(0, 0, 0, 0), out_dtype: int = CF_FP32,
             key_split: int = 0) -> cf_b2b_desc:
    """B2BGEMM descriptor (version 2); ``key_split`` 0 = chosen per shape,
    1 = off, 2..8 = CTAs per query block (attention shape)."""
    d = cf_b2b_desc()
    d.version = 2
    d.key_split = key_split
    d.mid_op = MID_CODES[op]
    d.mid_scale = float(scale)
    d.out_dtype = out_dtype
    d.batch = batch
    d.strideA, d.strideW1, d.strideW2, d.strideOut = strides
    return d


def _b2b_views(A, W1, W2, w1_trans, out):
    """Per-problem 2-D views of possibly batched [b, r, c] tensors."""
    def first(t):
        return t[0] if t.dim() == 3 else t

    def bstride(t):
        return t.stride(0) if t.dim() == 3 else 0
    batch = A.shape[0] if A.dim() == 3 else 1
    a, w1, w2, o = matrix(first(A)), matrix(first(W1), w1_trans), matrix(first(W2)), matrix(first(out))
    return batch, (a, w1, w2, o), (bstride(A), bstride(W1), bstride(W2), bstride(out))


def cf_b2bgemm(A: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, op: str, scale: float = 1.0,
               w1_trans: bool = False, out: Optional[torch.Tensor] = None, stream=None,
               out_dtype: torch.dtype = torch.float32, key_split: int = 0) -> torch.Tensor:
    """out = bf16(F(A @ W1)) @ W2, fused; tensors may carry a leading batch
    dim.  ``out`` is fp32 or bf16 (``out_dtype`` when it is allocated here).
    ``key_split`` (attention shape): 0 = chosen per shape, 1 = one CTA per
    query block, 2..8 = CTAs of a cluster sharing a block's key range."""
    lib = load_library()
    if out is None:
        shape = A.shape[:-1] + (W2.shape[-1],)
        out = torch.empty(shape, dtype=out_dtype, device=A.device)
    batch, (a, w1, w2, o), strides = _b2b_views(A, W1, W2, w1_trans, out)
    d = b2b_desc(op, scale, batch, strides, _dtype_code(out), key_split)
    st = lib.cf_b2bgemm(ctypes.byref(a), ctypes.byref(w1), ctypes.byref(w2), ctypes.byref(d), ctypes.byref(o),
                        _stream(stream))
    _check(st, "cf_b2bgemm")
    return out


def cf_unfused_gemm_epilogue(A, B, ops, bias=None, gamma=None, beta=None, out=None, b_trans=False,
                             intermediate=None, stream=None, residual=None, stage0_gamma=None, stage0_beta=None,
                             axis: str = "row"):
    """Comparison path: cuBLASLt GEMM to an fp32 intermediate, then a separate
    epilogue kernel (row or column reductions)."""
    lib = load_library()
    M = A.shape[0]
    N = B.shape[0] if b_trans else B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    if intermediate is None:
        intermediate = torch.empty((M, N), dtype=torch.float32, device=A.device)
    a, b, o, d = (matrix(A), matrix(B, b_trans), matrix(out),
                  epi_desc(ops, residual=residual, stage0_gamma=stage0_gamma, stage0_beta=stage0_beta, axis=axis))
    st = lib.cf_unfused_gemm_epilogue(ctypes.byref(a), ctypes.byref(b), _ptr(bias), _ptr(gamma), _ptr(beta),
                                      ctypes.byref(d), ctypes.byref(o), _ptr(intermediate), _stream(stream))
    _check(st, "cf_unfused_gemm_epilogue")
    return out


def cf_unfused_b2bgemm(A, W1, W2, op, scale=1.0, w1_trans=False, out=None, s_buf=None, p_buf=None, stream=None):
    """Comparison path: cuBLASLt GEMM1, a mid-op kernel writing bf16 S', cuBLASLt GEMM2."""
    lib = load_library()
    if out is None:
        out = torch.empty(A.shape[:-1] + (W2.shape[-1],), dtype=torch.float32, device=A.device)
    n1 = W1.shape[-2] if w1_trans else W1.shape[-1]
    mid_shape = A.shape[:-1] + (n1,)
    if s_buf is None:
        s_buf = torch.empty(mid_shape, dtype=torch.float32, device=A.device)
    if p_buf is None:
        p_buf = torch.empty(mid_shape, dtype=torch.bfloat16, device=A.device)
    batch, (a, w1, w2, o), strides = _b2b_views(A, W1, W2, w1_trans, out)
    d = b2b_desc(op, scale, batch, strides, _dtype_code(out))
    st = lib.cf_unfused_b2bgemm(ctypes.byref(a), ctypes.byref(w1), ctypes.byref(w2), ctypes.byref(d),
                                ctypes.byref(o), _ptr(s_buf), _ptr(p_buf), _stream(stream))
    _check(st, "cf_unfused_b2bgemm")
    return out


def _device_model(device: Optional[dict]) -> cf_device_model:
    dm = cf_device_model(0.0, 0.0, 0, 0.0, -1.0)  # library defaults (a GB300)
    for k, v in (device or {}).items():
        setattr(dm, k, v)
    return dm


def _cost_dict(c: cf_cost) -> dict:
    return {name: getattr(c, name) for name, _ in cf_cost._fields_}


def cf_cost_gemm_epilogue(M: int, N: int, K: int, ops: Sequence[Tuple], b_trans: bool = False,
                          axis: str = "row", device: Optional[dict] = None) -> dict:
    """Predicted fused and unfused times of a GEMM + epilogue of this shape
    (host only; ``device`` overrides cf_device_model fields)."""
    lib = load_library()
    a = cf_matrix(0, CF_BF16, 0, M, K, K)
    b = cf_matrix(0, CF_BF16, 1, K, N, K) if b_trans else cf_matrix(0, CF_BF16, 0, K, N, N)
    d, c, dm = epi_desc(ops, axis=axis), cf_cost(), _device_model(device)
    _check(lib.cf_cost_gemm_epilogue(ctypes.byref(a), ctypes.byref(b), ctypes.byref(d), ctypes.byref(dm),
                                     ctypes.byref(c)), "cf_cost_gemm_epilogue")
    return _cost_dict(c)


def cf_cost_b2bgemm(M: int, K: int, N1: int, N2: int, op: str, scale: float = 1.0, batch: int = 1,
                    w1_trans: bool = False, device: Optional[dict] = None) -> dict:
    """Predicted fused and unfused times of a B2BGEMM of this shape (host only)."""
    lib = load_library()
    a = cf_matrix(0, CF_BF16, 0, M, K, K)
    w1 = cf_matrix(0, CF_BF16, 1, K, N1, K) if w1_trans else cf_matrix(0, CF_BF16, 0, K, N1, N1)
    w2 = cf_matrix(0, CF_BF16, 0, N1, N2, N2)
    d, c, dm = b2b_desc(op, scale, batch), cf_cost(), _device_model(device)
    _check(lib.cf_cost_b2bgemm(ctypes.byref(a), ctypes.byref(w1), ctypes.byref(w2), ctypes.byref(d), ctypes.byref(dm),
                               ctypes.byref(c)), "cf_cost_b2bgemm")
    return _cost_dict(c)


def cf_last_device_status(stream=None) -> int:
    return int(load_library().cf_last_device_status(_stream(stream)))


def cf_status_string(status: int) -> str:
    return load_library().cf_status_string(status).decode()
