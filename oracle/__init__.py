"""CPU oracle for the weight-quantized linear layers (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
this package.  The library path never does: it shares no code with the CUDA sources and the
CUDA path never falls back to it.

The arithmetic lives in ``wql_oracle.c`` (plain C, ``-O2 -ffp-contract=off``, optional OpenMP);
this module only compiles it on first use and marshals numpy arrays through ctypes.  Every
function names the passage of the source pages it restates; see the header of the C file.

Parity status: every function here is pinned by ``tests/test_oracle.py`` against facts that do
not come from the oracle itself (numpy's binary16 conversion, exact rational arithmetic,
Python integers, closed forms and invariants of the method, the one worked example printed
on the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wql_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libwql_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float

_SIGS = {
    "wql_oracle_half_to_float_n": (None, [_P, _P, _I64]),
    "wql_oracle_float_to_half_n": (None, [_P, _P, _I64]),
    "wql_oracle_num_threads": (_I, []),
    "wql_oracle_awq_quantize": (None, [_P, _I, _I, _I, _P, _P, _P]),
    "wql_oracle_awq_unpack": (None, [_P, _P, _I, _I, _I, _P, _P]),
    "wql_oracle_awq_dequant": (None, [_P, _P, _P, _I, _I, _I, _P]),
    "wql_oracle_w4a16_linear": (None, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _P]),
    "wql_oracle_sumsq": (_F, [_P, _I]),
    "wql_oracle_rmsnorm": (None, [_P, _P, _F, _I, _I, _P]),
    "wql_oracle_qrmsnorm_quant_i8": (None, [_P, _P, _F, _I, _I, _P, _P]),
    "wql_oracle_act_absmax": (None, [_P, _P, _F, _I, _I, _P]),
    "wql_oracle_smooth": (None, [_P, _P, _P, _I, _I, _P, _P, _P]),
    "wql_oracle_per_channel_quant_i8": (None, [_P, _I, _I, _P, _P]),
    "wql_oracle_w8a8_acc": (_I, [_P, _P, _I, _I, _P, _I, _P]),
    "wql_oracle_w8a8_epilogue": (None, [_P, _P, _P, _I, _I, _P]),
    "wql_oracle_w8a8_epilogue_fused": (None, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "wql_oracle_add_qrmsnorm_quant_i8": (None, [_P, _P, _P, _F, _I, _I, _P, _P, _P]),
    "wql_oracle_per_token_quant_i8": (None, [_P, _I, _I, _P, _P]),
    "wql_oracle_per_token_quant_fp8": (None, [_P, _I, _I, _P, _P]),
    "wql_oracle_w8a8_epilogue_f64": (None, [_P, _P, _P, _I, _I, _P]),
    "wql_oracle_sym_int4_per_tensor": (_F, [_P, _I64, _P]),
    "wql_oracle_e4m3_to_float_n": (None, [_P, _P, _I64]),
    "wql_oracle_float_to_e4m3_n": (None, [_P, _P, _I64]),
    "wql_oracle_qrmsnorm_quant_fp8": (None, [_P, _P, _F, _I, _I, _P, _P]),
    "wql_oracle_add_qrmsnorm_quant_fp8": (None, [_P, _P, _P, _F, _I, _I, _P, _P, _P]),
    "wql_oracle_per_channel_quant_fp8": (None, [_P, _I, _I, _P, _P]),
    "wql_oracle_fp8_acc": (_I, [_P, _P, _I, _I, _P, _I, _P, _P]),
    "wql_oracle_fp8_epilogue_f64": (None, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "wql_oracle_silu_mul_f64": (None, [_P, _I64, _I, _P]),
    "wql_oracle_kv_quant_i8": (None, [_P, _I64, _I, _P, _P]),
    "wql_oracle_kv_dequant_i8": (None, [_P, _P, _I64, _I, _P]),
}


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libwql_oracle.so`` (gcc, no GPU needed)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
           "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _half_bits(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        return np.ascontiguousarray(a).view(np.uint16)
    assert a.dtype == np.uint16, "fp16 data must be float16 or its uint16 bit pattern"
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return int(_load().wql_oracle_num_threads())


# ---- binary16 ------------------------------------------------------------------------

def half_to_float(h) -> np.ndarray:
    h = _half_bits(h)
    out = np.empty(h.shape, np.float32)
    _load().wql_oracle_half_to_float_n(_ptr(h), _ptr(out), h.size)
    return out


def float_to_half(x) -> np.ndarray:
    """Round fp32 values to binary16 (ties to even); returns float16 array."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _load().wql_oracle_float_to_half_n(_ptr(x), _ptr(out), x.size)
    return out.view(np.float16)


# ---- AWQ W4A16 -------------------------------------------------------------------------

def awq_quantize(W, group: int):
    """Asymmetric per-group int4 quantisation and packing of W [K, N] fp32.

    Returns (qweight u32 [K, N/8], scales f16 [K/G, N], qzeros u32 [K/G, N/8]).
    """
    W = _c(W, np.float32)
    K, N = W.shape
    assert K % group == 0 and N % 8 == 0
    qweight = np.empty((K, N // 8), np.uint32)
    scales = np.empty((K // group, N), np.uint16)
    qzeros = np.empty((K // group, N // 8), np.uint32)
    _load().wql_oracle_awq_quantize(_ptr(W), K, N, group, _ptr(qweight), _ptr(scales), _ptr(qzeros))
    return qweight, scales.view(np.float16), qzeros


def awq_unpack(qweight, qzeros, K: int, N: int, group: int):
    """Codes q [K, N] and zero points z [K/G, N] as uint8."""
    qweight = _c(qweight, np.uint32)
    qzeros = _c(qzeros, np.uint32)
    q = np.empty((K, N), np.uint8)
    z = np.empty((K // group, N), np.uint8)
    _load().wql_oracle_awq_unpack(_ptr(qweight), _ptr(qzeros), K, N, group, _ptr(q), _ptr(z))
    return q, z


def awq_dequant(qweight, scales, qzeros, K: int, N: int, group: int) -> np.ndarray:
    """w[k, n] = (q - z) * s in fp32, shape [K, N]."""
    w = np.empty((K, N), np.float32)
    _load().wql_oracle_awq_dequant(_ptr(_c(qweight, np.uint32)), _ptr(_half_bits(scales)),
                                   _ptr(_c(qzeros, np.uint32)), K, N, group, _ptr(w))
    return w


def w4a16_linear(X, qweight, scales, qzeros, group: int, rows=None) -> np.ndarray:
    """Y = X @ dequant(W) with fp64 accumulation; X fp16 [M, K]; returns fp64 [len(rows), N]."""
    Xb = _half_bits(X)
    M, K = Xb.shape
    N = qweight.shape[1] * 8
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    Y = np.empty((rows.size, N), np.float64)
    _load().wql_oracle_w4a16_linear(_ptr(Xb), _ptr(_c(qweight, np.uint32)), _ptr(_half_bits(scales)),
                                    _ptr(_c(qzeros, np.uint32)), K, N, group, _ptr(rows),
                                    rows.size, _ptr(Y))
    return Y


# ---- SmoothQuant W8A8 --------------------------------------------------------------------

def sumsq(x) -> float:
    xb = _half_bits(x)
    return float(_load().wql_oracle_sumsq(_ptr(xb), xb.size))


def rmsnorm(X, gamma, eps: float) -> np.ndarray:
    Xb = _half_bits(X)
    M, K = Xb.shape
    out = np.empty((M, K), np.float32)
    _load().wql_oracle_rmsnorm(_ptr(Xb), _ptr(_half_bits(gamma)), eps, M, K, _ptr(out))
    return out


def qrmsnorm_quant_i8(X, gamma, eps: float):
    """Returns (q int8 [M, K], xs fp32 [M])."""
    Xb = _half_bits(X)
    M, K = Xb.shape
    q = np.empty((M, K), np.int8)
    xs = np.empty((M,), np.float32)
    _load().wql_oracle_qrmsnorm_quant_i8(_ptr(Xb), _ptr(_half_bits(gamma)), eps, M, K, _ptr(q), _ptr(xs))
    return q, xs


def add_qrmsnorm_quant_i8(X, R, gamma, eps: float):
    """Residual-fused QRMSNorm: returns (h fp16 [M, K] = fp16(x + r), q int8 [M, K], xs fp32 [M])."""
    Xb, Rb = _half_bits(X), _half_bits(R)
    M, K = Xb.shape
    h = np.empty((M, K), np.uint16)
    q = np.empty((M, K), np.int8)
    xs = np.empty((M,), np.float32)
    _load().wql_oracle_add_qrmsnorm_quant_i8(_ptr(Xb), _ptr(Rb), _ptr(_half_bits(gamma)), eps, M, K, _ptr(h),
                                             _ptr(q), _ptr(xs))
    return h.view(np.float16), q, xs


def per_token_quant_i8(X):
    """[W8A8] per_token_quant_int8 of plain fp16 activations: returns (q int8 [M, K], xs fp32 [M])."""
    Xb = _half_bits(X)
    M, K = Xb.shape
    q = np.empty((M, K), np.int8)
    xs = np.empty((M,), np.float32)
    _load().wql_oracle_per_token_quant_i8(_ptr(Xb), M, K, _ptr(q), _ptr(xs))
    return q, xs


def per_token_quant_fp8(X):
    """fp8 (e4m3) twin of per_token_quant_i8: returns (q e4m3 codes uint8 [M, K], xs fp32 [M])."""
    Xb = _half_bits(X)
    M, K = Xb.shape
    q = np.empty((M, K), np.uint8)
    xs = np.empty((M,), np.float32)
    _load().wql_oracle_per_token_quant_fp8(_ptr(Xb), M, K, _ptr(q), _ptr(xs))
    return q, xs


def act_absmax(X, gamma, eps: float) -> np.ndarray:
    Xb = _half_bits(X)
    M, K = Xb.shape
    out = np.empty((K,), np.float32)
    _load().wql_oracle_act_absmax(_ptr(Xb), _ptr(_half_bits(gamma)), eps, M, K, _ptr(out))
    return out


def smooth(absmax, gamma, W):
    """Returns (s fp32 [K], gamma' fp16 [K], W' fp32 [K, N])."""
    W = _c(W, np.float32)
    K, N = W.shape
    s = np.empty((K,), np.float32)
    g = np.empty((K,), np.uint16)
    Wo = np.empty((K, N), np.float32)
    _load().wql_oracle_smooth(_ptr(_c(absmax, np.float32)), _ptr(_half_bits(gamma)), _ptr(W), K, N,
                              _ptr(s), _ptr(g), _ptr(Wo))
    return s, g.view(np.float16), Wo


def per_channel_quant_i8(W):
    """W [K, N] fp32 -> (qW int8 [N, K], ws fp32 [N])."""
    W = _c(W, np.float32)
    K, N = W.shape
    qW = np.empty((N, K), np.int8)
    ws = np.empty((N,), np.float32)
    _load().wql_oracle_per_channel_quant_i8(_ptr(W), K, N, _ptr(qW), _ptr(ws))
    return qW, ws


def w8a8_acc(q, qW, rows=None) -> np.ndarray:
    """int32 accumulators [len(rows), N] of q [M, K] times qW [N, K]^T (exact; raises on int32 overflow)."""
    q = _c(q, np.int8)
    qW = _c(qW, np.int8)
    M, K = q.shape
    N = qW.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    acc = np.empty((rows.size, N), np.int32)
    ovf = _load().wql_oracle_w8a8_acc(_ptr(q), _ptr(qW), K, N, _ptr(rows), rows.size, _ptr(acc))
    if ovf:
        raise OverflowError("int8 GEMM accumulator exceeds int32")
    return acc


def w8a8_epilogue(acc, xs, ws) -> np.ndarray:
    """fp16 [R, N] = fp16((float(acc) * xs) * ws); xs are the per-row scales of acc's rows."""
    acc = _c(acc, np.int32)
    R, N = acc.shape
    y = np.empty((R, N), np.uint16)
    _load().wql_oracle_w8a8_epilogue(_ptr(acc), _ptr(_c(xs, np.float32)), _ptr(_c(ws, np.float32)), R, N, _ptr(y))
    return y.view(np.float16)


def w8a8_epilogue_fused(acc, xs, ws, bias=None, residual=None) -> np.ndarray:
    """fp16 [R, N] = fp16(((float(acc) * xs) * ws + bias) + residual); a None term is left out."""
    acc = _c(acc, np.int32)
    R, N = acc.shape
    y = np.empty((R, N), np.uint16)
    b = None if bias is None else _half_bits(bias).reshape(N)
    r = None if residual is None else _half_bits(residual).reshape(R, N)
    _load().wql_oracle_w8a8_epilogue_fused(_ptr(acc), _ptr(_c(xs, np.float32)), _ptr(_c(ws, np.float32)),
                                           None if b is None else _ptr(b), None if r is None else _ptr(r), R, N,
                                           _ptr(y))
    return y.view(np.float16)


def w8a8_epilogue_f64(acc, xs, ws) -> np.ndarray:
    acc = _c(acc, np.int32)
    R, N = acc.shape
    y = np.empty((R, N), np.float64)
    _load().wql_oracle_w8a8_epilogue_f64(_ptr(acc), _ptr(_c(xs, np.float32)), _ptr(_c(ws, np.float32)), R, N, _ptr(y))
    return y


# ---- SmoothQuant W8A8, fp8 (e4m3) variant --------------------------------------------------

def _e4m3_bits(a) -> np.ndarray:
    """float8_e4m3fn codes as uint8 (torch float8 tensors are passed as their uint8 view)."""
    a = np.asarray(a)
    assert a.dtype == np.uint8, "e4m3 data must be its uint8 bit pattern"
    return np.ascontiguousarray(a)


def e4m3_to_float(b) -> np.ndarray:
    b = _e4m3_bits(b)
    out = np.empty(b.shape, np.float32)
    _load().wql_oracle_e4m3_to_float_n(_ptr(b), _ptr(out), b.size)
    return out


def float_to_e4m3(x) -> np.ndarray:
    """Nearest e4m3 code (ties to even, saturating at +-448) of fp32 values, as uint8."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().wql_oracle_float_to_e4m3_n(_ptr(x), _ptr(out), x.size)
    return out


def qrmsnorm_quant_fp8(X, gamma, eps: float):
    """Returns (q e4m3 codes uint8 [M, K], xs fp32 [M]) with xs = absmax / 448."""
    Xb = _half_bits(X)
    M, K = Xb.shape
    q = np.empty((M, K), np.uint8)
    xs = np.empty((M,), np.float32)
    _load().wql_oracle_qrmsnorm_quant_fp8(_ptr(Xb), _ptr(_half_bits(gamma)), eps, M, K, _ptr(q), _ptr(xs))
    return q, xs


def add_qrmsnorm_quant_fp8(X, R, gamma, eps: float):
    """Residual-fused fp8 QRMSNorm: returns (h fp16 [M, K], q e4m3 uint8 [M, K], xs fp32 [M])."""
    Xb, Rb = _half_bits(X), _half_bits(R)
    M, K = Xb.shape
    h = np.empty((M, K), np.uint16)
    q = np.empty((M, K), np.uint8)
    xs = np.empty((M,), np.float32)
    _load().wql_oracle_add_qrmsnorm_quant_fp8(_ptr(Xb), _ptr(Rb), _ptr(_half_bits(gamma)), eps, M, K, _ptr(h),
                                              _ptr(q), _ptr(xs))
    return h.view(np.float16), q, xs


def per_channel_quant_fp8(W):
    """W [K, N] fp32 -> (qW e4m3 uint8 [N, K], ws fp32 [N]) with ws = absmax / 448."""
    W = _c(W, np.float32)
    K, N = W.shape
    qW = np.empty((N, K), np.uint8)
    ws = np.empty((N,), np.float32)
    _load().wql_oracle_per_channel_quant_fp8(_ptr(W), K, N, _ptr(qW), _ptr(ws))
    return qW, ws


def fp8_acc(q, qW, rows=None):
    """Exact fp64 sums [len(rows), N] of e4m3 q [M, K] times qW [N, K]^T, and the sums of |products|."""
    q = _e4m3_bits(q)
    qW = _e4m3_bits(qW)
    M, K = q.shape
    N = qW.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    acc = np.empty((rows.size, N), np.float64)
    absacc = np.empty((rows.size, N), np.float64)
    if _load().wql_oracle_fp8_acc(_ptr(q), _ptr(qW), K, N, _ptr(rows), rows.size, _ptr(acc), _ptr(absacc)):
        raise ValueError("fp8 GEMM reference: K > 65536 or a NaN code")
    return acc, absacc


def fp8_epilogue_f64(acc, xs, ws, bias=None, residual=None) -> np.ndarray:
    """fp64 [R, N] = ((acc * xs) * ws + bias) + residual, unrounded; a None term is left out."""
    acc = _c(acc, np.float64)
    R, N = acc.shape
    y = np.empty((R, N), np.float64)
    b = None if bias is None else _half_bits(bias).reshape(N)
    r = None if residual is None else _half_bits(residual).reshape(R, N)
    _load().wql_oracle_fp8_epilogue_f64(_ptr(acc), _ptr(_c(xs, np.float32)), _ptr(_c(ws, np.float32)),
                                        None if b is None else _ptr(b), None if r is None else _ptr(r), R, N, _ptr(y))
    return y


# ---- fused gate/up: SiLU(gate) * up ------------------------------------------------------------

def silu_mul_f64(y) -> np.ndarray:
    """y [R, N] fp64 with gate j at column 2j and up j at 2j + 1 -> silu(gate) * up, [R, N / 2] fp64."""
    y = _c(y, np.float64)
    R, N = y.shape
    assert N % 2 == 0
    out = np.empty((R, N // 2), np.float64)
    _load().wql_oracle_silu_mul_f64(_ptr(y), R, N, _ptr(out))
    return out


# ---- KV-cache int8, groups of 128 ------------------------------------------------------------

def kv_quant_i8(kv):
    """kv [rows, D] fp16 (D % 128 == 0) -> (q int8 [rows, D], scales fp32 [rows, D / 128])."""
    kb = _half_bits(kv)
    rows, D = kb.shape
    assert D % 128 == 0
    q = np.empty((rows, D), np.int8)
    s = np.empty((rows, D // 128), np.float32)
    _load().wql_oracle_kv_quant_i8(_ptr(kb), rows, D, _ptr(q), _ptr(s))
    return q, s


def kv_dequant_i8(q, scales) -> np.ndarray:
    """fp16 [rows, D] = fp16(q * scale of the element's group)."""
    q = _c(q, np.int8)
    rows, D = q.shape
    out = np.empty((rows, D), np.uint16)
    _load().wql_oracle_kv_dequant_i8(_ptr(q), _ptr(_c(scales, np.float32)), rows, D, _ptr(out))
    return out.view(np.float16)


def sym_int4_per_tensor(w):
    """Off-path symmetric per-tensor int4 of the tutorial's section 2 example; returns (scale, q)."""
    w = _c(w, np.float32)
    q = np.empty(w.shape, np.int8)
    scale = _load().wql_oracle_sym_int4_per_tensor(_ptr(w), w.size, _ptr(q))
    return float(scale), q
