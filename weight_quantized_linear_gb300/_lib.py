"""ctypes binding of libwql.so: argument marshalling only.

Every computation happens in the CUDA kernels behind the C ABI declared in ``include/wql.h``.
Tensors are torch CUDA tensors (torch is used for device memory and streams only); the calls are
enqueued on the current torch stream of the tensors' device.  There is no CPU fallback: if the
library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libwql.so")

WQL_OK, WQL_EINVAL, WQL_EUNSUPPORTED, WQL_ECUDA, WQL_ETIMEOUT = range(5)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); this list is also what the export test checks against wql.h
SIGNATURES = {
    "wql_status_string": (ctypes.c_char_p, [_I]),
    "wql_last_error": (ctypes.c_char_p, []),
    "wql_version": (_I, []),
    "wql_device_status": (_I, [_P]),
    "wql_diag_expire_wait": (_I, [_P]),
    "wql_trace_setup": (_I, [_P, _P, ctypes.c_uint64, _I, _I]),
    "wql_awq_pack": (_I, [_P, _I, _I, _I, _P, _P, _P, _P]),
    "wql_w4a16_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "wql_w4a16_kernel_for": (_I, [_I, _I, _I, _I]),
    "wql_w4a16_gemm_silu_mul": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "wql_qrmsnorm_quant_i8": (_I, [_P, _P, _F, _I, _I, _P, _P, _P]),
    "wql_add_qrmsnorm_quant_i8": (_I, [_P, _P, _P, _F, _I, _I, _P, _P, _P, _P]),
    "wql_per_token_quant_i8": (_I, [_P, _I, _I, _P, _P, _P]),
    "wql_per_token_quant_fp8": (_I, [_P, _I, _I, _P, _P, _P]),
    "wql_w8a8_workspace_bytes": (_SZ, [_I, _I, _I]),
    "wql_w8a8_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "wql_w8a8_gemm_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "wql_w8a8_gemm_fused": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "wql_act_absmax": (_I, [_P, _P, _F, _I, _I, _P, _P]),
    "wql_smooth": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P]),
    "wql_per_channel_quant_i8": (_I, [_P, _I, _I, _P, _P, _P]),
    "wql_qrmsnorm_quant_fp8": (_I, [_P, _P, _F, _I, _I, _P, _P, _P]),
    "wql_add_qrmsnorm_quant_fp8": (_I, [_P, _P, _P, _F, _I, _I, _P, _P, _P, _P]),
    "wql_per_channel_quant_fp8": (_I, [_P, _I, _I, _P, _P, _P]),
    "wql_w8a8_gemm_fp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P]),
    "wql_kv_quant_i8": (_I, [_P, ctypes.c_int64, _I, _P, _P, _P]),
    "wql_kv_dequant_i8": (_I, [_P, _P, ctypes.c_int64, _I, _P, _P]),
}

_lock = threading.Lock()
_lib = None


class WQLError(RuntimeError):
    def __init__(self, status: int, fn: str, detail: str):
        self.status = status
        super().__init__(f"{fn}: status {status}: {detail}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libwql.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libwql.so not found at {p}; build it with weight_quantized_linear_gb300.build.build()")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _check(status: int, fn: str) -> None:
    if status != WQL_OK:
        lib = load()
        detail = lib.wql_last_error().decode() or lib.wql_status_string(status).decode()
        raise WQLError(status, fn, detail)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------------------------------------
# AWQ W4A16
# ---------------------------------------------------------------------------------------------

def awq_pack(w: torch.Tensor, group: int):
    """fp32 w [K, N] -> (qweight int32 [K, N/8], scales fp16 [K/G, N], qzeros int32 [K/G, N/8]).

    qweight / qzeros hold uint32 bit patterns in int32 tensors (torch has no uint32 arithmetic).
    """
    K, N = w.shape
    _need(w, "w", torch.float32, (K, N))
    dev = w.device
    qweight = torch.empty((K, N // 8), dtype=torch.int32, device=dev)
    scales = torch.empty((K // group, N), dtype=torch.float16, device=dev)
    qzeros = torch.empty((K // group, N // 8), dtype=torch.int32, device=dev)
    _check(load().wql_awq_pack(_ptr(w), K, N, group, _ptr(qweight), _ptr(scales), _ptr(qzeros), _stream(dev)),
           "wql_awq_pack")
    return qweight, scales, qzeros


def w4a16_gemm(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor, group: int,
               out: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp16 = x [M, K] fp16 @ dequant(qweight, scales, qzeros)."""
    M, K = x.shape
    N = qweight.shape[1] * 8
    _need(x, "x", torch.float16, (M, K))
    _need(qweight, "qweight", torch.int32, (K, N // 8))
    _need(scales, "scales", torch.float16, (K // group, N))
    _need(qzeros, "qzeros", torch.int32, (K // group, N // 8))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _need(out, "out", torch.float16, (M, N))
    _check(load().wql_w4a16_gemm(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(qzeros), M, K, N, group, _ptr(out),
                                 _stream(x.device)), "wql_w4a16_gemm")
    return out


def w4a16_gemm_silu_mul(x: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor,
                        group: int, out: torch.Tensor | None = None) -> torch.Tensor:
    """Fused gate/up projection: the packed weight has N = 2I channels with gate j at channel 2j and
    up j at 2j + 1; returns y [M, I] fp16 = fp16(silu(g) * u) of the GEMM's fp16 gate and up."""
    M, K = x.shape
    N = qweight.shape[1] * 8
    _need(x, "x", torch.float16, (M, K))
    _need(qweight, "qweight", torch.int32, (K, N // 8))
    _need(scales, "scales", torch.float16, (K // group, N))
    _need(qzeros, "qzeros", torch.int32, (K // group, N // 8))
    if out is None:
        out = torch.empty((M, N // 2), dtype=torch.float16, device=x.device)
    _need(out, "out", torch.float16, (M, N // 2))
    _check(load().wql_w4a16_gemm_silu_mul(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(qzeros), M, K, N, group,
                                          _ptr(out), _stream(x.device)), "wql_w4a16_gemm_silu_mul")
    return out


def interleave_gate_up(w_gate: torch.Tensor, w_up: torch.Tensor) -> torch.Tensor:
    """[K, I] gate and up weights -> the [K, 2I] fused weight that w4a16_gemm_silu_mul expects
    (column 2j = gate j, column 2j + 1 = up j); pack it with awq_pack."""
    if w_gate.shape != w_up.shape or w_gate.dim() != 2:
        raise ValueError("gate and up weights must both be [K, I]")
    return torch.stack([w_gate, w_up], dim=2).reshape(w_gate.shape[0], 2 * w_gate.shape[1]).contiguous()


# ---------------------------------------------------------------------------------------------
# SmoothQuant W8A8
# ---------------------------------------------------------------------------------------------

def qrmsnorm_quant_i8(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6,
                      q: torch.Tensor | None = None, xs: torch.Tensor | None = None):
    """x [M, K] fp16, gamma [K] fp16 -> (q int8 [M, K], xs fp32 [M])."""
    M, K = x.shape
    _need(x, "x", torch.float16, (M, K))
    _need(gamma, "gamma", torch.float16, (K,))
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if xs is None:
        xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(q, "q", torch.int8, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _check(load().wql_qrmsnorm_quant_i8(_ptr(x), _ptr(gamma), float(eps), M, K, _ptr(q), _ptr(xs), _stream(x.device)),
           "wql_qrmsnorm_quant_i8")
    return q, xs


def per_token_quant_i8(x: torch.Tensor, q: torch.Tensor | None = None, xs: torch.Tensor | None = None):
    """x [M, K] fp16 -> (q int8 [M, K], xs fp32 [M]): per-token int8 of the row itself (no norm)."""
    M, K = x.shape
    _need(x, "x", torch.float16, (M, K))
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if xs is None:
        xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(q, "q", torch.int8, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _check(load().wql_per_token_quant_i8(_ptr(x), M, K, _ptr(q), _ptr(xs), _stream(x.device)), "wql_per_token_quant_i8")
    return q, xs


def per_token_quant_fp8(x: torch.Tensor, q: torch.Tensor | None = None, xs: torch.Tensor | None = None):
    """x [M, K] fp16 -> (q float8_e4m3fn [M, K], xs fp32 [M]) with xs = absmax / 448."""
    M, K = x.shape
    _need(x, "x", torch.float16, (M, K))
    if q is None:
        q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=x.device)
    if xs is None:
        xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(q, "q", torch.float8_e4m3fn, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _check(load().wql_per_token_quant_fp8(_ptr(x), M, K, _ptr(q), _ptr(xs), _stream(x.device)),
           "wql_per_token_quant_fp8")
    return q, xs


def add_qrmsnorm_quant_i8(x: torch.Tensor, residual: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6,
                          residual_out: torch.Tensor | None = None, q: torch.Tensor | None = None,
                          xs: torch.Tensor | None = None):
    """Residual-fused QRMSNorm: h = fp16(x + residual) -> (h [M, K] fp16, q int8 [M, K], xs fp32 [M]).

    residual_out receives h (it may be `residual` itself, for an in-place update)."""
    M, K = x.shape
    _need(x, "x", torch.float16, (M, K))
    _need(residual, "residual", torch.float16, (M, K))
    _need(gamma, "gamma", torch.float16, (K,))
    if residual_out is None:
        residual_out = torch.empty((M, K), dtype=torch.float16, device=x.device)
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if xs is None:
        xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(residual_out, "residual_out", torch.float16, (M, K))
    _need(q, "q", torch.int8, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _check(load().wql_add_qrmsnorm_quant_i8(_ptr(x), _ptr(residual), _ptr(gamma), float(eps), M, K, _ptr(residual_out),
                                            _ptr(q), _ptr(xs), _stream(x.device)), "wql_add_qrmsnorm_quant_i8")
    return residual_out, q, xs


def w4a16_kernel_for(M: int, K: int, N: int, group: int) -> str:
    """The kernel w4a16_gemm runs for this shape and group size: "decode" or "prefill"."""
    return "prefill" if load().wql_w4a16_kernel_for(M, K, N, group) else "decode"


def w8a8_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(load().wql_w8a8_workspace_bytes(M, K, N))


def w8a8_gemm(q: torch.Tensor, xs: torch.Tensor, qw: torch.Tensor, ws: torch.Tensor,
              out: torch.Tensor | None = None, acc_out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp16 = fp16((float(q @ qw^T) * xs) * ws); optional exact int32 acc_out [M, N]."""
    M, K = q.shape
    N = qw.shape[0]
    _need(q, "q", torch.int8, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _need(qw, "qw", torch.int8, (N, K))
    _need(ws, "ws", torch.float32, (N,))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=q.device)
    _need(out, "out", torch.float16, (M, N))
    if acc_out is not None:
        _need(acc_out, "acc_out", torch.int32, (M, N))
    need = w8a8_workspace_bytes(M, K, N)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().wql_w8a8_gemm(_ptr(q), _ptr(xs), _ptr(qw), _ptr(ws), M, K, N, _ptr(out), _ptr(acc_out),
                                _ptr(workspace), ws_bytes, _stream(q.device)), "wql_w8a8_gemm")
    return out


def w8a8_gemm_fused(q: torch.Tensor, xs: torch.Tensor, qw: torch.Tensor, ws: torch.Tensor,
                    bias: torch.Tensor | None = None, residual: torch.Tensor | None = None,
                    out: torch.Tensor | None = None, acc_out: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp16 = fp16(((float(q @ qw^T) * xs) * ws + bias) + residual); bias [N] and residual
    [M, N] fp16 are optional (None leaves the term out); `out` may be `residual` (in place)."""
    M, K = q.shape
    N = qw.shape[0]
    _need(q, "q", torch.int8, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _need(qw, "qw", torch.int8, (N, K))
    _need(ws, "ws", torch.float32, (N,))
    if bias is not None:
        _need(bias, "bias", torch.float16, (N,))
    if residual is not None:
        _need(residual, "residual", torch.float16, (M, N))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=q.device)
    _need(out, "out", torch.float16, (M, N))
    if acc_out is not None:
        _need(acc_out, "acc_out", torch.int32, (M, N))
    need = w8a8_workspace_bytes(M, K, N)
    if workspace is None and need > 0:
        workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().wql_w8a8_gemm_fused(_ptr(q), _ptr(xs), _ptr(qw), _ptr(ws), _ptr(bias), _ptr(residual), M, K, N,
                                      _ptr(out), _ptr(acc_out), _ptr(workspace), ws_bytes, _stream(q.device)),
           "wql_w8a8_gemm_fused")
    return out


def w8a8_gemm_noalloc(q: torch.Tensor, xs: torch.Tensor, qw: torch.Tensor, ws: torch.Tensor,
                      out: torch.Tensor, acc_out: torch.Tensor | None = None) -> torch.Tensor:
    """w8a8_gemm for callers that cannot allocate: the library uses its built-in scratch array.

    The caller passes every input and output (``out`` is required); the call itself allocates
    nothing.  Limits and sharing rules: see wql_w8a8_gemm_noalloc in include/wql.h.
    """
    M, K = q.shape
    N = qw.shape[0]
    _need(q, "q", torch.int8, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _need(qw, "qw", torch.int8, (N, K))
    _need(ws, "ws", torch.float32, (N,))
    _need(out, "out", torch.float16, (M, N))
    if acc_out is not None:
        _need(acc_out, "acc_out", torch.int32, (M, N))
    _check(load().wql_w8a8_gemm_noalloc(_ptr(q), _ptr(xs), _ptr(qw), _ptr(ws), M, K, N, _ptr(out), _ptr(acc_out),
                                        _stream(q.device)), "wql_w8a8_gemm_noalloc")
    return out


def act_absmax(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    M, K = x.shape
    _need(x, "x", torch.float16, (M, K))
    _need(gamma, "gamma", torch.float16, (K,))
    out = torch.empty((K,), dtype=torch.float32, device=x.device)
    _check(load().wql_act_absmax(_ptr(x), _ptr(gamma), float(eps), M, K, _ptr(out), _stream(x.device)),
           "wql_act_absmax")
    return out


def smooth(absmax: torch.Tensor, gamma: torch.Tensor, w: torch.Tensor):
    """Returns (s fp32 [K], gamma' fp16 [K], w' fp32 [K, N])."""
    K, N = w.shape
    _need(absmax, "absmax", torch.float32, (K,))
    _need(gamma, "gamma", torch.float16, (K,))
    _need(w, "w", torch.float32, (K, N))
    s = torch.empty((K,), dtype=torch.float32, device=w.device)
    g = torch.empty((K,), dtype=torch.float16, device=w.device)
    wo = torch.empty_like(w)
    _check(load().wql_smooth(_ptr(absmax), _ptr(gamma), _ptr(w), K, N, _ptr(s), _ptr(g), _ptr(wo), _stream(w.device)),
           "wql_smooth")
    return s, g, wo


def per_channel_quant_i8(w: torch.Tensor):
    """w [K, N] fp32 -> (qw int8 [N, K], ws fp32 [N])."""
    K, N = w.shape
    _need(w, "w", torch.float32, (K, N))
    qw = torch.empty((N, K), dtype=torch.int8, device=w.device)
    ws = torch.empty((N,), dtype=torch.float32, device=w.device)
    _check(load().wql_per_channel_quant_i8(_ptr(w), K, N, _ptr(qw), _ptr(ws), _stream(w.device)),
           "wql_per_channel_quant_i8")
    return qw, ws


def device_status(device: torch.device | None = None) -> None:
    """Synchronise the current stream and raise if a kernel abandoned a bounded wait."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    _check(load().wql_device_status(_stream(dev)), "wql_device_status")


def diag_expire_wait(device: torch.device | None = None) -> None:
    """Launch the failure-path diagnostic: a bounded wait that gives up (about 2 s); the next
    device_status() then raises WQLError with WQL_ETIMEOUT."""
    dev = device or torch.device("cuda", torch.cuda.current_device())
    _check(load().wql_diag_expire_wait(_stream(dev)), "wql_diag_expire_wait")


# ---- fp8 (float8_e4m3fn) variant of W8A8 ------------------------------------------------------

E4M3 = torch.float8_e4m3fn


def qrmsnorm_quant_fp8(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, q: torch.Tensor | None = None,
                       xs: torch.Tensor | None = None):
    """QRMSNorm + per-token fp8: x [M, K] fp16 -> (q float8_e4m3fn [M, K], xs fp32 [M]), xs = absmax / 448."""
    M, K = x.shape
    _need(x, "x", torch.float16, (M, K))
    _need(gamma, "gamma", torch.float16, (K,))
    if q is None:
        q = torch.empty((M, K), dtype=E4M3, device=x.device)
    if xs is None:
        xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(q, "q", E4M3, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _check(load().wql_qrmsnorm_quant_fp8(_ptr(x), _ptr(gamma), float(eps), M, K, _ptr(q), _ptr(xs), _stream(x.device)),
           "wql_qrmsnorm_quant_fp8")
    return q, xs


def add_qrmsnorm_quant_fp8(x: torch.Tensor, residual: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6,
                           residual_out: torch.Tensor | None = None, q: torch.Tensor | None = None,
                           xs: torch.Tensor | None = None):
    """Residual-fused fp8 QRMSNorm: h = fp16(x + residual) -> (h, q float8_e4m3fn [M, K], xs fp32 [M]).

    residual_out receives h (it may be `residual` itself, for an in-place update)."""
    M, K = x.shape
    _need(x, "x", torch.float16, (M, K))
    _need(residual, "residual", torch.float16, (M, K))
    _need(gamma, "gamma", torch.float16, (K,))
    if residual_out is None:
        residual_out = torch.empty((M, K), dtype=torch.float16, device=x.device)
    if q is None:
        q = torch.empty((M, K), dtype=E4M3, device=x.device)
    if xs is None:
        xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(residual_out, "residual_out", torch.float16, (M, K))
    _need(q, "q", E4M3, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _check(load().wql_add_qrmsnorm_quant_fp8(_ptr(x), _ptr(residual), _ptr(gamma), float(eps), M, K,
                                             _ptr(residual_out), _ptr(q), _ptr(xs), _stream(x.device)),
           "wql_add_qrmsnorm_quant_fp8")
    return residual_out, q, xs


def per_channel_quant_fp8(w: torch.Tensor, qw: torch.Tensor | None = None, ws: torch.Tensor | None = None):
    """w [K, N] fp32 -> (qw float8_e4m3fn [N, K], ws fp32 [N]) with ws = absmax / 448."""
    K, N = w.shape
    _need(w, "w", torch.float32, (K, N))
    if qw is None:
        qw = torch.empty((N, K), dtype=E4M3, device=w.device)
    if ws is None:
        ws = torch.empty((N,), dtype=torch.float32, device=w.device)
    _need(qw, "qw", E4M3, (N, K))
    _need(ws, "ws", torch.float32, (N,))
    _check(load().wql_per_channel_quant_fp8(_ptr(w), K, N, _ptr(qw), _ptr(ws), _stream(w.device)),
           "wql_per_channel_quant_fp8")
    return qw, ws


def w8a8_gemm_fp8(q: torch.Tensor, xs: torch.Tensor, qw: torch.Tensor, ws: torch.Tensor,
                  bias: torch.Tensor | None = None, residual: torch.Tensor | None = None,
                  out: torch.Tensor | None = None, acc_out: torch.Tensor | None = None) -> torch.Tensor:
    """y [M, N] fp16 = fp16(((acc * xs) * ws + bias) + residual), acc the fp32 sum of e4m3 products of
    q [M, K] and qw [N, K]; bias [N] and residual [M, N] fp16 optional; optional fp32 acc_out [M, N]."""
    M, K = q.shape
    N = qw.shape[0]
    _need(q, "q", E4M3, (M, K))
    _need(xs, "xs", torch.float32, (M,))
    _need(qw, "qw", E4M3, (N, K))
    _need(ws, "ws", torch.float32, (N,))
    if bias is not None:
        _need(bias, "bias", torch.float16, (N,))
    if residual is not None:
        _need(residual, "residual", torch.float16, (M, N))
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=q.device)
    _need(out, "out", torch.float16, (M, N))
    if acc_out is not None:
        _need(acc_out, "acc_out", torch.float32, (M, N))
    _check(load().wql_w8a8_gemm_fp8(_ptr(q), _ptr(xs), _ptr(qw), _ptr(ws), _ptr(bias), _ptr(residual), M, K, N,
                                    _ptr(out), _ptr(acc_out), _stream(q.device)), "wql_w8a8_gemm_fp8")
    return out


# ---- KV cache int8, groups of 128 channels ------------------------------------------------------

def kv_quant_i8(kv: torch.Tensor, q: torch.Tensor | None = None, scales: torch.Tensor | None = None):
    """kv [..., D] fp16 (D % 128 == 0) -> (q int8 [..., D], scales fp32 [..., D / 128]); s = absmax / 127."""
    D = kv.shape[-1]
    rows = kv.numel() // D if D else 0
    _need(kv, "kv", torch.float16, tuple(kv.shape))
    if q is None:
        q = torch.empty(kv.shape, dtype=torch.int8, device=kv.device)
    if scales is None:
        scales = torch.empty(tuple(kv.shape[:-1]) + (D // 128,), dtype=torch.float32, device=kv.device)
    _need(q, "q", torch.int8, tuple(kv.shape))
    _need(scales, "scales", torch.float32, tuple(kv.shape[:-1]) + (D // 128,))
    _check(load().wql_kv_quant_i8(_ptr(kv), rows, D, _ptr(q), _ptr(scales), _stream(kv.device)), "wql_kv_quant_i8")
    return q, scales


def kv_dequant_i8(q: torch.Tensor, scales: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """fp16 [..., D] = fp16(q * the scale of the element's group of 128)."""
    D = q.shape[-1]
    rows = q.numel() // D if D else 0
    _need(q, "q", torch.int8, tuple(q.shape))
    _need(scales, "scales", torch.float32, tuple(q.shape[:-1]) + (D // 128,))
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, device=q.device)
    _need(out, "out", torch.float16, tuple(q.shape))
    _check(load().wql_kv_dequant_i8(_ptr(q), _ptr(scales), rows, D, _ptr(out), _stream(q.device)), "wql_kv_dequant_i8")
    return out
