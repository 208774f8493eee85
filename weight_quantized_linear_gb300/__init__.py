"""GB300-native weight-quantized linear layers (AWQ W4A16, SmoothQuant W8A8 with int8 or fp8 codes).

The compute lives in ``libwql.so`` (hand-written CUDA for sm_103a behind the C ABI of
``include/wql.h``); this package only marshals torch tensors into that ABI.  Build it with
``weight_quantized_linear_gb300.build.build()``.  Importing the package does not load the library;
the first call does, and raises if it is missing.
"""
from ._lib import (  # noqa: F401
    E4M3,
    WQLError,
    act_absmax,
    add_qrmsnorm_quant_fp8,
    add_qrmsnorm_quant_i8,
    awq_pack,
    device_status,
    diag_expire_wait,
    interleave_gate_up,
    kv_dequant_i8,
    kv_quant_i8,
    load,
    per_channel_quant_fp8,
    per_channel_quant_i8,
    per_token_quant_fp8,
    per_token_quant_i8,
    qrmsnorm_quant_fp8,
    qrmsnorm_quant_i8,
    smooth,
    w4a16_gemm,
    w4a16_gemm_silu_mul,
    w4a16_kernel_for,
    w8a8_gemm,
    w8a8_gemm_fp8,
    w8a8_gemm_fused,
    w8a8_gemm_noalloc,
    w8a8_workspace_bytes,
)

__all__ = [
    "E4M3", "WQLError", "act_absmax", "add_qrmsnorm_quant_fp8", "add_qrmsnorm_quant_i8", "awq_pack", "device_status",
    "diag_expire_wait", "interleave_gate_up", "kv_dequant_i8", "kv_quant_i8", "load", "per_channel_quant_fp8", "per_channel_quant_i8",
    "per_token_quant_fp8", "per_token_quant_i8", "qrmsnorm_quant_fp8", "qrmsnorm_quant_i8", "smooth",
    "w4a16_gemm", "w4a16_gemm_silu_mul", "w4a16_kernel_for", "w8a8_gemm", "w8a8_gemm_fp8", "w8a8_gemm_fused", "w8a8_gemm_noalloc",
    "w8a8_workspace_bytes",
]
