"""Host-side checks of the C ABI (no GPU needed): the library builds for sm_103a, loads, and
exports every function that include/wql.h declares, with the binding's table matching the header."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wql.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(wql_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("wql_awq_pack", "wql_w4a16_gemm", "wql_qrmsnorm_quant_i8", "wql_w8a8_gemm"):
        assert required in names


def test_library_exports_every_declared_symbol(wql_lib):
    from weight_quantized_linear_gb300 import _lib
    lib = ctypes.CDLL(_lib.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in wql.h but not exported"
    assert sorted(_lib.SIGNATURES) == _declared_functions()


def test_host_only_entry_points(wql_lib):
    lib = wql_lib.load()
    assert lib.wql_version() == 100
    assert lib.wql_status_string(0) == b"ok"
    assert lib.wql_status_string(4) == b"device-side wait timed out"
    assert lib.wql_w8a8_workspace_bytes(16, 4096, 4096) >= 0
    # kernel choice: decode up to 16 tokens, tcgen05 from 33, in between by shape
    assert lib.wql_w4a16_kernel_for(1, 4096, 4096, 128) == 0
    assert lib.wql_w4a16_kernel_for(16, 4096, 22016, 32) == 0
    assert lib.wql_w4a16_kernel_for(33, 4096, 4096, 128) == 1
    assert lib.wql_w4a16_kernel_for(32, 11008, 4096, 128) == 1   # long K: split-K pays
    assert lib.wql_w4a16_kernel_for(32, 4096, 4096, 128) == 0    # 32 output tiles: decode
    assert lib.wql_w4a16_kernel_for(32, 4096, 4096, 32) == 1     # G = 32: four group epilogues per stage
    assert lib.wql_w4a16_kernel_for(24, 4096, 22016, 64) == 1    # G = 64 beyond one wave
    assert lib.wql_w4a16_kernel_for(24, 4096, 22016, 128) == 0
    # the phase trace exists only in the developer build; the default library refuses it
    assert lib.wql_trace_setup(None, None, 0, 0, 0) == 2  # WQL_EUNSUPPORTED
    assert b"WQL_PHASE_TRACE" in lib.wql_last_error()


def test_validation_rejects_bad_arguments_without_a_gpu(wql_lib):
    # Validation runs before anything touches the device, so these calls are safe on a CPU host.
    lib = wql_lib.load()
    fake = ctypes.c_void_p(1 << 20)
    # group 48 is not a valid AWQ group size
    assert lib.wql_w4a16_gemm(fake, fake, fake, fake, 1, 4096, 4096, 48, fake, None) == 1
    assert b"group" in lib.wql_last_error()
    # N not a multiple of 32
    assert lib.wql_w4a16_gemm(fake, fake, fake, fake, 1, 4096, 4008, 128, fake, None) == 1
    # misaligned pointer
    bad = ctypes.c_void_p((1 << 20) + 2)
    assert lib.wql_w4a16_gemm(bad, fake, fake, fake, 1, 4096, 4096, 128, fake, None) == 1
    # K beyond the register-resident norm kernel
    assert lib.wql_qrmsnorm_quant_i8(fake, fake, ctypes.c_float(1e-6), 1, 32768, fake, fake, None) == 2
    # M = 0 is an empty call
    assert lib.wql_w4a16_gemm(None, None, None, None, 0, 4096, 4096, 128, None, None) == 0
    assert lib.wql_w8a8_gemm(None, None, None, None, 0, 4096, 4096, None, None, None, 0, None) == 0
    # K not a multiple of 16 for the int8 GEMM
    assert lib.wql_w8a8_gemm(fake, fake, fake, fake, 1, 4100, 4096, fake, None, None, 0, None) == 1
    # the follow-up entry points validate the same way
    assert lib.wql_w4a16_gemm_silu_mul(fake, fake, fake, fake, 1, 4096, 96, 128, fake, None) == 1  # N % 64
    assert b"64" in lib.wql_last_error()
    assert lib.wql_w8a8_gemm_fp8(fake, fake, fake, fake, None, None, 1, 4100, 4096, fake, None, None) == 1
    assert lib.wql_w8a8_gemm_fp8(None, None, None, None, None, None, 0, 4096, 4096, None, None, None) == 0
    bad_bias = ctypes.c_void_p((1 << 20) + 8)  # bias must be 16-byte aligned
    assert lib.wql_w8a8_gemm_fused(fake, fake, fake, fake, bad_bias, None, 1, 4096, 4096, fake, None, None, 0,
                                   None) == 1
    assert lib.wql_kv_quant_i8(fake, 4, 192, fake, fake, None) == 1  # D % 128
    assert lib.wql_kv_quant_i8(None, 0, 256, None, None, None) == 0
    assert lib.wql_kv_dequant_i8(fake, fake, -1, 256, fake, None) == 1
    assert lib.wql_qrmsnorm_quant_fp8(fake, fake, ctypes.c_float(1e-6), 1, 32768, fake, fake, None) == 2
    assert lib.wql_add_qrmsnorm_quant_fp8(fake, None, fake, ctypes.c_float(1e-6), 1, 4096, fake, fake, fake,
                                          None) == 1  # residual required
    assert lib.wql_per_channel_quant_fp8(fake, 4096, 48, fake, fake, None) == 1  # N % 32


def test_binding_raises_without_library(tmp_path):
    from weight_quantized_linear_gb300 import _lib
    with pytest.raises(RuntimeError):
        # a fresh loader pointed at a missing file must fail loudly, never fall back
        saved = _lib._lib
        _lib._lib = None
        try:
            _lib.load(str(tmp_path / "missing.so"))
        finally:
            _lib._lib = saved


def test_inputs_recipe_counts():
    import numpy as np
    from weight_quantized_linear_gb300 import inputs
    W = inputs.weight(256, 512, seed=0, outliers=True)
    W0 = inputs.weight(256, 512, seed=0, outliers=False)
    changed = np.count_nonzero(W != W0)
    assert changed == round(0.001 * 256 * 512)
    X = inputs.activations(4, 1000, seed=0, outlier_channels=True)
    X0 = inputs.activations(4, 1000, seed=0, outlier_channels=False)
    assert np.count_nonzero(np.any(X != X0, axis=0)) == 10
    assert np.array_equal(inputs.gamma(64, seed=1), inputs.gamma(64, seed=1))
    assert len(inputs.sweep_cases()) == 45 and len(inputs.w8a8_cases()) == 8 and len(inputs.prefill_cases()) == 6


def test_header_is_plain_c99(tmp_path):
    """The boundary is a C ABI: include/wql.h must compile as strict C99 with no warnings."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_wql.c"
    src.write_text('#include "wql.h"\nint main(void) { return wql_version() > 0 ? 0 : 1; }\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, "-c", str(src),
                        "-o", str(tmp_path / "use_wql.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_phase_trace_build_compiles_and_exports_its_setup():
    # The developer build with the W4A16 kernels' phase stamps (-DWQL_PHASE_TRACE) is compiled only
    # on demand (bench.py --trace): check here that it still builds and exports the same C ABI.
    # Registering a buffer needs a GPU; without one the call fails with a CUDA error, not EUNSUPPORTED.
    from weight_quantized_linear_gb300 import build, _lib
    path = build.build(trace=True)
    lib = ctypes.CDLL(path)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    lib.wql_trace_setup.restype = ctypes.c_int
    lib.wql_trace_setup.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int, ctypes.c_int]
    assert lib.wql_trace_setup(None, None, 0, 0, 0) != _lib.WQL_EUNSUPPORTED
