"""GPU parity of the residual/bias fusions of the W8A8 block, through the C ABI.

Residual-fused QRMSNorm (h = fp16(x + r), then QRMSNorm + per-token int8 of h) and the int8 GEMM
epilogue with an optional bias and residual (y = fp16(((acc * xs) * ws + bias) + residual)) must
match the oracle bit for bit: the new residual h, the codes, the per-token scales and the fp16
outputs, on both GEMM kernels (decode up to 16 tokens, tcgen05 from 17), in place or not.
GEMM outputs not written in place go into NaN-poisoned buffers with guard bands: every element must
be written and neither guard touched.
"""
import numpy as np
import pytest

import oracle
from weight_quantized_linear_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from _gpu_util import Guarded, tile_rows  # noqa: E402


@pytest.fixture(scope="module")
def wql(wql_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return wql_lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 4096), (16, 4096), (37, 1032), (300, 4096), (5, 16384), (2048, 4096)])
def test_add_qrmsnorm_bit_exact(wql, M, K):
    X = inputs.activations(M, K, seed=21, outlier_channels=True)
    R = inputs.activations(M, K, seed=22)
    g = inputs.gamma(K, seed=21)
    h, q, xs = wql.add_qrmsnorm_quant_i8(dev(X), dev(R), dev(g), inputs.EPS)
    h_r, q_r, xs_r = oracle.add_qrmsnorm_quant_i8(X, R, g, inputs.EPS)
    assert np.array_equal(host(h).view(np.uint16), h_r.view(np.uint16))
    assert np.array_equal(host(q), q_r)
    assert np.array_equal(host(xs).view(np.uint32), xs_r.view(np.uint32))
    wql.device_status()


def test_add_qrmsnorm_in_place_and_cancelling(wql):
    M, K = 64, 4096
    X = inputs.activations(M, K, seed=23, outlier_channels=True)
    R = inputs.activations(M, K, seed=24)
    g = inputs.gamma(K, seed=23)
    r = dev(R)
    h, q, xs = wql.add_qrmsnorm_quant_i8(dev(X), r, dev(g), inputs.EPS, residual_out=r)
    h_r, q_r, xs_r = oracle.add_qrmsnorm_quant_i8(X, R, g, inputs.EPS)
    assert h.data_ptr() == r.data_ptr()
    assert np.array_equal(host(r).view(np.uint16), h_r.view(np.uint16))
    assert np.array_equal(host(q), q_r) and np.array_equal(host(xs), xs_r)
    # r = -x cancels every row: codes 0, scale 1
    h0, q0, xs0 = wql.add_qrmsnorm_quant_i8(dev(X), dev(-X), dev(g), inputs.EPS)
    assert np.all(host(h0) == 0) and np.all(host(q0) == 0) and np.all(host(xs0) == 1.0)
    wql.device_status()


@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (7, 1024, 352), (16, 4096, 11008), (17, 1024, 256),
                                   (100, 4096, 1056), (512, 4096, 4096)])
@pytest.mark.parametrize("terms", ["bias", "residual", "both", "none"])
def test_w8a8_fused_epilogue_bit_exact(wql, M, K, N, terms):
    rng = np.random.default_rng(M + K + N)
    q = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    qW = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    xs = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    bias = rng.normal(0, 1, N).astype(np.float16) if terms in ("bias", "both") else None
    res = rng.normal(0, 2, (M, N)).astype(np.float16) if terms in ("residual", "both") else None
    acc = Guarded((M, N), torch.int32)
    y = Guarded((M, N), torch.float16)
    wql.w8a8_gemm_fused(dev(q), dev(xs), dev(qW), dev(ws), None if bias is None else dev(bias),
                        None if res is None else dev(res), out=y.t, acc_out=acc.t)
    acc.check()
    y.check()
    assert acc.unwritten() == 0 and y.unwritten() == 0
    rows = tile_rows(M, 8)
    acc_r = oracle.w8a8_acc(q, qW, rows=rows)
    assert np.array_equal(host(acc.t)[rows], acc_r)
    y_r = oracle.w8a8_epilogue_fused(acc_r, xs[rows], ws, bias, None if res is None else res[rows])
    assert np.array_equal(host(y.t)[rows].view(np.uint16), y_r.view(np.uint16))
    wql.device_status()


@pytest.mark.parametrize("M", [4, 64])
def test_w8a8_fused_in_place_on_the_residual(wql, M):
    K, N = 2048, 1024
    rng = np.random.default_rng(M)
    q = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    qW = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    xs = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    bias = rng.normal(0, 1, N).astype(np.float16)
    res = rng.normal(0, 2, (M, N)).astype(np.float16)
    r = dev(res)
    y = wql.w8a8_gemm_fused(dev(q), dev(xs), dev(qW), dev(ws), dev(bias), r, out=r)
    assert y.data_ptr() == r.data_ptr()
    y_r = oracle.w8a8_epilogue_fused(oracle.w8a8_acc(q, qW), xs, ws, bias, res)
    assert np.array_equal(host(r).view(np.uint16), y_r.view(np.uint16))
    wql.device_status()
