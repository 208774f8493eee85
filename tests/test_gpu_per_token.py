"""GPU parity of the per-token quantisers of plain fp16 activations (per_token_quant_int8 and its
fp8 twin), through the C ABI: codes and scales bit-exact against the oracle, and the quantised row
feeding the int8 GEMM as QLinear.forward does with an input that is not a QRMSNorm output.
"""
import numpy as np
import pytest

import oracle
from weight_quantized_linear_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from _gpu_util import ROW_TOL, Guarded, dev, host, row_rel_err, tile_rows  # noqa: E402


@pytest.fixture(scope="module")
def wql(wql_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return wql_lib


def _rows(M, K, seed):
    X = inputs.activations(M, K, seed=seed, outlier_channels=True)
    if M >= 4:
        X[1] = 0                      # an all-zero row
        X[2] = np.float16(-0.375)     # a constant row
        X[3] *= np.float16(1e-3)      # a small row next to large ones
    return X


@pytest.mark.parametrize("M,K", [(1, 8), (4, 4096), (16, 4096), (33, 1032), (512, 4096), (4096, 4096),
                                 (3, 11008), (2, 16384)])
def test_per_token_quant_i8_bit_exact(wql, M, K):
    X = _rows(M, K, seed=M + K)
    q_r, xs_r = oracle.per_token_quant_i8(X)
    q = Guarded((M, K), torch.int8)
    xs = Guarded((M,), torch.float32)
    wql.per_token_quant_i8(dev(X), q=q.t, xs=xs.t)
    q.check()
    xs.check()
    assert np.array_equal(host(xs.t).view(np.uint32), xs_r.view(np.uint32))
    assert np.array_equal(host(q.t), q_r)
    wql.device_status()


def test_per_token_quant_i8_ties_go_to_even(wql):
    # scale exactly 1 (absmax 127): every half-integer in [-126.5, 126.5] is a rounding tie
    ties = np.arange(-126.5, 127.0, 1.0)
    row = np.concatenate([[127.0], ties, np.zeros(8 - (1 + ties.size) % 8)]).astype(np.float16)
    X = np.stack([row, -row, row * np.float16(0.5)])
    q_r, xs_r = oracle.per_token_quant_i8(X)
    q, xs = wql.per_token_quant_i8(dev(X))
    assert np.array_equal(host(q), q_r) and np.array_equal(host(xs), xs_r)
    assert host(xs)[0] == 1.0


@pytest.mark.parametrize("M,K", [(1, 64), (16, 4096), (512, 4096), (5, 16384)])
def test_per_token_quant_fp8_bit_exact(wql, M, K):
    X = _rows(M, K, seed=2 * M + K)
    q_r, xs_r = oracle.per_token_quant_fp8(X)
    q, xs = wql.per_token_quant_fp8(dev(X))
    assert np.array_equal(host(xs).view(np.uint32), xs_r.view(np.uint32))
    assert np.array_equal(host(q.view(torch.uint8)), q_r)
    wql.device_status()


@pytest.mark.parametrize("M,N", [(1, 4096), (16, 11008), (512, 4096)])
def test_plain_input_through_the_int8_gemm(wql, M, N):
    # QLinear.forward on a plain tensor: per-token int8 of x, then the int8 GEMM with per-channel
    # weights -- accumulators and outputs bit-exact, and within the fp16 tolerance of fp64
    K = 4096
    X = inputs.activations(M, K, seed=M + N, outlier_channels=True)
    qW_r, ws_r = oracle.per_channel_quant_i8(inputs.weight(K, N, seed=M + N))
    q_r, xs_r = oracle.per_token_quant_i8(X)
    q, xs = wql.per_token_quant_i8(dev(X))
    acc = Guarded((M, N), torch.int32)
    y = Guarded((M, N), torch.float16)
    wql.w8a8_gemm(q, xs, dev(qW_r), dev(ws_r), out=y.t, acc_out=acc.t)
    acc.check()
    y.check()
    assert acc.unwritten() == 0 and y.unwritten() == 0
    rows = tile_rows(M)
    acc_r = oracle.w8a8_acc(q_r, qW_r, rows=rows)
    assert np.array_equal(host(acc.t)[rows], acc_r)
    yh = host(y.t)[rows]
    assert np.array_equal(yh.view(np.uint16), oracle.w8a8_epilogue(acc_r, xs_r[rows], ws_r).view(np.uint16))
    assert row_rel_err(yh, oracle.w8a8_epilogue_f64(acc_r, xs_r[rows], ws_r)) <= ROW_TOL
    wql.device_status()


def test_per_token_quant_rejects_bad_shapes(wql):
    with pytest.raises(wql.WQLError):
        wql.per_token_quant_i8(torch.zeros((2, 12), dtype=torch.float16, device="cuda"))  # K % 8 != 0
    with pytest.raises(wql.WQLError) as ei:
        wql.per_token_quant_i8(torch.zeros((1, 16392), dtype=torch.float16, device="cuda"))
    assert ei.value.status == 2  # K > 16384: unsupported
    q, xs = wql.per_token_quant_i8(torch.zeros((0, 64), dtype=torch.float16, device="cuda"))
    assert q.shape == (0, 64) and xs.shape == (0,)
