"""GPU parity of the fp8 (float8_e4m3fn) variant of the W8A8 path, through the C ABI.

* QRMSNorm + per-token fp8 codes (plain and residual-fused) and the per-channel fp8 weights take
  their rounding decisions in fp32 on both sides, so codes and scales must match the oracle bit
  for bit.
* The fp8 GEMM accumulates in fp32 in the kernel's own order, so it is compared with the oracle's
  exact sum through the error bound of fp32 summation: |acc - exact| <= K * 2^-23 * sum_k |p_k|
  (one rounding of at most 2^-23 relative per addition, whatever the order or rounding mode).  Its
  fp16 output must lie within that bound, carried through the epilogue, plus the epilogue's own
  roundings (three fp32 roundings and the final fp16 one) of the unrounded fp64 value.
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


def dev8(a):
    """uint8 e4m3 codes -> a float8_e4m3fn device tensor."""
    return dev(a).view(torch.float8_e4m3fn)


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def host8(t):
    torch.cuda.synchronize()
    return t.view(torch.uint8).cpu().numpy()


def sample_rows(M, n=16):
    if M <= n:
        return np.arange(M, dtype=np.int64)
    return np.unique(np.concatenate([np.linspace(0, M - 1, n).astype(np.int64), [M - 1]]))


# ------------------------------------------------------------------------------------------------
# quantisers: bit-exact
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("M,K", [(1, 4096), (16, 4096), (37, 1032), (300, 4096), (5, 16384), (2048, 4096), (3, 8)])
def test_qrmsnorm_fp8_bit_exact(wql, M, K):
    X = inputs.activations(M, K, seed=31, outlier_channels=True)
    g = inputs.gamma(K, seed=31)
    q, xs = wql.qrmsnorm_quant_fp8(dev(X), dev(g), inputs.EPS)
    q_r, xs_r = oracle.qrmsnorm_quant_fp8(X, g, inputs.EPS)
    assert np.array_equal(host(xs).view(np.uint32), xs_r.view(np.uint32))
    assert np.array_equal(host8(q), q_r)
    wql.device_status()


def test_qrmsnorm_fp8_zero_rows_ties_and_signed_zeros(wql):
    M, K = 8, 1024
    X = inputs.activations(M, K, seed=32, outlier_channels=True)
    X[2] = 0
    X[5, ::3] = -0.0  # signed zeros become code 0x80
    # values whose quotient lands exactly on an e4m3 tie: a row of powers of two times 1 + 1/16
    X[6] = np.float16(1.0)
    X[6, ::7] = np.float16(1.0625)
    X[6, 0] = np.float16(4.0)
    g = inputs.gamma(K, seed=32)
    g[:] = np.float16(1.0)
    q, xs = wql.qrmsnorm_quant_fp8(dev(X), dev(g), inputs.EPS)
    q_r, xs_r = oracle.qrmsnorm_quant_fp8(X, g, inputs.EPS)
    assert np.array_equal(host(xs).view(np.uint32), xs_r.view(np.uint32))
    assert np.array_equal(host8(q), q_r)
    assert xs_r[2] == 1.0 and np.all(q_r[2] == 0)
    wql.device_status()


@pytest.mark.parametrize("M,K", [(1, 4096), (16, 4096), (37, 1032), (300, 4096), (5, 16384), (2048, 4096)])
def test_add_qrmsnorm_fp8_bit_exact(wql, M, K):
    X = inputs.activations(M, K, seed=33, outlier_channels=True)
    R = inputs.activations(M, K, seed=34)
    g = inputs.gamma(K, seed=33)
    h, q, xs = wql.add_qrmsnorm_quant_fp8(dev(X), dev(R), dev(g), inputs.EPS)
    h_r, q_r, xs_r = oracle.add_qrmsnorm_quant_fp8(X, R, g, inputs.EPS)
    assert np.array_equal(host(h).view(np.uint16), h_r.view(np.uint16))
    assert np.array_equal(host(xs).view(np.uint32), xs_r.view(np.uint32))
    assert np.array_equal(host8(q), q_r)
    wql.device_status()


def test_add_qrmsnorm_fp8_in_place(wql):
    M, K = 64, 4096
    X = inputs.activations(M, K, seed=35, outlier_channels=True)
    R = inputs.activations(M, K, seed=36)
    g = inputs.gamma(K, seed=35)
    r = dev(R)
    h, q, xs = wql.add_qrmsnorm_quant_fp8(dev(X), r, dev(g), inputs.EPS, residual_out=r)
    h_r, q_r, xs_r = oracle.add_qrmsnorm_quant_fp8(X, R, g, inputs.EPS)
    assert h.data_ptr() == r.data_ptr()
    assert np.array_equal(host(r).view(np.uint16), h_r.view(np.uint16))
    assert np.array_equal(host8(q), q_r) and np.array_equal(host(xs), xs_r)
    wql.device_status()


@pytest.mark.parametrize("K,N", [(4096, 4096), (1040, 96), (64, 11008), (4096, 352)])
def test_per_channel_quant_fp8_bit_exact(wql, K, N):
    W = inputs.weight(K, N, seed=37, outliers=True)
    W[:, 5] = 0  # an all-zero column gets scale 1
    qW, ws = wql.per_channel_quant_fp8(dev(W))
    qW_r, ws_r = oracle.per_channel_quant_fp8(W)
    assert np.array_equal(host(ws).view(np.uint32), ws_r.view(np.uint32))
    assert np.array_equal(host8(qW), qW_r)
    wql.device_status()


def test_fp8_prep_chain_bit_exact(wql):
    """Smoothing (shared with int8), then fp8 weights and fp8 activations."""
    M, K, N = 16, 4096, 4096
    X = inputs.activations(M, K, seed=38, outlier_channels=True)
    g = inputs.gamma(K, seed=38)
    W = inputs.weight(K, N, seed=38)
    a_r = oracle.act_absmax(X, g, inputs.EPS)
    _, g2_r, W2_r = oracle.smooth(a_r, g, W)
    qW_r, ws_r = oracle.per_channel_quant_fp8(W2_r)
    q_r, xs_r = oracle.qrmsnorm_quant_fp8(X, g2_r, inputs.EPS)
    Xd, gd = dev(X), dev(g)
    a = wql.act_absmax(Xd, gd, inputs.EPS)
    _, g2, W2 = wql.smooth(a, gd, dev(W))
    qW, ws = wql.per_channel_quant_fp8(W2)
    q, xs = wql.qrmsnorm_quant_fp8(Xd, g2, inputs.EPS)
    assert np.array_equal(host8(qW), qW_r) and np.array_equal(host(ws).view(np.uint32), ws_r.view(np.uint32))
    assert np.array_equal(host8(q), q_r) and np.array_equal(host(xs).view(np.uint32), xs_r.view(np.uint32))
    wql.device_status()


# ------------------------------------------------------------------------------------------------
# fp8 GEMM: within the fp32 summation bound of the exact sum
# ------------------------------------------------------------------------------------------------

def _fp8_codes(rng, shape, scale):
    """e4m3 codes of normal samples (spread over the format's range), via the oracle's encoder."""
    return oracle.float_to_e4m3((rng.standard_normal(shape) * scale).astype(np.float32))


def check_fp8_gemm(y, acc, q, qW, xs, ws, K, rows, bias=None, res=None):
    acc_r, absacc = oracle.fp8_acc(q, qW, rows=rows)
    e_acc = K * 2.0 ** -23 * absacc
    err = np.abs(acc[rows].astype(np.float64) - acc_r)
    assert np.all(err <= e_acc), f"acc error / bound up to {np.max(err / np.maximum(e_acc, 1e-300)):.3g}"
    r = None if res is None else res[rows]
    y_ref = oracle.fp8_epilogue_f64(acc_r, xs[rows], ws, bias, r)
    scale = np.abs(xs[rows].astype(np.float64))[:, None] * np.abs(ws.astype(np.float64))[None, :]
    terms = np.abs(acc_r) * scale
    if bias is not None:
        terms = terms + np.abs(bias.astype(np.float64))[None, :]
    if r is not None:
        terms = terms + np.abs(r.astype(np.float64))
    carried = e_acc * scale + 2.0 ** -21 * terms
    tol = (1 + 2.0 ** -11) * carried + 2.0 ** -11 * np.abs(y_ref) + 2.0 ** -24
    yerr = np.abs(y[rows].astype(np.float64) - y_ref)
    assert np.all(yerr <= tol), f"y error / tolerance up to {np.max(yerr / tol):.3g}"
    # the method's stated tolerance as well: row-relative L2 against the fp64 value
    num = np.linalg.norm(y[rows].astype(np.float64) - y_ref, axis=1)
    den = np.maximum(np.linalg.norm(y_ref, axis=1), 1e-30)
    assert np.max(num / den) <= 1e-2


@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (7, 1040, 352), (16, 4096, 11008), (17, 1024, 256),
                                   (64, 4096, 1056), (100, 2048, 4096), (300, 4096, 4096), (512, 4096, 11008),
                                   (1000, 1040, 352)])
def test_fp8_gemm_within_fp32_summation_bound(wql, M, K, N):
    rng = np.random.default_rng(M * 7 + K + N)
    q = _fp8_codes(rng, (M, K), 60.0)
    qW = _fp8_codes(rng, (N, K), 60.0)
    xs = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    acc = Guarded((M, N), torch.float32)
    yg = Guarded((M, N), torch.float16)
    y = wql.w8a8_gemm_fp8(dev8(q), dev(xs), dev8(qW), dev(ws), out=yg.t, acc_out=acc.t)
    acc.check()
    yg.check()
    assert np.isfinite(host(y)).all() and np.isfinite(host(acc.t)).all()  # every element written
    rows = tile_rows(M, 8)
    check_fp8_gemm(host(y), host(acc.t), q, qW, xs, ws, K, rows)
    # deterministic: a second call gives the same bits
    y2 = wql.w8a8_gemm_fp8(dev8(q), dev(xs), dev8(qW), dev(ws))
    assert torch.equal(y, y2)
    wql.device_status()


@pytest.mark.parametrize("M,K,N", [(4, 2048, 1024), (64, 4096, 4096), (300, 1024, 352)])
@pytest.mark.parametrize("terms", ["bias", "residual", "both"])
def test_fp8_gemm_bias_residual(wql, M, K, N, terms):
    rng = np.random.default_rng(M + K + N + len(terms))
    q = _fp8_codes(rng, (M, K), 60.0)
    qW = _fp8_codes(rng, (N, K), 60.0)
    xs = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    bias = rng.normal(0, 1, N).astype(np.float16) if terms in ("bias", "both") else None
    res = rng.normal(0, 2, (M, N)).astype(np.float16) if terms in ("residual", "both") else None
    acc = torch.empty((M, N), dtype=torch.float32, device="cuda")
    r = None if res is None else dev(res)
    y = wql.w8a8_gemm_fp8(dev8(q), dev(xs), dev8(qW), dev(ws), None if bias is None else dev(bias), r,
                          out=r, acc_out=acc)
    if r is not None:
        assert y.data_ptr() == r.data_ptr()  # in place on the residual
    rows = sample_rows(M, 24)
    check_fp8_gemm(host(y), host(acc), q, qW, xs, ws, K, rows, bias, res)
    wql.device_status()


def test_fp8_gemm_extremes_and_signed_zero_codes(wql):
    """Every code at +-448 (the largest products, |acc| = K * 448^2), subnormal codes and -0 codes."""
    M, K, N = 20, 8192, 128
    rng = np.random.default_rng(39)
    q = rng.choice(np.array([0x7e, 0xfe, 0x80, 0x00, 0x01, 0x81, 0x07], np.uint8), size=(M, K))
    qW = rng.choice(np.array([0x7e, 0xfe, 0x80, 0x08], np.uint8), size=(N, K))
    q[0] = 0x7e
    qW[0] = 0x7e
    qW[1] = 0xfe
    xs = np.full((M,), 1e-3, np.float32)
    ws = np.full((N,), 1e-4, np.float32)
    acc = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y = wql.w8a8_gemm_fp8(dev8(q), dev(xs), dev8(qW), dev(ws), acc_out=acc)
    a = host(acc)
    # 448^2 = 49 * 2^12: a partial sum of j equal products is 49 j 2^12, exact in fp32 for j <= 8192
    assert a[0, 0] == 448.0 * 448.0 * K and a[0, 1] == -448.0 * 448.0 * K
    check_fp8_gemm(host(y), a, q, qW, xs, ws, K, np.arange(M, dtype=np.int64))
    wql.device_status()


def test_fp8_full_block_against_oracle(wql):
    """The whole fp8 block at the SmoothQuant workload shape: smoothing, fp8 weights, the residual-fused
    fp8 norm and the GEMM with bias and residual, sampled rows against the oracle."""
    M, K, N = 512, 4096, 4096
    X = inputs.activations(M, K, seed=40, outlier_channels=True)
    R = inputs.activations(M, K, seed=41)
    g = inputs.gamma(K, seed=40)
    W = inputs.weight(K, N, seed=40)
    rng = np.random.default_rng(40)
    bias = rng.normal(0, 0.5, N).astype(np.float16)
    RY = rng.normal(0, 1, (M, N)).astype(np.float16)
    # oracle
    a_r = oracle.act_absmax(X, g, inputs.EPS)
    _, g2_r, W2_r = oracle.smooth(a_r, g, W)
    qW_r, ws_r = oracle.per_channel_quant_fp8(W2_r)
    h_r, q_r, xs_r = oracle.add_qrmsnorm_quant_fp8(X, R, g2_r, inputs.EPS)
    # CUDA path
    Xd, gd = dev(X), dev(g)
    a = wql.act_absmax(Xd, gd, inputs.EPS)
    _, g2, W2 = wql.smooth(a, gd, dev(W))
    qW, ws = wql.per_channel_quant_fp8(W2)
    h, q, xs = wql.add_qrmsnorm_quant_fp8(Xd, dev(R), g2, inputs.EPS)
    acc = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y = wql.w8a8_gemm_fp8(q, xs, qW, ws, dev(bias), dev(RY), acc_out=acc)
    assert np.array_equal(host(h).view(np.uint16), h_r.view(np.uint16))
    assert np.array_equal(host8(q), q_r) and np.array_equal(host8(qW), qW_r)
    rows = sample_rows(M, 16)
    check_fp8_gemm(host(y), host(acc), q_r, qW_r, xs_r, ws_r, K, rows, bias, RY)
    wql.device_status()


def test_fp8_empty_and_invalid(wql):
    q = torch.empty((0, 256), dtype=torch.float8_e4m3fn, device="cuda")
    qW = torch.zeros((64, 256), dtype=torch.float8_e4m3fn, device="cuda")
    xs = torch.empty((0,), dtype=torch.float32, device="cuda")
    ws = torch.ones((64,), dtype=torch.float32, device="cuda")
    y = wql.w8a8_gemm_fp8(q, xs, qW, ws)
    assert y.shape == (0, 64)
    with pytest.raises(wql.WQLError):
        wql.per_channel_quant_fp8(dev(inputs.weight(256, 48, seed=0)))  # N not a multiple of 32
    wql.device_status()


def test_fp8_decode_back_to_back_stress(wql):
    """Graph-replayed chains of fp8 decode GEMMs stay fault-free and bit-identical."""
    M, K, N = 16, 4096, 4096
    rng = np.random.default_rng(42)
    q = dev8(_fp8_codes(rng, (M, K), 60.0))
    xs = dev(rng.uniform(1e-3, 1e-2, M).astype(np.float32))
    qW = dev8(_fp8_codes(rng, (N, K), 60.0))
    ws = dev(rng.uniform(1e-4, 1e-3, N).astype(np.float32))
    ref = wql.w8a8_gemm_fp8(q, xs, qW, ws).clone()
    layers, reps = 16, 100
    stack = [qW.clone() for _ in range(layers)]
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in range(layers)]
    stream = torch.cuda.Stream()

    def step():
        for i, w in enumerate(stack):
            wql.w8a8_gemm_fp8(q, xs, w, ws, out=ys[i])

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    torch.cuda.synchronize()
    wql.device_status()
    for y in ys:
        assert torch.equal(y, ref)
