"""GPU parity of the tcgen05 prefill kernels (token counts from 17 up), through the C ABI.

W4A16: fp16 output within 1e-2 of the fp64 oracle (row-relative L2), on ragged tiles.
W8A8: int32 accumulators and fp16 outputs bit-exact, including adversarial extremes whose sums
leave the range where fp32 holds integers exactly (checks the 1024-k chunk folding).
GEMM outputs go into NaN-poisoned buffers with guard bands: every element must be written (finite)
and neither guard touched.
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


def row_rel_err(y, ref):
    num = np.linalg.norm(y.astype(np.float64) - ref, axis=1)
    return float((num / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)).max())


@pytest.mark.parametrize("M,K,N,G", [(17, 256, 128, 32), (64, 512, 96, 64), (65, 4096, 4096, 128),
                                     (128, 4096, 12288, 64), (200, 11008, 4096, 128), (257, 4096, 160, 32),
                                     (300, 96, 4096, 32),
                                     # split-K over clusters of 2, 4 and 8 CTAs, with uneven k splits,
                                     # owner column ranges down to 4 tokens, and ragged token tails
                                     (20, 4096, 256, 32), (31, 4160, 2048, 64), (64, 4096, 8192, 128),
                                     (33, 8192, 1024, 128),
                                     # 192-token tiles: one per CTA, several per CTA, a ragged last tile
                                     (576, 4096, 4096, 128), (448, 4096, 12288, 64), (500, 4096, 12288, 32)])
def test_w4a16_prefill_ragged(wql, monkeypatch, M, K, N, G):
    monkeypatch.setenv("WQL_FORCE_KERNEL", "prefill")  # below 33 tokens the choice depends on the shape
    W = inputs.weight(K, N, seed=2, outliers=True)
    X = inputs.activations(M, K, seed=2, outlier_channels=True)
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    rows = tile_rows(M)
    out = Guarded((M, N), torch.float16)
    wql.w4a16_gemm(dev(X), dev(qw_r.view(np.int32)), dev(s_r), dev(qz_r.view(np.int32)), G, out=out.t)
    out.check()
    y = host(out.t)
    ref = oracle.w4a16_linear(X, qw_r, s_r, qz_r, G, rows=rows)
    assert np.isfinite(y).all()
    assert row_rel_err(y[rows], ref) <= 1e-2
    wql.device_status()


@pytest.mark.parametrize("M,K,N,G,kernel", [(24, 4096, 12288, 64, "prefill"), (32, 11008, 4096, 128, "prefill"),
                                            (32, 4096, 4096, 128, "decode"), (16, 4096, 12288, 32, "decode"),
                                            (20, 4096, 4096, 32, "prefill"), (24, 4096, 22016, 64, "prefill"),
                                            (24, 4096, 22016, 128, "decode")])
def test_w4a16_default_kernel_choice(wql, M, K, N, G, kernel):
    # between 17 and 32 tokens w4a16_gemm picks the kernel by shape; the default path must be correct
    assert wql.w4a16_kernel_for(M, K, N, G) == kernel
    W = inputs.weight(K, N, seed=6, outliers=True)
    X = inputs.activations(M, K, seed=6, outlier_channels=True)
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    y = host(wql.w4a16_gemm(dev(X), dev(qw_r.view(np.int32)), dev(s_r), dev(qz_r.view(np.int32)), G))
    rows = np.array([0, M // 2, M - 1], dtype=np.int64)
    assert row_rel_err(y[rows], oracle.w4a16_linear(X, qw_r, s_r, qz_r, G, rows=rows)) <= 1e-2
    wql.device_status()


@pytest.mark.parametrize("M,K,N", [(17, 64, 32), (64, 1024, 128), (130, 4096, 256), (512, 4096, 4096),
                                   (96, 3008, 160)])
def test_w8a8_prefill_bit_exact(wql, M, K, N):
    rng = np.random.default_rng(M + K + N)
    q = rng.integers(-128, 128, size=(M, K), dtype=np.int8)
    qW = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    xs = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    acc = Guarded((M, N), torch.int32)
    y = Guarded((M, N), torch.float16)
    wql.w8a8_gemm(dev(q), dev(xs), dev(qW), dev(ws), out=y.t, acc_out=acc.t)
    acc.check()
    y.check()
    assert acc.unwritten() == 0 and y.unwritten() == 0
    rows = tile_rows(M)
    acc_r = oracle.w8a8_acc(q, qW, rows=rows)
    assert np.array_equal(host(acc.t)[rows], acc_r)
    assert np.array_equal(host(y.t)[rows].view(np.uint16), oracle.w8a8_epilogue(acc_r, xs[rows], ws).view(np.uint16))
    wql.device_status()


@pytest.mark.parametrize("K", [4096, 8192])
def test_w8a8_prefill_exact_beyond_fp32_integer_range(wql, K):
    M, N = 40, 256
    q = np.full((M, K), -128, np.int8)
    q[1::3] = 127
    q[2::3, ::2] = -128
    q[2::3, 1::2] = 127
    qW = np.full((N, K), -127, np.int8)
    qW[1::2] = 127
    qW[::5, : K // 2] = -128
    xs = np.full((M,), 0.01, np.float32)
    ws = np.full((N,), 0.001, np.float32)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    wql.w8a8_gemm(dev(q), dev(xs), dev(qW), dev(ws), acc_out=acc)
    ref = oracle.w8a8_acc(q, qW)
    assert np.abs(ref.astype(np.int64)).max() > 2 ** 24
    assert np.array_equal(host(acc), ref)
    wql.device_status()


@pytest.mark.parametrize("over", [False, True])
def test_w8a8_prefill_one_chunk_bound(wql, over):
    # One fp32 accumulator takes the whole of K when 128 x every row's L1 norm stays within 2^24.
    # At the bound (every |q| = 32, K = 4096: L1 = 2^17) against weights of -128 the partial sums
    # reach exactly 2^24 in magnitude; one code more in one row (over) switches the launch to
    # 1024-k chunks.  Both must be bit-exact.
    M, K, N = 64, 4096, 256
    q = np.full((M, K), 32, np.int8)
    q[1::2] = -32
    if over:
        q[5, 0] = 33
    qW = np.full((N, K), -128, np.int8)
    qW[1::2, ::2] = 127
    xs = np.full((M,), 0.01, np.float32)
    ws = np.full((N,), 0.001, np.float32)
    acc = Guarded((M, N), torch.int32)
    y = Guarded((M, N), torch.float16)
    wql.w8a8_gemm(dev(q), dev(xs), dev(qW), dev(ws), out=y.t, acc_out=acc.t)
    acc.check()
    y.check()
    ref = oracle.w8a8_acc(q, qW)
    assert np.abs(ref.astype(np.int64)).max() >= 2 ** 24
    assert np.array_equal(host(acc.t), ref)
    assert np.array_equal(host(y.t).view(np.uint16), oracle.w8a8_epilogue(ref, xs, ws).view(np.uint16))
    wql.device_status()


def test_w8a8_smoothquant_block_full_size_sampled(wql):
    # the W8A8 block at a full prefill size: prep chain on the GPU, GEMM through the tcgen05 path
    M, K, N = 4096, 4096, 11008
    X = inputs.activations(M, K, seed=5, outlier_channels=True)
    g = inputs.gamma(K, seed=5)
    W = inputs.weight(K, N, seed=5)
    Xd, gd, Wd = dev(X), dev(g), dev(W)
    a = wql.act_absmax(Xd, gd, inputs.EPS)
    s, g2, W2 = wql.smooth(a, gd, Wd)
    qW, ws = wql.per_channel_quant_i8(W2)
    q, xs = wql.qrmsnorm_quant_i8(Xd, g2, inputs.EPS)
    acc = Guarded((M, N), torch.int32)
    y = Guarded((M, N), torch.float16)
    wql.w8a8_gemm(q, xs, qW, ws, out=y.t, acc_out=acc.t)
    acc.check()
    y.check()
    assert acc.unwritten() == 0 and y.unwritten() == 0
    rows = tile_rows(M)  # first and last row of every 32-row block: both edges of every token tile
    qh, qWh, xsh, wsh = host(q), host(qW), host(xs), host(ws)
    acc_r = oracle.w8a8_acc(qh, qWh, rows=rows)
    assert np.array_equal(host(acc.t)[rows], acc_r)
    assert np.array_equal(host(y.t)[rows].view(np.uint16), oracle.w8a8_epilogue(acc_r, xsh[rows], wsh).view(np.uint16))
    wql.device_status()


@pytest.mark.parametrize("K", [1024, 4096])
def test_w8a8_prefill_most_negative_codes_fill_a_chunk(wql, K):
    """q = qw = -128 everywhere: every product is 2^14, a 1024-k chunk sums to exactly 2^24 (the largest
    integer range fp32 holds exactly), and K = 4096 folds four such chunks into 2^26 in int32."""
    M, N = 40, 96
    q = np.full((M, K), -128, np.int8)
    qW = np.full((N, K), -128, np.int8)
    xs = np.full((M,), 1e-3, np.float32)
    ws = np.full((N,), 1e-4, np.float32)
    acc = Guarded((M, N), torch.int32)
    y = Guarded((M, N), torch.float16)
    wql.w8a8_gemm(dev(q), dev(xs), dev(qW), dev(ws), out=y.t, acc_out=acc.t)
    acc.check()
    y.check()
    ref = oracle.w8a8_acc(q, qW)
    assert int(ref[0, 0]) == K * 16384
    assert np.array_equal(host(acc.t), ref)
    assert np.array_equal(host(y.t).view(np.uint16), oracle.w8a8_epilogue(ref, xs, ws).view(np.uint16))
    wql.device_status()


@pytest.mark.parametrize("M,K,N,G", [(32, 11008, 4096, 32), (256, 11008, 4096, 128)])
def test_w4a16_prefill_split_k_is_deterministic(wql, M, K, N, G):
    # the cluster split-K path adds the partial sums in a fixed order: repeated calls agree bit for bit
    W = inputs.weight(K, N, seed=4)
    X = inputs.activations(M, K, seed=4, outlier_channels=True)
    qw, s, qz = wql.awq_pack(dev(W), G)
    x = dev(X)
    y0 = host(wql.w4a16_gemm(x, qw, s, qz, G))
    for _ in range(3):
        assert np.array_equal(host(wql.w4a16_gemm(x, qw, s, qz, G)).view(np.uint16), y0.view(np.uint16))
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    rows = np.array([0, M // 2, M - 1], dtype=np.int64)
    assert row_rel_err(y0[rows], oracle.w4a16_linear(X, qw_r, s_r, qz_r, G, rows=rows)) <= 1e-2
    wql.device_status()


@pytest.mark.parametrize("kernel,M,K,N,G", [("prefill", 17, 4096, 256, 32), ("prefill", 20, 4096, 1024, 64),
                                            ("prefill", 32, 4160, 4096, 64), ("decode", 17, 4096, 512, 128),
                                            ("decode", 32, 2048, 1024, 32), ("decode", 64, 4096, 256, 64)])
def test_w4a16_both_kernels_across_the_dispatch_threshold(wql, monkeypatch, kernel, M, K, N, G):
    # w4a16_gemm picks the kernel by token count; each kernel must be correct on either side of it
    monkeypatch.setenv("WQL_FORCE_KERNEL", kernel)
    W = inputs.weight(K, N, seed=3, outliers=True)
    X = inputs.activations(M, K, seed=3, outlier_channels=True)
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    out = Guarded((M, N), torch.float16)
    wql.w4a16_gemm(dev(X), dev(qw_r.view(np.int32)), dev(s_r), dev(qz_r.view(np.int32)), G, out=out.t)
    out.check()
    y = host(out.t)
    assert np.isfinite(y).all()
    rows = tile_rows(M, 8)
    assert row_rel_err(y[rows], oracle.w4a16_linear(X, qw_r, s_r, qz_r, G, rows=rows)) <= 1e-2
    wql.device_status()
