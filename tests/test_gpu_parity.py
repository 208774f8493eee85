"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs.

Bars: packed weights, int8 activations and scales, per-channel weights and int32 accumulators
bit-exact; fp16 outputs within 1e-2 of the fp64 oracle, normalised by each row's L2 norm.
Every output of a GEMM under test is written into a NaN-poisoned buffer with guard bands on both
sides: all of it must come out finite (no tile left unwritten) and both guards untouched.
"""
import ctypes

import numpy as np
import pytest

import oracle
from weight_quantized_linear_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from _gpu_util import ROW_TOL, Guarded, tile_rows  # noqa: E402  (max over rows of ||y - y_ref|| / ||y_ref||)


@pytest.fixture(scope="module")
def wql(wql_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return wql_lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def u32_to_i32(a):
    return np.ascontiguousarray(a).view(np.int32)


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def row_rel_err(y, ref):
    y = y.astype(np.float64)
    num = np.linalg.norm(y - ref, axis=1)
    den = np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    return float((num / den).max())


def sample_rows(M, n=16):
    if M <= n:
        return np.arange(M, dtype=np.int64)
    r = np.unique(np.concatenate([[0, M - 1], np.linspace(0, M - 1, n - 2).astype(np.int64)]))
    return r.astype(np.int64)


# ------------------------------------------------------------------------------------------------
# awq_pack: bit-exact
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("K,N,G,outl", [(512, 512, 128, False), (256, 96, 32, True), (128, 160, 64, True),
                                        (4096, 4096, 128, True), (11008, 4096, 64, True), (4096, 22016, 32, True)])
def test_awq_pack_bit_exact(wql, K, N, G, outl):
    W = inputs.weight(K, N, seed=0, outliers=outl)
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    qw, s, qz = wql.awq_pack(dev(W), G)
    assert np.array_equal(host(qw), u32_to_i32(qw_r))
    assert np.array_equal(host(s).view(np.uint16), s_r.view(np.uint16))
    assert np.array_equal(host(qz), u32_to_i32(qz_r))


def test_awq_pack_degenerate_groups(wql):
    K, N, G = 64, 32, 32
    W = np.zeros((K, N), np.float32)
    W[G:, :16] = 0.5  # constant nonzero group
    W[G:, 16:] = inputs.weight(G, 16, seed=1)
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    qw, s, qz = wql.awq_pack(dev(W), G)
    assert np.array_equal(host(qw), u32_to_i32(qw_r))
    assert np.array_equal(host(s).view(np.uint16), s_r.view(np.uint16))
    assert np.array_equal(host(qz), u32_to_i32(qz_r))


# ------------------------------------------------------------------------------------------------
# w4a16_gemm: fp16 output vs fp64 oracle
# ------------------------------------------------------------------------------------------------

def _w4a16_case(wql, M, K, N, G, w_out=True, x_out=False, seed=0, rows=None):
    W = inputs.weight(K, N, seed=seed, outliers=w_out)
    X = inputs.activations(M, K, seed=seed, outlier_channels=x_out)
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    out = Guarded((M, N), torch.float16)
    wql.w4a16_gemm(dev(X), dev(u32_to_i32(qw_r)), dev(s_r), dev(u32_to_i32(qz_r)), G, out=out.t)
    out.check()
    y = host(out.t)
    assert np.isfinite(y).all(), f"{int((~np.isfinite(y)).sum())} outputs left unwritten or not finite"
    rows = np.arange(M, dtype=np.int64) if rows is None else rows
    ref = oracle.w4a16_linear(X, qw_r, s_r, qz_r, G, rows=rows)
    return y[rows], ref


TINY_AND_EDGE = [
    (1, 512, 512, 128),   # tiny config
    (1, 32, 32, 32),      # smallest legal shape: one group, one word column group
    (3, 256, 96, 32),     # ragged N (not a multiple of the 128-column strip)
    (17, 128, 160, 128),  # K == G, ragged M and N
    (33, 512, 64, 64),    # M just above a 32-token block
    (8, 4096, 4096, 128),
    (5, 11008, 4096, 128),  # K with 172 stages of 64 rows
    # K % 128 == 64: the last 128-row stage is half past K (activations loaded by the consumer
    # warps must be zero there), with zero token rows past M inside a 16-token block
    (1, 4160, 1024, 64),
    (13, 4160, 512, 32),
    (20, 192, 256, 64),
]


@pytest.mark.parametrize("M,K,N,G", TINY_AND_EDGE)
def test_w4a16_parity_small_and_edge(wql, M, K, N, G):
    y, ref = _w4a16_case(wql, M, K, N, G)
    assert np.isfinite(y).all()
    assert row_rel_err(y, ref) <= ROW_TOL


@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a16_parity_decode_qproj(wql, M):
    y, ref = _w4a16_case(wql, M, 4096, 4096, 128)
    err = row_rel_err(y, ref)
    assert err <= ROW_TOL
    # the kernel's own arithmetic (exact products, fp32 sums, one fp16 rounding) is far tighter
    assert err <= 2e-3


@pytest.mark.parametrize("case", inputs.sweep_cases(), ids=lambda c: f"M{c['M']}K{c['K']}N{c['N']}G{c['G']}")
def test_w4a16_parity_layer_sweep(wql, case):
    rows = sample_rows(case["M"], 16)
    y, ref = _w4a16_case(wql, case["M"], case["K"], case["N"], case["G"], rows=rows)
    assert row_rel_err(y, ref) <= ROW_TOL


@pytest.mark.parametrize("case", inputs.prefill_cases(), ids=lambda c: f"M{c['M']}N{c['N']}")
def test_w4a16_parity_prefill_every_token_tile(wql, case):
    # the first and last row of every 32-row block: both edges of every token tile the kernel uses;
    # the rest of the output is checked for being written (finite, guards intact)
    rows = tile_rows(case["M"])
    y, ref = _w4a16_case(wql, case["M"], case["K"], case["N"], case["G"], w_out=False, x_out=True, rows=rows)
    assert row_rel_err(y, ref) <= ROW_TOL


def test_w4a16_zero_activations_give_zero(wql):
    K, N, G = 256, 64, 32
    W = inputs.weight(K, N, seed=3)
    qw, s, qz = wql.awq_pack(dev(W), G)
    y = host(wql.w4a16_gemm(torch.zeros((4, K), dtype=torch.float16, device="cuda"), qw, s, qz, G))
    assert np.all(y == 0)
    wql.device_status()


def test_pack_then_gemm_on_one_stream_without_sync(wql):
    """The GEMMs copy their weights before waiting for the preceding kernel (programmatic dependent
    launch); the packing kernel makes its writes visible before it exits, so a GEMM enqueued right
    after it reads the new weights.  Two weights are packed alternately into the same buffers, each
    pack followed at once by a GEMM (no synchronisation in between): every GEMM must see the weights
    of the pack just before it, never the other ones."""
    M, K, N, G = 4, 4096, 4096, 128
    Ws = [dev(inputs.weight(K, N, seed=40 + i, outliers=True)) for i in range(2)]
    x = dev(inputs.activations(M, K, seed=40))
    qw = torch.empty((K, N // 8), dtype=torch.int32, device="cuda")
    s = torch.empty((K // G, N), dtype=torch.float16, device="cuda")
    qz = torch.empty((K // G, N // 8), dtype=torch.int32, device="cuda")
    refs = []
    for W in Ws:  # each weight's output, computed with a synchronisation in between
        a, b, c = wql.awq_pack(W, G)
        refs.append(wql.w4a16_gemm(x, a, b, c, G).clone())
    torch.cuda.synchronize()
    assert not torch.equal(refs[0], refs[1])
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in range(40)]
    for i, y in enumerate(ys):
        W = Ws[i % 2]
        K_, N_ = W.shape
        lib = wql.load()
        st = torch.cuda.current_stream().cuda_stream
        assert lib.wql_awq_pack(ctypes.c_void_p(W.data_ptr()), K_, N_, G, ctypes.c_void_p(qw.data_ptr()),
                                ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(qz.data_ptr()),
                                ctypes.c_void_p(st)) == 0
        wql.w4a16_gemm(x, qw, s, qz, G, out=y)
    torch.cuda.synchronize()
    for i, y in enumerate(ys):
        assert torch.equal(y, refs[i % 2]), f"GEMM {i} did not see the weights packed just before it"
    wql.device_status()


# ------------------------------------------------------------------------------------------------
# QRMSNorm + per-token int8: bit-exact
# ------------------------------------------------------------------------------------------------

# M >= 2048 takes the row groups of 128 threads (K <= 4096) or 64 threads (K <= 2048), with
# ragged lanes at K = 1032 (129 chunks of 8 for 256 lanes) and one chunk at K = 8
@pytest.mark.parametrize("M,K", [(1, 8), (7, 512), (33, 4096), (3, 11008), (2, 16384), (512, 4096), (2048, 4096),
                                 (2304, 2048), (4096, 1032), (2048, 8), (2048, 11008)])
def test_qrmsnorm_quant_bit_exact(wql, M, K):
    X = inputs.activations(M, K, seed=1, outlier_channels=True)
    g = inputs.gamma(K, seed=1)
    if M >= 3:
        X[1] = 0  # all-zero row
        X[2] = np.float16(0.375)  # constant row
    q_r, xs_r = oracle.qrmsnorm_quant_i8(X, g, inputs.EPS)
    q, xs = wql.qrmsnorm_quant_i8(dev(X), dev(g), inputs.EPS)
    assert np.array_equal(host(q), q_r)
    assert np.array_equal(host(xs).view(np.uint32), xs_r.view(np.uint32))


# ------------------------------------------------------------------------------------------------
# SmoothQuant W8A8: prep chain bit-exact, int32 accumulators bit-exact, fp16 output bit-exact
# ------------------------------------------------------------------------------------------------

def _w8a8_chain(wql, M, K, N, seed=0):
    X = inputs.activations(M, K, seed=seed, outlier_channels=True)
    g = inputs.gamma(K, seed=seed)
    W = inputs.weight(K, N, seed=seed)
    # oracle
    a_r = oracle.act_absmax(X, g, inputs.EPS)
    s_r, g2_r, W2_r = oracle.smooth(a_r, g, W)
    qW_r, ws_r = oracle.per_channel_quant_i8(W2_r)
    q_r, xs_r = oracle.qrmsnorm_quant_i8(X, g2_r, inputs.EPS)
    # CUDA path
    Xd, gd, Wd = dev(X), dev(g), dev(W)
    a = wql.act_absmax(Xd, gd, inputs.EPS)
    s, g2, W2 = wql.smooth(a, gd, Wd)
    qW, ws = wql.per_channel_quant_i8(W2)
    q, xs = wql.qrmsnorm_quant_i8(Xd, g2, inputs.EPS)
    got = dict(a=host(a), s=host(s), g2=host(g2), W2=host(W2), qW=host(qW), ws=host(ws), q=host(q), xs=host(xs))
    ref = dict(a=a_r, s=s_r, g2=g2_r, W2=W2_r, qW=qW_r, ws=ws_r, q=q_r, xs=xs_r)
    return got, ref, (q, xs, qW, ws)


@pytest.mark.parametrize("M,K,N", [(1, 512, 64), (16, 4096, 4096), (37, 1024, 96), (2048, 2048, 64)])
def test_w8a8_prep_chain_bit_exact(wql, M, K, N):
    got, ref, _ = _w8a8_chain(wql, M, K, N)
    for k in ("a", "s", "W2", "ws", "xs"):
        assert np.array_equal(got[k].view(np.uint32), ref[k].view(np.uint32)), k
    assert np.array_equal(got["g2"].view(np.uint16), ref["g2"].view(np.uint16))
    assert np.array_equal(got["qW"], ref["qW"])
    assert np.array_equal(got["q"], ref["q"])


W8A8_BLOCK_CELLS = [(c["M"], c["K"], c["N"]) for c in inputs.w8a8_cases()]  # all eight (M, N) cells


@pytest.mark.parametrize("M,K,N", W8A8_BLOCK_CELLS + [(5, 512, 96), (33, 1024, 160)])
def test_w8a8_gemm_bit_exact(wql, M, K, N):
    got, ref, (q, xs, qW, ws) = _w8a8_chain(wql, M, K, N, seed=2)
    acc = Guarded((M, N), torch.int32)
    yg = Guarded((M, N), torch.float16)
    wql.w8a8_gemm(q, xs, qW, ws, out=yg.t, acc_out=acc.t)
    acc.check()
    yg.check()
    y = host(yg.t)
    assert np.isfinite(y).all(), f"{int((~np.isfinite(y)).sum())} outputs left unwritten"
    assert acc.unwritten() == 0  # 0x7F7F7F7F exceeds any sum of K <= 2^17 int8 products
    rows = tile_rows(M)
    acc_r = oracle.w8a8_acc(ref["q"], ref["qW"], rows=rows)
    y_r = oracle.w8a8_epilogue(acc_r, ref["xs"][rows], ref["ws"])
    assert np.array_equal(host(acc.t)[rows], acc_r)
    assert np.array_equal(y[rows].view(np.uint16), y_r.view(np.uint16))
    y64 = oracle.w8a8_epilogue_f64(acc_r, ref["xs"][rows], ref["ws"])
    assert row_rel_err(y[rows], y64) <= ROW_TOL


@pytest.mark.parametrize("K", [4096, 16384])
def test_w8a8_int32_exact_beyond_fp32_integer_range(wql, K):
    # all products at the extreme: |acc| = K * 128 * 127 > 2^24, where plain fp32 sums lose integers
    M, N = 3, 64
    q = np.full((M, K), -128, np.int8)
    q[1] = 127
    q[2, ::2] = -128
    q[2, 1::2] = 127
    qW = np.full((N, K), -127, np.int8)
    qW[1::2] = 127
    xs = np.full((M,), 0.01, np.float32)
    ws = np.full((N,), 0.001, np.float32)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    wql.w8a8_gemm(dev(q), dev(xs), dev(qW), dev(ws), acc_out=acc)
    assert np.array_equal(host(acc), oracle.w8a8_acc(q, qW))


def test_w8a8_random_extremes_bit_exact(wql):
    rng = np.random.default_rng(5)
    M, K, N = 9, 8192, 128
    q = rng.choice(np.array([-128, -127, 127, 0, 1], np.int8), size=(M, K))
    qW = rng.choice(np.array([-127, 127, 0, -1], np.int8), size=(N, K))
    xs = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    ws = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    y = wql.w8a8_gemm(dev(q), dev(xs), dev(qW), dev(ws), acc_out=acc)
    acc_r = oracle.w8a8_acc(q, qW)
    assert np.array_equal(host(acc), acc_r)
    assert np.array_equal(host(y).view(np.uint16), oracle.w8a8_epilogue(acc_r, xs, ws).view(np.uint16))
    wql.device_status()


# ------------------------------------------------------------------------------------------------
# boundary behaviour on the device
# ------------------------------------------------------------------------------------------------

def test_empty_calls_and_errors(wql):
    x = torch.empty((0, 256), dtype=torch.float16, device="cuda")
    W = inputs.weight(256, 64, seed=0)
    qw, s, qz = wql.awq_pack(dev(W), 32)
    y = wql.w4a16_gemm(x, qw, s, qz, 32)
    assert y.shape == (0, 64)
    with pytest.raises(wql.WQLError):
        wql.awq_pack(dev(W[:, :48].copy()), 32)  # N not a multiple of 32
    wql.device_status()


# ------------------------------------------------------------------------------------------------
# long back-to-back launch chains (programmatic dependent launch, graph replay): the pipelined
# kernels must stay correct and fault-free over thousands of launches
# ------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,N,G", [(1, 4096, 4096, 128), (16, 4096, 4096, 128), (4, 11008, 4096, 32)])
def test_w4a16_decode_back_to_back_stress(wql, M, K, N, G):
    layers, reps = 16, 150
    W = inputs.weight(K, N, seed=1)
    qw, s, qz = wql.awq_pack(dev(W), G)
    stack = [(qw.clone(), s.clone(), qz.clone()) for _ in range(layers)]
    x = dev(inputs.activations(M, K, seed=1))
    ref = wql.w4a16_gemm(x, qw, s, qz, G).clone()
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in range(layers)]
    stream = torch.cuda.Stream()

    def step():
        for i, (a, b, c) in enumerate(stack):
            wql.w4a16_gemm(x, a, b, c, G, out=ys[i])

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
        assert torch.equal(y, ref)  # deterministic: bit-identical to the single call


def test_w8a8_decode_back_to_back_stress(wql):
    M, K, N = 16, 4096, 4096
    rng = np.random.default_rng(3)
    q = dev(rng.integers(-128, 128, size=(M, K), dtype=np.int8))
    xs = dev(rng.uniform(1e-3, 1e-2, M).astype(np.float32))
    qW = dev(rng.integers(-127, 128, size=(N, K), dtype=np.int8))
    ws = dev(rng.uniform(1e-4, 1e-3, N).astype(np.float32))
    ref = wql.w8a8_gemm(q, xs, qW, ws).clone()
    layers, reps = 16, 150
    stack = [qW.clone() for _ in range(layers)]
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in range(layers)]
    stream = torch.cuda.Stream()

    def step():
        for i, w in enumerate(stack):
            wql.w8a8_gemm(q, xs, w, ws, out=ys[i])

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


@pytest.mark.parametrize("M", [1, 8])
def test_decode_split_k_repeatable_at_many_strips(wql, M):
    """N = 22016 gives 172 strips and a 3-way cluster split-K: every call must give the same bits.
    (Before the consumers fenced their generic-proxy reads of a stage ahead of its TMA refill, 1-4 %
    of such calls came out with one column group's partial sums computed from a refilled stage.)"""
    K, N, G = 4096, 22016, 128
    W = inputs.weight(K, N, seed=M + N, outliers=True)
    x = dev(inputs.activations(M, K, seed=M + N, outlier_channels=True))
    qw, s, qz = wql.awq_pack(dev(W), G)
    ref = wql.w4a16_gemm(x, qw, s, qz, G).clone()
    y = torch.empty_like(ref)
    bad = 0
    for _ in range(300):
        wql.w4a16_gemm(x, qw, s, qz, G, out=y)
        bad += int(not torch.equal(y, ref))
    assert bad == 0, f"{bad} of 300 calls differ"
    rng = np.random.default_rng(M)
    q = dev(rng.integers(-128, 128, size=(M, K), dtype=np.int8))
    xs = dev(rng.uniform(1e-3, 1e-2, M).astype(np.float32))
    qW = dev(rng.integers(-127, 128, size=(N, K), dtype=np.int8))
    ws = dev(rng.uniform(1e-4, 1e-3, N).astype(np.float32))
    ref8 = wql.w8a8_gemm(q, xs, qW, ws).clone()
    y8 = torch.empty_like(ref8)
    bad8 = 0
    for _ in range(300):
        wql.w8a8_gemm(q, xs, qW, ws, out=y8)
        bad8 += int(not torch.equal(y8, ref8))
    assert bad8 == 0, f"{bad8} of 300 int8 calls differ"
    wql.device_status()
