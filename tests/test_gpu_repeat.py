"""Repeatability of the pipelined tensor-core kernels: the same call, repeated back to back, gives
the same bits every time.  A pipeline that reads a stage before its copy has landed, or after its
refill has begun, shows up here as an occasional difference (each kernel's reduction order is
fixed, so any difference is a race).
"""
import numpy as np
import pytest

from weight_quantized_linear_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

REPS = 100


@pytest.fixture(scope="module")
def wql(wql_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return wql_lib


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _repeat(fn, out):
    ref = fn().clone()
    bad = 0
    for _ in range(REPS):
        fn()
        bad += int(not torch.equal(out, ref))
    return bad


# tcgen05 W4A16: 64- and 128-token tiles with split-K (few tiles; the exchange through bulk copies
# between the CTAs of a cluster), 128-token tiles, 256-token tiles (one accumulator: the epilogue
# hands it back to the MMAs of the next tile), up to 18 tiles per persistent CTA
@pytest.mark.parametrize("M,K,N", [(64, 4096, 1024), (128, 4096, 4096), (256, 11008, 4096), (512, 4096, 4096),
                                   (2048, 4096, 11008), (8192, 4096, 11008)])
def test_w4a16_prefill_repeatable(wql, M, K, N):
    G = 128
    qw, s, qz = wql.awq_pack(dev(inputs.weight(K, N, seed=N, outliers=True)), G)
    x = dev(inputs.activations(M, K, seed=M, outlier_channels=True))
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    assert wql.w4a16_kernel_for(M, K, N, G) == "prefill"
    bad = _repeat(lambda: wql.w4a16_gemm(x, qw, s, qz, G, out=y), y)
    assert bad == 0, f"{bad} of {REPS} calls differ"
    assert bool(torch.isfinite(y).all())
    wql.device_status()


# tcgen05 int8 (64- and 128-token tiles, bias + residual) and fp8 (one and two CTAs per SM)
@pytest.mark.parametrize("M,N", [(48, 4096), (512, 11008)])
def test_w8a8_prefill_repeatable(wql, M, N):
    K = 4096
    rng = np.random.default_rng(M)
    q = dev(rng.integers(-128, 128, size=(M, K), dtype=np.int8))
    xs = dev(rng.uniform(1e-3, 1e-2, M).astype(np.float32))
    qW = dev(rng.integers(-127, 128, size=(N, K), dtype=np.int8))
    ws = dev(rng.uniform(1e-4, 1e-3, N).astype(np.float32))
    bias = dev(rng.normal(0, 1, N).astype(np.float16))
    res = dev(rng.normal(0, 1, (M, N)).astype(np.float16))
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    bad = _repeat(lambda: wql.w8a8_gemm_fused(q, xs, qW, ws, bias, res, out=y), y)
    assert bad == 0, f"{bad} of {REPS} int8 calls differ"
    wql.device_status()


@pytest.mark.parametrize("M,N", [(512, 4096), (4096, 4096)])  # 128 tiles (one CTA per SM), 1024 (two)
def test_fp8_prefill_repeatable(wql, M, N):
    K = 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(M + N)
    q = (torch.randn(M, K, device="cuda", generator=g) * 60).to(torch.float8_e4m3fn)
    qW = (torch.randn(N, K, device="cuda", generator=g) * 60).to(torch.float8_e4m3fn)
    xs = torch.full((M,), 0.01, device="cuda")
    ws = torch.full((N,), 0.001, device="cuda")
    res = torch.randn(M, N, device="cuda", generator=g).half()
    y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    bad = _repeat(lambda: wql.w8a8_gemm_fp8(q, xs, qW, ws, None, res, out=y), y)
    assert bad == 0, f"{bad} of {REPS} fp8 calls differ"
    wql.device_status()
