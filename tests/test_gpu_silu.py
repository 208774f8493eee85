"""GPU parity of the fused gate/up activation of the W4A16 GEMM (w4a16_gemm_silu_mul).

* Against the oracle: silu(gate) * up of the fp64 GEMM output, within the W4A16 tolerance
  (row-relative L2 <= 1e-2).
* Against the unfused composition on the device: the same library's fp16 GEMM output followed by
  silu(g) * u in fp32, which the fusion reproduces up to the last-bit difference of exp
  implementations (at most one fp16 unit).
Both kernels (the streaming decode kernel and the tcgen05 kernel, with and without split-K) are
covered, by shape and by the kernel-forcing switch.
"""
import numpy as np
import pytest

import oracle
from weight_quantized_linear_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from _gpu_util import Guarded  # noqa: E402

ROW_TOL = 1e-2


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


def sample_rows(M, n=12):
    if M <= n:
        return np.arange(M, dtype=np.int64)
    return np.unique(np.concatenate([np.linspace(0, M - 1, n).astype(np.int64), [M - 1]]))


def _case(wql, M, K, N, G, seed):
    """The weights in the oracle's packing (nothing the oracle sees comes from the CUDA path), and the
    same packed tensors on the device for the kernels under test."""
    W = inputs.weight(K, N, seed=seed, outliers=True)  # columns 2j / 2j + 1 act as gate j / up j
    X = inputs.activations(M, K, seed=seed, outlier_channels=True)
    packed = oracle.awq_quantize(W, G)
    qw_r, s_r, qz_r = packed
    return X, packed, dev(qw_r.view(np.int32)), dev(s_r), dev(qz_r.view(np.int32))


def _check(wql, X, packed, qw, s, qz, G, M, N):
    x = dev(X)
    out = Guarded((M, N // 2), torch.float16)
    y = wql.w4a16_gemm_silu_mul(x, qw, s, qz, G, out=out.t)
    out.check()
    assert y.shape == (M, N // 2) and np.isfinite(host(y)).all()
    rows = sample_rows(M)
    # the oracle: fp64 GEMM of the oracle-packed weight, then silu(gate) * up in fp64
    qw_r, s_r, qz_r = packed
    y2 = oracle.w4a16_linear(X, qw_r, s_r, qz_r, G, rows=rows)
    ref = oracle.silu_mul_f64(y2)
    got = host(y)[rows].astype(np.float64)
    num = np.linalg.norm(got - ref, axis=1)
    den = np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert np.max(num / den) <= ROW_TOL
    # the unfused composition on the device, from the same kernel's fp16 outputs
    y16 = wql.w4a16_gemm(x, qw, s, qz, G).float()
    g, u = y16[:, 0::2], y16[:, 1::2]
    comp = (g / (1.0 + torch.exp(-g)) * u).half()
    diff = (y.float() - comp.float()).abs()
    ulp = torch.maximum(comp.float().abs() * 2.0 ** -10, torch.full_like(diff, 2.0 ** -24))
    bad = (~(diff <= ulp * 1.001)).nonzero()
    if bad.shape[0]:
        r, j = bad[0].tolist()
        raise AssertionError(f"{bad.shape[0]} of {diff.numel()} outputs off by more than one fp16 unit; first "
                             f"[{r}, {j}]: fused {y[r, j].item()} composed {comp[r, j].item()} "
                             f"g {g[r, j].item()} u {u[r, j].item()}")
    wql.device_status()


# decode (M <= 16), the tcgen05 kernel (split-K for few tiles, 128-, 192- and 256-token tiles), ragged
@pytest.mark.parametrize("M,K,N,G", [(1, 4096, 22016, 128), (8, 4096, 22016, 64), (16, 1024, 1024, 32),
                                     (128, 4096, 1024, 128), (300, 4096, 22016, 128), (2048, 4096, 4096, 128),
                                     (37, 1024, 192, 64), (560, 4096, 11008, 128)])
def test_w4a16_silu_mul(wql, M, K, N, G):
    X, packed, qw, s, qz = _case(wql, M, K, N, G, seed=M + N)
    _check(wql, X, packed, qw, s, qz, G, M, N)


@pytest.mark.parametrize("force", ["decode", "prefill"])
def test_w4a16_silu_mul_both_kernels_mid_m(wql, monkeypatch, force):
    M, K, N, G = 24, 2048, 1024, 128
    monkeypatch.setenv("WQL_FORCE_KERNEL", force)
    X, packed, qw, s, qz = _case(wql, M, K, N, G, seed=7)
    _check(wql, X, packed, qw, s, qz, G, M, N)


def test_w4a16_silu_mul_gate_up_interleave_helper(wql):
    K, I, G, M = 512, 256, 128, 4
    wg = inputs.weight(K, I, seed=11)
    wu = inputs.weight(K, I, seed=12)
    fused = wql.interleave_gate_up(dev(wg), dev(wu))
    f = host(fused)
    assert np.array_equal(f[:, 0::2], wg) and np.array_equal(f[:, 1::2], wu)
    packed = oracle.awq_quantize(np.concatenate([wg[:, :, None], wu[:, :, None]], axis=2).reshape(K, 2 * I), G)
    qw, s, qz = wql.awq_pack(fused, G)
    assert np.array_equal(host(qw), packed[0].view(np.int32))  # the device packing agrees bit for bit
    X = inputs.activations(M, K, seed=13)
    _check(wql, X, packed, qw, s, qz, G, M, 2 * I)


def test_w4a16_silu_mul_rejects_odd_pairs(wql):
    W = inputs.weight(256, 96, seed=1)
    qw, s, qz = wql.awq_pack(dev(W), 128)
    x = dev(inputs.activations(2, 256, seed=1))
    with pytest.raises(wql.WQLError):
        wql.w4a16_gemm_silu_mul(x, qw, s, qz, 128)  # N = 96 is not a multiple of 64
    wql.device_status()
