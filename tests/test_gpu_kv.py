"""GPU parity of the KV-cache int8 quantisation (groups of 128 channels) and its dequantisation.

Both sides take every rounding decision in fp32 (the scale absmax / 127, the quotient, the product
q * s) and round the same way, so codes, scales and dequantised fp16 values must match the oracle
bit for bit, including at exact rounding ties.
"""
import numpy as np
import pytest

import oracle
from weight_quantized_linear_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


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


def _kv(rows, D, seed):
    """K/V-like rows: per-row magnitudes spread over four decades, a few outlier channels."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, D)) * rng.uniform(0.05, 50.0, size=(rows, 1))
    x[:, rng.choice(D, size=max(1, D // 100), replace=False)] *= 20.0
    return np.clip(x, -60000, 60000).astype(np.float16)


# rows x D: single group, ragged row counts, Llama-7B K+V per token (2 x 32 heads x 128) for a
# 4096-token prefill, and a long row
@pytest.mark.parametrize("rows,D", [(1, 128), (7, 256), (33, 4096), (4096, 8192), (3, 16384), (1000, 384)])
def test_kv_quant_and_dequant_bit_exact(wql, rows, D):
    x = _kv(rows, D, seed=rows + D)
    q, s = wql.kv_quant_i8(dev(x))
    q_r, s_r = oracle.kv_quant_i8(x)
    assert np.array_equal(host(s).view(np.uint32), s_r.view(np.uint32))
    assert np.array_equal(host(q), q_r)
    out = wql.kv_dequant_i8(q, s)
    assert np.array_equal(host(out).view(np.uint16), oracle.kv_dequant_i8(q_r, s_r).view(np.uint16))
    wql.device_status()


def test_kv_quant_ties_zero_groups_and_signed_zeros(wql):
    rows, D = 5, 512
    x = _kv(rows, D, seed=3)
    x[1, 128:256] = 0  # all-zero group: scale 1, codes 0
    x[2, :128] = -0.0
    # a group with scale exactly 2^-7 (absmax 127 * 2^-7) whose values sit on exact ties (c + 0.5) * 2^-7
    c = np.arange(-63, 65, dtype=np.float64)
    x[3, 256:384] = ((c + 0.5) * 2.0 ** -7).astype(np.float16)
    x[3, 256] = np.float16(127 * 2.0 ** -7)
    q, s = wql.kv_quant_i8(dev(x))
    q_r, s_r = oracle.kv_quant_i8(x)
    assert s_r[3, 2] == np.float32(2.0 ** -7)
    assert np.array_equal(host(s).view(np.uint32), s_r.view(np.uint32))
    assert np.array_equal(host(q), q_r)
    assert np.all(q_r[1, 128:256] == 0) and s_r[1, 1] == 1.0
    wql.device_status()


def test_kv_leading_dims_empty_and_invalid(wql):
    x = _kv(2 * 3 * 4, 256, seed=4).reshape(2, 3, 4, 256)  # [layers, tokens, heads, ...] style leading dims
    q, s = wql.kv_quant_i8(dev(x))
    assert q.shape == (2, 3, 4, 256) and s.shape == (2, 3, 4, 2)
    q_r, s_r = oracle.kv_quant_i8(x.reshape(-1, 256))
    assert np.array_equal(host(q).reshape(-1, 256), q_r)
    e = torch.empty((0, 128), dtype=torch.float16, device="cuda")
    q0, s0 = wql.kv_quant_i8(e)
    assert q0.shape == (0, 128) and s0.shape == (0, 1)
    with pytest.raises(wql.WQLError):
        wql.kv_quant_i8(dev(_kv(2, 192, seed=5)))  # D not a multiple of 128
    wql.device_status()


def test_kv_round_trip_error_bound(wql):
    x = _kv(512, 8192, seed=6)
    q, s = wql.kv_quant_i8(dev(x))
    out = host(wql.kv_dequant_i8(q, s)).astype(np.float64)
    step = np.repeat(host(s).astype(np.float64), 128, axis=1)
    # half a quantisation step, plus the fp16 rounding of the dequantised value
    bound = 0.5 * step * (1 + 1e-6) + np.abs(out) * 2.0 ** -11 + 2.0 ** -25
    assert np.all(np.abs(out - x.astype(np.float64)) <= bound)
    wql.device_status()
