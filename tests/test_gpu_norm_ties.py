"""QRMSNorm + int8 on rows built so that many quotients y / xs sit on or next to half-integers,
where round-half-even is decided by the last bit of the fp32 quotient.  The kernel must still
match the oracle's definition (a correctly rounded division, then round-half-even) bit for bit."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wql(wql_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return wql_lib


def _tie_rows(K, seed):
    rng = np.random.default_rng(seed)
    rows = []
    # with gamma = 1 and the row maximum 127, y / xs is 127 x / max|x| = x up to rounding: half-integers
    # in x land on (or within an ulp of) the rounding ties of the int8 codes
    halves = (np.arange(-254, 255) / 2.0).astype(np.float16)
    r = rng.choice(halves, size=K)
    r[0] = 127.0
    rows.append(r)
    r2 = rng.choice(halves, size=K) * np.float16(0.25)  # same ties after a power-of-two scaling
    r2[1] = np.float16(-31.75)
    rows.append(r2)
    # values one fp16 ulp away from half-integers
    near = halves.astype(np.float32)
    near = np.nextafter(near.astype(np.float16), np.float16(np.inf)).astype(np.float16)
    r3 = rng.choice(near, size=K)
    r3[2] = 127.0
    rows.append(r3)
    return np.stack(rows).astype(np.float16)


@pytest.mark.parametrize("K", [512, 4096])
def test_qrmsnorm_half_integer_quotients_bit_exact(wql, K):
    X = _tie_rows(K, seed=K)
    g = np.ones(K, np.float16)
    q_r, xs_r = oracle.qrmsnorm_quant_i8(X, g, 0.0)
    q, xs = wql.qrmsnorm_quant_i8(torch.from_numpy(X).cuda(), torch.from_numpy(g).cuda(), 0.0)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), q_r)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), xs_r.view(np.uint32))
    # the rows really exercise ties: many exact .5 quotients in fp64
    y64 = oracle.rmsnorm(X, g, 0.0).astype(np.float64)
    t = y64 / xs_r[:, None].astype(np.float64)
    assert np.mean(np.abs(np.abs(t - np.floor(t)) - 0.5) < 1e-4) > 0.2
