"""Weight quantisation on values whose quotients w / s fall on, or one ulp beside, the rounding
ties of round-half-to-even.  The kernels divide by multiplying with 1 / s and fall back to the
exact division near a tie; the codes must still equal the oracle's (a correctly rounded division,
then round-half-even) bit for bit."""
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


def _ties(shape, lo, hi, seed):
    rng = np.random.default_rng(seed)
    halves = np.arange(2 * lo + 1, 2 * hi, 2, dtype=np.float32) / 2  # lo + 0.5 .. hi - 0.5
    v = rng.choice(halves, size=shape).astype(np.float32)
    pick = rng.integers(0, 3, size=shape)
    v = np.where(pick == 1, np.nextafter(v, np.float32(np.inf)), v)
    v = np.where(pick == 2, np.nextafter(v, np.float32(-np.inf)), v)
    return v.astype(np.float32)


@pytest.mark.parametrize("G", [32, 64, 128])
def test_awq_pack_on_rounding_ties(wql, G):
    K, N = 2 * G, 96
    W = _ties((K, N), 0, 15, seed=G)
    W[::G] = 0.0        # every group holds 0 and 15: s = 1 exactly, z = 0, so w / s = w
    W[1::G] = 15.0
    W[:, 8:16] *= np.float32(0.25)  # a power-of-two scale: the same ties at s = 0.25
    qw_r, s_r, qz_r = oracle.awq_quantize(W, G)
    qw, s, qz = wql.awq_pack(torch.from_numpy(W).cuda(), G)
    torch.cuda.synchronize()
    assert np.array_equal(qw.cpu().numpy(), qw_r.view(np.int32))
    assert np.array_equal(s.cpu().numpy().view(np.uint16), s_r.view(np.uint16))
    assert np.array_equal(qz.cpu().numpy(), qz_r.view(np.int32))


def test_per_channel_quant_on_rounding_ties(wql):
    K, N = 256, 64
    W = _ties((K, N), -127, 127, seed=7)
    W[0] = 127.0                    # column maxima 127: ws = 1 exactly, so w / ws = w
    W[:, 32:] *= np.float32(0.5)    # and 0.5 for the second half of the columns
    qw_r, ws_r = oracle.per_channel_quant_i8(W)
    qw, ws = wql.per_channel_quant_i8(torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(ws.cpu().numpy().view(np.uint32), ws_r.view(np.uint32))
    assert np.array_equal(qw.cpu().numpy(), qw_r)
