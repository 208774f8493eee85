"""Concurrent first calls from several host threads, each on its own stream: the launchers' per-device
caches (kernel attributes, the norm's ring size and occupancy, the SM count) must stay consistent,
and every result must still match the oracle bit for bit."""
import threading

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


def test_norm_from_many_threads(wql):
    # row lengths that need different rings (and hence cache updates), interleaved across threads
    Ks = [1032, 4096, 8192, 16384, 2048, 6144, 12288, 4104]
    cases = [(17 + 3 * i, Ks[i % len(Ks)], i) for i in range(16)]
    want = {}
    for (M, K, seed) in cases:
        X = inputs.activations(M, K, seed=seed, outlier_channels=True)
        g = inputs.gamma(K, seed=seed)
        want[seed] = (X, g, oracle.qrmsnorm_quant_i8(X, g, inputs.EPS))
    got, errors = {}, []
    barrier = threading.Barrier(8)

    def worker(tid):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream()
            barrier.wait()
            with torch.cuda.stream(stream):
                for (M, K, seed) in cases[tid::8]:
                    X, g, _ = want[seed]
                    q, xs = wql.qrmsnorm_quant_i8(torch.from_numpy(X).cuda(), torch.from_numpy(g).cuda(), inputs.EPS)
                    stream.synchronize()
                    got[seed] = (q.cpu().numpy(), xs.cpu().numpy())
        except Exception as e:  # noqa: BLE001 -- reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (M, K, seed) in cases:
        q_r, xs_r = want[seed][2]
        q, xs = got[seed]
        assert np.array_equal(q, q_r) and np.array_equal(xs.view(np.uint32), xs_r.view(np.uint32)), (M, K)
    wql.device_status()
