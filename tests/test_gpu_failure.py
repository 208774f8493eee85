"""Failure detection without a GPU fault: a bounded on-chip wait that runs out must come back to the
host as WQL_ETIMEOUT through the device error word, once, and leave the context usable."""
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


def test_expired_wait_is_reported_once_and_the_context_survives(wql):
    wql.device_status()  # start clean
    wql.diag_expire_wait()  # one thread waits on a barrier nothing completes; it gives up (~2 s)
    with pytest.raises(wql.WQLError) as exc:
        wql.device_status()
    assert exc.value.status == 4  # WQL_ETIMEOUT
    wql.device_status()  # the error word was cleared
    # the context still runs kernels, with correct results
    X = inputs.activations(4, 512, seed=9, outlier_channels=True)
    g = inputs.gamma(512, seed=9)
    q, xs = wql.qrmsnorm_quant_i8(torch.from_numpy(X).cuda(), torch.from_numpy(g).cuda(), inputs.EPS)
    q_r, xs_r = oracle.qrmsnorm_quant_i8(X, g, inputs.EPS)
    assert np.array_equal(q.cpu().numpy(), q_r) and np.array_equal(xs.cpu().numpy(), xs_r)
    wql.device_status()
