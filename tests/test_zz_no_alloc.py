"""The int8 GEMM entry point that allocates nothing, checked against the workspace-taking one.

wql_w8a8_gemm_noalloc is for callers that cannot allocate device memory when they call the layer
(an engine whose memory is all reserved by its own pool, a plugin whose host framework owns every
allocation, a loop that cannot afford the allocator's synchronisation).  It runs the same kernels
as wql_w8a8_gemm with the library's built-in scratch array in place of a caller workspace, so its
results must be identical.  This file is named to be collected last: a run that stops at its first
failure has then already run every other test.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from _gpu_util import tile_rows  # noqa: E402


@pytest.fixture(scope="module")
def wql(wql_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return wql_lib


def _case(M, K, N, seed):
    rng = np.random.default_rng(seed)
    q = torch.from_numpy(rng.integers(-128, 128, size=(M, K), dtype=np.int8)).cuda()
    qw = torch.from_numpy(rng.integers(-127, 128, size=(N, K), dtype=np.int8)).cuda()
    xs = torch.from_numpy(rng.uniform(1e-3, 1e-2, M).astype(np.float32)).cuda()
    ws = torch.from_numpy(rng.uniform(1e-4, 1e-3, N).astype(np.float32)).cuda()
    return q, xs, qw, ws


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(wql):
    # Problems back to back through the C ABI: each call reuses the shared scratch the previous one
    # filled, and each must equal the workspace-taking entry point bit for bit.  The third problem
    # is smaller than the second, so the scratch still holds the second call's data past its own
    # M * K elements: nothing left over from an earlier call may leak into a result.  The oracle
    # checks the accumulators and outputs on the first and last row of every 32-row block.
    for M, K, N, seed in [(257, 4096, 4096, 1), (1024, 2048, 4160, 2), (300, 1024, 256, 3)]:
        q, xs, qw, ws = _case(M, K, N, seed)
        y_ref = wql.w8a8_gemm(q, xs, qw, ws)
        acc_ref = torch.empty((M, N), dtype=torch.int32, device="cuda")
        wql.w8a8_gemm(q, xs, qw, ws, acc_out=acc_ref)
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        acc = torch.zeros((M, N), dtype=torch.int32, device="cuda")
        wql.w8a8_gemm_noalloc(q, xs, qw, ws, out=y, acc_out=acc)
        torch.cuda.synchronize()
        assert torch.equal(acc, acc_ref)
        assert torch.equal(y, y_ref)
        rows = tile_rows(M)
        qh, qwh, xsh, wsh = q.cpu().numpy(), qw.cpu().numpy(), xs.cpu().numpy(), ws.cpu().numpy()
        acc_o = oracle.w8a8_acc(qh, qwh, rows=rows)
        assert np.array_equal(acc.cpu().numpy()[rows], acc_o)
        y_o = oracle.w8a8_epilogue(acc_o, xsh[rows], wsh)
        assert np.array_equal(y.cpu().numpy()[rows].view(np.uint16), y_o.view(np.uint16))
    wql.device_status()


def test_noalloc_decode_shape_needs_no_scratch(wql):
    q, xs, qw, ws = _case(4, 4096, 4096, 3)
    y = torch.empty((4, 4096), dtype=torch.float16, device="cuda")
    wql.w8a8_gemm_noalloc(q, xs, qw, ws, out=y)
    assert torch.equal(y, wql.w8a8_gemm(q, xs, qw, ws))
    wql.device_status()


def test_noalloc_rejects_calls_beyond_the_static_scratch(wql):
    # M * K * 2 + 16384 = 34422784 bytes > 32 MiB + 64 KiB: rejected before anything is launched
    q = torch.zeros((4200, 4096), dtype=torch.int8, device="cuda")
    xs = torch.ones((4200,), dtype=torch.float32, device="cuda")
    qw = torch.zeros((64, 4096), dtype=torch.int8, device="cuda")
    ws = torch.ones((64,), dtype=torch.float32, device="cuda")
    y = torch.empty((4200, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(wql.WQLError) as ei:
        wql.w8a8_gemm_noalloc(q, xs, qw, ws, out=y)
    assert ei.value.status == 2
    assert "static scratch" in str(ei.value)
