"""The allocation-free GEMM entry point.

minfer_op_gemm_noalloc serves callers that cannot call cudaMalloc: a process
whose own allocator already holds nearly all device memory, or code that must
not trigger the device-wide synchronization of cudaFree.  It keeps its operand
planes and split-K partials in a fixed 32 MiB device array inside the library.
This file is collected last on purpose, so a run that stops at the first
failure has run every other test first; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def qp():
    import quantized_transformer_prefill_gb300 as qp
    qp.lib()
    return qp


def _operands(seed, M, N, K):
    rng = np.random.default_rng(seed)
    nb = (K + 31) // 32
    xq = rng.integers(-127, 128, (M, nb * 32)).astype(np.int8)
    wq = rng.integers(-127, 128, (N, nb * 32)).astype(np.int8)
    xq[:, K:] = 0
    wq[:, K:] = 0
    xd = np.float16(rng.uniform(1e-3, 3e-2, (M, nb))).view(np.uint16)
    wd = np.float16(rng.uniform(1e-4, 1e-3, (N, nb))).view(np.uint16)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dev(xq), dev(xd.view(np.int16)), dev(wq), dev(wd.view(np.int16))


def test_noalloc_gemm_matches_allocating_gemm_twice(qp):
    """Two calls in a row (different shapes, the second finds the first's
    leftovers in the shared array) each match minfer_op_gemm."""
    for seed, (M, N, K) in enumerate([(300, 520, 688), (512, 896, 4864)]):
        xq, xd, wq, wd = _operands(seed, M, N, K)
        ref = qp.op_gemm(xq, xd, wq, wd, K).cpu().numpy()
        got = qp.op_gemm_noalloc(xq, xd, wq, wd, K).cpu().numpy()
        np.testing.assert_allclose(got, ref, rtol=2e-6, atol=2e-6 * np.abs(ref).max())


def test_noalloc_gemm_rejects_oversize(qp):
    """A problem whose scratch exceeds the fixed array is refused before any
    device work, with a dedicated error code."""
    M, N, K = 4096, 4096, 4096
    nb = K // 32
    xq = torch.zeros((M, nb * 32), dtype=torch.int8, device="cuda")
    xd = torch.zeros((M, nb), dtype=torch.int16, device="cuda")
    wq = torch.zeros((N, nb * 32), dtype=torch.int8, device="cuda")
    wd = torch.zeros((N, nb), dtype=torch.int16, device="cuda")
    y = torch.full((M, N), 5.0, dtype=torch.float32, device="cuda")
    rc = qp.lib().minfer_op_gemm_noalloc(xq.data_ptr(), xd.data_ptr(), M, wq.data_ptr(),
                                         wd.data_ptr(), N, K, y.data_ptr())
    assert rc == -10
    assert qp.lib().minfer_strerror(rc).decode()
    assert bool(torch.all(y == 5.0))
