"""The allocation-free GEMM entry point.

minfer_op_gemm_noalloc is for callers that cannot call cudaMalloc: a process
whose own memory pool reserved nearly all of HBM at start-up, or code that
must not stall the whole device the way cudaFree does.  It keeps its operand
planes and split-K partials in a fixed 32 MiB device array inside the library
and runs on a stream of its own.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test first; it also passes on its own in a fresh
process.
"""
import numpy as np
import pytest

from helpers import check_q8_sum

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
    return xq, xd, wq, wd


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_noalloc_gemm_matches_oracle_twice(qp, oracle_mod):
    """Two calls in a row (different shapes; the second finds the first's
    leftovers in the shared array), each within the f32 rounding bound of the
    oracle's Q8_0 matmul on sampled rows, and equal to the allocating entry
    point's result (same kernels, same split plan)."""
    for seed, (M, N, K) in enumerate([(300, 520, 688), (512, 896, 4864)]):
        xq, xd, wq, wd = _operands(seed, M, N, K)
        args = (_dev(xq), _dev(xd.view(np.int16)), _dev(wq), _dev(wd.view(np.int16)), K)
        got = qp.op_gemm_noalloc(*args).cpu().numpy()
        rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 37)), [M - 1]]))
        check_q8_sum(oracle_mod, got[rows], xq[rows], xd[rows], wq, wd, K)
        ref = qp.op_gemm(*args).cpu().numpy()
        assert np.array_equal(got, ref)


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
    for m, n in ((M, N), (2 ** 31, 16), (16, 2 ** 40)):
        rc = qp.lib().minfer_op_gemm_noalloc(xq.data_ptr(), xd.data_ptr(), m, wq.data_ptr(),
                                             wd.data_ptr(), n, K, y.data_ptr())
        assert rc == -10, (m, n, rc)
    assert qp.lib().minfer_strerror(-10).decode()
    torch.cuda.synchronize()
    assert bool(torch.all(y == 5.0))
