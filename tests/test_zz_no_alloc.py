"""qgemv_run_noalloc: the handle-free entry point for callers that may not allocate device
memory (a host application that owns all device memory, a capped or instrumented
allocator, a latency-critical path that cannot afford an allocation's synchronisation).
It keeps its scratch in fixed arrays inside the library, so these checks call it through
the C-ABI twice in a row, on the same and on different shapes, and compare each result with
qgemv_run's on the same inputs, within the GEMV tolerance used by every parity test
(|y - y_ref| <= 2e-3 * sum|x w| + 1e-5, with sum|x w| from the oracle).  The file is named
to be collected last; it also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import ATOL, RTOL, dev_bytes, dev_x
from quantized_weight_dequant_gb300 import qgemv, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_weight_dequant_gb300.build import build_library
    build_library()
    handle = qgemv.create(0)
    yield handle
    handle.close()


def _inputs(fmt, N, K, seed):
    W = synth.make_weights(fmt, N, K, seed)
    x = synth.make_x(fmt, K, seed)
    Wd, _ = dev_bytes(W)
    _, S = oracle.gemv(fmt, x, W, N, K)
    return Wd, dev_x(x), S


def _close(a, b, S):
    err = np.abs(a.astype(np.float64) - b.astype(np.float64))
    bad = np.nonzero(~(err <= RTOL * S + ATOL))[0]
    assert bad.size == 0, (bad[:5], err[bad[:5]])


CASES = [(synth.Q4_K, 4096, 14336), (synth.NVFP4, 700, 14336), (synth.Q4_K, 2000, 4096),
         (synth.Q6_K, 129, 12288), (synth.Q8_0, 300, 6144), (synth.TQ1_0, 77, 4096),
         (synth.Q5_K, 50, 2048)]


def test_noalloc_matches_run_on_two_calls_in_a_row(h):
    prev = None
    for fmt, N, K in CASES:
        Wd, xd, S = _inputs(fmt, N, K, seed=N + K + fmt)
        y_ref = torch.empty(N, dtype=torch.float32, device="cuda")
        qgemv.run(h, fmt, xd, Wd, N, K, y_ref)
        for call in range(2):  # the second call finds the scratch as the first left it
            y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
            qgemv.run_noalloc(fmt, xd, Wd, N, K, y)
            torch.cuda.synchronize()
            _close(y.cpu().numpy(), y_ref.cpu().numpy(), S)
            if call == 1:
                assert torch.equal(y, prev), "results differ between two calls in a row"
            prev = y.clone()
    assert qgemv.check_error(h) == qgemv.OK


def test_noalloc_rejects_shapes_beyond_its_scratch(h):
    N, K = qgemv.NOALLOC_MAX_COLUMN_SUMS // 7 + 1, 14336  # 7 K-columns
    y = torch.empty(16, dtype=torch.float32, device="cuda")
    x = torch.zeros(K, dtype=torch.int16, device="cuda")
    W = torch.zeros(64, dtype=torch.uint8, device="cuda")  # never read: rejected before launch
    st = qgemv.run_noalloc(synth.Q4_K, x, W, N, K, y, check=False)
    assert st == qgemv.ERR_TOO_LARGE
    assert "scratch" in qgemv.status_string(st)
    assert qgemv.run_noalloc(synth.Q4_K, x, W, 5, 1000, y, check=False) == qgemv.ERR_BAD_SHAPE
    torch.cuda.synchronize()
