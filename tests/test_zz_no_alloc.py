"""qgemv_run_noalloc: the handle-free entry point for callers that may not allocate device
memory (a host application that owns all device memory, a capped or instrumented
allocator, a latency-critical path that cannot afford an allocation's synchronisation).
It keeps its scratch in fixed arrays inside the library, so these checks call it through
the C-ABI twice in a row and compare every result with the CPU oracle on the same inputs,
within the GEMV tolerance of every parity test (|y - y_ref| <= 2e-3 * sum|x w| + 1e-5),
and with qgemv_run's result within the same tolerance; two calls in a row give the same
bits.  Covered: the shapes at
the scratch limit exactly (N * ceil(K / 2048) equal to its capacity) and at the longest K
(16 K-columns), a call on a side stream, and a call captured in a CUDA graph on a side
stream and replayed.  The file is named to be collected last; it also passes on its own in
a fresh process."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_parity, dev_bytes, dev_x, sample_rows
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


CASES = [(synth.Q4_K, 4096, 14336), (synth.NVFP4, 700, 14336), (synth.Q4_K, 2000, 4096),
         (synth.Q6_K, 129, 12288), (synth.Q8_0, 300, 6144), (synth.TQ1_0, 77, 4096),
         (synth.Q5_K, 50, 2048), (synth.Q4_K, 40, 32768)]


def _two_calls(h, fmt, N, K, seed, rows=None, stream=None):
    W = synth.make_weights(fmt, N, K, seed)
    x = synth.make_x(fmt, K, seed)
    Wd, _ = dev_bytes(W)
    xd = dev_x(x)
    if rows is None:
        y_ref, S = oracle.gemv(fmt, x, W, N, K)
        rows = np.arange(N)
    else:
        y_ref, S = oracle.gemv_rows(fmt, x, W, N, K, rows)
    y_run = torch.empty(N, dtype=torch.float32, device="cuda")
    qgemv.run(h, fmt, xd, Wd, N, K, y_run)
    torch.cuda.synchronize()
    prev = None
    for call in range(2):  # the second call finds the scratch as the first left it
        y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
        if stream is None:
            qgemv.run_noalloc(fmt, xd, Wd, N, K, y)
        else:
            stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                qgemv.run_noalloc(fmt, xd, Wd, N, K, y, stream=stream)
            stream.synchronize()
        torch.cuda.synchronize()
        yh = y.cpu().numpy()
        assert_parity(yh[rows], y_ref, S, f"noalloc {synth.FORMAT_NAMES[fmt]} {N}x{K} call {call}")
        # against the existing entry point, within the same tolerance (their launch plans can
        # differ, e.g. fused K-columns in qgemv_run, so the bits may too)
        assert_parity(yh[rows], y_run.cpu().numpy()[rows].astype(np.float64), S,
                      f"noalloc against qgemv_run {synth.FORMAT_NAMES[fmt]} {N}x{K} call {call}")
        if prev is not None:
            assert torch.equal(y, prev), "results differ between two calls in a row"
        prev = y.clone()


@pytest.mark.parametrize("fmt,N,K", CASES)
def test_noalloc_matches_oracle_on_two_calls_in_a_row(h, fmt, N, K):
    _two_calls(h, fmt, N, K, seed=N + K + fmt)


def test_noalloc_at_the_scratch_limit_exactly(h):
    """N * ceil(K / 2048) = 16384 * 16 = the scratch capacity: accepted, and correct on sampled
    rows (the last row range ends at the last column sum of the scratch)."""
    N, K = qgemv.NOALLOC_MAX_COLUMN_SUMS // 16, 32768
    assert N * (K // 2048) == qgemv.NOALLOC_MAX_COLUMN_SUMS
    _two_calls(h, synth.Q4_K, N, K, seed=5, rows=sample_rows(N, 96, seed=5))
    torch.cuda.empty_cache()


def test_noalloc_on_a_side_stream(h):
    _two_calls(h, synth.Q4_K, 1000, 14336, seed=8, stream=torch.cuda.Stream())


def test_noalloc_in_a_cuda_graph_on_a_side_stream(h):
    """Captured on a side stream after a warm-up call, then replayed twice with new activations
    copied in between: each replay reads the x it finds and matches the oracle and qgemv_run on
    that x."""
    fmt, N, K = synth.Q4_K, 1000, 14336
    W = synth.make_weights(fmt, N, K, 21)
    Wd, _ = dev_bytes(W)
    xs = [synth.make_x(fmt, K, 21 + i) for i in range(2)]
    xd = dev_x(xs[0])
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    qgemv.run_noalloc(fmt, xd, Wd, N, K, y)  # the library's one-time set-up happens outside the capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        qgemv.run_noalloc(fmt, xd, Wd, N, K, y, stream=side)
    torch.cuda.synchronize()
    for i, x in enumerate(xs):
        xd.copy_(dev_x(x))
        y.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        y_ref, S = oracle.gemv(fmt, x, W, N, K)
        yh = y.cpu().numpy()
        assert_parity(yh, y_ref, S, f"noalloc graph replay {i}")
        y_run = torch.empty(N, dtype=torch.float32, device="cuda")
        qgemv.run(h, fmt, xd, Wd, N, K, y_run)
        torch.cuda.synchronize()
        assert_parity(yh, y_run.cpu().numpy().astype(np.float64), S, f"noalloc graph replay {i} against qgemv_run")


def test_noalloc_rejects_shapes_beyond_its_scratch(h):
    N, K = qgemv.NOALLOC_MAX_COLUMN_SUMS // 7 + 1, 14336  # 7 K-columns
    y = torch.empty(16, dtype=torch.float32, device="cuda")
    x = torch.zeros(K, dtype=torch.int16, device="cuda")
    W = torch.zeros(64, dtype=torch.uint8, device="cuda")  # never read: rejected before launch
    st = qgemv.run_noalloc(synth.Q4_K, x, W, N, K, y, check=False)
    assert st == qgemv.ERR_TOO_LARGE
    assert "scratch" in qgemv.status_string(st)
    N2 = qgemv.NOALLOC_MAX_COLUMN_SUMS // 16 + 1  # one row past the limit at 16 K-columns
    assert qgemv.run_noalloc(synth.Q4_K, torch.zeros(32768, dtype=torch.int16, device="cuda"), W, N2, 32768, y,
                             check=False) == qgemv.ERR_TOO_LARGE
    assert qgemv.run_noalloc(synth.Q4_K, x, W, 5, 1000, y, check=False) == qgemv.ERR_BAD_SHAPE
    torch.cuda.synchronize()
