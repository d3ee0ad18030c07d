"""GPU parity of qgemv_run_gemm, the product for any number M of activation rows.  NVFP4 with
M > 8 runs the tcgen05 tensor-core kernel (tiles of 128 weight rows x 256 or 128 rows of X, X
by TMA, the weights dequantised to bf16 into tensor memory as the A operand, fp32 accumulation
in TMEM); the other
formats and shapes go through the batch path in chunks of 8.  Every checked output row meets
|y - y_ref| <= 2e-3 * sum|x w| + 1e-5 against the oracle's GEMV of its own activation row;
large cases check sampled rows of X (always the first, middle and last)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import ATOL, RTOL, dev_bytes, sample_rows
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


def _xs(fmt, M, K, seed):
    return np.stack([synth.make_x(fmt, K, seed + 17 * m) for m in range(M)])


def _dev_x(X):
    return torch.from_numpy(np.ascontiguousarray(X).view(np.int16)).cuda()


def _run(h, fmt, X, Wd, N, K):
    M = X.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qgemv.run_gemm(h, fmt, _dev_x(X), M, Wd, N, K, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _check(Y, X, fmt, W, N, K, ms, what):
    for m in ms:
        ref, S = oracle.gemv(fmt, X[m], W, N, K)
        err = np.abs(Y[m].astype(np.float64) - ref)
        bad = np.nonzero(~(err <= RTOL * S + ATOL))[0]
        assert bad.size == 0, f"{what} row {m}: {bad.size} outside, first {bad[:5]} err {err[bad[:5]]}"


# (N, K, M): one K-block; ragged N and M; 129 rows (a 256-row tile, mostly outside X); long K
# at M = 64 (64-row tiles, 128-wide stages, 8 K splits); K-blocks not a multiple of the ring
# depth (128- and 64-wide stages); a full prefill shape (2 splits); tiles enough for every SM
# (no split); one 64-wide K-block on 256-row tiles; 4096 rows of X with one K-block; 65 rows
# (the first 128-row tile); 20000 rows of X; 30000 weight rows
TC_CASES = [(128, 128, 9), (200, 4096, 300), (1000, 2048, 129), (256, 14336, 64), (333, 1152, 77),
            (200, 960, 150), (4096, 4096, 512), (130, 1024, 1000), (4096, 1024, 1100),
            (384, 64, 300), (128, 128, 4096), (520, 2048, 65), (256, 1024, 20000), (30000, 256, 300)]


@pytest.mark.parametrize("N,K,M", TC_CASES)
def test_tensor_core_gemm_matches_oracle(h, N, K, M):
    fmt = synth.NVFP4
    W = synth.make_weights(fmt, N, K, seed=N + K)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=M)
    Y = _run(h, fmt, X, Wd, N, K)
    assert not np.isnan(Y).any(), "unwritten outputs"
    ms = range(M) if M * N * K <= 2e9 and M <= 4096 else sample_rows(M, 24, seed=M)
    _check(Y, X, fmt, W, N, K, ms, f"NVFP4 {N}x{K} M={M}")
    assert qgemv.check_error(h) == qgemv.OK


@pytest.mark.parametrize("fmt,N,K,M", [(synth.NVFP4, 50, 4016, 20), (synth.NVFP4, 60, 960, 40),
                                       (synth.Q4_K, 300, 4096, 20),
                                       (synth.TQ1_0, 64, 4096, 11), (synth.Q8_0, 40, 1280, 9),
                                       (synth.NVFP4, 96, 2048, 8), (synth.NVFP4, 64, 512, 1)])
def test_gemm_batch_path(h, fmt, N, K, M):
    W = synth.make_weights(fmt, N, K, seed=4 + fmt)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=3)
    Y = _run(h, fmt, X, Wd, N, K)
    _check(Y, X, fmt, W, N, K, range(M), f"{synth.FORMAT_NAMES[fmt]} {N}x{K} M={M}")


def test_tensor_core_gemm_is_deterministic_and_rows_are_independent(h):
    """Repeated calls give identical bits; an all-zero row of X gives exact zeros; a row's
    result does not depend on the other rows of its tile (within the GEMV bound)."""
    fmt, N, K, M = synth.NVFP4, 384, 2048, 200
    W = synth.make_weights(fmt, N, K, seed=5)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=6)
    X[7] = 0
    Y1 = _run(h, fmt, X, Wd, N, K)
    Y2 = _run(h, fmt, X, Wd, N, K)
    assert np.array_equal(Y1, Y2)
    assert np.all(Y1[7] == 0)
    X2 = X.copy()
    X2[8:] = _xs(fmt, M - 8, K, seed=99)  # same first rows, different rest
    Y3 = _run(h, fmt, X2, Wd, N, K)
    for m in (0, 5):
        _, S = oracle.gemv(fmt, X[m], W, N, K)
        assert np.all(np.abs(Y3[m].astype(np.float64) - Y1[m]) <= 2 * (RTOL * S + ATOL))


def test_tensor_core_gemm_wide_range_rows(h):
    """Rows of X scaled by 2^-60 .. 2^60 (bf16 keeps them exactly): the bf16 operand path has
    no per-row exponent window to lose."""
    fmt, N, K, M = synth.NVFP4, 256, 1024, 16
    W = synth.make_weights(fmt, N, K, seed=8)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=8)
    for m in range(M):
        e = -60 + 8 * m
        v = torch.from_numpy(X[m].view(np.int16).copy()).view(torch.bfloat16).float() * (2.0 ** e)
        X[m] = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    Y = _run(h, fmt, X, Wd, N, K)
    _check(Y, X, fmt, W, N, K, range(M), "wide range")


def test_gemm_rejects_bad_arguments(h):
    K, N = 1024, 128
    x = torch.zeros((32, K), dtype=torch.int16, device="cuda")
    W = torch.zeros(synth.packed_bytes(synth.NVFP4, N, K), dtype=torch.uint8, device="cuda")
    y = torch.zeros((32, N), dtype=torch.float32, device="cuda")
    assert qgemv.run_gemm(h, synth.NVFP4, x, 0, W, N, K, y, check=False) == qgemv.ERR_INVALID_ARG
    assert qgemv.run_gemm(h, synth.NVFP4, x.data_ptr() + 2, 16, W, N, K, y, check=False) == qgemv.ERR_MISALIGNED
    assert qgemv.run_gemm(h, synth.NVFP4, x, 16, W, N, 1000, y, check=False) == qgemv.ERR_BAD_SHAPE
    torch.cuda.synchronize()
    assert qgemv.check_error(h) == qgemv.OK


def test_tensor_core_gemm_wait_times_out_and_the_context_stays_usable(h):
    """The test hook withholds one stage's arrivals in the first CTA: its bounded waits run out,
    the error word reports QGEMV_ERR_TIMEOUT, and the next call is correct."""
    fmt, N, K, M = synth.NVFP4, 256, 1024, 32
    W = synth.make_weights(fmt, N, K, seed=9)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=9)
    qgemv.set_option(h, qgemv.OPT_SPIN_LIMIT_NS, 2_000_000)
    qgemv.set_option(h, qgemv.OPT_TEST_STALL, 1)
    try:
        _run(h, fmt, X, Wd, N, K)
        assert qgemv.check_error(h) == qgemv.ERR_TIMEOUT
    finally:
        qgemv.set_option(h, qgemv.OPT_TEST_STALL, 0)
        qgemv.set_option(h, qgemv.OPT_SPIN_LIMIT_NS, 1_000_000_000)
    assert qgemv.check_error(h) == qgemv.OK
    Y = _run(h, fmt, X, Wd, N, K)
    _check(Y, X, fmt, W, N, K, range(M), "after timeout")
    assert qgemv.check_error(h) == qgemv.OK
