"""GPU parity of the small-batch GEMV (qgemv_run_batch): M = 1..8 activation vectors against
the oracle, one vector at a time, each output within |y - y_ref| <= 2e-3 * sum|x w| + 1e-5
of its own vector.  Every format runs the mma.sync kernel for M >= 2 (one to fourteen
K-columns, ragged row counts, partial last K-columns; TQ1_0 and Q6_K, whose blocks are not
16-byte aligned, through copy windows at every window offset); M = 1 and rows whose byte
length is not a multiple of 16 run the single-vector path per vector."""
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


def _check(Y, X, fmt, W, N, K, rows=None, what=""):
    for m in range(X.shape[0]):
        if rows is None:
            ref, S = oracle.gemv(fmt, X[m], W, N, K)
            got = Y[m]
        else:
            ref, S = oracle.gemv_rows(fmt, X[m], W, N, K, rows)
            got = Y[m][rows]
        err = np.abs(got.astype(np.float64) - ref)
        bad = np.nonzero(~(err <= RTOL * S + ATOL))[0]
        assert bad.size == 0, f"{what} vector {m}: {bad.size} outside, first {bad[:5]} err {err[bad[:5]]}"


def _run(h, fmt, X, W_dev, N, K, force=1):
    """force=1: the batch kernel for every M >= 2 (the automatic choice sends two or three
    vectors of fewer than 4096 rows to the single-vector path)."""
    M = X.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qgemv.set_option(h, qgemv.OPT_FORCE_PATH, force)
    try:
        qgemv.run_batch(h, fmt, _dev_x(X), M, W_dev, N, K, y)
        torch.cuda.synchronize()
    finally:
        qgemv.set_option(h, qgemv.OPT_FORCE_PATH, 0)
    return y.cpu().numpy()


SHAPES = [(synth.Q4_K, 77, 2048), (synth.Q4_K, 300, 4096), (synth.Q4_K, 129, 14336), (synth.Q4_K, 8, 2304),
          (synth.Q4_K, 1, 256), (synth.NVFP4, 65, 2048), (synth.NVFP4, 40, 14336), (synth.NVFP4, 333, 4352),
          (synth.NVFP4, 3, 256), (synth.Q5_K, 77, 4096), (synth.Q5_K, 33, 12288), (synth.Q5_K, 5, 768),
          (synth.Q8_0, 65, 4096), (synth.Q8_0, 40, 12288), (synth.Q8_0, 17, 1280),
          (synth.TQ1_0, 77, 4096), (synth.TQ1_0, 300, 2048), (synth.TQ1_0, 33, 14336), (synth.TQ1_0, 9, 6144),
          (synth.Q6_K, 65, 4096), (synth.Q6_K, 40, 12288), (synth.Q6_K, 129, 2048), (synth.Q6_K, 7, 6144)]


@pytest.mark.parametrize("fmt,N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
def test_batch_matches_oracle(h, fmt, N, K, M):
    W = synth.make_weights(fmt, N, K, seed=N + K + fmt)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=M + N)
    Y = _run(h, fmt, X, Wd, N, K)
    _check(Y, X, fmt, W, N, K, what=f"{synth.FORMAT_NAMES[fmt]} {N}x{K} M={M}")
    assert qgemv.check_error(h) == qgemv.OK


@pytest.mark.parametrize("fmt,N,K", [(synth.Q6_K, 40, 2816), (synth.TQ1_0, 33, 2304), (synth.Q8_0, 50, 4000),
                                     (synth.Q6_K, 17, 1024), (synth.TQ1_0, 20, 4352), (synth.NVFP4, 9, 4016)])
def test_batch_on_the_single_vector_path(h, fmt, N, K):
    W = synth.make_weights(fmt, N, K, seed=5 + fmt)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, 3, K, seed=9)
    Y = _run(h, fmt, X, Wd, N, K)
    _check(Y, X, fmt, W, N, K, what=f"{synth.FORMAT_NAMES[fmt]} {N}x{K}")


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.NVFP4, synth.TQ1_0, synth.Q6_K])
def test_batch_vectors_are_independent_and_deterministic(h, fmt):
    """Vector m of a batch equals the single-vector batch of the same x (the other vectors do
    not leak into it), within the GEMV bound, and repeated calls are bit-identical."""
    N, K = 200, 6144
    W = synth.make_weights(fmt, N, K, seed=3)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, 8, K, seed=4)
    X[3] = 0  # an all-zero vector gives exact zeros
    Y1 = _run(h, fmt, X, Wd, N, K)
    Y2 = _run(h, fmt, X, Wd, N, K)
    assert np.array_equal(Y1, Y2)
    assert np.all(Y1[3] == 0)
    for m in (0, 5):
        Ys = _run(h, fmt, X[m:m + 1], Wd, N, K)
        _, S = oracle.gemv(fmt, X[m], W, N, K)
        assert np.all(np.abs(Ys[0].astype(np.float64) - Y1[m]) <= 2 * (RTOL * S + ATOL))


@pytest.mark.parametrize("fmt,N,M", [(synth.Q6_K, 1024, 2), (synth.Q5_K, 1024, 3), (synth.Q4_K, 4096, 2),
                                     (synth.Q6_K, 1024, 4)])
def test_batch_automatic_path_choice(h, fmt, N, M):
    """The automatic choice (both ways of it) meets the same bound."""
    K = 4096
    W = synth.make_weights(fmt, N, K, seed=6 + fmt)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=12)
    Y = _run(h, fmt, X, Wd, N, K, force=0)
    _check(Y, X, fmt, W, N, K, what=f"auto {synth.FORMAT_NAMES[fmt]} {N}x{K} M={M}")


def test_batch_q6k_full_range_scales(h):
    """Q6_K scales over the whole int8 range: (q6 - 32) sc then exceeds 2048 in magnitude and
    is rounded once to fp16 in the batch kernel (relative error <= 2^-11 per weight), still
    within the GEMV bound against the oracle's exact weights."""
    fmt, N, K = synth.Q6_K, 96, 4096
    W = synth.make_weights(fmt, N, K, seed=13).copy()
    blocks = W.reshape(-1, 210)
    rng = np.random.default_rng(13)
    blocks[:, 192:208] = rng.integers(-128, 128, size=(blocks.shape[0], 16)).astype(np.int8).view(np.uint8)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, 8, K, seed=13)
    Y = _run(h, fmt, X, Wd, N, K)
    _check(Y, X, fmt, W, N, K, what="Q6_K full-range scales")


def test_batch_nvfp4_wide_range_vectors(h):
    """Vectors whose magnitudes differ by 2^40 get their own fp16 exponent window."""
    fmt, N, K = synth.NVFP4, 64, 4096
    W = synth.make_weights(fmt, N, K, seed=8)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, 4, K, seed=8)
    for m, e in enumerate([-30, 0, 10, 30]):
        v = torch.from_numpy(X[m].view(np.int16).copy()).view(torch.bfloat16).float() * (2.0 ** e)
        X[m] = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    Y = _run(h, fmt, X, Wd, N, K)
    _check(Y, X, fmt, W, N, K, what="nvfp4 wide range")


def test_batch_rejects_bad_arguments(h):
    K = 4096
    x = torch.zeros((9, K), dtype=torch.int16, device="cuda")
    W = torch.zeros(synth.packed_bytes(synth.Q4_K, 4, K), dtype=torch.uint8, device="cuda")
    y = torch.zeros((9, 16), dtype=torch.float32, device="cuda")
    assert qgemv.run_batch(h, synth.Q4_K, x, 0, W, 4, K, y, check=False) == qgemv.ERR_INVALID_ARG
    assert qgemv.run_batch(h, synth.Q4_K, x, 9, W, 4, K, y, check=False) == qgemv.ERR_INVALID_ARG
    assert qgemv.run_batch(h, synth.Q4_K, x.data_ptr() + 2, 2, W, 4, K, y, check=False) == qgemv.ERR_MISALIGNED
    assert qgemv.run_batch(h, synth.Q4_K, x, 2, W, 4, 1000, y, check=False) == qgemv.ERR_BAD_SHAPE
    torch.cuda.synchronize()
    assert qgemv.check_error(h) == qgemv.OK


@pytest.mark.parametrize("fmt,N,K,M", [(synth.Q4_K, 4096, 14336, 8), (synth.Q4_K, 28672, 4096, 4),
                                       (synth.NVFP4, 4096, 14336, 8), (synth.NVFP4, 14336, 4096, 2),
                                       (synth.TQ1_0, 11008, 4096, 8), (synth.Q6_K, 4096, 12288, 8)])
def test_batch_full_size_sampled_rows(h, fmt, N, K, M):
    W = synth.make_weights(fmt, N, K, seed=21 + fmt)
    Wd, _ = dev_bytes(W)
    X = _xs(fmt, M, K, seed=22)
    qgemv.set_option(h, qgemv.OPT_PDL, 1)
    try:
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        xd = _dev_x(X)
        for _ in range(2):
            qgemv.run_batch(h, fmt, xd, M, Wd, N, K, y)
        torch.cuda.synchronize()
    finally:
        qgemv.set_option(h, qgemv.OPT_PDL, 0)
    _check(y.cpu().numpy(), X, fmt, W, N, K, rows=sample_rows(N, 48, seed=N), what="full size")
    assert qgemv.check_error(h) == qgemv.OK


def _q80_small_scales(N, K, seed, lo, hi, codes=None):
    """Q8_0 weights whose block scales d are drawn log-uniformly from [lo, hi] (fp16, many of
    them fp16 subnormals below 6.1e-5) and, with `codes`, whose int8 codes all lie in that set:
    small codes against all-positive activations make rounding errors of the operand add up
    instead of cancelling."""
    W = synth.make_weights(synth.Q8_0, N, K, seed).reshape(N, K // 32, 34).copy()
    rng = np.random.default_rng(seed)
    d = np.exp(rng.uniform(np.log(lo), np.log(hi), size=W.shape[:2])).astype(np.float16)
    W[:, :, 0:2] = d.view(np.uint8).reshape(N, K // 32, 2)
    if codes is not None:
        W[:, :, 2:] = rng.choice(np.array(codes, dtype=np.int8), size=(N, K // 32, 32)).view(np.uint8)
    return W.reshape(-1)


@pytest.mark.parametrize("lo,hi,codes", [(1e-7, 3e-6, [1, 2, 3]), (2e-8, 1e-5, None), (1e-6, 1e-3, [1, -1, 2]),
                                         (6e-8, 6e-8, [1])])
def test_q80_batch_tiny_block_scales(h, lo, hi, codes):
    """Block scales in and around the fp16 subnormals: the operand d q is scaled per row and
    superblock into fp16's normal range, so its rounding stays relative (at most 2^-11 of each
    weight) and every output stays inside the GEMV bound, where a subnormal operand's absolute
    rounding would not."""
    N, K = 96, 4096
    W = _q80_small_scales(N, K, seed=71, lo=lo, hi=hi, codes=codes)
    Wd, _ = dev_bytes(W)
    for M in (2, 5):
        X = np.abs(_xs(synth.Q8_0, M, K, seed=73).view(np.float16)).astype(np.float16).view(np.uint16)
        Y = _run(h, synth.Q8_0, X, Wd, N, K)
        _check(Y, X, synth.Q8_0, W, N, K, what=f"Q8_0 d in [{lo}, {hi}] M={M}")
