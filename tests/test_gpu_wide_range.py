"""Wide-range activations against the oracle, with the GEMV bound itself:
|y - y_ref| <= 2e-3 * sum|x w| + 1e-5 per output, for every format and launch path.

The inputs are the hard case for any kernel that scales x per block: one large outlier per
32-element chunk among small values.  With the weights meeting the outliers set to exactly
zero (Q4_K/Q5_K code 0 and group minimum 0, Q6_K code 32, Q8_0 and NVFP4 code 0, TQ1_0
digit 1), an outlier sets its chunk's scale but adds nothing to sum |x w|, so any rounding
of the small values relative to the outlier shows up against the bound.  Also covered: the
outliers with their own weights, the whole fp16 range (65504 beside subnormals) and a bf16
range of 2^200 for NVFP4."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_parity, dev_bytes, dev_x, run_gemv
from quantized_weight_dequant_gb300 import qgemv, synth
from wide_range import outlier_x, zero_weight_columns

pytestmark = pytest.mark.gpu

ALL = [synth.Q4_K, synth.NVFP4, synth.TQ1_0, synth.Q5_K, synth.Q6_K, synth.Q8_0]


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_weight_dequant_gb300.build import build_library
    build_library()
    handle = qgemv.create(0)
    yield handle
    handle.close()


def _check(h, fmt, x, W, N, K, what, pdl=0, path=0):
    Wd, _ = dev_bytes(W)
    qgemv.set_option(h, qgemv.OPT_PDL, pdl)
    qgemv.set_option(h, qgemv.OPT_FORCE_PATH, path)
    try:
        y = run_gemv(h, fmt, dev_x(x), Wd, N, K).cpu().numpy()
    finally:
        qgemv.set_option(h, qgemv.OPT_PDL, 0)
        qgemv.set_option(h, qgemv.OPT_FORCE_PATH, 0)
    assert qgemv.check_error(h) == qgemv.OK
    y_ref, S = oracle.gemv(fmt, x, W, N, K)
    assert_parity(y, y_ref, S, f"{synth.FORMAT_NAMES[fmt]} {N}x{K} {what}")
    return y, y_ref, S


SHAPES = [(64, 4096), (40, 14336), (33, 2048)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("fmt", ALL)
def test_outliers_meeting_zero_weights(h, fmt, N, K):
    x, cols = outlier_x(fmt, K, seed=7 + fmt + K)
    W = zero_weight_columns(fmt, synth.make_weights(fmt, N, K, seed=17 + fmt), N, K, cols)
    wd = oracle.dequant_rows(fmt, W, N, K, np.arange(N))
    assert np.all(wd[:, cols] == 0.0)
    for pdl in (0, 1):
        _check(h, fmt, x, W, N, K, f"outliers on zero weights pdl={pdl}", pdl=pdl)


@pytest.mark.parametrize("fmt", ALL)
def test_outliers_meeting_zero_weights_plain_row_path(h, fmt):
    N, K = 37, 4096
    x, cols = outlier_x(fmt, K, seed=3 + fmt)
    W = zero_weight_columns(fmt, synth.make_weights(fmt, N, K, seed=5 + fmt), N, K, cols)
    _check(h, fmt, x, W, N, K, "rowwarp", path=2)


@pytest.mark.parametrize("fmt", ALL)
def test_outliers_with_their_weights(h, fmt):
    N, K = 50, 8192
    x, _ = outlier_x(fmt, K, seed=11 + fmt)
    _check(h, fmt, x, synth.make_weights(fmt, N, K, seed=13 + fmt), N, K, "outliers")


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.TQ1_0, synth.Q5_K, synth.Q6_K, synth.Q8_0])
def test_the_whole_fp16_range(h, fmt):
    """65504 beside fp16 subnormals (down to 2^-24) and everything in between, in every chunk;
    half of the large values meet zero weights."""
    N, K = 40, 4096
    rng = np.random.default_rng(23 + fmt)
    mag = 2.0 ** rng.uniform(-24, 16, size=K)
    xf = np.sign(rng.standard_normal(K)) * np.minimum(mag, 65504.0)
    cols = np.arange(0, K, 64)
    xf[cols] = 65504.0 * np.sign(rng.standard_normal(cols.size))
    xf[cols + 1] = 2.0 ** -24
    x = xf.astype(np.float16).view(np.uint16).copy()
    W = zero_weight_columns(fmt, synth.make_weights(fmt, N, K, seed=29 + fmt), N, K, cols[::2])
    _check(h, fmt, x, W, N, K, "fp16 range")


def test_nvfp4_bf16_range_beyond_fp16(h):
    """bf16 activations spanning 2^-100 .. 2^100 within chunks: values more than ~2^30 below
    their chunk's largest one do not fit the scaled f16 staging and take the residual path."""
    N, K = 48, 4096
    rng = np.random.default_rng(31)
    xf = np.sign(rng.standard_normal(K)) * 2.0 ** rng.uniform(-100, 100, size=K)
    cols = np.arange(0, K, 32)
    xf[cols] = 2.0 ** 100
    x = torch.tensor(xf, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    W = zero_weight_columns(synth.NVFP4, synth.make_weights(synth.NVFP4, N, K, seed=37), N, K, cols)
    for pdl in (0, 1):
        _check(h, synth.NVFP4, x, W, N, K, f"bf16 range pdl={pdl}", pdl=pdl)


@pytest.mark.parametrize("fmt", ALL)
def test_outliers_grouped_and_epilogue_launch(h, fmt):
    """The grouped kernel (qgemv_run_ex, alpha = 1, beta = 0, fp32 out) on the same inputs."""
    N, K = 64, 4096
    x, cols = outlier_x(fmt, K, seed=41 + fmt)
    W = zero_weight_columns(fmt, synth.make_weights(fmt, N, K, seed=43 + fmt), N, K, cols)
    Wd, _ = dev_bytes(W)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    qgemv.run_ex(h, fmt, dev_x(x), Wd, N, K, y)
    torch.cuda.synchronize()
    y_ref, S = oracle.gemv(fmt, x, W, N, K)
    assert_parity(y.cpu().numpy(), y_ref, S, "run_ex outliers")


@pytest.mark.parametrize("fmt", ALL)
def test_outliers_noalloc(h, fmt):
    N, K = 50, 6144
    x, cols = outlier_x(fmt, K, seed=47 + fmt)
    W = zero_weight_columns(fmt, synth.make_weights(fmt, N, K, seed=53 + fmt), N, K, cols)
    Wd, _ = dev_bytes(W)
    y = torch.empty(N, dtype=torch.float32, device="cuda")
    qgemv.run_noalloc(fmt, dev_x(x), Wd, N, K, y)
    torch.cuda.synchronize()
    y_ref, S = oracle.gemv(fmt, x, W, N, K)
    assert_parity(y.cpu().numpy(), y_ref, S, "noalloc outliers")


@pytest.mark.parametrize("fmt", ALL)
def test_outliers_small_batch(h, fmt):
    """Two and five activation vectors (qgemv_run_batch, the tensor-core batch kernel)."""
    N, K = 4096, 4096
    W = synth.make_weights(fmt, N, K, seed=59 + fmt)
    for M in (2, 5):
        xs, cols = zip(*[outlier_x(fmt, K, seed=61 + fmt + 7 * m) for m in range(M)])
        W2 = zero_weight_columns(fmt, W, N, K, cols[0]) if M == 2 else W
        Wd, _ = dev_bytes(W2)
        X = torch.from_numpy(np.stack(xs).view(np.int16)).cuda()
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        qgemv.run_batch(h, fmt, X, M, Wd, N, K, Y)
        torch.cuda.synchronize()
        rows = np.arange(0, N, 97)
        for m in range(M):
            y_ref, S = oracle.gemv_rows(fmt, xs[m], W2, N, K, rows)
            assert_parity(Y[m].cpu().numpy()[rows], y_ref, S, f"batch M={M} vector {m}")
