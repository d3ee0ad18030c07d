"""GPU parity: the CUDA path (through the C-ABI) against the CPU oracle on the same seeded
inputs.  Unpacked codes/scales/mins are compared bit for bit; GEMV outputs within
|y - y_ref| <= 2e-3 * sum|x w| + 1e-5 per output."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_parity, dev_bytes, dev_x, run_gemv, sample_rows
from quantized_weight_dequant_gb300 import qgemv, synth

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


def _check_full(h, fmt, N, K, seed, what=""):
    W = synth.make_weights(fmt, N, K, seed)
    x = synth.make_x(fmt, K, seed)
    Wd, _ = dev_bytes(W)
    y = run_gemv(h, fmt, dev_x(x), Wd, N, K).cpu().numpy()
    assert qgemv.check_error(h) == qgemv.OK
    y_ref, S = oracle.gemv(fmt, x, W, N, K)
    assert_parity(y, y_ref, S, f"{synth.FORMAT_NAMES[fmt]} {N}x{K} {what}")
    return y


# Small and mid shapes: several tiles, ragged tails, both paths.
SHAPES = {
    synth.Q4_K: [(1, 256), (3, 512), (37, 4096), (300, 2304), (64, 14336), (1024, 1024), (131, 6400), (5, 36864),
                 (2, 32768)],
    synth.Q5_K: [(1, 256), (33, 4096), (70, 2560), (16, 12288)],
    synth.Q6_K: [(1, 256), (9, 768), (40, 4096), (17, 12288), (5, 2048)],
    synth.Q8_0: [(1, 32), (3, 160), (50, 4096), (8, 12288), (2, 288)],
    synth.TQ1_0: [(1, 256), (9, 768), (50, 2048), (40, 4096), (3, 6144)],
    synth.NVFP4: [(1, 16), (3, 48), (7, 272), (33, 4096), (9, 14336), (20, 1024), (2, 4352)],
}


@pytest.mark.parametrize("fmt,N,K", [(f, n, k) for f, shapes in SHAPES.items() for n, k in shapes])
def test_gemv_matches_oracle_small_and_ragged(h, fmt, N, K):
    _check_full(h, fmt, N, K, seed=N * 7 + K + fmt)


@pytest.mark.parametrize("fmt", ALL)
def test_unpack_is_bit_exact(h, fmt):
    for N, K in [(5, 512), (3, 4096)] + ([(2, 48)] if fmt == synth.NVFP4 else []) + \
            ([(2, 96)] if fmt == synth.Q8_0 else []):
        W = synth.make_weights(fmt, N, K, seed=100 + fmt)
        Wd, _ = dev_bytes(W)
        G = qgemv.group_size(fmt)
        codes = torch.empty((N, K), dtype=torch.int8, device="cuda")
        scales = torch.empty((N, K // G), dtype=torch.float32, device="cuda")
        mins = torch.empty((N, K // G), dtype=torch.float32, device="cuda")
        qgemv.unpack(h, fmt, Wd, N, K, codes, scales, mins)
        c_ref, s_ref, m_ref = oracle.unpack(fmt, W, N, K)
        assert np.array_equal(codes.cpu().numpy(), c_ref)
        assert np.array_equal(scales.cpu().numpy().astype(np.float64), s_ref)
        assert np.array_equal(mins.cpu().numpy().astype(np.float64), m_ref)


@pytest.mark.parametrize("fmt,N,K", [(synth.Q4_K, 37, 4096), (synth.NVFP4, 33, 4096), (synth.TQ1_0, 40, 4096),
                                     (synth.Q5_K, 33, 4096), (synth.Q6_K, 40, 4096), (synth.Q8_0, 50, 4096)])
def test_plain_row_path_matches_oracle(h, fmt, N, K):
    qgemv.set_option(h, qgemv.OPT_FORCE_PATH, 2)
    try:
        assert "rowwarp" in qgemv.describe(h, fmt, N, K)
        _check_full(h, fmt, N, K, seed=5 + fmt, what="rowwarp")
    finally:
        qgemv.set_option(h, qgemv.OPT_FORCE_PATH, 0)


@pytest.mark.parametrize("ksplit", [0, 1])
@pytest.mark.parametrize("cps,pdl", [(2, 0), (1, 0), (1, 1), (2, 1)])
@pytest.mark.parametrize("fmt", ALL)
def test_launch_variants_match_oracle(h, fmt, cps, pdl, ksplit):
    """CTAs per SM, programmatic dependent launch, and split-K (one K-column per CTA, column
    sums added by the last CTA of each row range) against K-columns added in the CTA."""
    qgemv.set_option(h, qgemv.OPT_CTAS_PER_SM, cps)
    qgemv.set_option(h, qgemv.OPT_PDL, pdl)
    qgemv.set_option(h, qgemv.OPT_KSPLIT, ksplit)
    try:
        for N, K in [(70, 14336), (333, 4096), (5, 12288), (1, 32768), (600, 2304)]:
            d = qgemv.describe(h, fmt, N, K)
            assert "rowwarp" in d or f"split={int((ksplit == 0 and K > 4096) or K <= 2048)}" in d, d
            _check_full(h, fmt, N, K, seed=11 * cps + pdl + fmt + N, what=f"cps={cps} pdl={pdl} ksplit={ksplit}")
    finally:
        qgemv.set_option(h, qgemv.OPT_CTAS_PER_SM, 2)
        qgemv.set_option(h, qgemv.OPT_PDL, 0)
        qgemv.set_option(h, qgemv.OPT_KSPLIT, 0)


@pytest.mark.parametrize("depth,rows", [(2, 1), (3, 3), (8, 2), (4, 8)])
def test_ring_shapes_match_oracle(h, depth, rows):
    qgemv.set_option(h, qgemv.OPT_RING_DEPTH, depth)
    qgemv.set_option(h, qgemv.OPT_ROWS_PER_STAGE, rows)
    try:
        _check_full(h, synth.Q4_K, 261, 4096, seed=depth * 10 + rows, what=f"D={depth} R={rows}")
        _check_full(h, synth.NVFP4, 97, 14336, seed=depth * 10 + rows, what=f"D={depth} R={rows}")
    finally:
        qgemv.set_option(h, qgemv.OPT_RING_DEPTH, 0)
        qgemv.set_option(h, qgemv.OPT_ROWS_PER_STAGE, 0)


def _shape_cases():
    out = []
    for sname in ("q4k_llama8b_decode", "nvfp4_llama8b", "tq1_0", "layer", "layer_every_format"):
        for si, (name, fmt, N, K) in enumerate(synth.SHAPE_SETS[sname]):
            out.append(pytest.param(sname, si, fmt, N, K, id=f"{sname}:{name}"))
    return out


@pytest.mark.parametrize("sname,si,fmt,N,K", _shape_cases())
def test_full_size_workload_shapes_on_sampled_rows(h, sname, si, fmt, N, K):
    """Full sizes in the launch configuration the bench times (programmatic dependent
    launch on) and in the plain one, on sampled rows."""
    seed = synth.shape_seed(sname, si)
    W = synth.make_weights(fmt, N, K, seed)
    x = synth.make_x(fmt, K, seed)
    Wd, _ = dev_bytes(W)
    xd = dev_x(x)
    rows = sample_rows(N, 384, seed)
    y_ref, S = oracle.gemv_rows(fmt, x, W, N, K, rows)
    for pdl in (1, 0):
        qgemv.set_option(h, qgemv.OPT_PDL, pdl)
        try:
            y = run_gemv(h, fmt, xd, Wd, N, K).cpu().numpy()
        finally:
            qgemv.set_option(h, qgemv.OPT_PDL, 0)
        assert qgemv.check_error(h) == qgemv.OK
        assert_parity(y[rows], y_ref, S, f"{sname} {N}x{K} pdl={pdl}")
        assert np.all(np.isfinite(y))


@pytest.mark.parametrize("fmt,N,K,mode", [(synth.Q4_K, 1_500_007, 6144, "fused"), (synth.Q4_K, 1_300_001, 6144, "split"),
                                          (synth.NVFP4, 1_100_003, 4096, "fused"), (synth.Q8_0, 700_001, 14336, "fused")])
def test_huge_row_counts_on_sampled_rows(h, fmt, N, K, mode):
    """Millions of rows (5 to 11 GB of weights): the workspace limit (N * K-columns <= 4 Mi)
    sends the long-K case with the most rows to CTAs that add their K-columns themselves, the
    reduction-buffer budget raises the grid, and row indices pass 2^19 per launch.  The matrix
    is a seeded block of rows tiled on the device, so row r equals base row r % n0."""
    n0 = 4096
    W0 = synth.make_weights(fmt, n0, K, seed=77 + fmt)
    x = synth.make_x(fmt, K, seed=78)
    if fmt == synth.NVFP4:  # nibble rows then scale rows: tile each part
        nib = torch.from_numpy(W0[: n0 * (K // 2)]).cuda().view(n0, K // 2)
        sc = torch.from_numpy(W0[n0 * (K // 2):]).cuda().view(n0, K // 16)
        reps = (N + n0 - 1) // n0
        Wd = torch.cat([nib.repeat(reps, 1)[:N].reshape(-1), sc.repeat(reps, 1)[:N].reshape(-1)])
        del nib, sc
    else:
        rb = synth.packed_bytes(fmt, 1, K)
        base = torch.from_numpy(W0).cuda().view(n0, rb)
        Wd = base.repeat((N + n0 - 1) // n0, 1)[:N].reshape(-1).contiguous()
        del base
    assert Wd.numel() == synth.packed_bytes(fmt, N, K)
    d = qgemv.describe(h, fmt, N, K)
    assert f"split={int(mode == 'split')}" in d, d
    y = run_gemv(h, fmt, dev_x(x), Wd, N, K)
    assert qgemv.check_error(h) == qgemv.OK
    rows = np.unique(np.concatenate([sample_rows(N, 200, seed=N), [N - 1, N - 2, min(N - 3, (1 << 20) + 5)]]))
    y_ref, S = oracle.gemv_rows(fmt, x, W0, n0, K, rows % n0)
    assert_parity(y.cpu().numpy()[rows], y_ref, S, f"{synth.FORMAT_NAMES[fmt]} {N}x{K} {mode}")
    del Wd, y
    torch.cuda.empty_cache()


def test_q4k_1024x1024_full(h):
    name, fmt, N, K = synth.SHAPE_SETS["q4k_1024x1024"][0]
    _check_full(h, fmt, N, K, seed=synth.shape_seed("q4k_1024x1024", 0), what=name)


@pytest.mark.parametrize("fmt", ALL)
def test_deterministic_bitwise(h, fmt):
    N, K = 513, 4096 if fmt != synth.Q8_0 else 4096
    W = synth.make_weights(fmt, N, K, seed=3)
    x = synth.make_x(fmt, K, seed=3)
    Wd, _ = dev_bytes(W)
    xd = dev_x(x)
    first = run_gemv(h, fmt, xd, Wd, N, K).clone()
    for _ in range(9):
        assert torch.equal(run_gemv(h, fmt, xd, Wd, N, K), first)


@pytest.mark.parametrize("fmt", ALL)
def test_output_guards_and_poisoned_neighbours(h, fmt):
    N, K = 77, 4096
    W = synth.make_weights(fmt, N, K, seed=9)
    x = synth.make_x(fmt, K, seed=9)
    Wd, _ = dev_bytes(W, pad_front=4096, pad_back=4096, fill=0xFF)
    canary = -1234.5
    ybuf = torch.full((N + 64,), canary, dtype=torch.float32, device="cuda")
    y = ybuf[32:32 + N]
    run_gemv(h, fmt, dev_x(x), Wd, N, K, y=y)
    torch.cuda.synchronize()
    yb = ybuf.cpu().numpy()
    assert np.all(yb[:32] == canary) and np.all(yb[32 + N:] == canary)
    y_ref, S = oracle.gemv(fmt, x, W, N, K)
    assert_parity(yb[32:32 + N], y_ref, S, "guarded")


def test_invalid_arguments_return_status_and_launch_nothing(h):
    N, K = 8, 512
    W = torch.zeros(synth.packed_bytes(synth.Q4_K, N, K) + 64, dtype=torch.uint8, device="cuda")
    x = torch.zeros(K + 16, dtype=torch.int16, device="cuda")
    y = torch.full((N + 8,), 7.0, dtype=torch.float32, device="cuda")
    r = lambda *a: qgemv.run(h, *a, check=False)
    assert r(9, x, W, N, K, y) == qgemv.ERR_UNSUPPORTED_FORMAT
    assert r(synth.Q4_K, x, W, 0, K, y) == qgemv.ERR_BAD_SHAPE
    assert r(synth.Q4_K, x, W, N, 300, y) == qgemv.ERR_BAD_SHAPE
    assert r(synth.Q8_0, x, W, N, 48, y) == qgemv.ERR_BAD_SHAPE
    assert r(synth.NVFP4, x, W, N, 40, y) == qgemv.ERR_BAD_SHAPE
    assert r(synth.Q4_K, x, None, N, K, y) == qgemv.ERR_INVALID_ARG
    assert r(synth.Q4_K, None, W, N, K, y) == qgemv.ERR_INVALID_ARG
    assert r(synth.Q4_K, x, W, N, K, None) == qgemv.ERR_INVALID_ARG
    assert r(synth.Q4_K, x, W[1:], N, K, y) == qgemv.ERR_MISALIGNED
    assert r(synth.Q4_K, x[1:], W, N, K, y) == qgemv.ERR_MISALIGNED
    assert r(synth.Q4_K, x, W, N, K, y[1:]) == qgemv.ERR_MISALIGNED
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    assert qgemv.set_option(h, qgemv.OPT_RING_DEPTH, 1, check=False) == qgemv.ERR_INVALID_ARG
    assert qgemv.set_option(h, 77, 0, check=False) == qgemv.ERR_INVALID_ARG
    assert qgemv.check_error(h) == qgemv.OK


def test_bounded_wait_times_out_and_the_context_stays_usable(h):
    N, K = 512, 4096
    W = synth.make_weights(synth.Q4_K, N, K, seed=21)
    x = synth.make_x(synth.Q4_K, K, seed=21)
    Wd, _ = dev_bytes(W)
    xd = dev_x(x)
    qgemv.set_option(h, qgemv.OPT_SPIN_LIMIT_NS, 2_000_000)
    qgemv.set_option(h, qgemv.OPT_TEST_STALL, 1)
    try:
        run_gemv(h, synth.Q4_K, xd, Wd, N, K)
        assert qgemv.check_error(h) == qgemv.ERR_TIMEOUT
    finally:
        qgemv.set_option(h, qgemv.OPT_TEST_STALL, 0)
        qgemv.set_option(h, qgemv.OPT_SPIN_LIMIT_NS, 1_000_000_000)
    assert qgemv.check_error(h) == qgemv.OK
    y = run_gemv(h, synth.Q4_K, xd, Wd, N, K).cpu().numpy()
    assert qgemv.check_error(h) == qgemv.OK
    y_ref, S = oracle.gemv(synth.Q4_K, x, W, N, K)
    assert_parity(y, y_ref, S, "after timeout")


def test_pdl_launches_match_oracle(h):
    qgemv.set_option(h, qgemv.OPT_PDL, 1)
    try:
        ys = []
        for fmt in (synth.Q4_K, synth.NVFP4):
            ys.append(_check_full(h, fmt, 300, 4096, seed=31 + fmt, what="pdl"))
    finally:
        qgemv.set_option(h, qgemv.OPT_PDL, 0)


def test_runs_on_a_side_stream_and_in_a_cuda_graph(h):
    N, K = 1000, 4096
    fmt = synth.Q4_K
    W = synth.make_weights(fmt, N, K, seed=41)
    x = synth.make_x(fmt, K, seed=41)
    Wd, _ = dev_bytes(W)
    xd = dev_x(x)
    y = torch.zeros(N, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        qgemv.run(h, fmt, xd, Wd, N, K, y, stream=s)
    s.synchronize()
    y_ref, S = oracle.gemv(fmt, x, W, N, K)
    assert_parity(y.cpu().numpy(), y_ref, S, "side stream")
    y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        qgemv.run(h, fmt, xd, Wd, N, K, y, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert_parity(y.cpu().numpy(), y_ref, S, "graph replay")
