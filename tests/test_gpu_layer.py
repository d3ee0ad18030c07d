"""GPU parity of the layer entry points: the general epilogue y = alpha x.W^T + beta y in
fp32/fp16/bf16 (qgemv_run_ex), grouped launches of several matrices sharing x, with mixed
formats (qgemv_run_group), and the SwiGLU gate/up pair, against the CPU oracle.

Tolerances follow from the GEMV bound e = 2e-3 * S + 1e-5 (S = sum|x w| from the oracle):
  general:  |alpha| e + |beta c| 2^-22 + half an ulp of the output type at the result
  SwiGLU:   1.1 e_g (|u| + e_u) + |silu(g)| e_u + 1e-6 |h| (+ output half ulp), from
            |silu'| <= 1.0998 (pinned in the oracle tests) and the fp32 evaluation of silu.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import ATOL, RTOL, dev_bytes, dev_x, sample_rows
from quantized_weight_dequant_gb300 import qgemv, synth

pytestmark = pytest.mark.gpu

TORCH_OUT = {qgemv.OUT_F32: torch.float32, qgemv.OUT_F16: torch.float16, qgemv.OUT_BF16: torch.bfloat16}
# relative half ulp and absolute floor (half the smallest subnormal) of each output type
HALF_ULP = {qgemv.OUT_F32: (2.0 ** -24, 2.0 ** -150), qgemv.OUT_F16: (2.0 ** -11, 2.0 ** -25),
            qgemv.OUT_BF16: (2.0 ** -8, 2.0 ** -134)}


@pytest.fixture(scope="module")
def h():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from quantized_weight_dequant_gb300.build import build_library
    build_library()
    handle = qgemv.create(0)
    yield handle
    handle.close()


def _weights(fmt, N, K, seed):
    W = synth.make_weights(fmt, N, K, seed)
    Wd, _ = dev_bytes(W)
    return W, Wd


def _out_tol(out, ref):
    rel, floor = HALF_ULP[out]
    return rel * np.abs(ref) + floor


def _assert_within(got, ref, tol, what):
    err = np.abs(got - ref)
    bad = np.nonzero(~(err <= tol))[0]
    assert bad.size == 0, f"{what}: {bad.size} outside, first {bad[:5]} err {err[bad[:5]]} tol {tol[bad[:5]]}"


def _c_values(N, out, seed):
    """Initial y (the beta term's C) in the output type, and its exact values."""
    c = torch.from_numpy(np.random.default_rng(seed).normal(size=N).astype(np.float32)).to(TORCH_OUT[out])
    return c.cuda(), c.to(torch.float64).numpy()


def _check_general(fmt, x, W, N, K, alpha, beta, out, y_dev, c_vals, what):
    ref, S = oracle.gemv_general(fmt, x, W, N, K, alpha, beta, c_vals)
    got = y_dev.to(torch.float64).cpu().numpy()
    tol = (RTOL * S + abs(alpha) * ATOL) + abs(beta) * np.abs(c_vals) * 2.0 ** -22 + _out_tol(out, ref)
    _assert_within(got, ref, tol, what)


def _swiglu_tol(o, out):
    eg = RTOL * o["Sg"] + ATOL
    eu = RTOL * o["Su"] + ATOL
    sg = np.array([oracle.silu(v) for v in o["g"]])
    return 1.1 * eg * (np.abs(o["u"]) + eu) + np.abs(sg) * eu + 1e-6 * np.abs(o["h"]) + _out_tol(out, o["h"])


# K = 2048: one K-column per row (sums final in the loop); 4096: fused columns; 14336: split
# columns through the workspace; 4000 / 4016: shapes the streaming kernel does not take.
GENERAL = [(synth.Q4_K, 77, 2048), (synth.Q4_K, 300, 4096), (synth.Q4_K, 129, 14336), (synth.Q8_0, 50, 4000),
           (synth.NVFP4, 65, 4096), (synth.NVFP4, 40, 14336), (synth.NVFP4, 9, 4016), (synth.TQ1_0, 33, 4096),
           (synth.Q6_K, 21, 12288), (synth.Q5_K, 17, 2048)]
EPI = [(1.0, 0.0, qgemv.OUT_F32), (-0.5, 0.0, qgemv.OUT_F16), (2.0, 0.75, qgemv.OUT_F32),
       (1.0, -1.0, qgemv.OUT_BF16), (0.25, 2.0, qgemv.OUT_F16)]


@pytest.mark.parametrize("fmt,N,K", GENERAL)
def test_general_epilogue_matches_oracle(h, fmt, N, K):
    W, Wd = _weights(fmt, N, K, seed=N + K + fmt)
    x = synth.make_x(fmt, K, seed=N + fmt)
    xd = dev_x(x)
    for i, (alpha, beta, out) in enumerate(EPI):
        y, c_vals = _c_values(N, out, seed=i)
        if beta == 0.0:  # y must not be read: poison it
            y.fill_(float("nan"))
        qgemv.run_ex(h, fmt, xd, Wd, N, K, y, alpha, beta, out)
        torch.cuda.synchronize()
        _check_general(fmt, x, W, N, K, alpha, beta, out, y, c_vals,
                       f"{synth.FORMAT_NAMES[fmt]} {N}x{K} alpha={alpha} beta={beta} out={out}")
    assert qgemv.check_error(h) == qgemv.OK


@pytest.mark.parametrize("fmt,N,K", [(synth.Q4_K, 300, 4096), (synth.Q4_K, 129, 14336), (synth.NVFP4, 65, 2048),
                                     (synth.Q6_K, 40, 12288), (synth.TQ1_0, 200, 4096), (synth.TQ1_0, 70, 14336),
                                     (synth.TQ1_0, 9, 256)])
def test_general_epilogue_with_unit_alpha_equals_run_bitwise(h, fmt, N, K):
    """qgemv_run against the grouped kernel with out = 1 * r + 0: the same sums bit for bit."""
    _, Wd = _weights(fmt, N, K, seed=3 + fmt)
    xd = dev_x(synth.make_x(fmt, K, seed=3))
    y0 = torch.empty(N, dtype=torch.float32, device="cuda")
    y1 = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    qgemv.run(h, fmt, xd, Wd, N, K, y0)
    qgemv.run_ex(h, fmt, xd, Wd, N, K, y1, 1.0, 0.0, qgemv.OUT_F32)
    assert torch.equal(y0, y1)


SWIGLU = [(synth.Q4_K, 77, 2048), (synth.Q4_K, 301, 4096), (synth.Q4_K, 65, 14336), (synth.NVFP4, 33, 4096),
          (synth.NVFP4, 19, 14336), (synth.TQ1_0, 40, 4096), (synth.Q8_0, 21, 4000), (synth.Q6_K, 1, 12288)]


@pytest.mark.parametrize("fmt,N,K", SWIGLU)
def test_swiglu_pair_matches_oracle(h, fmt, N, K):
    Wg, Wgd = _weights(fmt, N, K, seed=N + K)
    Wu, Wud = _weights(fmt, N, K, seed=N + K + 1)
    x = synth.make_x(fmt, K, seed=K + fmt)
    o = oracle.swiglu(fmt, x, Wg, Wu, N, K)
    xd = dev_x(x)
    for out in (qgemv.OUT_F32, qgemv.OUT_BF16):
        y = torch.full((N,), float("nan"), dtype=TORCH_OUT[out], device="cuda")
        qgemv.run_group(h, xd, K, [qgemv.problem(fmt, Wgd, N, y, packed_W_up=Wud, out=out, swiglu=True)])
        torch.cuda.synchronize()
        _assert_within(y.to(torch.float64).cpu().numpy(), o["h"], _swiglu_tol(o, out),
                       f"swiglu {synth.FORMAT_NAMES[fmt]} {N}x{K} out={out}")
    assert qgemv.check_error(h) == qgemv.OK


def _run_and_check_group(h, specs, K, x, what, repeat=1):
    """specs: list of dicts fmt, N, seed, [swiglu, alpha, beta, out]; one run_group call."""
    probs, checks, keep = [], [], []  # keep: the device buffers that probs[] points into
    for s in specs:
        fmt, N = s["fmt"], s["N"]
        W, Wd = _weights(fmt, N, K, s["seed"])
        out = s.get("out", qgemv.OUT_F32)
        alpha, beta = s.get("alpha", 1.0), s.get("beta", 0.0)
        keep.append(Wd)
        if s.get("swiglu"):
            Wu, Wud = _weights(fmt, N, K, s["seed"] + 1)
            keep.append(Wud)
            y = torch.full((N,), float("nan"), dtype=TORCH_OUT[out], device="cuda")
            probs.append(qgemv.problem(fmt, Wd, N, y, packed_W_up=Wud, out=out, swiglu=True))
            checks.append(("swiglu", fmt, N, W, Wu, y, out, None, 1.0, 0.0))
        else:
            y, c_vals = _c_values(N, out, seed=s["seed"])
            if beta == 0.0:
                y.fill_(float("nan"))
            probs.append(qgemv.problem(fmt, Wd, N, y, alpha=alpha, beta=beta, out=out))
            checks.append(("gemv", fmt, N, W, None, y, out, c_vals, alpha, beta))
    xd = dev_x(x)
    results = []
    for _ in range(repeat):
        for kind, fmt, N, W, Wu, y, out, c_vals, alpha, beta in checks:
            if kind == "gemv" and beta != 0.0:  # restore C before each call
                y.copy_(torch.from_numpy(c_vals).to(TORCH_OUT[out]))
        qgemv.run_group(h, xd, K, probs)
        torch.cuda.synchronize()
        results.append([c[5].clone() for c in checks])
    for kind, fmt, N, W, Wu, y, out, c_vals, alpha, beta in checks:
        label = f"{what}: {kind} {synth.FORMAT_NAMES[fmt]} {N}x{K}"
        if kind == "swiglu":
            o = oracle.swiglu(fmt, x, W, Wu, N, K)
            _assert_within(y.to(torch.float64).cpu().numpy(), o["h"], _swiglu_tol(o, out), label)
        else:
            _check_general(fmt, x, W, N, K, alpha, beta, out, y, c_vals, label)
    for r in results[1:]:  # deterministic from call to call
        assert all(torch.equal(a, b) for a, b in zip(results[0], r))
    assert qgemv.check_error(h) == qgemv.OK


def test_group_mixed_format_qkv(h):
    K = 4096
    x = synth.make_x(synth.Q4_K, K, seed=11)
    specs = [dict(fmt=synth.Q4_K, N=512, seed=1), dict(fmt=synth.Q5_K, N=128, seed=2),
             dict(fmt=synth.Q6_K, N=128, seed=3)]
    _run_and_check_group(h, specs, K, x, "qkv", repeat=2)


@pytest.mark.parametrize("K", [2048, 4096, 12288])
def test_group_every_integer_format_with_epilogues_and_a_pair(h, K):
    x = synth.make_x(synth.Q4_K, K, seed=K)
    specs = [dict(fmt=synth.Q4_K, N=33, seed=10, swiglu=True, out=qgemv.OUT_BF16),
             dict(fmt=synth.Q5_K, N=1, seed=20, alpha=-2.0, out=qgemv.OUT_F16),
             dict(fmt=synth.Q6_K, N=70, seed=30, alpha=0.5, beta=1.5),
             dict(fmt=synth.Q8_0, N=9, seed=40),
             dict(fmt=synth.TQ1_0, N=65, seed=50, beta=-1.0, out=qgemv.OUT_BF16),
             dict(fmt=synth.Q4_K, N=300, seed=60),
             dict(fmt=synth.Q6_K, N=2, seed=70, swiglu=True),
             dict(fmt=synth.Q4_K, N=129, seed=80, out=qgemv.OUT_F16)]
    _run_and_check_group(h, specs, K, x, f"8 matrices K={K}", repeat=2)


def test_group_nvfp4_pair_and_plain(h):
    K = 14336
    x = synth.make_x(synth.NVFP4, K, seed=5)
    specs = [dict(fmt=synth.NVFP4, N=96, seed=1, swiglu=True), dict(fmt=synth.NVFP4, N=40, seed=3, alpha=0.5)]
    _run_and_check_group(h, specs, K, x, "nvfp4", repeat=2)


def test_group_with_a_shape_the_streaming_kernel_does_not_take(h):
    K = 4000  # Q8_0 only: not a multiple of 256, so every matrix runs warp per row
    x = synth.make_x(synth.Q8_0, K, seed=6)
    specs = [dict(fmt=synth.Q8_0, N=20, seed=1), dict(fmt=synth.Q8_0, N=7, seed=2, swiglu=True, out=qgemv.OUT_F16)]
    _run_and_check_group(h, specs, K, x, "rowwarp group")


def test_group_under_programmatic_dependent_launch_chain(h):
    qgemv.set_option(h, qgemv.OPT_PDL, 1)
    try:
        K = 4096
        x = synth.make_x(synth.Q4_K, K, seed=8)
        specs = [dict(fmt=synth.Q4_K, N=1024, seed=1, swiglu=True), dict(fmt=synth.Q6_K, N=256, seed=2)]
        _run_and_check_group(h, specs, K, x, "pdl", repeat=3)
    finally:
        qgemv.set_option(h, qgemv.OPT_PDL, 0)


def test_group_rejects_bad_arguments_before_launching(h):
    K = 4096
    x = torch.zeros(K, dtype=torch.int16, device="cuda")
    W = torch.zeros(synth.packed_bytes(synth.Q4_K, 4, K), dtype=torch.uint8, device="cuda")
    Wn = torch.zeros(synth.packed_bytes(synth.NVFP4, 4, K), dtype=torch.uint8, device="cuda")
    y = torch.zeros(16, dtype=torch.float32, device="cuda")
    ok = qgemv.problem(synth.Q4_K, W, 4, y)

    def st(probs, xx=x):
        return qgemv.run_group(h, xx, K, probs, check=False)
    assert st([]) == qgemv.ERR_INVALID_ARG
    assert st([ok] * (qgemv.MAX_GROUP + 1)) == qgemv.ERR_INVALID_ARG
    assert st([ok, qgemv.problem(synth.NVFP4, Wn, 4, y)]) == qgemv.ERR_INVALID_ARG  # one x for both
    assert st([qgemv.problem(synth.Q4_K, W, 4, y, swiglu=True)]) == qgemv.ERR_INVALID_ARG  # no up matrix
    assert st([qgemv.problem(synth.Q4_K, W, 4, y, out=3)]) == qgemv.ERR_INVALID_ARG
    assert st([qgemv.problem(synth.Q4_K, W, 4, None)]) == qgemv.ERR_INVALID_ARG
    assert st([qgemv.problem(synth.Q4_K, W, 4, y.data_ptr() + 4)]) == qgemv.ERR_MISALIGNED
    assert st([qgemv.problem(synth.Q4_K, W, 0, y)]) == qgemv.ERR_BAD_SHAPE
    assert st([qgemv.problem(9, W, 4, y)]) == qgemv.ERR_UNSUPPORTED_FORMAT
    assert st([ok], xx=x.data_ptr() + 2) == qgemv.ERR_MISALIGNED
    assert qgemv.run_ex(h, synth.Q4_K, x, W, 4, 1000, y, check=False) == qgemv.ERR_BAD_SHAPE
    torch.cuda.synchronize()
    assert qgemv.check_error(h) == qgemv.OK


def test_full_size_decoder_layer_groups_on_sampled_rows(h):
    """The mixed-format attention projections (Q Q4_K 4096, K Q5_K 1024, V Q6_K 1024 rows) in one
    launch, and the MLP gate/up pair (12288 x 4096 Q4_K each) as SwiGLU, at full size, under
    programmatic dependent launch as a decode loop runs them; sampled rows against the oracle."""
    K = 4096
    x = synth.make_x(synth.Q4_K, K, seed=1234)
    xd = dev_x(x)
    qkv = [(synth.Q4_K, 4096), (synth.Q5_K, 1024), (synth.Q6_K, 1024)]
    mats = [synth.make_weights(f, N, K, seed=400 + i) for i, (f, N) in enumerate(qkv)]
    dev = [dev_bytes(W)[0] for W in mats]
    ys = [torch.full((N,), float("nan"), dtype=torch.float32, device="cuda") for _, N in qkv]
    Ng = 12288
    Wg = synth.make_weights(synth.Q4_K, Ng, K, seed=500)
    Wu = synth.make_weights(synth.Q4_K, Ng, K, seed=501)
    Wgd, Wud = dev_bytes(Wg)[0], dev_bytes(Wu)[0]
    hy = torch.full((Ng,), float("nan"), dtype=torch.bfloat16, device="cuda")
    qgemv.set_option(h, qgemv.OPT_PDL, 1)
    try:
        for _ in range(2):
            qgemv.run_group(h, xd, K, [qgemv.problem(f, d, N, y) for (f, N), d, y in zip(qkv, dev, ys)])
            qgemv.run_group(h, xd, K, [qgemv.problem(synth.Q4_K, Wgd, Ng, hy, packed_W_up=Wud,
                                                     out=qgemv.OUT_BF16, swiglu=True)])
        torch.cuda.synchronize()
    finally:
        qgemv.set_option(h, qgemv.OPT_PDL, 0)
    for (f, N), W, y in zip(qkv, mats, ys):
        rows = sample_rows(N, 48, seed=N + f)
        ref, S = oracle.gemv_rows(f, x, W, N, K, rows)
        got = y.cpu().numpy().astype(np.float64)[rows]
        _assert_within(got, ref, RTOL * S + ATOL, f"qkv {synth.FORMAT_NAMES[f]}")
    rows = sample_rows(Ng, 64, seed=9)
    g, Sg = oracle.gemv_rows(synth.Q4_K, x, Wg, Ng, K, rows)
    u, Su = oracle.gemv_rows(synth.Q4_K, x, Wu, Ng, K, rows)
    o = {"g": g, "u": u, "Sg": Sg, "Su": Su, "h": np.array([oracle.silu(a) for a in g]) * u}
    got = hy.to(torch.float64).cpu().numpy()[rows]
    _assert_within(got, o["h"], _swiglu_tol(o, qgemv.OUT_BF16), "gate/up swiglu")
    assert qgemv.check_error(h) == qgemv.OK
