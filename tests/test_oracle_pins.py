"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test fixes part of the oracle by an independent route: a library conversion,
numbers printed on the pages, a different formulation of the same mathematics, or a
test-side encoder.  A dropped term, a wrong sign, a swapped nibble or index in the
oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from block_encoders import q4k_block, q5k_block, q6k_block, q80_block
from conftest import read_golden
from quantized_weight_dequant_gb300 import synth

F16_ALL = np.arange(65536, dtype=np.uint16)


# ---------------------------------------------------------------- minifloat decoders
def _same(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)]) \
        and np.array_equal(np.signbit(a[~np.isnan(a)]), np.signbit(b[~np.isnan(b)]))


def test_fp16_decoder_matches_numpy_on_every_code():
    mine = np.array([oracle.fp16(int(h)) for h in F16_ALL])
    ref = F16_ALL.view(np.float16).astype(np.float64)
    assert _same(mine, ref)


def test_bf16_decoder_matches_torch_on_every_code():
    mine = np.array([oracle.bf16(int(h)) for h in F16_ALL])
    ref = torch.from_numpy(F16_ALL.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same(mine, ref)


@pytest.mark.parametrize("dtype,fn", [(torch.float8_e4m3fn, "e4m3"), (torch.float8_e5m2, "e5m2")])
def test_fp8_decoders_match_torch_on_every_code(dtype, fn):
    codes = np.arange(256, dtype=np.uint8)
    mine = np.array([getattr(oracle, fn)(int(c)) for c in codes])
    ref = torch.from_numpy(codes.copy()).view(dtype).to(torch.float64).numpy()
    assert _same(mine, ref)


def test_e2m1_decoder_matches_the_mx_specification_table():
    table = {int(c): float(v) for c, v in read_golden("e2m1_magnitudes.txt")}
    for c in range(16):
        v = oracle.e2m1(c)
        want = table[c & 7] * (-1.0 if c & 8 else 1.0)
        assert v == want and math.copysign(1.0, v) == math.copysign(1.0, want)
    # The same generic routine, given E2M1's parameters, is what decodes it.
    for c in range(16):
        assert oracle.minifloat(c, 2, 1, 1, 0) == oracle.e2m1(c)


# ---------------------------------------------------------------- TQ1_0 digits
def test_tq1_digits_equal_base3_expansion_of_the_byte_level():
    # A byte b stands for the level v = floor(243 b / 256); its digits, most significant
    # first, must be what the floor pair returns.
    for b in range(256):
        v = (243 * b) // 256
        want = [(v // 3 ** (4 - n)) % 3 for n in range(5)]
        assert [oracle.tq1_digit(b, n) for n in range(5)] == want


def test_tq1_fp16_digit_extraction_fails_as_the_page_reports():
    g = {k: int(v) for k, v in read_golden("tq1_0_fp16_digit_extraction.txt")}
    f16 = np.float16
    wrong = []
    for b in range(256):
        for n in range(5):
            hi = np.floor(f16(f16(3 ** (n + 1)) * f16(b)) / f16(256))
            lo = np.floor(f16(f16(3 ** n) * f16(b)) / f16(256))
            d16 = int(hi) - 3 * int(lo)
            if d16 != oracle.tq1_digit(b, n):
                wrong.append((b, n, d16))
    assert 256 * 5 == g["total_digits"]
    assert len(wrong) == g["wrong_digits"]
    hit = [w for w in wrong if w[0] == g["example_byte"] and w[1] == g["example_digit"]]
    assert hit and hit[0][2] == g["example_fp16_value"]
    assert oracle.tq1_digit(g["example_byte"], g["example_digit"]) == g["example_reference_value"]


def test_tq1_five_digit_collapse_with_zero_padding_over_all_bytes():
    # sum_n y_n t_n(b) == sum_{k=1..5} g_k floor(3^k b/256), g_k = y_{k-1} - 3 y_k, y_5 = 0;
    # with y_4 = 0 the same expression gives the four-digit (qh) form.
    rng = np.random.default_rng(5)
    for pad in (False, True):
        for _ in range(20):
            y = rng.standard_normal(5)
            if pad:
                y[4] = 0.0
            g = [y[k - 1] - 3 * (y[k] if k < 5 else 0.0) for k in range(1, 6)]
            for b in range(256):
                lhs = sum(y[n] * oracle.tq1_digit(b, n) for n in range(5))
                rhs = sum(g[k - 1] * ((3 ** k * b) // 256) for k in range(1, 6))
                assert abs(lhs - rhs) <= 1e-12 * (1 + abs(lhs))


def test_tq1_generator_bytes_round_trip_through_the_oracle_digits():
    rng = np.random.default_rng(11)
    digits = rng.integers(0, 3, size=(4000, 5))
    b = synth._tq1_bytes(digits)
    got = np.array([[oracle.tq1_digit(int(bb), n) for n in range(5)] for bb in b])
    assert np.array_equal(got, digits)
    # every one of the 243 levels round-trips
    all_digits = np.array([[(v // 3 ** (4 - n)) % 3 for n in range(5)] for v in range(243)])
    b = synth._tq1_bytes(all_digits)
    assert np.array_equal(np.array([[oracle.tq1_digit(int(bb), n) for n in range(5)] for bb in b]), all_digits)


def test_tq1_element_order_matches_the_dequantize_index_description():
    # The dequantize produces 16 elements per index il: il < 10 -> 16 consecutive bytes of
    # the 32-byte region at digit il/2; 10 <= il < 15 -> the 16-byte region at digit il-10;
    # il == 15 -> the qh tail (four bytes, digit-major: our reading of the page).
    W = synth.make_weights(synth.TQ1_0, 1, 256, seed=42)
    blk = W[:54]
    d = int(blk[52]) | (int(blk[53]) << 8)
    dv = float(np.array([d], dtype=np.uint16).view(np.float16)[0])
    want = np.zeros(256)
    for il in range(16):
        for e in range(16):
            if il < 10:
                byte, n = blk[16 * (il % 2) + e], il // 2
            elif il < 15:
                byte, n = blk[32 + e], il - 10
            else:
                byte, n = blk[48 + e % 4], e // 4
            want[16 * il + e] = dv * (oracle.tq1_digit(int(byte), n) - 1)
    got = oracle.dequant_rows(synth.TQ1_0, W, 1, 256, [0])[0]
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- Q4_K
def _q4k_dense(blk):
    return oracle.dequant_rows(synth.Q4_K, blk, 1, 256, [0])[0]


def test_q4k_known_blocks():
    g = {k: float(v) for k, v in read_golden("q4k_known_blocks.txt")}
    w = _q4k_dense(q4k_block([15] * 256, [63] * 8, [0] * 8, 1.0, 0.0))
    assert np.all(w == g["all_max_scale"])
    w = _q4k_dense(q4k_block([0] * 256, [0] * 8, [63] * 8, 0.0, 1.0))
    assert np.all(w == g["all_min_only"])
    w = _q4k_dense(q4k_block([1] * 256, [1] * 8, [1] * 8, 0.5, 0.25))
    assert np.all(w == g["unit_codes"])


def test_q4k_each_element_and_group_lands_where_the_layout_says():
    rng = np.random.default_rng(1)
    s = rng.integers(1, 64, 8)
    m = rng.integers(0, 64, 8)
    for i in list(range(0, 256, 7)) + [31, 32, 63, 64, 255]:
        q = np.zeros(256, dtype=int)
        q[i] = 9
        w = _q4k_dense(q4k_block(q, s, m, 1.0, 0.5))
        want = -0.5 * m[np.arange(256) // 32]
        want[i] += 9 * s[i // 32]
        assert np.array_equal(w, want), i


def test_q4k_scale_packing_round_trip_over_all_six_bit_values():
    for v in range(64):
        for g in range(8):
            s = np.zeros(8, dtype=int)
            m = np.zeros(8, dtype=int)
            s[g] = v
            m[7 - g] = (v * 5) % 64
            blk = q4k_block([1] * 256, s, m, 1.0, 1.0)
            w = _q4k_dense(blk)
            # with q = 1 and d = dmin = 1: w = s_g - m_g
            want = (s - m)[np.arange(256) // 32]
            assert np.array_equal(w, want.astype(float))


def _page_kernel_q4k_gemv(x16, W, N, K):
    """Float32 restatement of the Q4_K page's kernel arithmetic ("Kernel code").

    Per 256-weight block, 32 lanes split as 4 cohorts x 2 teams x 4 lanes: team t reads
    the 16-bit scale words at t, t+2, t+4 and unpacks s and m for groups {2t, 2t+1, 2t+4,
    2t+5} with the 0x3f3f / 0x0f0f / 0xc0c0 masks; each lane reads two 8-byte quant runs
    64 bytes apart, multiplies activations by the masked but unshifted nibble and undoes
    the 2^8 and 2^4 factors once per block; the min term uses per-lane activation sums.
    Here every lane of every block is evaluated at once with numpy, in float32.
    """
    nb = K // 256
    x = x16.view(np.float16).astype(np.float32)
    Wb = W.reshape(N, nb, 144)
    y = np.zeros(N, dtype=np.float32)
    t = np.repeat(np.arange(2), 4)          # team of each lane in a cohort (8 lanes)
    r = np.tile(np.arange(4), 2)            # lane within the team
    for n in range(N):
        tot = np.float32(0)
        for b in range(nb):
            blk = Wb[n, b]
            xb = x[256 * b: 256 * (b + 1)]
            u16 = blk.view(np.uint16)                     # whole block as 72 ushorts
            sc = np.stack([u16[2 + t + 2 * j] for j in range(3)])  # scale words at t, t+2, t+4
            s16 = np.stack([sc[0] & 0x3F3F, sc[1] & 0x3F3F,
                            (sc[2] & 0x0F0F) | ((sc[0] & 0xC0C0) >> 2),
                            ((sc[2] >> 4) & 0x0F0F) | ((sc[1] & 0xC0C0) >> 2)])
            sc8 = np.stack([s16 & 0xFF, s16 >> 8], axis=1).reshape(8, -1).astype(np.float32)  # [8 bytes, lanes]
            base = 64 * t + 8 * r
            part = np.zeros(8, dtype=np.float32)
            for half, off in ((0, 0), (1, 128)):        # first and second 8-byte run (q1, q2)
                q = np.stack([u16[8 + 16 * t + 4 * r + 32 * half + i] for i in range(4)])  # [4, lanes]
                lo_idx = base + off
                xl = np.stack([xb[lo_idx + k] for k in range(8)])        # activations paired with low nibbles
                xh = np.stack([xb[lo_idx + 32 + k] for k in range(8)])   # ... with high nibbles
                a0 = (xl[0::2] * (q & 0x000F)).sum(0, dtype=np.float32)
                a1 = (xl[1::2] * (q & 0x0F00)).sum(0, dtype=np.float32)
                a2 = (xh[0::2] * (q & 0x00F0)).sum(0, dtype=np.float32)
                a3 = (xh[1::2] * (q & 0xF000)).sum(0, dtype=np.float32)
                part += (a0 + a1 / np.float32(256)) * sc8[4 * half + 0] \
                    + (a2 + a3 / np.float32(256)) * sc8[4 * half + 1] / np.float32(16)
            sumy = np.stack([xb[base + k * 32 + j] for k in (0, 1, 4, 5) for j in range(8)]).reshape(4, 8, -1).sum(1)
            mins = np.stack([sc8[2], sc8[3], sc8[6], sc8[7]])
            d = np.float32(blk[0:2].view(np.float16)[0])
            dmin = np.float32(blk[2:4].view(np.float16)[0])
            tot += (d * part - dmin * (sumy * mins).sum(0)).sum(dtype=np.float32)
        y[n] = tot
    return y


def test_q4k_oracle_agrees_with_the_page_kernel_arithmetic():
    N, K = 6, 1024
    W = synth.make_weights(synth.Q4_K, N, K, seed=77)
    x = synth.make_x(synth.Q4_K, K, seed=77)
    y_ref, S = oracle.gemv(synth.Q4_K, x, W, N, K)
    y_page = _page_kernel_q4k_gemv(x, W, N, K)
    assert np.all(np.abs(y_page - y_ref) <= 1e-5 * S + 1e-6)
    # and a mistake in either (dropping the min term) would show
    assert np.max(np.abs(y_ref)) > 1e-3


# ---------------------------------------------------------------- Q5_K, Q6_K, Q8_0 (layout pins)
def test_q5k_hand_built_blocks():
    rng = np.random.default_rng(2)
    for _ in range(20):
        q = rng.integers(0, 32, 256)
        s = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        blk = q5k_block(q, s, m, 0.5, 0.125)
        w = oracle.dequant_rows(synth.Q5_K, blk, 1, 256, [0])[0]
        g = np.arange(256) // 32
        assert np.array_equal(w, 0.5 * s[g] * q - 0.125 * m[g])


def test_q6k_hand_built_blocks():
    rng = np.random.default_rng(4)
    for _ in range(20):
        q = rng.integers(0, 64, 256)
        sc = rng.integers(-32, 32, 16)
        blk = q6k_block(q, sc, 0.25)
        w = oracle.dequant_rows(synth.Q6_K, blk, 1, 256, [0])[0]
        assert np.array_equal(w, 0.25 * sc[np.arange(256) // 16] * (q - 32))


def test_q80_hand_built_blocks():
    rng = np.random.default_rng(6)
    q = rng.integers(-128, 128, 32)
    blk = q80_block(q, 0.375)
    w = oracle.dequant_rows(synth.Q8_0, blk, 1, 32, [0])[0]
    assert np.array_equal(w, 0.375 * q)


# ---------------------------------------------------------------- NVFP4
def test_nvfp4_nibble_order_scale_blocks_and_abs_scale():
    N, K = 2, 64
    nib = np.zeros(N * K // 2, dtype=np.uint8)
    sc = np.zeros(N * K // 16, dtype=np.uint8)
    # element (1, 37): odd -> high nibble of byte 1*32 + 18; code 0xB = -1.5
    nib[32 + 18] = 0xB0
    # element (0, 4): even -> low nibble of byte 2; code 0x7 = 6
    nib[2] = 0x07
    e4 = lambda v: int(torch.tensor([v]).to(torch.float8_e4m3fn).view(torch.uint8)[0])
    sc[0] = e4(0.25)                  # row 0, block 0 (elements 0..15)
    sc[4 + 2] = e4(-2.0)              # row 1, block 2 (elements 32..47): negative scale, |.| used
    W = np.concatenate([nib, sc])
    w = oracle.dequant_rows(synth.NVFP4, W, N, K, [0, 1])
    want = np.zeros((N, K))
    want[0, 4] = 6 * 0.25
    want[1, 37] = -1.5 * 2.0
    assert np.array_equal(w, want)


def test_nvfp4_subnormal_e4m3_scales_decode_exactly():
    for code in range(1, 8):  # E4M3 subnormals m * 2^-9
        assert oracle.e4m3(code) == code * 2.0 ** -9


# ---------------------------------------------------------------- GEMV and unpack
@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.Q8_0, synth.TQ1_0, synth.NVFP4])
def test_gemv_is_the_plain_dot_product_of_the_dequantised_rows(fmt):
    N, K = 5, 512
    W = synth.make_weights(fmt, N, K, seed=10 + fmt)
    x = synth.make_x(fmt, K, seed=10 + fmt)
    xv = np.array([oracle.bf16(int(v)) if fmt == synth.NVFP4 else oracle.fp16(int(v)) for v in x])
    dense = oracle.dequant_rows(fmt, W, N, K, range(N))
    y, S = oracle.gemv(fmt, x, W, N, K)
    assert np.allclose(y, dense @ xv, rtol=1e-12, atol=1e-12)
    assert np.allclose(S, np.abs(dense * xv).sum(1), rtol=1e-12)
    # one-hot activations pick single weights
    e = np.zeros(K, dtype=np.uint16)
    e[K - 3] = 0x3C00 if fmt != synth.NVFP4 else 0x3F80  # 1.0 in fp16 / bf16
    y1, _ = oracle.gemv(fmt, e, W, N, K)
    assert np.array_equal(y1, dense[:, K - 3])


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q5_K, synth.Q6_K, synth.Q8_0, synth.TQ1_0, synth.NVFP4])
def test_unpack_reconstructs_every_weight_and_fits_fp32(fmt):
    N, K = 3, 512
    W = synth.make_weights(fmt, N, K, seed=20 + fmt)
    codes, scales, mins = oracle.unpack(fmt, W, N, K)
    G = oracle.group_size(fmt)
    w = scales.repeat(G, axis=1) * codes - mins.repeat(G, axis=1)
    assert np.array_equal(w, oracle.dequant_rows(fmt, W, N, K, range(N)))
    # scales and mins are exactly representable in fp32 (the GPU reports them as fp32)
    assert np.array_equal(scales.astype(np.float32).astype(np.float64), scales)
    assert np.array_equal(mins.astype(np.float32).astype(np.float64), mins)


def test_generator_distributions_and_determinism():
    W1 = synth.make_weights(synth.Q4_K, 64, 1024, seed=3)
    W2 = synth.make_weights(synth.Q4_K, 64, 1024, seed=3)
    assert np.array_equal(W1, W2) and W1.size == synth.packed_bytes(synth.Q4_K, 64, 1024)
    codes, _, _ = oracle.unpack(synth.Q4_K, W1, 64, 1024)
    counts = np.bincount(codes.ravel().astype(np.int64), minlength=16)
    assert counts.min() > 0.9 * counts.mean()
    Wt = synth.make_weights(synth.TQ1_0, 64, 1024, seed=3)
    ct, _, _ = oracle.unpack(synth.TQ1_0, Wt, 64, 1024)
    c3 = np.bincount((ct.ravel() + 1).astype(np.int64), minlength=3)
    assert c3.min() > 0.95 * c3.mean()
    Wf = synth.make_weights(synth.NVFP4, 16, 1024, seed=3)
    assert Wf.size == synth.packed_bytes(synth.NVFP4, 16, 1024)
    _, sf, _ = oracle.unpack(synth.NVFP4, Wf, 16, 1024)
    # about a quarter of |N(0,1)|*0.05 falls below 2^-6, the E4M3 subnormal range
    frac_sub = np.mean(2 * sf < 2.0 ** -6)
    assert 0.1 < frac_sub < 0.45


# ---------------------------------------------------------------- layer epilogues
def _x_values(fmt, x):
    """Activations as fp64 by numpy / torch (not by the oracle's own decoder)."""
    if fmt == synth.NVFP4:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    return x.view(np.float16).astype(np.float64)


def test_silu_is_x_times_scipy_logistic_and_has_the_odd_part_x():
    expit = pytest.importorskip("scipy.special").expit
    g = np.concatenate([np.linspace(-40, 40, 801), [-800.0, -1e-300, 0.0, 1e-300, 800.0]])
    mine = np.array([oracle.silu(v) for v in g])
    np.testing.assert_allclose(mine, g * expit(g), rtol=1e-14, atol=0)
    assert oracle.silu(-800.0) == 0.0 and oracle.silu(800.0) == 800.0
    # logistic(x) + logistic(-x) = 1, so silu(x) - silu(-x) = x
    for v in np.linspace(-30, 30, 61):
        assert abs((oracle.silu(v) - oracle.silu(-v)) - v) <= 1e-14 * max(1.0, abs(v))
    # the slope bound the SwiGLU tolerance relies on: max |silu'| is about 1.0998 (near x = 2.4)
    t = np.linspace(-20, 20, 40001)
    s = np.array([oracle.silu(v) for v in t])
    slope = np.abs(np.diff(s) / np.diff(t)).max()
    assert 1.09 < slope < 1.1


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.Q6_K, synth.NVFP4])
def test_general_gemv_is_alpha_times_the_dense_product_plus_beta_c(fmt):
    N, K = 6, 512
    W = synth.make_weights(fmt, N, K, seed=40 + fmt)
    x = synth.make_x(fmt, K, seed=40 + fmt)
    dense = oracle.dequant_rows(fmt, W, N, K, range(N))
    xv = _x_values(fmt, x)
    c = np.random.default_rng(7).normal(size=N)
    y, S = oracle.gemv_general(fmt, x, W, N, K, -0.75, 2.5, c)
    ref = -0.75 * (dense @ xv) + 2.5 * c
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, 0.75 * np.abs(dense * xv).sum(1), rtol=1e-12)
    y1, S1 = oracle.gemv_general(fmt, x, W, N, K, 1.0, 0.0, np.full(N, np.nan))  # beta = 0 never reads c
    y0, S0 = oracle.gemv(fmt, x, W, N, K)
    assert np.array_equal(y1, y0) and np.array_equal(S1, S0)


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.TQ1_0, synth.NVFP4])
def test_swiglu_gates_the_up_rows_with_silu_of_the_gate_rows(fmt):
    expit = pytest.importorskip("scipy.special").expit
    N, K = 7, 512
    Wg = synth.make_weights(fmt, N, K, seed=50 + fmt)
    Wu = synth.make_weights(fmt, N, K, seed=60 + fmt)
    x = synth.make_x(fmt, K, seed=50 + fmt)
    xv = _x_values(fmt, x)
    g = oracle.dequant_rows(fmt, Wg, N, K, range(N)) @ xv
    u = oracle.dequant_rows(fmt, Wu, N, K, range(N)) @ xv
    out = oracle.swiglu(fmt, x, Wg, Wu, N, K)
    np.testing.assert_allclose(out["g"], g, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["u"], u, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["h"], g * expit(g) * u, rtol=1e-11, atol=1e-12)
    # the two matrices play different roles: swapping them changes the result
    swapped = oracle.swiglu(fmt, x, Wu, Wg, N, K)["h"]
    assert not np.allclose(swapped, out["h"], rtol=1e-3)


@pytest.mark.parametrize("fmt", [synth.Q4_K, synth.NVFP4, synth.TQ1_0, synth.Q5_K, synth.Q6_K, synth.Q8_0])
def test_zero_weight_column_edit_is_exact(fmt):
    """The wide-range tests' weight edit: the chosen columns dequantise (by the oracle) to
    exactly zero in every row, every other weight outside the edited Q4_K/Q5_K groups keeps
    its value, and the edited bytes still decode with the oracle's layout."""
    from wide_range import zero_weight_columns
    N, K = 3, 512
    W = synth.make_weights(fmt, N, K, seed=5 + fmt)
    cols = np.array([0, 37, 64, 255, 256, 300, 511])
    W2 = zero_weight_columns(fmt, W, N, K, cols)
    a = oracle.dequant_rows(fmt, W, N, K, np.arange(N))
    b = oracle.dequant_rows(fmt, W2, N, K, np.arange(N))
    assert np.all(b[:, cols] == 0.0)
    keep = np.ones(K, dtype=bool)
    if fmt in (synth.Q4_K, synth.Q5_K):  # the group minimum of an edited column's group is 0
        for c in cols:
            keep[(c // 32) * 32:(c // 32) * 32 + 32] = False
    else:
        keep[cols] = False
    assert np.array_equal(a[:, keep], b[:, keep])
