"""Test inputs for wide-range activations: x with one large outlier per 32-element chunk
among small values, and packed weights edited so that the weights meeting chosen columns
are exactly zero (the case where an outlier sets the scale of its chunk but adds nothing
to sum |x w|).  The byte edits follow the layout descriptions (the same ones the test-side
block builders encode); every caller checks the result with the oracle's own dequantiser.
"""
import numpy as np
import torch

from block_encoders import pack_kquant_scales
from quantized_weight_dequant_gb300 import synth


def _kquant_scales_mins(S):
    s, m = np.zeros(8, dtype=np.int64), np.zeros(8, dtype=np.int64)
    for g in range(8):
        if g < 4:
            s[g], m[g] = S[g] & 63, S[g + 4] & 63
        else:
            s[g] = (S[g + 4] & 15) | ((S[g - 4] >> 6) << 4)
            m[g] = (S[g + 4] >> 4) | ((S[g] >> 6) << 4)
    return s, m


def _tq1_digits(b):
    return [((3 ** (n + 1) * int(b)) // 256) % 3 for n in range(5)]


def _tq1_byte(digits):
    v = 0
    for t in digits:
        v = v * 3 + t
    return (256 * v + 242) // 243


def _tq1_pos(i):
    """Element i of a TQ1_0 block -> (byte index, digit)."""
    if i < 160:
        return i % 32, i // 32
    if i < 240:
        return 32 + (i - 160) % 16, (i - 160) // 16
    return 48 + (i - 240) % 4, (i - 240) // 4


def zero_weight_columns(fmt, W: np.ndarray, N: int, K: int, cols) -> np.ndarray:
    """A copy of the packed matrix W (N x K) whose weights in columns `cols` are exactly 0 in
    every row: code 0 with a zero group minimum (Q4_K, Q5_K), code 32 (Q6_K), code 0 (Q8_0,
    NVFP4), digit 1 (TQ1_0)."""
    W = W.copy()
    cols = sorted(set(int(c) for c in cols))
    if fmt == synth.NVFP4:
        nib = W[: N * (K // 2)].reshape(N, K // 2)
        for k in cols:
            nib[:, k // 2] &= np.uint8(0xF0 if k % 2 == 0 else 0x0F)
        return W
    bw, bb = synth.BLOCK[fmt]
    blk = W.reshape(N, K // bw, bb)
    for k in cols:
        b, i = k // bw, k % bw
        for n in range(N):
            p = blk[n, b]
            if fmt in (synth.Q4_K, synth.Q5_K):
                c, h, j = i // 64, (i // 32) % 2, i % 32
                s, m = _kquant_scales_mins(p[4:16])
                m[i // 32] = 0
                p[4:16] = pack_kquant_scales(s, m)
                qoff = 16 if fmt == synth.Q4_K else 48
                p[qoff + 32 * c + j] &= np.uint8(0xF0 if h == 0 else 0x0F)
                if fmt == synth.Q5_K:
                    p[16 + j] &= np.uint8(~(1 << (2 * c + h)) & 0xFF)
            elif fmt == synth.Q6_K:  # stored value 32: low nibble 0, top bits 2
                H, r, l = i // 128, (i % 128) // 32, i % 32
                lo = 64 * H + l + 32 * (r & 1)
                p[lo] &= np.uint8(0xF0 if r < 2 else 0x0F)
                qh = 128 + 32 * H + l
                p[qh] = (p[qh] & np.uint8(~(3 << (2 * r)) & 0xFF)) | np.uint8(2 << (2 * r))
            elif fmt == synth.Q8_0:
                p[2 + i] = 0
            elif fmt == synth.TQ1_0:
                byte, digit = _tq1_pos(i)
                d = _tq1_digits(p[byte])
                d[digit] = 1
                if byte >= 48:
                    d[4] = 0
                p[byte] = _tq1_byte(d)
    return blk.reshape(-1)


def outlier_x(fmt, K: int, seed: int, big: float = 3000.0, small: float = 1e-3, every: int = 32):
    """x bits: small * N(0,1) with one +-big outlier at the start of every `every` elements;
    returns (bits, outlier columns)."""
    rng = np.random.default_rng(seed)
    xf = rng.standard_normal(K) * small
    cols = np.arange(0, K, every)
    xf[cols] = big * np.sign(rng.standard_normal(cols.size))
    if fmt == synth.NVFP4:
        bits = torch.tensor(xf, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    else:
        bits = xf.astype(np.float16).view(np.uint16)
    return bits.copy(), cols
