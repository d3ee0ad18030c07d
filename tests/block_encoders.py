"""Test-side block builders: place known codes/scales into the byte layouts.

These are the encoding direction of each layout (value -> byte position), written from
the layout descriptions, and are used to hand-build blocks with known weights.  They
share nothing with the oracle's decoders, so a round trip checks one against the other.
"""
import numpy as np


def f16_bytes(v):
    b = np.array([v], dtype=np.float16).view(np.uint8)
    return int(b[0]), int(b[1])


def pack_kquant_scales(s, m):
    """8 six-bit scales s and mins m -> the 12 packed bytes of a Q4_K/Q5_K block.

    Groups 0..3 keep their low 6 bits in bytes 0..3 (scales) and 4..7 (mins); groups 4..7
    put their low nibbles in bytes 8..11 (scale low, min high) and their top two bits in
    bits 6..7 of bytes 0..3 (scales) and 4..7 (mins).
    """
    S = np.zeros(12, dtype=np.uint8)
    for g in range(4):
        S[g] = (s[g] & 63) | ((s[g + 4] >> 4) << 6)
        S[g + 4] = (m[g] & 63) | ((m[g + 4] >> 4) << 6)
        S[g + 8] = (s[g + 4] & 15) | ((m[g + 4] & 15) << 4)
    return S


def q4k_block(q, s, m, d, dmin):
    """q[256] in 0..15, s/m[8] in 0..63 -> 144 bytes."""
    b = np.zeros(144, dtype=np.uint8)
    b[0], b[1] = f16_bytes(d)
    b[2], b[3] = f16_bytes(dmin)
    b[4:16] = pack_kquant_scales(s, m)
    for i in range(256):
        c, h, j = i // 64, (i // 32) % 2, i % 32
        b[16 + 32 * c + j] |= (q[i] & 15) << (4 * h)
    return b


def q5k_block(q, s, m, d, dmin):
    """q[256] in 0..31 -> 176 bytes."""
    b = np.zeros(176, dtype=np.uint8)
    b[0], b[1] = f16_bytes(d)
    b[2], b[3] = f16_bytes(dmin)
    b[4:16] = pack_kquant_scales(s, m)
    for i in range(256):
        c, h, j = i // 64, (i // 32) % 2, i % 32
        b[48 + 32 * c + j] |= (q[i] & 15) << (4 * h)
        b[16 + j] |= ((q[i] >> 4) & 1) << (2 * c + h)
    return b


def q6k_block(q, sc, d):
    """q[256] in 0..63 (stored value, the weight uses q-32), sc[16] int8 -> 210 bytes."""
    b = np.zeros(210, dtype=np.uint8)
    for i in range(256):
        H, r, l = i // 128, (i % 128) // 32, i % 32
        b[64 * H + l + 32 * (r & 1)] |= (q[i] & 15) << (4 * (r >> 1))
        b[128 + 32 * H + l] |= ((q[i] >> 4) & 3) << (2 * r)
    b[192:208] = np.asarray(sc, dtype=np.int8).view(np.uint8)
    b[208], b[209] = f16_bytes(d)
    return b


def q80_block(q, d):
    b = np.zeros(34, dtype=np.uint8)
    b[0], b[1] = f16_bytes(d)
    b[2:34] = np.asarray(q, dtype=np.int8).view(np.uint8)
    return b
