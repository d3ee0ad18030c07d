"""Seeded synthetic inputs for the batch-1 dequant GEMV (packed weight bytes and activations).

This module is shared by the CPU oracle's tests, the CUDA parity tests and the benchmark.
It holds no part of the decode or dot-product arithmetic: it only draws random bytes and
random numbers and writes them in the block layouts described below.  The decode side
(what a byte means) lives separately in the oracle and in the CUDA kernels.

Block layouts (byte offsets inside one block, little-endian fp16):

* Q4_K  (256 weights, 144 B): d fp16 @0, dmin fp16 @2, 12 bytes of packed 6-bit
  group scales/mins @4, 128 bytes of 4-bit quants @16.  ("Writing a high performant
  GEMV + dequant for Metal", sections "What is a weight block?" and "Kernel code".)
* Q5_K  (256 weights, 176 B): d @0, dmin @2, scales[12] @4, qh[32] @16, qs[128] @48.
* Q6_K  (256 weights, 210 B): ql[128] @0, qh[64] @128, int8 scales[16] @192, d @208.
* Q8_0  (32 weights, 34 B):   d @0, int8 qs[32] @2.
  (Q5_K, Q6_K and Q8_0 are only named on the Metal GEMV page, section "UD-Q4_K_XL";
  their layouts are taken to be the standard ggml ones: a reading, not on the pages.)
* TQ1_0 (256 weights, 54 B):  qs[48] @0 (5 base-3 digits per byte), qh[4] @48
  (4 digits per byte), d fp16 @52.  ("metal: TQ1_0 kernel performance", section 1.)
* NVFP4 W4A16 (Mojo ``fp4_gemv`` page): E2M1 nibbles [N, K/2] (low nibble = even
  element) followed by E4M3 scales [N, K/16] in one buffer.

Distributions follow the benchmark configurations: Q4_K quants uniform 0..15, 6-bit
scales/mins uniform 0..63, d and dmin = fp16(|N(0,1)| * 1e-2); NVFP4 codes uniform over
all 16 values, scales e4m3(|N(0,1)| * 0.05); TQ1_0 digits uniform over {0,1,2} with
d = fp16(|N(0,1)| * 1e-2); x = fp16(N(0,1)) (bf16 for NVFP4).
"""
from __future__ import annotations

import numpy as np

# Format ids: must equal the C enum qgemv_format_t.
Q4_K, NVFP4, TQ1_0, Q5_K, Q6_K, Q8_0 = 0, 1, 2, 3, 4, 5
FORMAT_NAMES = {Q4_K: "Q4_K", NVFP4: "NVFP4", TQ1_0: "TQ1_0", Q5_K: "Q5_K", Q6_K: "Q6_K", Q8_0: "Q8_0"}
FORMAT_IDS = {v: k for k, v in FORMAT_NAMES.items()}

# (weights per block, bytes per block).  NVFP4 is described per 16-element scale block.
BLOCK = {
    Q4_K: (256, 144),
    Q5_K: (256, 176),
    Q6_K: (256, 210),
    Q8_0: (32, 34),
    TQ1_0: (256, 54),
    NVFP4: (16, 9),
}
K_MULTIPLE = {Q4_K: 256, Q5_K: 256, Q6_K: 256, TQ1_0: 256, Q8_0: 32, NVFP4: 16}


def fmt_id(fmt) -> int:
    return FORMAT_IDS[fmt] if isinstance(fmt, str) else int(fmt)


def packed_bytes(fmt, N: int, K: int) -> int:
    f = fmt_id(fmt)
    if f == NVFP4:
        return N * (K // 2) + N * (K // 16)
    bw, bb = BLOCK[f]
    return N * (K // bw) * bb


def bytes_per_weight(fmt) -> float:
    f = fmt_id(fmt)
    bw, bb = BLOCK[f]
    return bb / bw


def _fp16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 -> IEEE binary16 (round-to-nearest-even, numpy) and return the bits."""
    return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.asarray(v, dtype=np.float32).copy())
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _e4m3_bits(v: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.asarray(v, dtype=np.float32).copy())
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def _put_u16(blocks: np.ndarray, off: int, bits: np.ndarray) -> None:
    blocks[:, off] = (bits & 0xFF).astype(np.uint8)
    blocks[:, off + 1] = (bits >> 8).astype(np.uint8)


# TQ1_0 encoder (value -> byte).  A byte b stores the 5-digit base-3 number v through
# b = ceil(256 v / 243); the decoder side reads digit n as floor(3^(n+1) b / 256) mod 3.
_TQ_ENCODE = np.array([(256 * v + 242) // 243 for v in range(243)], dtype=np.uint8)


def _tq1_bytes(digits: np.ndarray) -> np.ndarray:
    """digits [..., 5] in {0,1,2}, most significant first -> encoded bytes [...]."""
    v = np.zeros(digits.shape[:-1], dtype=np.int64)
    for n in range(digits.shape[-1]):
        v = v * 3 + digits[..., n]
    return _TQ_ENCODE[v]


def make_weights(fmt, N: int, K: int, seed: int) -> np.ndarray:
    """Packed weight bytes for an N x K matrix, rows contiguous, as a flat uint8 array."""
    f = fmt_id(fmt)
    assert K % K_MULTIPLE[f] == 0 and N >= 1
    rng = np.random.default_rng(seed)
    if f == NVFP4:
        nib = rng.integers(0, 256, size=N * (K // 2), dtype=np.uint8)
        sc = _e4m3_bits(np.abs(rng.standard_normal(N * (K // 16))) * 0.05)
        return np.concatenate([nib, sc])
    bw, bb = BLOCK[f]
    nblk = N * (K // bw)
    out = np.empty((nblk, bb), dtype=np.uint8)
    if f in (Q4_K, Q5_K):
        _put_u16(out, 0, _fp16_bits(np.abs(rng.standard_normal(nblk)) * 1e-2))
        _put_u16(out, 2, _fp16_bits(np.abs(rng.standard_normal(nblk)) * 1e-2))
        # 12 uniform random bytes == 16 independent uniform 6-bit scales and mins.
        out[:, 4:bb] = rng.integers(0, 256, size=(nblk, bb - 4), dtype=np.uint8)
    elif f == Q6_K:
        out[:, 0:192] = rng.integers(0, 256, size=(nblk, 192), dtype=np.uint8)
        out[:, 192:208] = rng.integers(-32, 32, size=(nblk, 16)).astype(np.int8).view(np.uint8)
        _put_u16(out, 208, _fp16_bits(np.abs(rng.standard_normal(nblk)) * 1e-2))
    elif f == Q8_0:
        _put_u16(out, 0, _fp16_bits(np.abs(rng.standard_normal(nblk)) * 1e-2))
        out[:, 2:34] = rng.integers(0, 256, size=(nblk, 32), dtype=np.uint8)
    elif f == TQ1_0:
        qs_digits = rng.integers(0, 3, size=(nblk, 48, 5))
        qh_digits = rng.integers(0, 3, size=(nblk, 4, 5))
        qh_digits[..., 4] = 0  # the qh bytes carry four digits; the fifth position is empty
        out[:, 0:48] = _tq1_bytes(qs_digits)
        out[:, 48:52] = _tq1_bytes(qh_digits)
        _put_u16(out, 52, _fp16_bits(np.abs(rng.standard_normal(nblk)) * 1e-2))
    return out.reshape(-1)


def make_x(fmt, K: int, seed: int) -> np.ndarray:
    """Activation bits (uint16): fp16 N(0,1), or bf16 N(0,1) for NVFP4."""
    f = fmt_id(fmt)
    rng = np.random.default_rng(seed + 7919)
    v = rng.standard_normal(K)
    return _bf16_bits(v) if f == NVFP4 else _fp16_bits(v)


def x_dtype_name(fmt) -> str:
    return "bf16" if fmt_id(fmt) == NVFP4 else "fp16"


# Shapes of the benchmark configurations (name, fmt, N, K).
# Shape sets of the measured workloads (one entry per GEMV: name, format, N, K), by name.
SHAPE_SETS = {
    "q4k_1024x1024": [("q4k_1024x1024", Q4_K, 1024, 1024)],
    "q4k_llama8b_decode": [("q4k_qkv_6144x4096", Q4_K, 6144, 4096),
                           ("q4k_gateup_28672x4096", Q4_K, 28672, 4096),
                           ("q4k_down_4096x14336", Q4_K, 4096, 14336)],
    "nvfp4_llama8b": [("nvfp4_4096x14336", NVFP4, 4096, 14336),
                      ("nvfp4_14336x4096", NVFP4, 14336, 4096)],
    "tq1_0": [("tq1_0_4096x4096", TQ1_0, 4096, 4096),
              ("tq1_0_11008x4096", TQ1_0, 11008, 4096)],
}
# Decoder layer, hidden 4096, MLP 12288, 8 KV heads x 128.
LAYER_SHAPES = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
                ("gate", 12288, 4096), ("up", 12288, 4096), ("down", 4096, 12288)]
LAYER_MIXED = {"q": Q4_K, "k": Q5_K, "v": Q6_K, "o": Q8_0, "gate": Q4_K, "up": Q4_K, "down": Q6_K}
SHAPE_SETS["layer"] = [(f"layer_{p}_{FORMAT_NAMES[LAYER_MIXED[p]]}_{n}x{k}", LAYER_MIXED[p], n, k)
                       for p, n, k in LAYER_SHAPES]
# The same layer with every projection in every integer-code format (7 x 4 GEMVs).
LAYER_FORMATS = (Q4_K, Q5_K, Q6_K, Q8_0)
SHAPE_SETS["layer_every_format"] = [(f"layer_{p}_{FORMAT_NAMES[f]}_{n}x{k}", f, n, k)
                                    for p, n, k in LAYER_SHAPES for f in LAYER_FORMATS]


def shape_seed(set_name: str, shape_index: int) -> int:
    """Seed of the synthetic weights of entry `shape_index` of a shape set: 1000 per set (in the
    order above) plus the entry."""
    return 1000 * list(SHAPE_SETS).index(set_name) + shape_index
