"""Helpers for the GPU tests: upload seeded inputs, run through the C-ABI, compare."""
import numpy as np
import torch

import oracle
from quantized_weight_dequant_gb300 import qgemv, synth

RTOL = 2e-3   # |y - y_ref| <= 2e-3 * sum|x w| + 1e-5 per output
ATOL = 1e-5


def dev_bytes(a: np.ndarray, pad_front: int = 0, pad_back: int = 0, fill: int = 0xA5):
    """uint8 device tensor holding `a` (optionally inside poisoned padding); returns (view, base)."""
    base = torch.full((pad_front + a.size + pad_back,), fill, dtype=torch.uint8, device="cuda")
    view = base[pad_front:pad_front + a.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)).cuda())
    return view, base


def dev_x(x_bits: np.ndarray):
    return torch.from_numpy(x_bits.view(np.int16).copy()).cuda()


def run_gemv(h, fmt, x_dev, W_dev, N, K, y=None):
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device="cuda")
    qgemv.run(h, fmt, x_dev, W_dev, N, K, y)
    return y


def assert_parity(y_gpu: np.ndarray, y_ref: np.ndarray, S: np.ndarray, what: str = ""):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    bound = RTOL * S + ATOL
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{what}: {bad.size} outputs out of tolerance, first {bad[:5]}, "
                           f"err {err[bad[:5]]}, bound {bound[bad[:5]]}")


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    rows = set([0, N - 1, N // 2]) | set(rng.integers(0, N, size=min(count, N)).tolist())
    return np.array(sorted(rows), dtype=np.int64)
