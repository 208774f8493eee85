"""Helpers shared by the GPU parity tests: device transfers, the row-relative error of the W4A16
tolerance, the rows at which tiled outputs are compared, and poisoned output buffers with guard
bands (an output element a kernel never writes stays poison, a write past either end of the output
lands in a guard band).
"""
from __future__ import annotations

import numpy as np
import torch

# the fp16 tolerance of the W4A16 and fp16 W8A8 outputs: max over rows of ||y - y_ref|| / ||y_ref||
ROW_TOL = 1e-2

_POISON = {
    torch.float16: 0x7E00,      # quiet NaN
    torch.float32: 0x7FC00000,  # quiet NaN
    torch.int32: 0x7F7F7F7F,    # beyond any int32 accumulator of K <= 2^17 int8 products
    torch.int8: 0x5A,
    torch.uint8: 0x5A,
}
_INT_VIEW = {torch.float16: torch.int16, torch.float32: torch.int32, torch.int32: torch.int32,
             torch.int8: torch.int8, torch.uint8: torch.uint8}


def dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def row_rel_err(y, ref) -> float:
    y = np.asarray(y, dtype=np.float64)
    num = np.linalg.norm(y - ref, axis=1)
    den = np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    return float((num / den).max())


def tile_rows(M: int, block: int = 32) -> np.ndarray:
    """The first and last row of every `block`-row block of M rows (and row M - 1): every token tile
    of the tiled kernels (32, 64, 128 or 256 rows, all aligned to multiples of 32) starts and ends at
    one of them."""
    r = np.arange(0, M, block, dtype=np.int64)
    return np.unique(np.concatenate([r, np.minimum(r + block - 1, M - 1), [M - 1]]))


class Guarded:
    """A contiguous output tensor of `shape` inside a larger allocation, with `band` elements of
    guard on each side; the whole allocation starts filled with a poison pattern (NaN for floating
    point, 0x7F7F7F7F for int32).  `t` is the tensor to pass as the output; `check()` asserts that
    both guard bands are untouched."""

    def __init__(self, shape, dtype, band: int = 4096):
        n = int(np.prod(shape)) if len(shape) else 1
        self.band, self.n, self.dtype = band, n, dtype
        self.buf = torch.empty((n + 2 * band,), dtype=dtype, device="cuda")
        pat = _POISON[dtype]
        iv = _INT_VIEW[dtype]
        if iv == torch.int16 and pat >= 0x8000:
            pat -= 0x10000
        self.buf.view(iv).fill_(pat)
        self.poison = pat
        self.t = self.buf[band:band + n].view(shape)

    def check(self):
        iv = _INT_VIEW[self.dtype]
        lo = self.buf[:self.band].view(iv)
        hi = self.buf[self.band + self.n:].view(iv)
        torch.cuda.synchronize()
        assert bool((lo == self.poison).all()), "a kernel wrote below the start of its output"
        assert bool((hi == self.poison).all()), "a kernel wrote past the end of its output"

    def unwritten(self) -> int:
        """How many output elements still hold the poison pattern."""
        torch.cuda.synchronize()
        return int((self.t.view(_INT_VIEW[self.dtype]) == self.poison).sum().item())
