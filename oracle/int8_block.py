"""INT8 optimizer states with one absmax scale per block of 64 elements.

FORGE summary, §2 Precision and fidelity, third low-precision point: INT8
optimizer states use blocks of 64 elements (instead of the 2048 of common 8-bit
optimizers) to lower the quantisation error.  The summary fixes only the block
length; the rest is our plainest reading:

* a block is 64 consecutive elements of one weight row (d_in % 64 == 0);
* the code is signed symmetric linear: scale s = absmax / 127 (binary32, IEEE
  division), code q = clamp(rne(x / s), -127, 127) with x / s a binary32 IEEE
  division and rne round-half-to-even; a block whose absmax is 0 gets s = 0 and
  all codes 0;
* dequantisation is the binary32 product q * s;
* m and v use the same code (v >= 0, so its codes are 0..127).

The quantisation decision is taken in binary32, the precision the kernel takes
it in, so that both sides map equal inputs to equal codes.

Pinned by: round-trip error <= s/2, the absmax element mapping to +-127, the
all-zero block, and a brute-force nearest-code search (tests/test_oracle_int8.py).
"""
from __future__ import annotations

import numpy as np

BLOCK = 64
QMAX = 127


def quantize(x) -> tuple:
    """binary32 values of shape (..., 64k) -> (int8 codes, binary32 scales of shape (..., k))."""
    x = np.asarray(x, dtype=np.float32)
    blocks = x.reshape(x.shape[:-1] + (x.shape[-1] // BLOCK, BLOCK))
    absmax = np.max(np.abs(blocks), axis=-1)
    s = (absmax / np.float32(QMAX)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    ratio = (blocks / safe[..., None]).astype(np.float32)
    q = np.clip(np.rint(ratio), -QMAX, QMAX)
    q = np.where((s > 0)[..., None], q, 0).astype(np.int8)
    return q.reshape(x.shape), s


def dequantize(q, s) -> np.ndarray:
    """int8 codes (..., 64k) and binary32 scales (..., k) -> binary32 values."""
    q = np.asarray(q, dtype=np.int8)
    s = np.asarray(s, dtype=np.float32)
    blocks = q.reshape(q.shape[:-1] + (q.shape[-1] // BLOCK, BLOCK)).astype(np.float32)
    return (blocks * s[..., None]).astype(np.float32).reshape(q.shape)
