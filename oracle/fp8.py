"""fp64 CPU oracle of the 8-bit floating-point contraction.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA path.

What the pages fix (nanochat hub page, pomoai.com, section "核心技术亮点",
FP8 mixed-precision training item): the latest version trains with 8-bit
floating point, halving the memory of the quantised tensors.  They name no
format, no scaling rule and no place in the model.

Readings, stated where used:

  * the operand format is E4M3 of the OCP 8-bit floating point specification
    (the format meant for forward-pass operands): a code is s.eeee.mmm with
    exponent bias 7; e = 0 encodes the subnormals (-1)^s 2^-6 (m / 8); e > 0
    encodes (-1)^s 2^(e-7) (1 + m / 8); there are no infinities and only
    s.1111.111 is NaN, so the largest finite magnitude is 2^8 * 1.75 = 448;
  * the contraction is C = scale * A . B^T with per-tensor dequantisation
    folded into one scalar; products of two E4M3 values are exact in fp32
    and the sum is the plain sum (here in fp64).
"""
from __future__ import annotations

import numpy as np

E4M3_BIAS = 7
E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of every E4M3 code (uint8 array) as float64; NaN codes give NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - E4M3_BIAS).astype(np.int64))
    sub = sign * np.ldexp(m / 8.0, 1 - E4M3_BIAS)
    out = np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, out)


def gemm_e4m3(a_codes: np.ndarray, b_codes: np.ndarray, scale: float) -> np.ndarray:
    """C = scale * decode(A) . decode(B)^T for A (M, K) and B (N, K) code arrays."""
    return float(scale) * (e4m3_decode(a_codes) @ e4m3_decode(b_codes).T)
