"""Oracle for block-scaled FP8 (MXFP8, E4M3 elements with E8M0 block scales).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py.  The product package never imports it.

What it follows.  The pages name FP8 only as a tensor-core input type; the
block-scaled form is the OCP "Microscaling Formats (MX) Specification" v1.0:
  * an MX block is 32 consecutive elements sharing one scale (section 5, the
    MXFP8 rows of its format table: E4M3 elements, block size 32, E8M0 scale);
  * E8M0 (section 5.4): an unsigned 8-bit exponent with bias 127, no sign and no
    mantissa: code x means 2^(x - 127); 0xFF is NaN;
  * the value of element i of a block is scale · element (section 5.2), so the
    dot product of two MX vectors is the plain dot product of those values.
For the GEMM C = act(alpha·A·B + bias) (+ R) the blocks run along K: A's scale
SA[m, k // 32] multiplies A[m, k] and B's scale SB[k // 32, n] multiplies
B[k, n] (reading taken: scales keep their operand's orientation with K divided
by 32; a ragged last block of K keeps its scale).

Everything is fp64: the dequantized values (E4M3 value · 2^(s-127)) are exact in
fp64 for every code pair, the product is numpy's fp64 matrix product (a library
primitive), and the epilogue is the same elementwise chain as the plain oracle
(bias over rows, ReLU, erf GELU, then + R).
"""
from __future__ import annotations

import math

import numpy as np

from . import fp8

BLOCK = 32
EPI_NONE, EPI_BIAS, EPI_BIAS_RELU, EPI_BIAS_GELU = 0, 1, 2, 3


def e8m0_decode(code: int) -> float:
    """Value of one E8M0 scale byte: 2^(code - 127); NaN for 0xFF."""
    code &= 0xFF
    if code == 0xFF:
        return math.nan
    return math.ldexp(1.0, code - 127)


def e8m0_table() -> np.ndarray:
    return np.array([e8m0_decode(c) for c in range(256)], dtype=np.float64)


def _codes(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach().cpu().contiguous()
            if t.dtype != torch.uint8:
                t = t.view(torch.uint8)
            return t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.uint8)


def kblocks(K: int) -> int:
    return (K + BLOCK - 1) // BLOCK


def dequantize_a(A_codes, SA) -> np.ndarray:
    """fp64 A[m, k] · 2^(SA[m, k // 32] - 127) for E4M3 codes A [M, K] and
    scales SA [M, ceil(K/32)]."""
    a = fp8.decode_codes(_codes(A_codes)).astype(np.float64)
    s = e8m0_table()[_codes(SA)]
    M, K = a.shape
    if s.shape != (M, kblocks(K)):
        raise ValueError(f"SA must be [{M}, {kblocks(K)}], got {s.shape}")
    return a * s[:, np.arange(K) // BLOCK]


def dequantize_b(B_codes, SB) -> np.ndarray:
    """fp64 B[k, n] · 2^(SB[k // 32, n] - 127) for E4M3 codes B [K, N] and
    scales SB [ceil(K/32), N]."""
    b = fp8.decode_codes(_codes(B_codes)).astype(np.float64)
    s = e8m0_table()[_codes(SB)]
    K, N = b.shape
    if s.shape != (kblocks(K), N):
        raise ValueError(f"SB must be [{kblocks(K)}, {N}], got {s.shape}")
    return b * s[np.arange(K) // BLOCK, :]


def _epilogue(x: np.ndarray, bias, epi: int) -> np.ndarray:
    act = epi - 3 if epi >= 4 else epi
    if act == EPI_NONE:
        return x
    x = x + _vec(bias)[None, :]
    if act == EPI_BIAS_RELU:
        return np.maximum(x, 0.0)
    if act == EPI_BIAS_GELU:
        erf = np.vectorize(math.erf, otypes=[np.float64])
        return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))
    return x


def _vec(v) -> np.ndarray:
    try:
        import torch
        if isinstance(v, torch.Tensor):
            return v.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(v, dtype=np.float64)


def mx_gemm(A, SA, B, SB, bias=None, epi: int = EPI_NONE, alpha: float = 1.0, residual=None) -> np.ndarray:
    """fp64 C = act(alpha·deq(A)·deq(B) + bias) (+ R for epilogues 4..6)."""
    if epi != EPI_NONE and bias is None:
        raise ValueError("the epilogue needs a bias")
    C = alpha * (dequantize_a(A, SA) @ dequantize_b(B, SB))
    C = _epilogue(C, bias, epi)
    if epi >= 4:
        if residual is None:
            raise ValueError("the residual epilogue needs R")
        C = C + _vec(residual)
    return C


def mx_gemm_entries(A, SA, B, SB, bias, epi: int, rows, cols, alpha: float = 1.0, residual=None) -> np.ndarray:
    """fp64 values of C at (rows[i], cols[i]), one dot product of a dequantized
    row of A and column of B each (for full-size checks)."""
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    a_codes, b_codes = _codes(A), _codes(B)
    sa, sb = _codes(SA), _codes(SB)
    out = np.empty(rows.shape[0], dtype=np.float64)
    bvec = _vec(bias) if bias is not None else None
    rvec = _vec(residual) if residual is not None else None
    for i, (m, n) in enumerate(zip(rows, cols)):
        arow = dequantize_a(a_codes[m:m + 1], sa[m:m + 1])[0]
        bcol = dequantize_b(b_codes[:, n:n + 1], sb[:, n:n + 1])[:, 0]
        x = alpha * float(np.dot(arow, bcol))
        act = epi - 3 if epi >= 4 else epi
        if act != EPI_NONE:
            x += float(bvec[n])
            if act == EPI_BIAS_RELU:
                x = max(x, 0.0)
            elif act == EPI_BIAS_GELU:
                x = 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0)))
        if epi >= 4:
            x += float(rvec[m, n])
        out[i] = x
    return out
