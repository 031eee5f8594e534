"""Pins of the block-scaled FP8 oracle (oracle/mx.py) to what the MX format's
definition fixes, checked against things other than the oracle itself: the
E8M0 code table of the OCP MX specification, the plain-GEMM oracle (C, pinned
on its own) on operands whose values are built as element · 2^scale block by
block, exact invariances of power-of-two scales, and NaN propagation."""
import math

import numpy as np
import pytest
import torch

from autotuning_tcgen05_tmem_gb300 import inputs
from oracle import fp8
from oracle import gemm as og
from oracle import mx


@pytest.mark.parametrize("code,value", [(127, 1.0), (128, 2.0), (126, 0.5), (0, 2.0 ** -127), (254, 2.0 ** 127),
                                        (131, 16.0), (120, 1.0 / 128)])
def test_e8m0_codes(code, value):
    assert mx.e8m0_decode(code) == value


def test_e8m0_nan_code():
    assert math.isnan(mx.e8m0_decode(255))
    t = mx.e8m0_table()
    assert np.isnan(t[255]) and np.all(np.isfinite(t[:255]))
    assert np.all(t[1:255] == 2 * t[0:254])            # each code doubles the last


def _codes(shape, rng, lo=-6, hi=6):
    """E4M3 codes of small normal values: sign, exponent field lo+7..hi+7, mantissa."""
    s = rng.integers(0, 2, size=shape)
    e = rng.integers(lo + 7, hi + 8, size=shape)
    m = rng.integers(0, 8, size=shape)
    return ((s << 7) | (e << 3) | m).astype(np.uint8)


def test_unit_scales_give_the_plain_fp8_product():
    rng = np.random.default_rng(1)
    M, N, K = 7, 9, 70
    A, B = _codes((M, K), rng), _codes((K, N), rng)
    SA = np.full((M, mx.kblocks(K)), 127, np.uint8)
    SB = np.full((mx.kblocks(K), N), 127, np.uint8)
    want = og.gemm(fp8.decode_codes(A), fp8.decode_codes(B))
    got = mx.mx_gemm(A, SA, B, SB)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=0)


@pytest.mark.parametrize("K", [32, 64, 40, 100, 1])
def test_block_scales_act_on_their_32_elements_of_k(K):
    """The value of an MX operand is element · 2^(scale - 127) with the scale of
    the element's 32-block along K; build those values directly (fp32 holds them
    exactly here) and compare with the plain oracle.  A wrong block index (k % 32,
    k // 16), a transposed SB, or a missing scale fails this."""
    rng = np.random.default_rng(K)
    M, N = 5, 6
    kb = mx.kblocks(K)
    A, B = _codes((M, K), rng, -3, 3), _codes((K, N), rng, -3, 3)
    ea = rng.integers(-5, 6, size=(M, kb))
    eb = rng.integers(-5, 6, size=(kb, N))
    Av = np.empty((M, K), np.float32)
    Bv = np.empty((K, N), np.float32)
    for m in range(M):
        for k in range(K):
            Av[m, k] = np.ldexp(fp8.e4m3_decode(int(A[m, k])), int(ea[m, k // 32]))
    for k in range(K):
        for n in range(N):
            Bv[k, n] = np.ldexp(fp8.e4m3_decode(int(B[k, n])), int(eb[k // 32, n]))
    bias = np.linspace(-1, 1, N).astype(np.float32)
    want = og.gemm(Av, Bv, bias, og.EPI_BIAS_GELU, alpha=0.5)
    got = mx.mx_gemm(A, (127 + ea).astype(np.uint8), B, (127 + eb).astype(np.uint8), bias, mx.EPI_BIAS_GELU,
                     alpha=0.5)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-300)


def test_moving_a_factor_of_two_between_a_and_b_blocks_changes_nothing():
    rng = np.random.default_rng(7)
    M, N, K = 6, 5, 96
    A, B = _codes((M, K), rng), _codes((K, N), rng)
    SA = rng.integers(120, 135, size=(M, 3)).astype(np.uint8)
    SB = rng.integers(120, 135, size=(3, N)).astype(np.uint8)
    base = mx.mx_gemm(A, SA, B, SB)
    SA2, SB2 = SA.copy(), SB.copy()
    SA2[:, 1] += 1            # × 2 on every row's block 1 ...
    SB2[1, :] -= 1            # ... ÷ 2 on every column's block 1
    assert np.array_equal(mx.mx_gemm(A, SA2, B, SB2), base)
    SA3 = SA.copy()
    SA3[2, :] += 3            # one row's scales × 8 scale that row of C by 8, exactly
    out = mx.mx_gemm(A, SA3, B, SB)
    assert np.array_equal(out[2], 8 * base[2]) and np.array_equal(np.delete(out, 2, 0), np.delete(base, 2, 0))


def test_nan_scale_poisons_exactly_its_row_and_column():
    rng = np.random.default_rng(3)
    M, N, K = 4, 5, 64
    A, B = _codes((M, K), rng), _codes((K, N), rng)
    SA = np.full((M, 2), 127, np.uint8)
    SB = np.full((2, N), 127, np.uint8)
    SA[1, 0] = 255
    SB[1, 3] = 255
    out = mx.mx_gemm(A, SA, B, SB)
    nan = np.isnan(out)
    assert nan[1].all() and nan[:, 3].all() and nan.sum() == N + M - 1


def test_entries_equal_the_full_product_and_residual():
    A, SA, B, SB, bias = inputs.make_mx_operands(40, 48, 200, "scaled_normal", seed=5)
    R = inputs.make_residual(40, 48, "mxfp8", "scaled_normal", seed=5)
    full = mx.mx_gemm(A, SA, B, SB, bias, 6, alpha=1.25, residual=R)
    rows = [0, 39, 17, 5]
    cols = [0, 47, 3, 30]
    ent = mx.mx_gemm_entries(A, SA, B, SB, bias, 6, rows, cols, alpha=1.25, residual=R)
    np.testing.assert_allclose(ent, full[rows, cols], rtol=1e-12)


def test_integer_inputs_are_exact_quarters():
    """With elements in [-2, 2] and scales 2^-1..2^1 every product is a multiple
    of 1/4, and so is every sum: the case the device must match bit for bit."""
    A, SA, B, SB, bias = inputs.make_mx_operands(33, 40, 300, "int", seed=9)
    assert A.dtype == torch.float8_e4m3fn and SA.dtype == torch.uint8 and SA.shape == (33, 10)
    assert SB.shape == (10, 40) and set(np.unique(SA.numpy())) <= {126, 127, 128}
    C = mx.mx_gemm(A, SA, B, SB)
    assert np.array_equal(C * 4, np.round(C * 4)) and np.abs(C).max() < 2 ** 20
