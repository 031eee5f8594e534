"""Pins for the fp64 GEMM oracle (oracle/gemm_ref.c) against facts that do not
come from the oracle itself: hand brute force, identity and permutation
matrices, exact integer sums, textbook values of the normal CDF, and torch's
own round-to-nearest-even bf16 conversion."""
import math
import random

import numpy as np
import pytest

from oracle import gemm as og


def _py_product(A, B):
    """Plain Python triple loop over lists of ints/floats (hand brute force)."""
    M, K, N = len(A), len(B), len(B[0])
    return [[sum(A[m][k] * B[k][n] for k in range(K)) for n in range(N)] for m in range(M)]


def test_one_by_one():
    C = og.gemm(np.array([[3.0]]), np.array([[-2.5]]))
    assert C.shape == (1, 1) and C[0, 0] == -7.5


def test_two_by_two_by_hand():
    A = np.array([[1.0, 2.0], [3.0, 4.0]])
    B = np.array([[5.0, 6.0], [7.0, 8.0]])
    # worked by hand: [[1·5+2·7, 1·6+2·8], [3·5+4·7, 3·6+4·8]]
    assert og.gemm(A, B).tolist() == [[19.0, 22.0], [43.0, 50.0]]


def test_three_five_seven_brute_force():
    rng = random.Random(7)
    A = [[rng.randint(-9, 9) for _ in range(5)] for _ in range(3)]
    B = [[rng.randint(-9, 9) for _ in range(7)] for _ in range(5)]
    want = _py_product(A, B)
    got = og.gemm(np.array(A, np.float32), np.array(B, np.float32))
    assert got.tolist() == [[float(v) for v in row] for row in want]


def test_identity_both_sides():
    rng = np.random.default_rng(1)
    B = rng.standard_normal((6, 9)).astype(np.float32)
    assert np.array_equal(og.gemm(np.eye(6, dtype=np.float32), B), B.astype(np.float64))
    assert np.array_equal(og.gemm(B, np.eye(9, dtype=np.float32)), B.astype(np.float64))


def test_permutation_matrices_permute_rows_and_columns():
    rng = np.random.default_rng(2)
    X = rng.standard_normal((7, 5)).astype(np.float32)
    p = rng.permutation(7)
    P = np.zeros((7, 7), np.float32)
    P[np.arange(7), p] = 1.0           # (P·X)[i] = X[p[i]]
    assert np.array_equal(og.gemm(P, X), X[p].astype(np.float64))
    q = rng.permutation(5)
    Q = np.zeros((5, 5), np.float32)
    Q[q, np.arange(5)] = 1.0           # (X·Q)[:, j] = X[:, q[j]]
    assert np.array_equal(og.gemm(X, Q), X[:, q].astype(np.float64))


def test_integer_inputs_are_exact_against_python_ints():
    rng = random.Random(3)
    M, K, N = 17, 129, 23
    A = [[rng.randint(-2, 2) for _ in range(K)] for _ in range(M)]
    B = [[rng.randint(-2, 2) for _ in range(N)] for _ in range(K)]
    bias = [rng.randint(-2, 2) for _ in range(N)]
    want = _py_product(A, B)
    got = og.gemm(np.array(A, np.float32), np.array(B, np.float32),
                  np.array(bias, np.float32), og.EPI_BIAS_RELU)
    for m in range(M):
        for n in range(N):
            assert got[m, n] == max(want[m][n] + bias[n], 0)


def test_bias_is_added_per_column_to_every_row():
    A = np.zeros((4, 3), np.float32)
    B = np.zeros((3, 5), np.float32)
    bias = np.arange(5, dtype=np.float32) - 2
    C = og.gemm(A, B, bias, og.EPI_BIAS)
    assert np.array_equal(C, np.tile(bias.astype(np.float64), (4, 1)))
    assert np.array_equal(og.gemm(A, B, bias, og.EPI_BIAS_RELU),
                          np.tile(np.maximum(bias, 0).astype(np.float64), (4, 1)))


def test_epilogue_none_ignores_bias():
    A = np.ones((2, 2), np.float32)
    B = np.ones((2, 2), np.float32)
    assert np.array_equal(og.gemm(A, B, np.full(2, 100, np.float32), og.EPI_NONE),
                          np.full((2, 2), 2.0))


@pytest.mark.parametrize("x,phi", [
    (0.0, 0.5),
    (1.0, 0.8413447460685429),     # textbook Φ(1)
    (-1.0, 0.15865525393145707),   # Φ(-1) = 1 - Φ(1)
    (2.0, 0.9772498680518208),     # Φ(2)
    (-3.0, 0.0013498980316300933), # Φ(-3)
])
def test_gelu_equals_x_times_normal_cdf(x, phi):
    C = og.gemm(np.array([[x]], np.float32), np.array([[1.0]], np.float32),
                np.array([0.0], np.float32), og.EPI_BIAS_GELU)
    assert C[0, 0] == pytest.approx(x * phi, rel=1e-14, abs=1e-300)


def test_gelu_limits():
    big = np.array([[30.0], [-30.0]], np.float32)
    C = og.gemm(big, np.array([[1.0]], np.float32), np.array([0.0], np.float32),
                og.EPI_BIAS_GELU)
    assert C[0, 0] == 30.0
    assert abs(C[1, 0]) < 1e-100


def test_entries_match_full_product_and_threads_do_not_matter():
    rng = np.random.default_rng(4)
    A = rng.standard_normal((37, 53)).astype(np.float32)
    B = rng.standard_normal((53, 29)).astype(np.float32)
    bias = rng.standard_normal(29).astype(np.float32)
    full1 = og.gemm(A, B, bias, og.EPI_BIAS_GELU, threads=1)
    full8 = og.gemm(A, B, bias, og.EPI_BIAS_GELU, threads=8)
    assert np.array_equal(full1, full8)
    rows = rng.integers(0, 37, 50)
    cols = rng.integers(0, 29, 50)
    ent = og.gemm_entries(A, B, bias, og.EPI_BIAS_GELU, rows, cols)
    assert np.array_equal(ent, full1[rows, cols])


def test_numpy_fp64_matmul_agrees_to_rounding():
    # a library routine as an independent check of the summation itself
    rng = np.random.default_rng(5)
    A = rng.standard_normal((64, 300)).astype(np.float32)
    B = rng.standard_normal((300, 48)).astype(np.float32)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    assert np.abs(og.gemm(A, B) - ref).max() < 1e-11


def test_empty_extents():
    assert og.gemm(np.zeros((0, 4), np.float32), np.zeros((4, 3), np.float32)).shape == (0, 3)
    C = og.gemm(np.zeros((2, 0), np.float32), np.zeros((0, 3), np.float32),
                np.array([1.0, -1.0, 0.5], np.float32), og.EPI_BIAS_RELU)
    assert C.tolist() == [[1.0, 0.0, 0.5]] * 2


def test_bf16_round_to_nearest_even_known_points():
    one_ulp = 2.0 ** -7
    vals = [1.0, 1.0 + one_ulp / 2, 1.0 + 1.5 * one_ulp, -2.0, 0.0, 3.0e38, 1e-45]
    bits = og.round_bf16_bits(vals)
    assert bits[0] == 0x3F80
    assert bits[1] == 0x3F80           # tie -> even (mantissa 0)
    assert bits[2] == 0x3F82           # tie -> even (mantissa 2)
    assert bits[3] == 0xC000
    assert bits[4] == 0x0000
    v5 = og.bf16_bits_to_f64([bits[5]])[0]  # within half an ulp (2^-8 relative) of 3e38
    assert abs(v5 - 3.0e38) <= 3.0e38 * 2.0 ** -8
    assert bits[6] == 0x0000           # far below the smallest bf16 subnormal 2^-133
    assert og.round_bf16_bits([3.5e38])[0] == 0x7F80   # past the largest finite: +inf


def test_bf16_rounding_agrees_with_torch():
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(6)
    x = (torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 8))
    x = x.to(torch.float32)
    ours = og.round_bf16_bits(x.double().numpy())
    theirs = x.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(ours, theirs)


def test_normalised_error_metric():
    A = np.array([[3.0, 4.0]], np.float32)       # ||a|| = 5
    B = np.array([[1.0], [0.0]], np.float32)     # ||b|| = 1
    assert og.normalised_error(np.array([[0.5]]), np.array([[0.0]]), A, B) == pytest.approx(0.1)


def test_planted_mistakes_are_caught():
    """Each plausible slip in a product routine fails one of the pins above."""
    A = np.array([[1.0, 2.0], [3.0, 4.0]])
    B = np.array([[5.0, 6.0], [7.0, 8.0]])
    hand = [[19.0, 22.0], [43.0, 50.0]]
    transposed_b = (A @ B.T).tolist()
    dropped_last_k = (A[:, :1] @ B[:1, :]).tolist()
    wrong_sign = (A @ (-B)).tolist()
    for wrong in (transposed_b, dropped_last_k, wrong_sign):
        assert wrong != hand
    assert math.isclose(0.5 * 1.0 * (1 + math.erf(1 / math.sqrt(2))), 0.8413447460685429)
    tanh_gelu = 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * (1 + 0.044715)))
    assert abs(tanh_gelu - 0.8413447460685429) > 1e-5


def test_e4m3_decode_from_its_definition_matches_torch_for_every_code():
    import torch
    from oracle import fp8
    table = fp8.e4m3_table()
    # hand values of the format: 1.0, -2.0, the largest finite 448, the smallest
    # subnormal 2^-9, the largest subnormal 7/8·2^-6, the smallest normal 2^-6
    assert table[0x38] == 1.0 and table[0xC0] == -2.0 and table[0x7E] == 448.0
    assert table[0x01] == 2.0 ** -9 and table[0x07] == 7 / 8 * 2.0 ** -6 and table[0x08] == 2.0 ** -6
    assert np.isnan(table[0x7F]) and np.isnan(table[0xFF]) and table[0x80] == 0.0
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    same = (table == ref) | (np.isnan(table) & np.isnan(ref))
    assert same.all(), np.nonzero(~same)
    # 254 finite values, symmetric, strictly increasing over the positive codes
    pos = table[:0x7F]
    assert np.all(np.diff(pos) > 0) and np.array_equal(table[0x80:0xFF], -pos)


def test_alpha_scales_the_product_before_bias_and_activation():
    rng = np.random.default_rng(3)
    A = rng.integers(-3, 4, size=(5, 7)).astype(np.float32)
    B = rng.integers(-3, 4, size=(7, 6)).astype(np.float32)
    bias = rng.integers(-2, 3, size=6).astype(np.float32)
    exact = A.astype(np.float64) @ B.astype(np.float64)
    for alpha in (1.0, 0.5, -0.25, 3.0):
        got = og.gemm(A, B, bias, og.EPI_BIAS_RELU, alpha=alpha)
        assert np.array_equal(got, np.maximum(alpha * exact + bias, 0.0))
        ent = og.gemm_entries(A, B, bias, og.EPI_BIAS_RELU, [0, 4], [5, 0], alpha=alpha)
        assert np.array_equal(ent, got[[0, 4], [5, 0]])


def test_fp8_operands_reach_the_oracle_as_their_decoded_values():
    import torch
    from autotuning_tcgen05_tmem_gb300 import inputs
    A, B, bias = inputs.make_operands(9, 10, 11, "fp8", "int", seed=1)
    assert A.dtype == torch.float8_e4m3fn and bias.dtype == torch.bfloat16
    Af = A.to(torch.float32).numpy().astype(np.float64)
    Bf = B.to(torch.float32).numpy().astype(np.float64)
    assert np.array_equal(og.gemm(A, B, None, og.EPI_NONE), Af @ Bf)
