"""Pins of the gated (GLU-style dual-output) oracle, oracle/gemm.py: glu().

C = act(A·B_gate + b_gate) ⊙ (A·B_up + b_up) over a fused gate+up weight whose
columns alternate in blocks of 32 ("Tiling the hierarchy", fusion: the
elementwise chain after a product is fused onto it; "CuTile Autotuning": fused
dual-GEMM kernels, Linear + GLU activation).  Pinned by a brute-force loop
from the definition, by its reduction to the plain GEMM oracle, by the column
mapping of the fused layout, by closed forms of SiLU and by exact integer
ReGLU; planted mistakes (gate and up swapped, a 64-column block) must fail."""
import math

import numpy as np
import pytest

from oracle import gemm as og


def _brute(A, B, bias, epi):
    """Triple loop from the definition, in Python floats (fp64)."""
    M, K = A.shape
    N = B.shape[1]
    out = np.zeros((M, N // 2))
    for i in range(M):
        for o in range(N // 2):
            gc = 64 * (o // 32) + o % 32
            uc = gc + 32
            g = sum(float(A[i, k]) * float(B[k, gc]) for k in range(K)) + float(bias[gc])
            u = sum(float(A[i, k]) * float(B[k, uc]) for k in range(K)) + float(bias[uc])
            if epi == og.EPI_BIAS_REGLU:
                a = max(g, 0.0)
            elif epi == og.EPI_BIAS_GEGLU:
                a = 0.5 * g * (1.0 + math.erf(g / math.sqrt(2.0)))
            else:
                a = g / (1.0 + math.exp(-g))
            out[i, o] = a * u
    return out


def _rand(M, N, K, seed):
    r = np.random.default_rng(seed)
    return (r.uniform(-1, 1, (M, K)).astype(np.float32), r.uniform(-1, 1, (K, N)).astype(np.float32),
            r.uniform(-1, 1, N).astype(np.float32))


@pytest.mark.parametrize("epi", og.GLU_EPILOGUES)
def test_glu_equals_a_brute_force_loop(epi):
    A, B, bias = _rand(3, 128, 5, 1)
    got = og.glu(A, B, bias, epi)
    assert got.shape == (3, 64)
    assert np.allclose(got, _brute(A, B, bias, epi), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("epi,plain", [(og.EPI_BIAS_REGLU, og.EPI_BIAS_RELU), (og.EPI_BIAS_GEGLU, og.EPI_BIAS_GELU)])
def test_glu_with_a_unit_up_path_is_the_plain_oracle(epi, plain):
    """Up weights 0 and up bias 1: C = act(A·B_gate + b_gate), the plain oracle's
    activation of the gate columns alone."""
    A, B, bias = _rand(7, 192, 33, 2)
    o = np.arange(96)
    gate = 64 * (o // 32) + o % 32          # the layout, written out here
    up = gate + 32
    B[:, up] = 0.0
    bias[up] = 1.0
    want = og.gemm(A, np.ascontiguousarray(B[:, gate]), bias[gate], plain)
    # (scipy's erf against the C library's: the same function, last-bit differences)
    assert np.allclose(og.glu(A, B, bias, epi), want, rtol=1e-14, atol=1e-300)


def test_glu_output_column_mapping():
    """A = I: C[i, o] = act(B[i, gate(o)] + bg)·(B[i, up(o)] + bu); the fused
    columns carry their own index, so each output picks the right pair."""
    N = 256
    K = 4
    A = np.eye(K, dtype=np.float32)
    B = np.tile(np.arange(N, dtype=np.float32), (K, 1))
    bias = np.zeros(N, dtype=np.float32)
    got = og.glu(A, B, bias, og.EPI_BIAS_REGLU)
    o = np.arange(N // 2)
    g = 64 * (o // 32) + o % 32
    assert np.array_equal(got[0], g * (g + 32.0))
    gate, up = og.glu_columns(N)
    assert np.array_equal(gate, g) and np.array_equal(up, g + 32)
    assert sorted(np.concatenate([gate, up]).tolist()) == list(range(N))


def test_silu_closed_forms():
    x = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 2.5])
    s = og.glu_act(x, og.EPI_BIAS_SWIGLU)
    assert s[0] == 0.0
    assert s[1] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), rel=1e-15)
    assert s[2] == pytest.approx(-1.0 / (1.0 + math.e), rel=1e-15)
    assert s[3] == pytest.approx(40.0, rel=1e-15) and abs(s[4]) < 1e-15
    assert s[5] - s[5] * 0 == pytest.approx(2.5 / (1 + math.exp(-2.5)), rel=1e-15)
    gl = og.glu_act(np.array([0.0, 1.0, -1.0]), og.EPI_BIAS_GEGLU)
    assert gl[0] == 0.0 and gl[1] == pytest.approx(0.8413447460685429, rel=1e-14)   # Φ(1)
    assert gl[2] == pytest.approx(-0.15865525393145707, rel=1e-14)                   # -Φ(-1)


def test_reglu_is_exact_on_small_integers():
    r = np.random.default_rng(3)
    A = r.integers(-2, 3, (9, 40)).astype(np.float32)
    B = r.integers(-2, 3, (40, 128)).astype(np.float32)
    bias = r.integers(-2, 3, 128).astype(np.float32)
    got = og.glu(A, B, bias, og.EPI_BIAS_REGLU)
    Ai, Bi, bi = A.astype(int), B.astype(int), bias.astype(int)
    gate, up = og.glu_columns(128)
    want = np.maximum(Ai @ Bi[:, gate] + bi[gate], 0) * (Ai @ Bi[:, up] + bi[up])
    assert np.array_equal(got, want.astype(np.float64))


def test_glu_entries_match_the_full_result():
    A, B, bias = _rand(11, 320, 17, 4)
    full = og.glu(A, B, bias, og.EPI_BIAS_GEGLU)
    rows, cols = [0, 5, 10, 3], [0, 31, 32, 159]
    assert np.allclose(og.gemm_entries(A, B, bias, og.EPI_BIAS_GEGLU, rows, cols), full[rows, cols],
                       rtol=1e-14, atol=1e-15)


def test_glu_pins_catch_swapped_gate_and_up(monkeypatch):
    real = og.glu_columns
    monkeypatch.setattr(og, "glu_columns", lambda N: tuple(reversed(real(N))))
    with pytest.raises(AssertionError):
        test_glu_with_a_unit_up_path_is_the_plain_oracle(og.EPI_BIAS_REGLU, og.EPI_BIAS_RELU)


def test_glu_pins_catch_a_wrong_block_size(monkeypatch):
    monkeypatch.setattr(og, "GLU_BLOCK", 64)
    with pytest.raises((AssertionError, ValueError)):
        test_glu_output_column_mapping()
