"""Gated (GLU-style dual-output) epilogues on the GPU, through the C ABI.

C [M, N/2] = act(A·B_gate + b_gate) ⊙ (A·B_up + b_up) over a fused gate+up
weight B [K, N] whose 32-column gate and up blocks alternate ("Tiling the
hierarchy", fusion; "CuTile Autotuning": fused dual-GEMM kernels, Linear + GLU
activation).  ReGLU on small integers is exact (each product below 2^24), so
the bits must equal the oracle's; GeGLU and SwiGLU are compared with the fp64
oracle within the error of the two dot products and the output's rounding."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import device_bits, operands
from oracle import gemm as og

pytestmark = pytest.mark.gpu

C = g.make_config
GLU = {"reglu": og.EPI_BIAS_REGLU, "geglu": og.EPI_BIAS_GEGLU, "swiglu": og.EPI_BIAS_SWIGLU}


def _run(A, B, bias, epi, cfg=None, dtype="bf16"):
    M, K = A.shape
    N = B.shape[1]
    out_dt = torch.float32 if dtype == "fp32" else torch.bfloat16
    buf = torch.full((M * (N // 2) + 128,), 777.0, dtype=out_dt, device="cuda")
    Cd = buf[64:64 + M * (N // 2)].view(M, N // 2)
    p = g.plan_with_config(M, N, K, dtype, epi, cfg) if cfg is not None else g.plan(M, N, K, dtype, epi)
    with p:
        p.run(A.cuda(), B.cuda(), bias.cuda(), Cd)
        assert p.status() == 0, g.last_error()
        used = p.config
    assert (buf[:64] == 777.0).all() and (buf[64 + M * (N // 2):] == 777.0).all()   # nothing written outside C
    return Cd.cpu(), used


def _within_tolerance(Cd, A, B, bias, epi):
    """|C - C_ref| <= 2^-7·|C_ref| + 2e-3·(||a_i||·(||b_gate||·max(1, |U|) + ||b_up||·max(1, |act(G)|)))."""
    ref = og.gemm(A, B, bias, GLU[epi])
    Af = og._as_f32_input(A).astype(np.float64)
    Bf = og._as_f32_input(B).astype(np.float64)
    bf = og._as_f32_input(bias).astype(np.float64)
    gate, up = og.glu_columns(Bf.shape[1])
    G = Af @ Bf[:, gate] + bf[gate]
    U = Af @ Bf[:, up] + bf[up]
    ra = np.sqrt((Af * Af).sum(axis=1))[:, None]
    sg = np.sqrt((Bf[:, gate] ** 2).sum(axis=0))[None, :]
    su = np.sqrt((Bf[:, up] ** 2).sum(axis=0))[None, :]
    scale = ra * (sg * np.maximum(1, np.abs(U)) + su * np.maximum(1, np.abs(og.glu_act(G, GLU[epi]))))
    err = np.abs(Cd.double().numpy() - ref)
    return float((err / (2.0 ** -7 * np.abs(ref) + 2e-3 * scale)).max())


CASES = [
    ((300, 320, 520), C(128, 128, 64, 4)),            # 128 x 128: two gate/up block pairs per tile
    ((257, 384, 1000), C(128, 192, 64, 4)),           # three pairs per tile, ragged M and K
    ((200, 512, 264), C(256, 256, 64, 2)),            # two stacked MMAs, four pairs
    ((300, 256, 520), C(128, 64, 64, 4, 1, 4)),       # one pair per tile, raster 1
    ((1000, 1024, 1000), C(256, 256, 128, 3, 0, 1, 1, 2)),   # CTA pair
    ((300, 384, 520), C(256, 128, 64, 4, 0, 1, 1, 2)),       # CTA pair, bn 128
]


@pytest.mark.parametrize("shape,cfg", CASES, ids=lambda x: "x".join(map(str, x)) if isinstance(x, tuple)
                         else "x".join(map(str, x.astuple())))
def test_reglu_bit_exact_on_integer_inputs(shape, cfg):
    M, N, K = shape
    A, B, bias = operands(M, N, K, "bf16", "int", seed=51)
    got, _ = _run(A, B, bias, "reglu", cfg)
    assert np.array_equal(device_bits(got), og.round_bf16_bits(og.gemm(A, B, bias, og.EPI_BIAS_REGLU)))


@pytest.mark.parametrize("dtype,cfg", [("fp32", C(128, 128, 32, 4)), ("fp8", C(128, 128, 128, 4))])
def test_reglu_bit_exact_other_dtypes(dtype, cfg):
    M, N, K = 200, 256, 256
    A, B, bias = operands(M, N, K, dtype, "int", seed=52)
    got, _ = _run(A, B, bias, "reglu", cfg, dtype)
    ref = og.gemm(A, B, bias, og.EPI_BIAS_REGLU)
    want = og.round_f32(ref).view(np.uint32) if dtype == "fp32" else og.round_bf16_bits(ref)
    assert np.array_equal(device_bits(got), want)


@pytest.mark.parametrize("epi", ["geglu", "swiglu"])
@pytest.mark.parametrize("shape,cfg", CASES[:3] + CASES[4:5], ids=lambda x: "x".join(map(str, x))
                         if isinstance(x, tuple) else "x".join(map(str, x.astuple())))
def test_gated_random_within_tolerance(epi, shape, cfg):
    M, N, K = shape
    A, B, bias = operands(M, N, K, "bf16", "scaled_normal", seed=53)
    got, _ = _run(A, B, bias, epi, cfg)
    assert _within_tolerance(got, A, B, bias, epi) <= 1.0


def test_tuned_gate_up_projection_every_element():
    """The fused gate+up projection of the transformer sweep at 512 tokens
    (4096 -> 2 x 14336) through the tuned GeGLU plan, every element."""
    M, N, K = 512, 28672, 4096
    A, B, bias = inputs.make_operands(M, N, K, "bf16", "scaled_normal", seed=54)
    got, cfg = _run(A, B, bias, "geglu")
    assert cfg.swap_ab == 0 and cfg.split_k == 1 and cfg.bn % 64 == 0
    assert _within_tolerance(got, A, B, bias, "geglu") <= 1.0


def test_gated_rules_and_host_path():
    rc, _ = g.plan_with_config_rc(256, 256, 256, "bf16", "geglu", C(128, 128, 64, 4, 0, 1, 2))
    assert rc == g.ERR_INFEASIBLE                       # no split-K
    rc, _ = g.plan_with_config_rc(16, 256, 256, "bf16", "geglu", C(128, 16, 64, 4, 0, 1, 1, 1, 1))
    assert rc == g.ERR_INFEASIBLE                       # no swap
    rc, _ = g.plan_with_config_rc(256, 288, 256, "bf16", "reglu", C(128, 96, 64, 4))
    assert rc == g.ERR_INFEASIBLE                       # whole 64-column block pairs
    M, N, K = 130, 256, 512
    A, B, bias = operands(M, N, K, "bf16", "int", seed=55)
    out = torch.empty(M, N // 2, dtype=torch.bfloat16).pin_memory()
    with g.plan_with_config(M, N, K, "bf16", "reglu", C(128, 128, 64, 4)) as p:
        p.run_host(A.pin_memory(), B.pin_memory(), bias.pin_memory(), out)
    assert np.array_equal(device_bits(out), og.round_bf16_bits(og.gemm(A, B, bias, og.EPI_BIAS_REGLU)))
