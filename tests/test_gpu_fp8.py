"""FP8 E4M3 operands (tcgen05.mma kind::f8f6f4, bf16 C) against the oracle,
which decodes the same bytes from the format's definition: bit-exact on
small-integer inputs (with and without the product scale alpha), within the
stated tolerance on random inputs, on the plain, swapped, split-K (each route)
and CTA-pair paths, with and without a residual."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import alloc_out, device_bits, guard_intact, sampled_error
from oracle import gemm as og

pytestmark = pytest.mark.gpu

C = g.make_config

CASES = [
    ((300, 320, 1024), C(128, 128, 128, 4), 0),
    ((300, 320, 1024), C(256, 256, 128, 3), 0),
    ((300, 320, 1024), C(128, 128, 256, 2), 0),
    ((520, 640, 384), C(128, 128, 128, 4, 1, 4), 0),              # grouped raster, ragged K blocks
    ((20, 320, 1024), C(128, 16, 128, 6, 0, 1, 1, 1, 1), 0),      # swapped
    ((40, 264, 1024), C(256, 64, 128, 2, 0, 1, 3, 1, 1), 0),      # swapped split-K
    ((300, 320, 2048), C(256, 128, 128, 4, 0, 1, 4), 0),          # split-K, cluster route
    ((300, 320, 2048), C(256, 128, 128, 4, 0, 1, 4), 1),          # split-K, cooperative route
    ((300, 320, 1024), C(256, 256, 128, 4, 0, 1, 1, 2), 0),       # CTA pair
    ((1000, 1000, 4096), C(256, 256, 128, 3, 0, 1, 4, 2), 0),     # CTA pair, split-K (cluster of 4 pairs)
    ((1000, 1000, 4096), C(256, 256, 128, 3, 0, 1, 4, 2), 1),     # CTA pair, split-K, cooperative route
]


def _id(c):
    (M, N, K), cfg, route = c
    return f"{M}x{N}x{K}-{'x'.join(str(v) for v in cfg.astuple())}-r{route}"


def _run(A, B, bias, epi, cfg, route=0, alpha=1.0, R=None, guard=64):
    M, K = A.shape
    N = B.shape[1]
    g.debug_set(3, route)
    try:
        p = g.plan_with_config(M, N, K, "fp8", epi, cfg)
    finally:
        g.debug_set(3, 0)
    with p:
        p.set_scale(alpha)
        Cd, buf = alloc_out(M, N, g.BF16, guard)
        bd = bias.cuda() if bias is not None and epi != "none" else None
        if R is None:
            p.run(A.cuda(), B.cuda(), bd, Cd)
        else:
            p.run_ex(A.cuda(), B.cuda(), bd, R.cuda(), Cd)
        assert p.status() == 0, g.last_error()
        info = p.launch_info
    return Cd.cpu(), guard_intact(buf, guard, M, N), info


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("epi,alpha", [("relu", 1.0), ("none", 0.5), ("bias", -0.25)])
def test_fp8_integer_inputs_bit_exact(case, epi, alpha):
    (M, N, K), cfg, route = case
    A, B, bias = inputs.make_operands(M, N, K, "fp8", "int", seed=31)
    out, ok, info = _run(A, B, bias, epi, cfg, route, alpha)
    assert ok, "write outside C"
    assert info.b_transposed == (0 if N % 16 == 0 else 1)   # in place, or a K-major copy when N % 16 != 0
    want = og.round_bf16_bits(og.gemm(A, B, bias if epi != "none" else None, g.EPILOGUES[epi], alpha=alpha))
    bad = np.argwhere(device_bits(out) != want)
    assert bad.size == 0, f"{len(bad)} mismatches ({g.SPLITK_ROUTES[info.splitk_route]}), first {bad[:5].tolist()}"


@pytest.mark.parametrize("case", [CASES[0], CASES[4], CASES[8]], ids=_id)
def test_fp8_k_major_copy_of_b_gives_the_same_bits(case):
    (M, N, K), cfg, route = case
    A, B, bias = inputs.make_operands(M, N, K, "fp8", "scaled_normal", seed=34)
    direct, _, i1 = _run(A, B, bias, "gelu", cfg, route, 1.5)
    g.debug_set(2, 1)          # B first copied K-major
    try:
        copied, _, i2 = _run(A, B, bias, "gelu", cfg, route, 1.5)
    finally:
        g.debug_set(2, 0)
    assert i1.b_transposed == 0 and i2.b_transposed == 1
    assert np.array_equal(device_bits(direct), device_bits(copied))


@pytest.mark.parametrize("case", CASES[::2], ids=_id)
def test_fp8_random_gelu_within_tolerance(case):
    (M, N, K), cfg, route = case
    A, B, bias = inputs.make_operands(M, N, K, "fp8", "decode", seed=32)
    alpha = 0.75
    out, ok, _ = _run(A, B, bias, "gelu", cfg, route, alpha)
    ref = og.gemm(A, B, bias, og.EPI_BIAS_GELU, alpha=alpha)
    Af = A.to(torch.float32).numpy().astype(np.float64)
    Bf = B.to(torch.float32).numpy().astype(np.float64)
    scale = abs(alpha) * np.sqrt((Af ** 2).sum(1))[:, None] * np.sqrt((Bf ** 2).sum(0))[None, :]
    err = np.abs(out.float().numpy() - ref) / np.maximum(scale, 1e-30)
    assert ok and float(err.max()) <= 2e-3, float(err.max())


def test_fp8_residual_bit_exact_and_tuned_plan():
    M, N, K = 512, 1024, 2048
    A, B, bias = inputs.make_operands(M, N, K, "fp8", "int", seed=33)
    R = inputs.make_residual(M, N, "fp8", "int", seed=33)
    assert R.dtype == torch.bfloat16
    with g.plan(M, N, K, "fp8", "relu_residual") as p:
        Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        p.run_ex(A.cuda(), B.cuda(), bias.cuda(), R.cuda(), Cd)
        assert p.status() == 0
        tuned = p.config.astuple()
    want = og.round_bf16_bits(og.gemm(A, B, bias, og.EPI_BIAS_RELU_RESIDUAL, residual=R))
    assert np.array_equal(device_bits(Cd.cpu()), want), tuned


@pytest.mark.parametrize("name", ["fp8_relu_8192", "fp8_decode_16x8192x28672", "fp8_gelu_1000x1000x8192"])
def test_fp8_full_size_tuned_plan_sampled(name):
    """The FP8 workloads at full size through tuned plans (the configurations
    the sweep times), checked on sampled entries."""
    w = inputs.WORKLOADS[name]
    A, B, bias = inputs.make_workload(w, seed=0)
    with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as p:
        Cd = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
        p.run(A.cuda(), B.cuda(), bias.cuda() if bias is not None else None, Cd)
        assert p.status() == 0, g.last_error()
        cfg = p.config.astuple()
    assert sampled_error(Cd.cpu(), A, B, bias, w.epi, n=2048) <= 2e-3, cfg


@pytest.mark.parametrize("shape,cfg,cluster", [((300, 320, 2048), C(256, 256, 128, 4, 0, 1, 4, 2), 8),
                                               ((300, 320, 2064), C(256, 256, 128, 4, 0, 1, 2, 2), 4)])
def test_fp8_pair_tiles_reduce_inside_a_cluster(shape, cfg, cluster):
    # A pair tile's K slices as one cluster of 2S CTAs (split-K through
    # distributed shared memory), bit-exact and equal to the cooperative route.
    M, N, K = shape
    A, B, bias = inputs.make_operands(M, N, K, "fp8", "int", seed=35)
    out, ok, info = _run(A, B, bias, "relu", cfg, 0, 0.5)
    assert ok and info.splitk_route == 3 and info.cluster == cluster
    want = og.round_bf16_bits(og.gemm(A, B, bias, g.EPILOGUES["relu"], alpha=0.5))
    assert np.array_equal(device_bits(out), want)
    coop, ok2, info2 = _run(A, B, bias, "relu", cfg, 1, 0.5)
    assert ok2 and info2.splitk_route == 2 and np.array_equal(device_bits(coop), device_bits(out))
