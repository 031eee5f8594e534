"""The allocation-free entry point (gemm_run_noalloc).

gemm_run_noalloc serves callers that cannot call cudaMalloc: code under a
framework whose caching allocator owns device memory (a raw cudaMalloc escapes
its accounting and may synchronise the device), and services that reserve all
device memory up front and must not fail or stall on an allocation.  It runs
the same kernel as a plan of the same configuration, with its scratch in a
fixed array inside the library.  Here it is called through the C ABI two times
in a row on different inputs; each result is compared bit for bit with the
oracle (integer inputs, whose sums are exact) and with gemm_plan_with_config +
gemm_run on the same configuration (both sum split-K partials in slice order,
so the bits agree on any input).  The limits of the fixed scratch are probed at
their edges.  This file is collected last so that a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import _build, inputs
from gpu_util import device_bits, oracle_rounded_bits

pytestmark = pytest.mark.gpu

MAX_TILES = 4096                      # GEMM_NOALLOC_MAX_TILES
WS_BYTES = 16 * 1024 * 1024           # GEMM_NOALLOC_WORKSPACE_BYTES


def _planned(M, N, K, epi, cfg, A, B, bias):
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with g.plan_with_config(M, N, K, "bf16", epi, cfg) as p:
        p.run(A, B, bias, C)
        torch.cuda.synchronize()
        assert p.status() == 0, g.last_error()
    return C


def _noalloc(M, N, K, epi, cfg, A, B, bias):
    got = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    rc = g.run_noalloc_rc(M, N, K, epi, cfg, A, B, bias, got)
    assert rc == 0, g.last_error()
    torch.cuda.synchronize()
    return got


CASES = [
    ((300, 320, 2048), g.make_config(128, 128, 64, 4, 0, 1, 3), "gelu"),          # split-K, unswapped
    ((16, 1024, 4096), g.make_config(128, 16, 64, 8, 0, 1, 8, 1, 1), "none"),     # split-K, swapped (decode)
    ((257, 384, 520), g.make_config(256, 128, 64, 3, 1, 4, 1), "relu"),            # no split
]


@pytest.mark.parametrize("shape,cfg,epi", CASES)
def test_noalloc_two_calls_in_a_row_equal_the_oracle_and_the_planned_path(shape, cfg, epi):
    _build.build()
    M, N, K = shape
    for call, seed in enumerate((21, 22)):
        # integer-valued inputs: exact sums, so the bits must equal the oracle's
        A, B, bias = inputs.make_operands(M, N, K, "bf16", "int", seed=seed)
        want = oracle_rounded_bits(A, B, bias, "relu" if epi == "gelu" else epi, g.BF16)
        e = "relu" if epi == "gelu" else epi
        Ad, Bd, bd = A.cuda(), B.cuda(), bias.cuda() if e != "none" else None
        got = _noalloc(M, N, K, e, cfg, Ad, Bd, bd)
        assert np.array_equal(device_bits(got.cpu()), want), call
        # random inputs, every epilogue: the same bits as the planned path
        A, B, bias = inputs.make_operands(M, N, K, "bf16", "scaled_normal", seed=seed, device="cuda")
        bias_arg = bias if epi != "none" else None
        got = _noalloc(M, N, K, epi, cfg, A, B, bias_arg)
        want_plan = _planned(M, N, K, epi, cfg, A, B, bias_arg)
        assert torch.equal(got.view(torch.int16), want_plan.view(torch.int16)), call


def test_noalloc_at_the_tile_limit():
    _build.build()
    # exactly GEMM_NOALLOC_MAX_TILES tiles of 128 x 256 (no split: no workspace)
    cfg = g.make_config(128, 256, 64, 4)
    M, N, K = 128 * 64, 256 * 64, 64
    assert (M // 128) * (N // 256) == MAX_TILES
    A, B, bias = inputs.make_operands(M, N, K, "bf16", "int", seed=23, device="cuda")
    got = _noalloc(M, N, K, "relu", cfg, A, B, bias)
    want = _planned(M, N, K, "relu", cfg, A, B, bias)
    assert torch.equal(got.view(torch.int16), want.view(torch.int16))
    # sampled rows against the oracle (integer inputs: exact)
    rows = [0, 1, 4097, M - 1]
    Ac, Bc, bc = A.cpu(), B.cpu(), bias.cpu()
    ref = oracle_rounded_bits(Ac[rows], Bc, bc, "relu", g.BF16)
    assert np.array_equal(device_bits(got[rows].cpu()), ref)


def test_noalloc_one_tile_over_the_limit_is_rejected():
    _build.build()
    cfg = g.make_config(128, 128, 64, 4)
    M, N, K = 128 * (MAX_TILES + 1), 128, 64        # 4097 tiles
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    assert g.run_noalloc_rc(M, N, K, "none", cfg, A, B, None, C) == g.ERR_INVALID_ARG
    assert "exceed the fixed scratch" in g.last_error()


def test_noalloc_workspace_exactly_at_the_limit():
    _build.build()
    # 64 tiles x 4 slices x 128 x 128 x 4 bytes = 16 MiB of partial tiles
    cfg = g.make_config(128, 128, 64, 4, 0, 1, 4)
    M, N, K = 1024, 1024, 2048
    assert (M // 128) * (N // 128) * 4 * 128 * 128 * 4 == WS_BYTES
    A, B, bias = inputs.make_operands(M, N, K, "bf16", "int", seed=24)
    got = _noalloc(M, N, K, "relu", cfg, A.cuda(), B.cuda(), bias.cuda())
    assert np.array_equal(device_bits(got.cpu()), oracle_rounded_bits(A, B, bias, "relu", g.BF16))


def test_noalloc_workspace_just_over_the_limit_is_rejected():
    _build.build()
    # 65 tiles x 4 slices x 64 KiB = 16.25 MiB of partial tiles
    cfg = g.make_config(128, 128, 64, 4, 0, 1, 4)
    M, N, K = 128 * 65, 128, 2048
    A = torch.zeros(M, K, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(K, N, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    assert g.run_noalloc_rc(M, N, K, "none", cfg, A, B, None, C) == g.ERR_INVALID_ARG
    assert "exceed the fixed scratch" in g.last_error()


def test_noalloc_checked_run_reports_an_expired_wait():
    _build.build()
    cfg = g.make_config(128, 128, 64, 4, 0, 1, 2)
    M, N, K = 256, 256, 512
    A, B, bias = inputs.make_operands(M, N, K, "bf16", "int", seed=25, device="cuda")
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.debug_set(4, 1)                  # checked runs
    g.debug_set(0, 50_000_000)         # 50 ms device wait limit
    g.debug_set(1, 1)                  # the epilogue waits on a barrier nothing signals
    try:
        rc = g.run_noalloc_rc(M, N, K, "relu", cfg, A, B, bias, C)
    finally:
        g.debug_set(1, 0)
        g.debug_set(0, 2_000_000_000)
        g.debug_set(4, 0)
    assert rc == g.ERR_TIMEOUT, g.last_error()
    # the next call clears the status word and runs normally
    got = _noalloc(M, N, K, "relu", cfg, A, B, bias)
    want = oracle_rounded_bits(A.cpu(), B.cpu(), bias.cpu(), "relu", g.BF16)
    assert np.array_equal(device_bits(got.cpu()), want)
