"""The allocation-free entry point (gemm_run_noalloc) against the planned path.

gemm_run_noalloc serves callers that cannot call cudaMalloc (code under a
framework whose caching allocator owns device memory, services that reserve all
memory up front); it runs the same split-K kernel with its scratch in a fixed
array inside the library.  Here it is called through the C ABI twice in a row,
on different inputs, and each result is compared with gemm_plan_with_config +
gemm_run on the same configuration.  This file is collected last so that a run
that stops at the first failure has already run every other test."""
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import _build, inputs
from oracle import gemm as og

pytestmark = pytest.mark.gpu

TOL = 2e-3   # max |C - C_ref| / (||a_i||·||b_j||), the tolerance of the parity tests


def _planned(M, N, K, epi, cfg, A, B, bias):
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with g.plan_with_config(M, N, K, "bf16", epi, cfg) as p:
        p.run(A, B, bias, C)
        torch.cuda.synchronize()
        assert p.status() == 0, g.last_error()
    return C


def _scaled_diff(C1, C2, A, B):
    return og.normalised_error(C1.float().cpu().numpy(), C2.float().cpu().numpy().astype("float64"),
                               A.cpu(), B.cpu())


@pytest.mark.parametrize("shape,cfg,epi", [
    ((300, 320, 2048), g.make_config(128, 128, 64, 4, 0, 1, 3), "gelu"),          # split-K, unswapped
    ((16, 1024, 4096), g.make_config(128, 16, 64, 8, 0, 1, 8, 1, 1), "none"),     # split-K, swapped (decode)
    ((257, 384, 520), g.make_config(256, 128, 64, 3, 1, 4, 1), "relu"),            # no split
])
def test_noalloc_matches_the_planned_path_on_two_calls_in_a_row(shape, cfg, epi):
    _build.build()
    M, N, K = shape
    for call, seed in enumerate((21, 22)):
        A, B, bias = inputs.make_operands(M, N, K, "bf16", "scaled_normal", seed=seed, device="cuda")
        bias_arg = bias if epi != "none" else None
        want = _planned(M, N, K, epi, cfg, A, B, bias_arg)
        got = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        rc = g.run_noalloc_rc(M, N, K, epi, cfg, A, B, bias_arg, got)
        assert rc == 0, (call, g.last_error())
        torch.cuda.synchronize()
        assert _scaled_diff(got, want, A, B) <= TOL, call


def test_noalloc_rejects_problems_beyond_its_fixed_scratch():
    _build.build()
    # 32 x 32 tiles x split 8 x 128 x 128 x 4 bytes = 512 MiB of partial tiles
    cfg = g.make_config(128, 128, 64, 4, 0, 1, 8)
    M = N = 4096
    A = torch.zeros(M, 1024, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1024, N, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    rc = g.run_noalloc_rc(M, N, 1024, "none", cfg, A, B, None, C)
    assert rc == g.ERR_INVALID_ARG
    assert "exceed the fixed scratch" in g.last_error()
