"""GPU parity of the tcgen05 GEMM against the fp64 oracle, through the C ABI.

Bars: bit-exact on small-integer inputs (sums exact in fp32; the output is the
exact value rounded once, so the device result and the oracle's rounding of
the exact value must have identical bits); normalised error
max |C - C_ref| / (||a_i||·||b_j||) <= 2e-3 on random inputs."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import (TOL, alloc_out, device_bits, normalised_error, operands, oracle_rounded_bits,
                      run_config, sampled_error)

pytestmark = pytest.mark.gpu

C = g.make_config

# (M, N, K) ragged against every tile size used below; configs cover both tile
# heights, every bn class, 1-4 K spans, shallow and deep rings, both rasters,
# grouping, split-K and the swapped (small-M) orientation.
BF16_CASES = [
    ((300, 320, 520), C(128, 128, 64, 4)),
    ((300, 320, 520), C(128, 64, 64, 6)),
    ((300, 320, 520), C(128, 192, 64, 4)),
    ((300, 320, 520), C(128, 256, 64, 3)),
    ((300, 320, 520), C(256, 128, 64, 3)),
    ((300, 320, 520), C(256, 64, 128, 2)),
    ((300, 320, 520), C(128, 128, 128, 3)),
    ((300, 320, 520), C(128, 64, 256, 2)),
    ((300, 320, 520), C(128, 128, 64, 2, 1, 2)),
    ((520, 640, 264), C(128, 64, 64, 4, 0, 4)),
    ((520, 640, 264), C(128, 128, 64, 4, 1, 16)),
    ((300, 320, 520), C(128, 128, 64, 4, 0, 1, 3)),
    ((300, 320, 520), C(256, 256, 64, 2, 0, 1, 4)),
    ((20, 320, 520), C(128, 16, 64, 6, 0, 1, 1, 1, 1)),
    ((20, 320, 520), C(128, 32, 64, 6, 0, 1, 2, 1, 1)),
    ((40, 264, 520), C(256, 64, 128, 2, 0, 1, 3, 1, 1)),
    ((16, 1024, 1024), C(128, 16, 64, 8, 0, 1, 8, 1, 1)),
    # CTA pairs (cta_group 2): 256-row tiles, each CTA 128 rows and half of B
    ((300, 320, 520), C(256, 256, 64, 4, 0, 1, 1, 2)),
    ((300, 320, 520), C(256, 128, 64, 6, 0, 1, 1, 2)),
    ((300, 320, 520), C(256, 256, 128, 3, 0, 1, 1, 2)),
    ((520, 640, 264), C(256, 128, 64, 4, 1, 4, 1, 2)),
    ((300, 320, 1032), C(256, 256, 64, 4, 0, 1, 4, 2)),
]

FP32_CASES = [
    ((200, 160, 136), C(128, 32, 32, 4)),
    ((200, 160, 136), C(128, 128, 32, 4)),
    ((200, 160, 136), C(256, 64, 64, 2)),
    ((200, 160, 136), C(128, 96, 64, 2)),
    ((200, 160, 136), C(128, 64, 32, 4, 0, 1, 2)),
    ((24, 160, 136), C(128, 16, 32, 4, 0, 1, 1, 1, 1)),
    ((24, 160, 136), C(128, 32, 64, 4, 0, 1, 3, 1, 1)),
    ((200, 160, 136), C(256, 64, 32, 4, 0, 1, 1, 2)),
    ((200, 160, 264), C(256, 128, 32, 4, 0, 1, 2, 2)),
    ((264, 256, 136), C(256, 256, 64, 2, 0, 1, 1, 2)),
]


def _cases_id(c):
    (M, N, K), cfg = c
    return f"{M}x{N}x{K}-{'x'.join(str(v) for v in cfg.astuple())}"


@pytest.mark.parametrize("case", BF16_CASES, ids=_cases_id)
@pytest.mark.parametrize("epi", ["relu", "none"])
def test_bf16_integer_inputs_bit_exact(case, epi):
    (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, "bf16", "int", seed=3)
    out, guard_ok = run_config(A, B, bias, epi, cfg)
    assert guard_ok, "write outside C"
    want = oracle_rounded_bits(A, B, bias, epi, g.BF16)
    got = device_bits(out)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("case", FP32_CASES, ids=_cases_id)
def test_fp32_integer_inputs_bit_exact(case):
    (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, "fp32", "int", seed=4)
    out, guard_ok = run_config(A, B, bias, "relu", cfg)
    assert guard_ok
    want = oracle_rounded_bits(A, B, bias, "relu", g.FP32_TF32)
    bad = np.argwhere(device_bits(out) != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("case", BF16_CASES[::2], ids=_cases_id)
@pytest.mark.parametrize("epi", ["none", "bias", "relu", "gelu"])
def test_bf16_random_within_tolerance(case, epi):
    (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, "bf16", "scaled_normal", seed=5)
    out, guard_ok = run_config(A, B, bias, epi, cfg)
    assert guard_ok
    assert normalised_error(out, A, B, bias, epi) <= TOL


@pytest.mark.parametrize("case", FP32_CASES, ids=_cases_id)
@pytest.mark.parametrize("epi", ["bias", "gelu"])
def test_fp32_random_within_tolerance(case, epi):
    (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, "fp32", "uniform", seed=6)
    out, guard_ok = run_config(A, B, bias, epi, cfg)
    assert guard_ok
    assert normalised_error(out, A, B, bias, epi) <= TOL


def test_every_candidate_of_the_256_cube_integer_fp32_relu():
    """Every feasible configuration the generator offers for the 256³ fp32
    ReLU workload is bit-exact on its integer variant."""
    w = inputs.WORKLOADS["fp32_relu_256_int"]
    A, B, bias = inputs.make_workload(w, seed=0)
    dev = g.device_params_query()
    cands = g.enumerate_configs(w.M, w.N, w.K, "fp32", "relu", dev)
    assert len(cands) > 50
    want = oracle_rounded_bits(A, B, bias, "relu", g.FP32_TF32)
    Ad, Bd, bd = A.cuda(), B.cuda(), bias.cuda()
    for cfg in cands:
        Cd, _ = alloc_out(w.M, w.N, g.FP32_TF32)
        with g.plan_with_config(w.M, w.N, w.K, "fp32", "relu", cfg) as p:
            p.run(Ad, Bd, bd, Cd)
            assert p.status() == 0, (cfg, g.last_error())
        assert np.array_equal(device_bits(Cd.cpu()), want), cfg


def test_split_k_is_deterministic():
    A, B, bias = operands(257, 384, 4096, "bf16", "scaled_normal", seed=8)
    cfg = C(128, 128, 64, 4, 0, 1, 6)
    a, _ = run_config(A, B, bias, "gelu", cfg)
    b, _ = run_config(A, B, bias, "gelu", cfg)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert normalised_error(a, A, B, bias, "gelu") <= TOL


# --- transformer sweep through tuned plans ----------------------------------------
# (the headline workloads are checked element by element in test_gpu_full_size.py)

def test_sweep_shapes_through_tuned_plans():
    """A slice of the 30-shape transformer sweep through tuned plans: every
    element where the oracle takes a few seconds at most, sampled entries on
    the largest shapes."""
    for w in inputs.SWEEP[::7]:
        A, B, bias = inputs.make_workload(w, seed=1)
        with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as p:
            Cd, _ = alloc_out(w.M, w.N, g.BF16)
            p.run(A.cuda(), B.cuda(), bias.cuda(), Cd)
            assert p.status() == 0
        if 2.0 * w.M * w.N * w.K <= 2.5e11:
            assert normalised_error(Cd.cpu(), A, B, bias, w.epi) <= TOL, w.name
        else:
            assert sampled_error(Cd.cpu(), A, B, bias, w.epi, n=4096) <= TOL, w.name


# --- edge cases ---------------------------------------------------------------------

def test_tiny_and_degenerate_extents():
    for (M, N, K) in [(1, 8, 8), (1, 8, 64), (129, 8, 8), (7, 24, 16)]:
        A, B, bias = operands(M, N, K, "bf16", "int", seed=9)
        out, ok = run_config(A, B, bias, "relu", C(128, 64, 64, 2))
        assert ok and np.array_equal(device_bits(out), oracle_rounded_bits(A, B, bias, "relu", g.BF16))


def test_k_zero_gives_act_of_bias():
    M, N = 70, 96
    bias = torch.arange(N, dtype=torch.float32).sub(48).div(8).to(torch.bfloat16)
    A = torch.empty(M, 0, dtype=torch.bfloat16)
    B = torch.empty(0, N, dtype=torch.bfloat16)
    Cd, _ = alloc_out(M, N, g.BF16)
    with g.plan_with_config(M, N, 0, "bf16", "relu", C(128, 64, 64, 2)) as p:
        p.run(None, None, bias.cuda(), Cd)
        assert p.status() == 0
    want = torch.relu(bias.float()).to(torch.bfloat16).expand(M, N)
    assert torch.equal(Cd.cpu(), want)


def test_empty_output_is_a_no_op():
    Cd, buf = alloc_out(0, 64, g.BF16, guard=64)
    with g.plan_with_config(0, 64, 64, "bf16", "none", C(128, 64, 64, 2)) as p:
        p.run(None, None, None, Cd)
    torch.cuda.synchronize()
    assert (buf == 12345.0).all()


def test_error_codes():
    cfg = C(128, 128, 64, 4)
    rc, _ = g.plan_with_config_rc(128, 128, 72 + 3, "bf16", "none", cfg)  # K·2 not a multiple of 16
    assert rc == g.ERR_MISALIGNED
    rc, _ = g.plan_with_config_rc(128, 128, 128, "bf16", "none", C(64, 128, 64, 4))
    assert rc == g.ERR_INFEASIBLE and "bm" in g.last_error()
    rc, _ = g.plan_with_config_rc(-1, 128, 128, "bf16", "none", cfg)
    assert rc == g.ERR_INVALID_ARG
    A, B, bias = operands(128, 128, 128, "bf16", "int")
    Ad, Bd = A.cuda(), B.cuda()
    Cd, _ = alloc_out(128, 128, g.BF16)
    with g.plan_with_config(128, 128, 128, "bf16", "relu", cfg) as p:
        assert p.run_rc(Ad, Bd, None, Cd) == g.ERR_INVALID_ARG           # bias required
        raw = torch.empty(128 * 128 + 8, dtype=torch.bfloat16, device="cuda")
        assert p.run_rc(Ad, Bd, bias.cuda(), raw[1:]) == g.ERR_MISALIGNED  # C not 16-byte aligned
        assert p.run_rc(Ad, None, bias.cuda(), Cd) == g.ERR_INVALID_ARG
        p.run(Ad, Bd, bias.cuda(), Cd)
        assert p.status() == 0


def test_run_host_matches_run():
    A, B, bias = operands(200, 192, 512, "bf16", "scaled_normal", seed=11)
    cfg = C(128, 64, 64, 4, 0, 1, 2)
    dev_out, _ = run_config(A, B, bias, "gelu", cfg)
    host_out = torch.empty(200, 192, dtype=torch.bfloat16).pin_memory()
    with g.plan_with_config(200, 192, 512, "bf16", "gelu", cfg) as p:
        p.run_host(A.pin_memory(), B.pin_memory(), bias.pin_memory(), host_out)
    assert torch.equal(dev_out.view(torch.int16), host_out.view(torch.int16))


@pytest.mark.parametrize("cfg", [C(128, 64, 64, 4, 0, 1, 2), C(128, 128, 64, 4)], ids=["split2", "nosplit"])
def test_run_host_many_matches_run(cfg):
    """gemm_run_host_many: five GEMMs from pinned host buffers, pipelined over
    two streams and two plans of the configuration; each C equals the device
    path's bits (integer inputs also the oracle's)."""
    M, N, K = 200, 192, 512
    ins = [operands(M, N, K, "bf16", "int" if i % 2 else "scaled_normal", seed=40 + i) for i in range(5)]
    outs = [torch.full((M, N), 3.0, dtype=torch.bfloat16).pin_memory() for _ in ins]
    with g.plan_with_config(M, N, K, "bf16", "relu", cfg) as p:
        p.run_host_many([a.pin_memory() for a, _, _ in ins], [b.pin_memory() for _, b, _ in ins],
                        [c.pin_memory() for _, _, c in ins], outs)
        assert p.status() == 0
    for i, (A, B, bias) in enumerate(ins):
        dev_out, _ = run_config(A, B, bias, "relu", cfg)
        assert torch.equal(dev_out.view(torch.int16), outs[i].view(torch.int16)), i
        if i % 2:
            assert np.array_equal(device_bits(outs[i]), oracle_rounded_bits(A, B, bias, "relu", g.BF16)), i


def test_gelu_epilogue_pointwise_accuracy():
    """C = gelu(x·1 + 0) over a sweep of x.  The device's erf (Abramowitz &
    Stegun 7.1.28) has absolute error <= 3e-7, and its fp32 evaluation (a
    sixteenth power) adds at most about 1.2e-5 of erfc <= 1, so |GELU_dev - GELU|
    <= 0.5·|x|·(3e-7 + 1.2e-5) before the bf16 rounding; the bf16 result may
    therefore differ from the exactly rounded one by at most one rounding step
    plus that bound (which is what matters far in the negative tail, where
    GELU ~ 0)."""
    M, N, K = 512, 64, 64
    xs = torch.linspace(-8, 8, M, dtype=torch.float64)
    A = torch.zeros(M, K, dtype=torch.float32)
    A[:, 0] = xs.float()
    A = A.to(torch.bfloat16)
    B = torch.zeros(K, N, dtype=torch.bfloat16)
    B[0, :] = 1.0
    bias = torch.zeros(N, dtype=torch.bfloat16)
    out, ok = run_config(A, B, bias, "gelu", C(128, 64, 64, 2))
    assert ok
    from oracle import gemm as og
    exact = og.gemm(A, B, bias, og.EPI_BIAS_GELU)
    got = out.double().numpy()
    x = A.double().numpy()[:, :1]
    step = np.abs(exact) * 2.0 ** -8 + 1e-38           # one bf16 rounding step
    allowed = step + 0.5 * np.abs(x) * (3e-7 + 1.2e-5) * 1.01
    assert np.all(np.abs(got - exact) <= allowed), np.argwhere(np.abs(got - exact) > allowed)[:5]
    want = oracle_rounded_bits(A, B, bias, "gelu", g.BF16)
    core = (x[:, 0] >= -1.0)                         # 1 + erf >= 0.31: the bound is relative here
    assert (device_bits(out)[core] == want[core]).mean() > 0.98
