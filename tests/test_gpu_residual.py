"""The residual epilogues, C = act(A·B + bias) + R, on every store path of the
kernel (plain, swapped, each split-K route, CTA pairs) against the oracle:
bit-exact on small-integer inputs, within the stated tolerance with GELU; in
place (R = C); and the argument rules of gemm_run / gemm_run_ex."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import alloc_out, device_bits, guard_intact, operands
from oracle import gemm as og

pytestmark = pytest.mark.gpu

C = g.make_config

CASES = [
    ("bf16", (300, 320, 520), C(128, 128, 64, 4), 0),                    # plain
    ("bf16", (300, 320, 520), C(256, 256, 64, 2), 0),                    # two 128-row halves, one accumulator
    ("bf16", (20, 320, 520), C(128, 16, 64, 6, 0, 1, 1, 1, 1), 0),       # swapped (small M)
    ("bf16", (40, 264, 520), C(256, 64, 128, 2, 0, 1, 3, 1, 1), 0),      # swapped split-K
    ("bf16", (40, 264, 520), C(128, 64, 64, 4, 0, 1, 2, 1, 1), 0),       # swapped split-K, cluster route
    ("bf16", (300, 320, 1032), C(256, 128, 64, 4, 0, 1, 4), 0),          # split-K, cluster route
    ("bf16", (300, 320, 1032), C(256, 128, 64, 4, 0, 1, 4), 1),          # split-K, cooperative route
    ("bf16", (2048, 2048, 512), C(128, 128, 64, 4, 0, 1, 2), 0),         # split-K, last arriver
    ("bf16", (300, 320, 520), C(256, 256, 64, 4, 0, 1, 1, 2), 0),        # CTA pair
    ("bf16", (1000, 1000, 2056), C(256, 256, 64, 6, 0, 1, 4, 2), 0),     # CTA pair, split-K, cluster route
    ("bf16", (1000, 1000, 2056), C(256, 256, 64, 6, 0, 1, 4, 2), 1),     # CTA pair, cooperative split-K
    ("fp32", (200, 160, 136), C(128, 64, 32, 4)),
]
CASES = [c if len(c) == 4 else c + (0,) for c in CASES]


def _id(c):
    dt, (M, N, K), cfg, route = c
    return f"{dt}-{M}x{N}x{K}-{'x'.join(str(v) for v in cfg.astuple())}-r{route}"


def _run(dt, A, B, bias, R, epi, cfg, route=0, in_place=False, guard=64):
    M, K = A.shape
    N = B.shape[1]
    dtc = g.BF16 if dt == "bf16" else g.FP32_TF32
    g.debug_set(3, route)
    try:
        p = g.plan_with_config(M, N, K, dtc, epi, cfg)
    finally:
        g.debug_set(3, 0)
    with p:
        Cd, buf = alloc_out(M, N, dtc, guard)
        Rd = R.cuda()
        if in_place:
            Cd.copy_(Rd)
            Rd = Cd
        p.run_ex(A.cuda(), B.cuda(), bias.cuda(), Rd, Cd)
        assert p.status() == 0, g.last_error()
        info = p.launch_info
    return Cd.cpu(), guard_intact(buf, guard, M, N), info


def _want_bits(A, B, bias, R, epi_code, dtc):
    ref = og.gemm(A, B, bias, epi_code, residual=R)
    return og.round_bf16_bits(ref) if dtc == g.BF16 else og.round_f32(ref).view(np.uint32)


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("epi", ["relu_residual", "bias_residual"])
def test_residual_integer_inputs_bit_exact(case, epi):
    dt, (M, N, K), cfg, route = case
    A, B, bias = operands(M, N, K, dt, "int", seed=21)
    R = inputs.make_residual(M, N, dt, "int", seed=21)
    out, ok, info = _run(dt, A, B, bias, R, epi, cfg, route)
    assert ok, "write outside C"
    dtc = g.BF16 if dt == "bf16" else g.FP32_TF32
    want = _want_bits(A, B, bias, R, g.EPILOGUES[epi], dtc)
    bad = np.argwhere(device_bits(out) != want)
    assert bad.size == 0, f"{len(bad)} mismatches ({g.SPLITK_ROUTES[info.splitk_route]}), first {bad[:5].tolist()}"


@pytest.mark.parametrize("case", CASES[::3], ids=_id)
def test_residual_in_place_equals_out_of_place(case):
    dt, (M, N, K), cfg, route = case
    A, B, bias = operands(M, N, K, dt, "scaled_normal", seed=22)
    R = inputs.make_residual(M, N, dt, "scaled_normal", seed=22)
    a, ok1, _ = _run(dt, A, B, bias, R, "gelu_residual", cfg, route)
    b, ok2, _ = _run(dt, A, B, bias, R, "gelu_residual", cfg, route, in_place=True)
    assert ok1 and ok2 and np.array_equal(device_bits(a), device_bits(b))
    ref = og.gemm(A, B, bias, g.EPI_BIAS_GELU_RESIDUAL, residual=R)
    # normalised error of the GEMM part (the residual itself is exact before rounding)
    scale = np.sqrt((A.float().numpy().astype(np.float64) ** 2).sum(1))[:, None] * \
        np.sqrt((B.float().numpy().astype(np.float64) ** 2).sum(0))[None, :]
    err = np.abs(a.float().numpy() - ref) / np.maximum(scale, 1e-30)
    # bf16 output of |R| ~ 1 carries 2^-9 relative rounding on top of the GEMM error
    assert (np.abs(a.float().numpy() - ref) <= 2e-3 * scale + 2.0 ** -8 * np.abs(ref) + 1e-6).all(), float(err.max())


def test_tuned_plan_with_a_residual_epilogue():
    M, N, K = 512, 1024, 2048
    A, B, bias = operands(M, N, K, "bf16", "int", seed=23)
    R = inputs.make_residual(M, N, "bf16", "int", seed=23)
    with g.plan(M, N, K, "bf16", "relu_residual") as p:
        Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        p.run_ex(A.cuda(), B.cuda(), bias.cuda(), R.cuda(), Cd)
        assert p.status() == 0
    assert np.array_equal(device_bits(Cd.cpu()), _want_bits(A, B, bias, R, g.EPI_BIAS_RELU_RESIDUAL, g.BF16))


def test_residual_argument_rules():
    M, N, K = 256, 256, 256
    A, B, bias = operands(M, N, K, "bf16", "int", seed=24)
    R = inputs.make_residual(M, N, "bf16", "int", seed=24).cuda()
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with g.plan_with_config(M, N, K, "bf16", "relu_residual", C(128, 128, 64, 4)) as p:
        assert p.run_rc(A.cuda(), B.cuda(), bias.cuda(), Cd) == g.ERR_INVALID_ARG      # R missing
        assert "residual" in g.last_error()
    with g.plan_with_config(M, N, K, "bf16", "relu", C(128, 128, 64, 4)) as p:
        rc = g.lib().gemm_run_ex(p.handle, g._ptr(A.cuda()), g._ptr(B.cuda()), g._ptr(bias.cuda()), g._ptr(R),
                                 g._ptr(Cd), None)
        assert rc == g.ERR_INVALID_ARG                                               # R on a plan without one
