"""One tensor copy per operand and stage (launch_info.span_copies).

A stage of an operand is a run of 128-byte spans along its contiguous extent
(K for a K-major operand, N for B read in place), laid out span after span in
shared memory.  Where that extent is a whole number of spans the tensor map
views the matrix as [spans][rows][one span] and a single 3-D box takes the
whole run ("Tiling the hierarchy": the tile moves to shared memory as one
block).  The bytes that land are the ones the per-span copies would land, so
the results must be the same bits either way, and bit-exact against the
oracle on integer inputs."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from gpu_util import alloc_out, device_bits, guard_intact, operands, oracle_rounded_bits

pytestmark = pytest.mark.gpu

C = g.make_config
DT = {"bf16": g.BF16, "fp32": g.FP32_TF32, "fp8": g.FP8_E4M3}

# (dtype, (M, N, K), config, expected span_copies bits: 1 = MMA-A, 2 = MMA-B)
CASES = [
    ("bf16", (300, 640, 1024), C(128, 128, 128, 3, 0, 1, 1), 3),          # A in K, B in N
    ("bf16", (300, 1000, 2048), C(128, 128, 128, 3, 0, 1, 1), 1),         # N = 1000: B per span
    ("bf16", (300, 640, 1000), C(128, 128, 128, 3, 0, 1, 1), 2),          # K = 1000: A per span
    ("bf16", (1000, 1024, 1032), C(256, 256, 64, 4, 0, 1, 1, 2), 2),      # pair: each CTA's 128 columns of B
    ("bf16", (300, 640, 2048), C(128, 128, 128, 3, 0, 1, 2), 3),          # split-K
    ("bf16", (16, 1024, 2048), C(128, 16, 128, 4, 0, 1, 1, 1, 1), 3),     # swapped: B rows in N, A in K
    ("fp32", (200, 160, 512), C(128, 64, 64, 3, 0, 1, 1), 3),             # tf32: A in K, B's K-major copy
    ("fp8", (256, 256, 1024), C(128, 128, 256, 2, 0, 1, 1), 1),           # E4M3 spans of 128
]


def _id(c):
    dt, (M, N, K), cfg, _ = c
    return f"{dt}-{M}x{N}x{K}-{'x'.join(str(v) for v in cfg.astuple())}"


def _run(dt, A, B, bias, epi, cfg, spans):
    M, K = A.shape
    N = B.shape[1]
    g.debug_set(7, spans)
    try:
        p = g.plan_with_config(M, N, K, DT[dt], epi, cfg)
    finally:
        g.debug_set(7, 1)
    with p:
        info = p.launch_info
        Cd, buf = alloc_out(M, N, g.BF16 if dt == "fp8" else DT[dt], 64)
        p.run(A.cuda(), B.cuda(), bias.cuda(), Cd)
        torch.cuda.synchronize()
        assert p.status() == 0, g.last_error()
        assert guard_intact(buf, 64, M, N)
        return Cd.cpu(), info


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_span_copies_bit_exact_on_integer_inputs(case):
    dt, (M, N, K), cfg, bits = case
    A, B, bias = operands(M, N, K, dt, "int", seed=81)
    got, info = _run(dt, A, B, bias, "relu", cfg, 1)
    assert info.span_copies == bits
    want = oracle_rounded_bits(A, B, bias, "relu", g.BF16 if dt == "fp8" else DT[dt])
    assert np.array_equal(device_bits(got), want)


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_span_copies_on_and_off_give_the_same_bits(case):
    dt, (M, N, K), cfg, _ = case
    A, B, bias = operands(M, N, K, dt, "scaled_normal", seed=82)
    on, i_on = _run(dt, A, B, bias, "gelu", cfg, 1)
    off, i_off = _run(dt, A, B, bias, "gelu", cfg, 0)
    assert i_off.span_copies == 0
    assert np.array_equal(device_bits(on), device_bits(off))
