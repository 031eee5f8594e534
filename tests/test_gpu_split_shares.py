"""One-wave split-K through global memory, finalised share by share (split-K
route 2).

Each K slice of a tile owns a share of the tile's blocks; a share's owner
finalises it once the other slices have arrived on it, and an owner whose peers
do not arrive within its bounded wait hands the share to whichever slice
arrives last.  No slice ever waits for one that may not be resident.  Checked
here:
  * parity with the oracle, bit-exact on integer inputs, for single CTAs, CTA
    pairs and swapped tiles, both with the owners' wait and with owners that
    hand every share over at once (gemm_debug_set(5, 0));
  * the two protocols give the same bits on random inputs (both sum the
    partials in slice order);
  * two such plans that each need more than half of the SMs, launched on two
    streams at once, so that some slices of each are not resident while the
    other kernel runs: status 0 under a short device wait limit, and
    bit-exact results (the page's under-filled 1000 x 1000 x 8192, "Compilers
    and Kernel Languages", "A different tile for every shape")."""
import time

import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from gpu_util import alloc_out, device_bits, guard_intact, operands, oracle_rounded_bits

pytestmark = pytest.mark.gpu

C = g.make_config
ROUTE_SHARES = 2

CASES = [
    ("bf16", (300, 320, 1032), C(256, 128, 64, 4, 0, 1, 4)),          # 2 halves, 4 shares
    ("bf16", (300, 320, 1032), C(128, 128, 64, 4, 0, 1, 3)),          # 3 shares
    ("bf16", (264, 320, 2056), C(128, 64, 64, 4, 0, 1, 6)),           # 2 chunks, 6 shares of 8 blocks
    ("bf16", (1000, 1000, 2056), C(256, 256, 64, 6, 0, 1, 4, 2)),     # CTA pair
    ("bf16", (300, 320, 2056), C(256, 128, 64, 4, 0, 1, 2, 2)),       # CTA pair, bn 128
    ("fp32", (200, 160, 264), C(128, 64, 32, 4, 0, 1, 2)),
    ("bf16", (16, 1024, 2048), C(128, 16, 128, 4, 0, 1, 12, 1, 1)),   # swapped, 12 shares
    ("bf16", (40, 264, 2056), C(256, 64, 64, 3, 0, 1, 4, 1, 1)),      # swapped, two halves
]


def _id(c):
    dt, (M, N, K), cfg = c
    return f"{dt}-{M}x{N}x{K}-{'x'.join(str(v) for v in cfg.astuple())}"


def _plan(M, N, K, dtc, epi, cfg):
    g.debug_set(3, 1)                   # global-memory exchange (no clusters)
    try:
        return g.plan_with_config(M, N, K, dtc, epi, cfg)
    finally:
        g.debug_set(3, 0)


def _run(dt, A, B, bias, epi, cfg, poll=None, guard=64):
    M, K = A.shape
    N = B.shape[1]
    dtc = g.BF16 if dt == "bf16" else g.FP32_TF32
    with _plan(M, N, K, dtc, epi, cfg) as p:
        assert p.launch_info.splitk_route == ROUTE_SHARES
        Cd, buf = alloc_out(M, N, dtc, guard)
        if poll is not None:
            g.debug_set(5, poll)
        try:
            for _ in range(2):          # the second launch starts from grown counts
                p.run(A.cuda(), B.cuda(), bias.cuda() if epi != "none" else None, Cd)
            st = p.status()
        finally:
            g.debug_set(5, 50000)
        assert st == 0, g.last_error()
        return Cd.cpu(), guard_intact(buf, guard, M, N)


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("poll", [None, 0], ids=["owners-wait", "owners-hand-over"])
def test_shares_bit_exact_on_integer_inputs(case, poll):
    dt, (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, dt, "int", seed=3)
    got, ok = _run(dt, A, B, bias, "relu", cfg, poll)
    assert ok
    dtc = g.BF16 if dt == "bf16" else g.FP32_TF32
    assert np.array_equal(device_bits(got), oracle_rounded_bits(A, B, bias, "relu", dtc))


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_owner_and_handover_give_the_same_bits(case):
    dt, (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, dt, "scaled_normal", seed=4)
    a, _ = _run(dt, A, B, bias, "gelu", cfg, None)
    b, _ = _run(dt, A, B, bias, "gelu", cfg, 0)
    assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("cfg", [C(256, 256, 128, 3, 0, 1, 4, 2),      # 64 pairs = 128 CTAs
                                 C(128, 128, 64, 4, 0, 1, 2)],         # 128 single CTAs
                         ids=["pairs", "single"])
def test_two_streams_each_over_half_the_sms(cfg):
    M, N, K = 1000, 1000, 8192
    props = torch.cuda.get_device_properties(0)
    A, B, bias = operands(M, N, K, "bf16", "int", seed=5)
    A2, B2, bias2 = operands(M, N, K, "bf16", "int", seed=6)
    want1 = oracle_rounded_bits(A, B, bias, "relu", g.BF16)
    want2 = oracle_rounded_bits(A2, B2, bias2, "relu", g.BF16)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    p1 = _plan(M, N, K, g.BF16, "relu", cfg)
    p2 = _plan(M, N, K, g.BF16, "relu", cfg)
    try:
        assert p1.launch_info.splitk_route == ROUTE_SHARES
        ctas = p1.launch_info.grid
        assert ctas > props.multi_processor_count // 2
        d1 = [t.cuda() for t in (A, B, bias)]
        d2 = [t.cuda() for t in (A2, B2, bias2)]
        C1 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        C2 = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        # a device wait limit far below the default 2 s: nothing may rely on it
        g.debug_set(0, 100_000_000)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(20):
            with torch.cuda.stream(s1):
                p1.run(*d1, C1, stream=s1)
            with torch.cuda.stream(s2):
                p2.run(*d2, C2, stream=s2)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        assert p1.status() == 0, g.last_error()
        assert p2.status() == 0, g.last_error()
    finally:
        g.debug_set(0, 2_000_000_000)
        p1.close()
        p2.close()
    assert wall < 1.0, wall
    assert np.array_equal(device_bits(C1.cpu()), want1)
    assert np.array_equal(device_bits(C2.cpu()), want2)
