"""Split-K through distributed shared memory: the K slices of a tile form one
thread-block cluster and push their fp32 partial tiles into the owning CTA's
shared memory.  Parity against the oracle (bit-exact on integer inputs), the
route actually taken (launch info), and bit-identity with the global-memory
exchange (both add the partials in slice order)."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from gpu_util import alloc_out, device_bits, guard_intact, normalised_error, operands, oracle_rounded_bits

pytestmark = pytest.mark.gpu

C = g.make_config
ROUTE_CLUSTER = 3

# Ragged M/N/K; cluster sizes 2, 4 and 8, both tile heights, bn 64..256, blocks
# owned in pairs and one by one, a grouped raster, swapped tiles; every launch
# fits one wave (the route is taken only then).
CASES = [
    ("bf16", (300, 320, 1032), C(256, 128, 64, 4, 0, 1, 4)),
    ("bf16", (300, 320, 1032), C(128, 256, 64, 4, 0, 1, 2)),
    ("bf16", (300, 320, 1032), C(256, 256, 64, 3, 0, 1, 2)),
    ("bf16", (300, 320, 1032), C(128, 128, 64, 4, 0, 1, 4)),
    ("bf16", (520, 640, 1032), C(128, 64, 64, 4, 0, 4, 2)),
    ("bf16", (1000, 1000, 2056), C(256, 128, 128, 2, 0, 1, 4)),
    ("bf16", (1024, 1024, 512), C(128, 128, 64, 4, 0, 1, 2)),   # 128 units
    ("bf16", (264, 136, 4096), C(128, 64, 64, 6, 0, 1, 8)),
    ("fp32", (200, 160, 264), C(128, 64, 32, 4, 0, 1, 2)),
    ("fp32", (200, 160, 264), C(128, 128, 32, 4, 0, 1, 4)),
    # Swapped (tokens along the MMA's N): blocks of 128 rows x 16 columns.
    ("bf16", (16, 4096, 1024), C(128, 16, 128, 4, 0, 1, 4, 1, 1)),   # one block per tile, one owner
    ("bf16", (20, 320, 1032), C(128, 32, 64, 4, 0, 1, 2, 1, 1)),     # ragged tokens, rows and K
    ("bf16", (40, 264, 2056), C(256, 64, 64, 3, 0, 1, 4, 1, 1)),     # two halves, blocks owned in pairs
    ("bf16", (16, 1024, 4096), C(128, 16, 128, 4, 0, 1, 8, 1, 1)),   # cluster of 8
    ("fp32", (24, 200, 264), C(128, 32, 32, 4, 0, 1, 2, 1, 1)),
    ("bf16", (100, 264, 1032), C(128, 128, 64, 4, 0, 1, 2, 1, 1)),   # eight chunks per half
]


def _id(c):
    dt, (M, N, K), cfg = c
    return f"{dt}-{M}x{N}x{K}-{'x'.join(str(v) for v in cfg.astuple())}"


def _run(dt, A, B, bias, epi, cfg, route, guard=64):
    M, K = A.shape
    N = B.shape[1]
    dtc = g.BF16 if dt == "bf16" else g.FP32_TF32
    g.debug_set(3, route)
    try:
        p = g.plan_with_config(M, N, K, dtc, epi, cfg)
    finally:
        g.debug_set(3, 0)
    with p:
        info = p.launch_info
        Cd, buf = alloc_out(M, N, dtc, guard)
        p.run(A.cuda(), B.cuda(), bias.cuda() if epi != "none" else None, Cd)
        assert p.status() == 0, g.last_error()
    return Cd.cpu(), guard_intact(buf, guard, M, N), info


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("epi", ["relu", "none"])
def test_cluster_route_integer_inputs_bit_exact(case, epi):
    dt, (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, dt, "int", seed=11)
    out, guard_ok, info = _run(dt, A, B, bias, epi, cfg, route=0)
    if info.splitk_route != ROUTE_CLUSTER:
        pytest.fail(f"expected the cluster route, got {g.SPLITK_ROUTES[info.splitk_route]}")
    assert info.cluster == cfg.split_k and info.grid == info.units
    assert guard_ok, "write outside C"
    want = oracle_rounded_bits(A, B, bias, epi, g.BF16 if dt == "bf16" else g.FP32_TF32)
    bad = np.argwhere(device_bits(out) != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


@pytest.mark.parametrize("case", CASES[::3], ids=_id)
def test_cluster_and_global_exchange_agree_bitwise(case):
    dt, (M, N, K), cfg = case
    A, B, bias = operands(M, N, K, dt, "scaled_normal", seed=12)
    c_cluster, ok1, i1 = _run(dt, A, B, bias, "gelu", cfg, route=0)
    c_global, ok2, i2 = _run(dt, A, B, bias, "gelu", cfg, route=1)
    assert i1.splitk_route == ROUTE_CLUSTER and i2.splitk_route in (1, 2)
    assert ok1 and ok2
    assert np.array_equal(device_bits(c_cluster), device_bits(c_global))
    assert normalised_error(c_cluster, A, B, bias, "gelu") <= 2e-3


def test_cluster_route_is_deterministic():
    dt, (M, N, K), cfg = CASES[0]
    A, B, bias = operands(M, N, K, dt, "scaled_normal", seed=13)
    runs = [device_bits(_run(dt, A, B, bias, "bias", cfg, route=0)[0]) for _ in range(3)]
    assert all(np.array_equal(runs[0], r) for r in runs[1:])


@pytest.mark.parametrize("shape,cfg", [
    ((300, 320, 1032), C(256, 256, 64, 3, 0, 1, 8)),   # an owner would receive 2 x 7 x 16 KB > its 192 KB ring
    ((2048, 2048, 512), C(128, 128, 64, 4, 0, 1, 2)),  # 512 units: more than one wave
])
def test_other_split_plans_keep_the_global_exchange(shape, cfg):
    M, N, K = shape
    A, B, bias = operands(M, N, K, "bf16", "int", seed=14)
    out, ok, info = _run("bf16", A, B, bias, "relu", cfg, route=0)
    assert info.splitk_route in (1, 2) and info.cluster == 1
    assert ok and np.array_equal(device_bits(out), oracle_rounded_bits(A, B, bias, "relu", g.BF16))


# CTA pairs: persistent pairs walking many units (accumulator hand-back between
# the two CTAs), and split-K on pairs through every route: the S pairs of a
# tile as one cluster of 2S CTAs (distributed shared memory), and, forced, the
# global-memory routes.
PAIR_CASES = [
    # (shape, config, forced route, expected route, expected cluster size)
    ((2048, 2048, 512), C(256, 128, 64, 6, 0, 1, 1, 2), 0, 0, 2),     # 128 units on at most 76 pairs
    ((300, 320, 2056), C(256, 256, 64, 6, 0, 1, 4, 2), 0, 3, 8),      # 4 pairs per cluster, few clusters
    ((1000, 1000, 2056), C(256, 256, 64, 6, 0, 1, 4, 2), 0, 2, 2),    # 16 clusters of 8 would not all fit: cooperative
    ((300, 320, 2056), C(256, 256, 64, 6, 0, 1, 4, 2), 1, 2, 2),      # forced global: cooperative
    ((520, 640, 1032), C(256, 128, 64, 4, 0, 1, 2, 2), 0, 3, 4),      # bn 128, 2 pairs per cluster
    ((2048, 2048, 1024), C(256, 256, 64, 4, 0, 1, 2, 2), 0, 1, 2),    # more units than pairs: last arriver
]


@pytest.mark.parametrize("shape,cfg,force,route,cluster", PAIR_CASES, ids=lambda v: str(v))
def test_cta_pair_plans_bit_exact(shape, cfg, force, route, cluster):
    M, N, K = shape
    A, B, bias = operands(M, N, K, "bf16", "int", seed=15)
    out, ok, info = _run("bf16", A, B, bias, "relu", cfg, route=force)
    assert info.cluster == cluster and info.grid % 2 == 0 and info.splitk_route == route
    assert ok and np.array_equal(device_bits(out), oracle_rounded_bits(A, B, bias, "relu", g.BF16))


@pytest.mark.parametrize("shape,cfg", [((300, 320, 2056), C(256, 256, 64, 6, 0, 1, 4, 2)),
                                       ((520, 640, 1032), C(256, 128, 64, 4, 0, 1, 2, 2))])
def test_pair_cluster_and_global_exchange_agree_bitwise(shape, cfg):
    M, N, K = shape
    A, B, bias = operands(M, N, K, "bf16", "scaled_normal", seed=17)
    c_cluster, ok1, i1 = _run("bf16", A, B, bias, "gelu", cfg, route=0)
    c_global, ok2, i2 = _run("bf16", A, B, bias, "gelu", cfg, route=1)
    assert i1.splitk_route == ROUTE_CLUSTER and i1.cluster == 2 * cfg.split_k and i2.splitk_route in (1, 2)
    assert ok1 and ok2
    assert np.array_equal(device_bits(c_cluster), device_bits(c_global))
    assert normalised_error(c_cluster, A, B, bias, "gelu") <= 2e-3


def test_cta_pair_agrees_with_single_cta_tiles_bitwise_on_integers_and_within_tolerance():
    M, N, K = 520, 1000, 2056
    A, B, bias = operands(M, N, K, "bf16", "scaled_normal", seed=16)
    pair, ok1, i1 = _run("bf16", A, B, bias, "gelu", C(256, 256, 64, 6, 0, 1, 1, 2), route=0)
    single, ok2, i2 = _run("bf16", A, B, bias, "gelu", C(256, 256, 64, 3, 0, 1, 1, 1), route=0)
    assert i1.cluster == 2 and i2.cluster == 1 and ok1 and ok2
    assert normalised_error(pair, A, B, bias, "gelu") <= 2e-3
    assert normalised_error(single, A, B, bias, "gelu") <= 2e-3
