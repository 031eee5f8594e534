"""Block-scaled FP8 (MX: E4M3 elements, one E8M0 scale per 32 elements of K;
tcgen05.mma kind::mxf8f6f4.block_scale, scales staged through TMEM) against the
oracle, which dequantizes the same bytes from the format's definition:
bit-exact on small-integer inputs, within the stated tolerance on random ones,
on every tile shape, K step, tile order, operand swap, CTA pair and split-K route the rules allow; the
scale packing against the documented layout; argument checks."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import alloc_out, device_bits, guard_intact
from oracle import gemm as og
from oracle import mx

pytestmark = pytest.mark.gpu

C = g.make_config

CASES = [
    ((256, 256, 512), C(128, 128, 128, 4), 0),
    ((300, 320, 1008), C(128, 128, 128, 4), 0),                # ragged M, N and a 16-element last block
    ((300, 320, 1024), C(128, 256, 128, 3), 0),                # two B scale atoms per stage
    ((300, 320, 1024), C(256, 128, 128, 3), 0),                # two A halves
    ((300, 320, 1024), C(128, 128, 256, 2), 0),                # two K atoms per stage
    ((520, 640, 384), C(128, 128, 128, 4, 1, 4), 0),           # grouped raster, K ragged to the stage
    ((300, 320, 2048), C(128, 128, 128, 4, 0, 1, 4), 0),       # split-K, cluster route
    ((300, 320, 2048), C(128, 128, 128, 4, 0, 1, 4), 1),       # split-K, cooperative route
    ((200, 136, 512), C(128, 128, 128, 4), 0),                 # N % 16 != 0: B from a K-major copy
    ((1000, 1000, 4096), C(128, 128, 128, 4, 0, 1, 3), 0),     # split-K over several waves (last arriver)
    ((20, 320, 1024), C(128, 32, 128, 6, 0, 1, 1, 1, 1), 0),   # swapped: tokens along N, one token tile
    ((40, 264, 1024), C(256, 64, 128, 2, 0, 1, 3, 1, 1), 0),   # swapped, split-K, B from a K-major copy
    ((200, 256, 512), C(128, 128, 128, 4, 0, 1, 1, 1, 1), 0),  # swapped, two token tiles of one atom each
    ((300, 320, 1024), C(256, 256, 128, 3, 0, 1, 1, 2), 0),    # CTA pair (each CTA holds all B scales)
    ((1000, 1000, 4096), C(256, 256, 128, 3, 0, 1, 4, 2), 0),  # CTA pair, split-K (cluster of 4 pairs), B K-major
    ((1000, 1000, 4096), C(256, 256, 128, 3, 0, 1, 4, 2), 1),  # the same on the cooperative route
    ((200, 136, 512), C(256, 128, 128, 4, 0, 1, 1, 2), 0),     # CTA pair, bn 128, two accumulators
]


def _id(c):
    (M, N, K), cfg, route = c
    return f"{M}x{N}x{K}-{'x'.join(str(v) for v in cfg.astuple())}-r{route}"


def _packed(SA, SB, M, N, K):
    sa = g.mx_pack_scales(SA.cuda(), M, K, False)
    sb = g.mx_pack_scales(SB.cuda(), N, K, True)
    return sa, sb


def _run(A, SA, B, SB, bias, epi, cfg, route=0, alpha=1.0, R=None, guard=64):
    M, K = A.shape
    N = B.shape[1]
    g.debug_set(3, route)
    try:
        p = g.plan_with_config(M, N, K, "mxfp8", epi, cfg)
    finally:
        g.debug_set(3, 0)
    with p:
        p.set_scale(alpha)
        sa, sb = _packed(SA, SB, M, N, K)
        Cd, buf = alloc_out(M, N, g.BF16, guard)
        bd = bias.cuda() if bias is not None and epi != "none" else None
        p.run_mx(A.cuda(), sa, B.cuda(), sb, bd, Cd, R.cuda() if R is not None else None)
        assert p.status() == 0, g.last_error()
        info = p.launch_info
    return Cd.cpu(), guard_intact(buf, guard, M, N), info


@pytest.mark.parametrize("case", CASES, ids=_id)
@pytest.mark.parametrize("epi,alpha", [("relu", 1.0), ("none", 0.5)])
def test_mxfp8_integer_inputs_bit_exact(case, epi, alpha):
    (M, N, K), cfg, route = case
    A, SA, B, SB, bias = inputs.make_mx_operands(M, N, K, "int", seed=41)
    out, ok, info = _run(A, SA, B, SB, bias, epi, cfg, route, alpha)
    assert ok, "write outside C"
    assert info.b_transposed == (0 if N % 16 == 0 else 1)
    want = og.round_bf16_bits(mx.mx_gemm(A, SA, B, SB, bias if epi != "none" else None, g.EPILOGUES[epi],
                                         alpha=alpha))
    bad = np.argwhere(device_bits(out) != want)
    assert bad.size == 0, f"{len(bad)} mismatches ({g.SPLITK_ROUTES[info.splitk_route]}), first {bad[:5].tolist()}"


def _normalised_error(out, A, SA, B, SB, ref, alpha):
    Ad = mx.dequantize_a(A, SA)
    Bd = mx.dequantize_b(B, SB)
    scale = abs(alpha) * np.sqrt((Ad ** 2).sum(1))[:, None] * np.sqrt((Bd ** 2).sum(0))[None, :]
    return float((np.abs(out.float().numpy() - ref) / np.maximum(scale, 1e-30)).max())


@pytest.mark.parametrize("case", CASES[::2] + [CASES[1]], ids=_id)
def test_mxfp8_random_gelu_within_tolerance(case):
    (M, N, K), cfg, route = case
    A, SA, B, SB, bias = inputs.make_mx_operands(M, N, K, "scaled_normal", seed=42)
    alpha = 0.75
    out, ok, _ = _run(A, SA, B, SB, bias, "gelu", cfg, route, alpha)
    ref = mx.mx_gemm(A, SA, B, SB, bias, mx.EPI_BIAS_GELU, alpha=alpha)
    assert ok and _normalised_error(out, A, SA, B, SB, ref, alpha) <= 2e-3


def test_mxfp8_scales_matter_per_block():
    """Scales that differ from block to block (decode-like spread) change the
    result, and the device follows each one: compared with the result of all
    unit scales, both sides move identically."""
    M, N, K = 256, 256, 1024
    A, SA, B, SB, bias = inputs.make_mx_operands(M, N, K, "int", seed=43)
    cfg = C(128, 128, 128, 4)
    out, _, _ = _run(A, SA, B, SB, bias, "none", cfg)
    ones_a, ones_b = torch.full_like(SA, 127), torch.full_like(SB, 127)
    plain, _, _ = _run(A, ones_a, B, ones_b, bias, "none", cfg)
    assert not np.array_equal(device_bits(out), device_bits(plain))
    want = og.round_bf16_bits(mx.mx_gemm(A, ones_a, B, ones_b))
    assert np.array_equal(device_bits(plain), want)


def test_mxfp8_residual_in_place_and_tuned_plan():
    M, N, K = 512, 1024, 2048
    A, SA, B, SB, bias = inputs.make_mx_operands(M, N, K, "int", seed=44)
    R = inputs.make_residual(M, N, "mxfp8", "int", seed=44)
    with g.plan(M, N, K, "mxfp8", "relu_residual") as p:
        tuned = p.config
        assert tuned.cta_group == 1 and tuned.swap_ab == 0 and tuned.bn in (128, 256)
        sa, sb = _packed(SA, SB, M, N, K)
        Cd = R.cuda().clone()                      # C += relu(A·B + bias), in place
        p.run_mx(A.cuda(), sa, B.cuda(), sb, bias.cuda(), Cd, Cd)
        assert p.status() == 0
    want = og.round_bf16_bits(mx.mx_gemm(A, SA, B, SB, bias, 5, residual=R))
    assert np.array_equal(device_bits(Cd.cpu()), want), tuned.astuple()


@pytest.mark.parametrize("name", ["mxfp8_gelu_1000x1000x8192", "mxfp8_decode_16x8192x28672", "mxfp8_relu_8192"])
def test_mxfp8_full_size_sampled_entries(name):
    w = inputs.WORKLOADS[name]
    A, SA, B, SB, bias = inputs.make_mx_workload(w, seed=0)
    with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as p:
        sa, sb = _packed(SA, SB, w.M, w.N, w.K)
        Cd = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
        p.run_mx(A.cuda(), sa, B.cuda(), sb, bias.cuda() if bias is not None else None, Cd)
        assert p.status() == 0
    rng = np.random.default_rng(0)
    rows = np.concatenate([[0, w.M - 1], rng.integers(0, w.M, 60)])
    cols = np.concatenate([[0, w.N - 1], rng.integers(0, w.N, 60)])
    ref = mx.mx_gemm_entries(A, SA, B, SB, bias, g.EPILOGUES[w.epi], rows, cols)
    got = Cd.cpu().float().numpy()[rows, cols]
    Ad = mx.dequantize_a(A.view(torch.uint8).numpy()[rows], SA.numpy()[rows])
    Bd = mx.dequantize_b(B.view(torch.uint8).numpy()[:, cols], SB.numpy()[:, cols])
    scale = np.sqrt((Ad ** 2).sum(1)) * np.sqrt((Bd ** 2).sum(0))
    assert float((np.abs(got - ref) / scale).max()) <= 2e-3


@pytest.mark.parametrize("rows,K,b_side", [(300, 1008, False), (136, 512, True), (1, 32, False), (257, 300, True)])
def test_scale_packing_follows_the_documented_layout(rows, K, b_side):
    kb = (K + 31) // 32
    gen = torch.Generator().manual_seed(rows + K)
    S = torch.randint(0, 255, (kb, rows) if b_side else (rows, kb), generator=gen, dtype=torch.uint8)
    packed = g.mx_pack_scales(S.cuda(), rows, K, b_side).cpu().numpy()
    nbytes = g.mx_scales_bytes(rows, K)
    KT = 2 * ((K + 255) // 256)
    assert nbytes == 2 * ((rows + 255) // 256) * KT * 512
    want = np.zeros(nbytes, np.uint8)
    Sn = S.numpy()
    for r in range(rows):
        for j in range(kb):
            off = ((r // 128) * KT + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
            want[off] = Sn[j, r] if b_side else Sn[r, j]
    assert np.array_equal(packed[:nbytes], want)


def test_mx_plan_rejects_the_unscaled_entry_points_and_vice_versa():
    M, N, K = 256, 256, 256
    A, SA, B, SB, bias = inputs.make_mx_operands(M, N, K, "int", seed=45)
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    with g.plan_with_config(M, N, K, "mxfp8", "relu", C(128, 128, 128, 4)) as p:
        with pytest.raises(g.GemmError) as e:
            p.run(A.cuda(), B.cuda(), bias.cuda(), Cd)
        assert e.value.code == g.ERR_INVALID_ARG
    with g.plan_with_config(M, N, K, "fp8", "relu", C(128, 128, 128, 4)) as p:
        sa, sb = _packed(SA, SB, M, N, K)
        with pytest.raises(g.GemmError) as e:
            p.run_mx(A.cuda(), sa, B.cuda(), sb, bias.cuda(), Cd)
        assert e.value.code == g.ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:       # B's scales come in 128-column atoms: bn 192 is refused
        g.plan_with_config(M, N, K, "mxfp8", "relu", C(128, 192, 128, 3))
    assert e.value.code == g.ERR_INFEASIBLE


@pytest.mark.parametrize("shape,cfg,cluster", [((300, 320, 2048), C(256, 256, 128, 3, 0, 1, 4, 2), 8),
                                               ((300, 320, 2048), C(256, 256, 128, 3, 0, 1, 2, 2), 4)])
def test_mxfp8_pair_tiles_reduce_inside_a_cluster(shape, cfg, cluster):
    # Block-scaled pair tiles whose K slices form one cluster of 2S CTAs: the
    # partials land in the ring that also held the scale atoms.
    M, N, K = shape
    A, SA, B, SB, bias = inputs.make_mx_operands(M, N, K, "int", seed=46)
    out, ok, info = _run(A, SA, B, SB, bias, "relu", cfg, 0, 0.5)
    assert ok and info.splitk_route == 3 and info.cluster == cluster
    want = og.round_bf16_bits(mx.mx_gemm(A, SA, B, SB, bias, g.EPILOGUES["relu"], alpha=0.5))
    assert np.array_equal(device_bits(out), want)
    coop, ok2, info2 = _run(A, SA, B, SB, bias, "relu", cfg, 1, 0.5)
    assert ok2 and info2.splitk_route == 2 and np.array_equal(device_bits(coop), device_bits(out))
