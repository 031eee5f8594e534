"""Launch ordering on one stream under programmatic overlap: chains where each
GEMM reads the previous one's output as A (nothing declared, or only B, the
weights, declared independent: B's first stages are copied early, A after the
previous kernel has finished) and independent GEMMs with both operands
declared, all captured in CUDA graphs, replayed many times and checked bit for
bit."""
import numpy as np
import pytest
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import device_bits, oracle_rounded_bits

pytestmark = pytest.mark.gpu
C = g.make_config


def _graph(fn, stream):
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        fn(torch.cuda.current_stream())
    return gr


# (M, second GEMM's config): unswapped with a cooperative split-K, a CTA pair,
# and swapped (the weights are then the kernel's first operand).
CHAIN = [(256, C(128, 64, 64, 4)), (256, C(128, 128, 64, 4, 0, 1, 3)), (256, C(256, 128, 64, 4, 0, 1, 1, 2)),
         (40, C(128, 64, 64, 4, 0, 1, 2, 1, 1))]


@pytest.mark.parametrize("declared", ["", "B"])
@pytest.mark.parametrize("M,cfg2", CHAIN, ids=lambda v: "x".join(str(x) for x in v.astuple()) if hasattr(v, "astuple") else str(v))
def test_chain_reads_its_producers_output(declared, M, cfg2):
    # C1 = relu(A·B1 + b1) feeds the next GEMM as its A: C2 = relu(C1·B2 + b2).
    K, N1, N2 = 2048, 384, 256
    A, B1, b1 = inputs.make_operands(M, N1, K, "bf16", "int", seed=60)
    _A2, B2, b2 = inputs.make_operands(M, N2, N1, "bf16", "int", seed=61)
    B2 = (B2.float() / 64).bfloat16()               # keep the second product's sums exact in fp32
    dA, dB1, db1, dB2, db2 = (t.cuda() for t in (A, B1, b1, B2, b2))
    C1 = torch.empty(M, N1, dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")
    p1 = g.plan_with_config(M, N1, K, "bf16", "relu", C(128, 128, 64, 4, 0, 1, 2, 1, 1 if M < 128 else 0))
    p2 = g.plan_with_config(M, N2, N1, "bf16", "relu", cfg2)
    p1.set_independent_operands(declared)
    p2.set_independent_operands(declared)
    s = torch.cuda.Stream()

    def chain(st):
        for _ in range(4):
            C1.zero_()
            p1.run(dA, dB1, db1, C1, st)
            p2.run(C1, dB2, db2, C2, st)

    with torch.cuda.stream(s):
        chain(s)
    torch.cuda.synchronize()
    gr = _graph(chain, s)
    for _ in range(20):
        gr.replay()
    torch.cuda.synchronize()
    assert p1.status() == 0 and p2.status() == 0
    want1 = oracle_rounded_bits(A, B1, b1, "relu", g.BF16)
    assert np.array_equal(device_bits(C1.cpu()), want1)
    assert np.array_equal(device_bits(C2.cpu()), oracle_rounded_bits(C1.cpu(), B2, b2, "relu", g.BF16))
    p1.close()
    p2.close()


@pytest.mark.parametrize("declared", ["B", "AB"])
@pytest.mark.parametrize("dtype,cfg", [("bf16", C(256, 256, 64, 4, 0, 1, 4, 2)), ("bf16", C(128, 16, 128, 5, 0, 1, 4, 1, 1)),
                                       ("fp32", C(128, 64, 32, 4, 0, 1, 2))])
def test_declared_operands_give_the_same_bits(declared, dtype, cfg):
    M, N, K = (40, 320, 2048) if cfg.swap_ab else (300, 320, 2048)
    sets = []
    for k in range(4):
        A, B, bias = inputs.make_operands(M, N, K, dtype, "int", seed=70 + k)
        sets.append((A, B, bias, A.cuda(), B.cuda(), bias.cuda(),
                     torch.empty(M, N, dtype=inputs.out_torch_dtype(dtype), device="cuda")))
    p = g.plan_with_config(M, N, K, dtype, "relu", cfg)
    p.set_independent_operands(declared)
    s = torch.cuda.Stream()

    def step(st):
        for (_A, _B, _b, dA, dB, db, dC) in sets:
            p.run(dA, dB, db, dC, st)

    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    gr = _graph(step, s)
    for _ in range(30):
        gr.replay()
    torch.cuda.synchronize()
    assert p.status() == 0, g.last_error()
    kind = g.BF16 if dtype == "bf16" else g.FP32_TF32
    for (A, B, bias, _dA, _dB, _db, dC) in sets:
        assert np.array_equal(device_bits(dC.cpu()), oracle_rounded_bits(A, B, bias, "relu", kind))
    p.close()


@pytest.mark.parametrize("declared", ["B", "AB"])
@pytest.mark.parametrize("cfg", [C(256, 256, 128, 3, 0, 1, 1, 2), C(128, 32, 128, 6, 0, 1, 1, 1, 1)])
def test_block_scaled_with_declared_operands_and_a_bias_written_just_before(declared, cfg):
    # A bf16 GEMM writes the bias vector's row that the block-scaled GEMM then
    # reads in its epilogue, which always waits for the previous kernel.
    from oracle import gemm as og
    from oracle import mx
    M, N, K = (20, 320, 1024) if cfg.swap_ab else (300, 256, 1024)
    A, SA, B, SB, _bias = inputs.make_mx_operands(M, N, K, "int", seed=80)
    Ab, Bb, bb = inputs.make_operands(1, N, 512, "bf16", "int", seed=81)
    dAb, dBb, dbb = Ab.cuda(), Bb.cuda(), bb.cuda()
    bias_row = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    pb = g.plan_with_config(1, N, 512, "bf16", "relu", C(128, 32, 64, 4, 0, 1, 1, 1, 1))
    p = g.plan_with_config(M, N, K, "mxfp8", "relu", cfg)
    p.set_independent_operands(declared)
    sa = g.mx_pack_scales(SA.cuda(), M, K, False)
    sb = g.mx_pack_scales(SB.cuda(), N, K, True)
    dA, dB = A.cuda(), B.cuda()
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()

    def step(st):
        for _ in range(3):
            bias_row.zero_()
            pb.run(dAb, dBb, dbb, bias_row, st)
            p.run_mx(dA, sa, dB, sb, bias_row.view(N), Cd, None, st)

    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    gr = _graph(step, s)
    for _ in range(20):
        gr.replay()
    torch.cuda.synchronize()
    assert p.status() == 0 and pb.status() == 0
    bias_bits = oracle_rounded_bits(Ab, Bb, bb, "relu", g.BF16)
    assert np.array_equal(device_bits(bias_row.cpu()), bias_bits)
    want = og.round_bf16_bits(mx.mx_gemm(A, SA, B, SB, bias_row.cpu().view(N), g.EPILOGUES["relu"]))
    assert np.array_equal(device_bits(Cd.cpu()), want)
    p.close()
    pb.close()


def test_operand_mask_is_checked():
    with g.plan_with_config(256, 256, 256, "bf16", "relu", C(128, 128, 64, 4)) as p:
        with pytest.raises(ValueError):
            p.set_independent_operands("C")
        with pytest.raises(g.GemmError) as e:
            g._check(g.lib().gemm_plan_set_independent_operands(p._h, 4))
        assert e.value.code == g.ERR_INVALID_ARG
