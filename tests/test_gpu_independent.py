"""Launch ordering on one stream: a chain where each GEMM reads the previous
one's output (the default, every launch waits for the previous kernel before
touching memory), and independent GEMMs declared as such (operand loads start
while the previous kernel drains), both captured in CUDA graphs and replayed
many times, checked bit for bit."""
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


def test_dependent_chain_waits_for_its_producer():
    # C1 = relu(A·B1 + b1) feeds the next GEMM as its A: C2 = relu(C1·B2 + b2).
    M, K, N1, N2 = 256, 512, 384, 256
    A, B1, b1 = inputs.make_operands(M, N1, K, "bf16", "int", seed=60)
    _A2, B2, b2 = inputs.make_operands(M, N2, N1, "bf16", "int", seed=61)
    B2 = (B2.float() / 64).bfloat16()               # keep the second product's sums exact in fp32
    dA, dB1, db1, dB2, db2 = (t.cuda() for t in (A, B1, b1, B2, b2))
    C1 = torch.empty(M, N1, dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty(M, N2, dtype=torch.bfloat16, device="cuda")
    p1 = g.plan_with_config(M, N1, K, "bf16", "relu", C(128, 128, 64, 4, 0, 1, 2))
    p2 = g.plan_with_config(M, N2, N1, "bf16", "relu", C(128, 64, 64, 4))
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


@pytest.mark.parametrize("dtype,cfg", [("bf16", C(256, 256, 64, 4, 0, 1, 4, 2)), ("bf16", C(128, 16, 128, 5, 0, 1, 4, 1, 1)),
                                       ("fp32", C(128, 64, 32, 4, 0, 1, 2))])
def test_independent_inputs_give_the_same_bits(dtype, cfg):
    M, N, K = (40, 320, 2048) if cfg.swap_ab else (300, 320, 2048)
    sets = []
    for k in range(4):
        A, B, bias = inputs.make_operands(M, N, K, dtype, "int", seed=70 + k)
        sets.append((A, B, bias, A.cuda(), B.cuda(), bias.cuda(),
                     torch.empty(M, N, dtype=inputs.out_torch_dtype(dtype), device="cuda")))
    p = g.plan_with_config(M, N, K, dtype, "relu", cfg)
    p.set_independent_inputs(True)
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
