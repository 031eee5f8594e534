"""Full-size parity through tuned plans: every element of the workloads the
targets are quoted on, against the fp64 oracle.

  * Random inputs of each workload's distribution through the tuned plan (the
    plan and launch the bench times): normalised error
    max |C - C_ref| / (||a_i||·||b_j||) <= 2e-3 over every element.
  * Integer-valued inputs ({-2..2}, whose sums are exact in fp32) through the
    tuned configuration of the same workload, with the ReLU epilogue: every
    element bit-exact against the oracle rounded to the output type.  This
    covers the exact tile, pair, K step and split-K route the headline runs.

Workloads: the 256³ fp32 case, the under-filled 1000 x 1000 x 8192 ("Compilers
and Kernel Languages", "A different tile for every shape"), the large square
8192³ and the 16-token decode 16 x 8192 x 28672."""
import numpy as np
import pytest

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from gpu_util import TOL, alloc_out, device_bits, normalised_error, oracle_rounded_bits

pytestmark = pytest.mark.gpu

NAMES = ["fp32_relu_256", "bf16_gelu_1000x1000x8192", "bf16_decode_16x8192x28672", "bf16_relu_8192"]


def _run(plan, w, A, B, bias):
    Cd, _ = alloc_out(w.M, w.N, g.DTYPES[w.dtype])
    plan.run(A.cuda(), B.cuda(), bias.cuda() if (bias is not None and plan.epi != 0) else None, Cd)
    assert plan.status() == 0, g.last_error()
    return Cd.cpu()


@pytest.mark.parametrize("name", NAMES)
def test_tuned_plan_every_element_within_tolerance(name):
    w = inputs.WORKLOADS[name]
    A, B, bias = inputs.make_workload(w, seed=0)
    with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as p:
        got = _run(p, w, A, B, bias)
    assert normalised_error(got, A, B, bias, w.epi) <= TOL


@pytest.mark.parametrize("name", NAMES)
def test_tuned_configuration_bit_exact_on_integer_inputs(name):
    w = inputs.WORKLOADS[name]
    with g.plan(w.M, w.N, w.K, w.dtype, w.epi) as tuned:
        cfg = tuned.config
        route = tuned.launch_info.splitk_route
    A, B, bias = inputs.make_operands(w.M, w.N, w.K, w.dtype, "int", seed=7)
    with g.plan_with_config(w.M, w.N, w.K, w.dtype, "relu", cfg) as p:
        assert p.launch_info.splitk_route == route          # the same exchange route as the tuned plan
        got = _run(p, w, A, B, bias)
    assert np.array_equal(device_bits(got), oracle_rounded_bits(A, B, bias, "relu", g.DTYPES[w.dtype]))
