"""The explicit configurations the GPU tests launch are all feasible under the
default device parameters (checked here on the CPU, before any GPU run)."""
import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import _build


def test_gpu_case_configs_are_feasible():
    _build.build()
    import test_gpu_parity as t
    d = g.device_params_default()
    for (M, N, K), cfg in t.BF16_CASES:
        assert g.check_config(M, N, K, "bf16", "relu", cfg, d) == 0, cfg
    for (M, N, K), cfg in t.FP32_CASES:
        assert g.check_config(M, N, K, "fp32", "relu", cfg, d) == 0, cfg
