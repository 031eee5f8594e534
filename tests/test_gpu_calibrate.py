"""Calibration on the GPU: exhaustive timing tables of small shapes through the
library, a refit that does not lose against the shipped coefficients, and the
coefficient file applied by device_params_query through GEMM_MODEL_PARAMS."""
import os

import pytest

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import calibrate

pytestmark = pytest.mark.gpu
pytest.importorskip("scipy")


def test_measure_fit_save_and_apply(tmp_path):
    shapes = [(256, 512, 1024, "bf16", "relu"), (16, 2048, 2048, "bf16", "none")]
    tables = calibrate.measure(shapes)
    assert [len(t["rows"]) > 10 for t in tables] == [True, True]
    assert all(us > 0 for t in tables for _c, us in t["rows"])
    dev = g.device_params_query()
    fitted, before, after = calibrate.fit(tables, dev, max_evals=400)
    assert after <= before
    path = tmp_path / "params.txt"
    calibrate.save(str(path), fitted)
    os.environ["GEMM_MODEL_PARAMS"] = str(path)
    try:
        q = g.device_params_query()
    finally:
        del os.environ["GEMM_MODEL_PARAMS"]
    for n in calibrate.COEFFS:
        assert getattr(q, n) == pytest.approx(getattr(fitted, n), rel=1e-6), n
    assert q.sm_count == dev.sm_count
