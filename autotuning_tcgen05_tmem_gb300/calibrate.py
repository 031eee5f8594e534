"""Per-device calibration of the cost model.

"Tile Selection: Cost Models Against Measurement" ("Selection is per device")
holds that the best tile depends on the device, and "Autotuning & cost models"
§6 pairs an analytical model with measurement.  This module closes that loop
for the library's own model: it times every candidate of a few shapes on the
current device (exhaustive, interleaved CUDA-event timing through the library),
fits the model's coefficients to those timings by least squares in log time,
and writes them as a "name value" file that `gemm_model_params_load` and the
GEMM_MODEL_PARAMS variable apply.  The model itself is always the library's
(`gemm_model_predict` through the C ABI); nothing here restates it.

    python -m autotuning_tcgen05_tmem_gb300.calibrate --workloads a,b,c --out params.txt
"""
from __future__ import annotations

import argparse
import json
import math
import sys

from . import (DeviceParams, SEARCH_EXHAUSTIVE, device_params_default, device_params_query, make_config,
               model_predict, rank_agreement, tune_search)

# Coefficients fitted by default: the ones the model cannot read off the device.
COEFFS = ("l2_gbs", "mma_issue_clk", "kblock_clk", "mem_latency_us", "epi_elems_per_clk", "epi_gelu_elems_per_clk",
          "splitk_gbs", "launch_us")


def measure(shapes) -> list:
    """Exhaustive timing tables: for each (M, N, K, dtype, epi) a dict with the
    shape and rows [(config tuple, measured microseconds)] (GPU required)."""
    tables = []
    for (M, N, K, dtype, epi) in shapes:
        r = tune_search(M, N, K, dtype, epi, SEARCH_EXHAUSTIVE, 0)
        rows = [(tuple(x.config.astuple()), float(x.measured_us)) for x in r.rows if x.measured_us > 0]
        tables.append({"M": M, "N": N, "K": K, "dtype": dtype, "epi": epi, "rows": rows})
    return tables


def _with(dev: DeviceParams, names, values) -> DeviceParams:
    d = DeviceParams()
    for f, _t in DeviceParams._fields_:
        setattr(d, f, getattr(dev, f))
    for n, v in zip(names, values):
        setattr(d, n, float(v))
    return d


def loss(tables, dev: DeviceParams) -> float:
    """Mean squared log error of the model's predictions against the tables."""
    err, n = 0.0, 0
    for t in tables:
        for cfg, us in t["rows"]:
            p = model_predict(t["M"], t["N"], t["K"], t["dtype"], t["epi"], make_config(*cfg), dev).predicted_us
            err += (math.log(p) - math.log(us)) ** 2
            n += 1
    return err / max(n, 1)


def rank_stats(tables, dev: DeviceParams) -> dict:
    """Median Kendall tau and mean top-1 hit of the model's ranking per table."""
    taus, hits = [], []
    for t in tables:
        pred = [model_predict(t["M"], t["N"], t["K"], t["dtype"], t["epi"], make_config(*cfg), dev).predicted_us
                for cfg, _us in t["rows"]]
        meas = [us for _cfg, us in t["rows"]]
        st = rank_agreement(pred, meas)
        taus.append(st.kendall_tau)
        hits.append(st.top1_hit)
    taus.sort()
    return {"kendall_tau_median": taus[len(taus) // 2] if taus else None,
            "top1_hits": int(sum(hits)), "tables": len(tables)}


def fit(tables, dev: DeviceParams | None = None, names=COEFFS, max_evals: int = 3000):
    """Coefficients minimising `loss`, searched in log space from `dev`'s values
    (Nelder-Mead); returns (fitted DeviceParams, loss before, loss after)."""
    from scipy.optimize import minimize
    dev = dev or device_params_default()
    x0 = [math.log(getattr(dev, n)) for n in names]

    def f(x):
        return loss(tables, _with(dev, names, [math.exp(v) for v in x]))

    before = f(x0)
    res = minimize(f, x0, method="Nelder-Mead",
                   options={"maxfev": max_evals, "xatol": 1e-4, "fatol": 1e-9, "adaptive": True})
    best = res.x if res.fun < before else x0
    fitted = _with(dev, names, [math.exp(v) for v in best])
    return fitted, before, min(res.fun, before)


def save(path: str, dev: DeviceParams, names=COEFFS) -> None:
    with open(path, "w") as f:
        f.write("# cost-model coefficients fitted to this device's timings\n")
        for n in names:
            f.write(f"{n} {getattr(dev, n):.9g}\n")


def main(argv=None) -> int:
    from . import inputs
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workloads", default="bf16_gelu_1000x1000x8192,bf16_gelu_out_t128,bf16_gelu_up_t512,"
                                           "bf16_gelu_qkv_t2048,bf16_decode_16x8192x28672,bf16_gelu_kv_t16")
    ap.add_argument("--out", required=True, help="coefficient file to write")
    ap.add_argument("--tables-out", default=None, help="also write the timing tables (JSON)")
    args = ap.parse_args(argv)
    shapes = [(w.M, w.N, w.K, w.dtype, w.epi) for w in (inputs.WORKLOADS[n] for n in args.workloads.split(","))]
    dev = device_params_query()
    tables = measure(shapes)
    if args.tables_out:
        with open(args.tables_out, "w") as f:
            json.dump(tables, f)
    fitted, before, after = fit(tables, dev)
    save(args.out, fitted)
    print(json.dumps({"loss_before": before, "loss_after": after, "before": rank_stats(tables, dev),
                      "after": rank_stats(tables, fitted),
                      "coefficients": {n: getattr(fitted, n) for n in COEFFS}}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
