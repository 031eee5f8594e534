"""Autotuned tcgen05 GEMM for GB300 — Python binding of the C ABI.

The library computes C = act(A·B + bias) with a tile configuration chosen per
shape by a cost model and by timing candidates on the device (tune once, cache
by shape).  Every step runs in the native library (include/gemm_gb300.h); this
module only marshals arguments with ctypes.  PyTorch supplies device memory and
streams.

There is no fallback: if the native library has not been built, every call
raises.  Build it with `autotuning_tcgen05_tmem_gb300._build.build()` (or
`__graft_entry__.build()`).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import _build

BF16, FP32_TF32, FP8_E4M3, MXFP8_E4M3 = 0, 1, 2, 3
OPERAND_A, OPERAND_B = 1, 2            # gemm_plan_set_independent_operands
EPI_NONE, EPI_BIAS, EPI_BIAS_RELU, EPI_BIAS_GELU = 0, 1, 2, 3
EPI_BIAS_RESIDUAL, EPI_BIAS_RELU_RESIDUAL, EPI_BIAS_GELU_RESIDUAL = 4, 5, 6
EPI_BIAS_REGLU, EPI_BIAS_GEGLU, EPI_BIAS_SWIGLU = 7, 8, 9
EPILOGUES = {"none": EPI_NONE, "bias": EPI_BIAS, "relu": EPI_BIAS_RELU, "gelu": EPI_BIAS_GELU,
             "bias_residual": EPI_BIAS_RESIDUAL, "relu_residual": EPI_BIAS_RELU_RESIDUAL,
             "gelu_residual": EPI_BIAS_GELU_RESIDUAL,
             "reglu": EPI_BIAS_REGLU, "geglu": EPI_BIAS_GEGLU, "swiglu": EPI_BIAS_SWIGLU}
DTYPES = {"bf16": BF16, "fp32": FP32_TF32, "tf32": FP32_TF32, "fp8": FP8_E4M3, "e4m3": FP8_E4M3,
          "mxfp8": MXFP8_E4M3}

OK = 0
STATUS_NAMES = {0: "GEMM_OK", -1: "GEMM_ERR_INVALID_ARG", -2: "GEMM_ERR_MISALIGNED",
                -3: "GEMM_ERR_UNSUPPORTED", -4: "GEMM_ERR_INFEASIBLE", -5: "GEMM_ERR_CUDA",
                -6: "GEMM_ERR_TIMEOUT", -7: "GEMM_ERR_NO_DEVICE"}
ERR_INVALID_ARG, ERR_MISALIGNED, ERR_UNSUPPORTED, ERR_INFEASIBLE, ERR_CUDA, ERR_TIMEOUT, ERR_NO_DEVICE = \
    -1, -2, -3, -4, -5, -6, -7

REASONS = ["FEASIBLE", "CTA_GROUP", "UMMA_M", "UMMA_N", "LAYOUT", "BK", "STAGES", "SCHEDULE",
           "SPLIT_K", "ALIGN", "TMEM", "SMEM", "REGS"]

# Names the header declares; the CPU test checks the library exports each one.
EXPORTS = ["gemm_version", "gemm_last_error", "gemm_device_params_default",
           "gemm_device_params_workshop", "gemm_check_config", "gemm_enumerate",
           "gemm_fixed_config", "gemm_model_predict", "gemm_rank_agreement",
           "gemm_schedule_unit", "gemm_device_params_query", "gemm_plan",
           "gemm_plan_with_config", "gemm_plan_config", "gemm_run", "gemm_run_host",
           "gemm_plan_status", "gemm_plan_destroy", "gemm_tune", "gemm_cache_stats",
           "gemm_cache_clear", "gemm_debug_set", "gemm_run_noalloc", "gemm_tune_search",
           "gemm_cache_save", "gemm_cache_load", "gemm_plan_launch_info", "gemm_select_config_set",
           "gemm_plan_from_list", "gemm_tune_batch", "gemm_run_ex", "gemm_plan_set_scale",
           "gemm_run_mx", "gemm_mx_scales_bytes", "gemm_mx_pack_scales", "gemm_model_params_load",
           "gemm_plan_set_independent_operands", "gemm_run_host_many", "gemm_plan_tuned_on", "gemm_tune_on"]


class GemmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("bm", "bn", "bk", "stages", "raster", "group", "split_k", "cta_group", "swap_ab")]

    def astuple(self):
        return tuple(getattr(self, f) for f, _ in self._fields_)

    def asdict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}

    def __repr__(self):
        return "Config(%s)" % ", ".join(f"{k}={v}" for k, v in self.asdict().items())


def make_config(bm, bn, bk, stages, raster=0, group=1, split_k=1, cta_group=1, swap_ab=0) -> Config:
    return Config(bm, bn, bk, stages, raster, group, split_k, cta_group, swap_ab)


class DeviceParams(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("model_kind", ctypes.c_int32),
                ("smem_per_block", ctypes.c_int64), ("l2_bytes", ctypes.c_int64)] + \
               [(n, ctypes.c_double) for n in
                ("peak_tflops_bf16", "peak_tflops_tf32", "peak_tflops_fp8", "hbm_gbs", "sm_clock_mhz", "l2_gbs", "mma_issue_clk",
                 "kblock_clk", "mem_latency_us", "epi_elems_per_clk", "epi_gelu_elems_per_clk", "splitk_gbs",
                 "launch_us")] + \
               [("kernel_regs", ctypes.c_int32), ("threads_per_cta", ctypes.c_int32)]

    def asdict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class ModelTerms(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in
                ("predicted_us", "mma_us", "l2_us", "hbm_us", "latency_us", "epilogue_us", "splitk_us",
                 "launch_us", "wave_eff", "tile_eff", "pad_eff", "hbm_bytes", "l2_bytes", "flops")] + \
               [(n, ctypes.c_int64) for n in ("tiles", "units", "waves", "ctas")]

    def asdict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class TuneRow(ctypes.Structure):
    _fields_ = [("config", Config), ("predicted_us", ctypes.c_double), ("measured_us", ctypes.c_double),
                ("measured_min_us", ctypes.c_double), ("model_rank", ctypes.c_int32),
                ("measured_rank", ctypes.c_int32), ("status", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class LaunchInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("grid", "block", "smem_bytes", "cluster", "splitk_route", "b_transposed", "units", "tiles",
                 "span_copies")]

    def asdict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


SPLITK_ROUTES = {0: "none", 1: "global_last_arriver", 2: "global_shares", 3: "cluster_dsmem"}


class RankStats(ctypes.Structure):
    _fields_ = [("kendall_tau", ctypes.c_double), ("spearman_rho", ctypes.c_double),
                ("regret", ctypes.c_double), ("tune_seconds", ctypes.c_double),
                ("best_us", ctypes.c_double), ("fixed_us", ctypes.c_double),
                ("top1_hit", ctypes.c_int32), ("n_measured", ctypes.c_int32),
                ("n_candidates", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    def asdict(self):
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


_LIB = None


def library_path() -> str:
    return _build.LIB


def _load_library(path: str):
    """ctypes handle of a library exporting the C ABI, with signatures set."""
    L = ctypes.CDLL(path)
    P = ctypes.POINTER
    i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    sig = {
        "gemm_version": (ctypes.c_char_p, []),
        "gemm_last_error": (ctypes.c_char_p, []),
        "gemm_device_params_default": (None, [P(DeviceParams)]),
        "gemm_device_params_workshop": (None, [P(DeviceParams)]),
        "gemm_check_config": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, P(Config),
                                             P(DeviceParams)]),
        "gemm_enumerate": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, P(DeviceParams),
                                          P(Config), i32, P(i32)]),
        "gemm_fixed_config": (ctypes.c_int, [ctypes.c_int, P(DeviceParams), P(Config)]),
        "gemm_model_predict": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, P(Config),
                                              P(DeviceParams), P(ModelTerms)]),
        "gemm_rank_agreement": (ctypes.c_int, [P(ctypes.c_double), P(ctypes.c_double), i32,
                                               P(RankStats)]),
        "gemm_schedule_unit": (ctypes.c_int, [i64, i32, i32, i32, i32, i32, i32, P(i32), P(i32),
                                              P(i32), P(i32), P(i32)]),
        "gemm_device_params_query": (ctypes.c_int, [P(DeviceParams)]),
        "gemm_plan": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, P(vp)]),
        "gemm_plan_with_config": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, P(Config),
                                                 P(vp)]),
        "gemm_plan_config": (ctypes.c_int, [vp, P(Config)]),
        "gemm_run": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
        "gemm_run_ex": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp]),
        "gemm_plan_set_scale": (ctypes.c_int, [vp, ctypes.c_float]),
        "gemm_plan_set_independent_operands": (ctypes.c_int, [vp, i32]),
        "gemm_run_mx": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "gemm_mx_scales_bytes": (i64, [i64, i64]),
        "gemm_mx_pack_scales": (ctypes.c_int, [vp, i64, i64, i32, vp, vp]),
        "gemm_model_params_load": (ctypes.c_int, [ctypes.c_char_p, P(DeviceParams)]),
        "gemm_run_host": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
        "gemm_plan_status": (ctypes.c_int, [vp]),
        "gemm_plan_launch_info": (ctypes.c_int, [vp, P(LaunchInfo)]),
        "gemm_select_config_set": (ctypes.c_int, [P(ctypes.c_double), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                  P(ctypes.c_int32), P(ctypes.c_int32), P(ctypes.c_double),
                                                  P(ctypes.c_double)]),
        "gemm_plan_from_list": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int, P(Config), ctypes.c_int32, P(vp)]),
        "gemm_tune_batch": (ctypes.c_int, [P(ctypes.c_int64), ctypes.c_int32, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_char_p, P(ctypes.c_int32)]),
        "gemm_plan_destroy": (None, [vp]),
        "gemm_tune": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, i32, P(TuneRow), i32,
                                     P(i32), P(RankStats)]),
        "gemm_cache_stats": (ctypes.c_int, [P(i64), P(i64), P(i64)]),
    "gemm_tune_search": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32,
                                        ctypes.c_uint64, P(TuneRow), i32, P(i32), P(RankStats)]),
    "gemm_cache_save": (ctypes.c_int, [ctypes.c_char_p, P(i64)]),
    "gemm_cache_load": (ctypes.c_int, [ctypes.c_char_p, P(i64)]),
        "gemm_cache_clear": (None, []),
        "gemm_debug_set": (ctypes.c_int, [i32, i64]),
        "gemm_run_noalloc": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, P(Config), vp, vp, vp, vp, vp]),
        "gemm_run_host_many": (ctypes.c_int, [vp, i32, P(vp), P(vp), P(vp), P(vp), vp]),
        "gemm_plan_tuned_on": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp,
                                              P(vp)]),
        "gemm_tune_on": (ctypes.c_int, [i64, i64, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, i32,
                                        P(TuneRow), i32, P(i32), P(RankStats)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """The loaded native library; raises if it has not been built for this machine."""
    global _LIB
    if _LIB is None:
        if not _build.is_current():
            raise RuntimeError(
                "the native GEMM library is not built for this machine (no CPU or eager fallback "
                "exists); run autotuning_tcgen05_tmem_gb300._build.build()")
        _LIB = _load_library(_build.LIB)
    return _LIB


def last_error() -> str:
    return lib().gemm_last_error().decode()


def _check(rc: int):
    if rc != OK:
        raise GemmError(rc, last_error())
    return rc


def version() -> str:
    return lib().gemm_version().decode()


def _dt(dtype) -> int:
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def _ep(epi) -> int:
    return EPILOGUES[epi] if isinstance(epi, str) else int(epi)


# --- host logic ----------------------------------------------------------------

def device_params_default() -> DeviceParams:
    d = DeviceParams()
    lib().gemm_device_params_default(ctypes.byref(d))
    return d


def device_params_workshop() -> DeviceParams:
    d = DeviceParams()
    lib().gemm_device_params_workshop(ctypes.byref(d))
    return d


def device_params_query() -> DeviceParams:
    d = DeviceParams()
    _check(lib().gemm_device_params_query(ctypes.byref(d)))
    return d


def model_params_load(path: str, dev: DeviceParams) -> DeviceParams:
    """dev with the cost-model coefficients of a "name value" file applied."""
    out = DeviceParams()
    ctypes.memmove(ctypes.byref(out), ctypes.byref(dev), ctypes.sizeof(DeviceParams))
    _check(lib().gemm_model_params_load(str(path).encode(), ctypes.byref(out)))
    return out


def check_config(M, N, K, dtype, epi, cfg: Config, dev: DeviceParams) -> int:
    rc = lib().gemm_check_config(M, N, K, _dt(dtype), _ep(epi), ctypes.byref(cfg), ctypes.byref(dev))
    if rc < 0:
        raise GemmError(rc, last_error())
    return rc


def enumerate_configs(M, N, K, dtype, epi, dev: DeviceParams) -> list[Config]:
    n = ctypes.c_int32(0)
    _check(lib().gemm_enumerate(M, N, K, _dt(dtype), _ep(epi), ctypes.byref(dev), None, 0, ctypes.byref(n)))
    arr = (Config * max(n.value, 1))()
    _check(lib().gemm_enumerate(M, N, K, _dt(dtype), _ep(epi), ctypes.byref(dev), arr, n.value,
                                ctypes.byref(n)))
    return [arr[i] for i in range(n.value)]


def fixed_config(dtype, dev: DeviceParams) -> Config:
    c = Config()
    _check(lib().gemm_fixed_config(_dt(dtype), ctypes.byref(dev), ctypes.byref(c)))
    return c


def model_predict(M, N, K, dtype, epi, cfg: Config, dev: DeviceParams) -> ModelTerms:
    t = ModelTerms()
    _check(lib().gemm_model_predict(M, N, K, _dt(dtype), _ep(epi), ctypes.byref(cfg), ctypes.byref(dev),
                                    ctypes.byref(t)))
    return t


def rank_agreement(predicted, measured) -> RankStats:
    n = len(predicted)
    P = (ctypes.c_double * n)(*predicted)
    Q = (ctypes.c_double * n)(*measured)
    s = RankStats()
    _check(lib().gemm_rank_agreement(P, Q, n, ctypes.byref(s)))
    return s


def schedule_unit(unit, tiles_m, tiles_n, split_k, raster, group, num_kb):
    out = [ctypes.c_int32() for _ in range(5)]
    _check(lib().gemm_schedule_unit(unit, tiles_m, tiles_n, split_k, raster, group, num_kb,
                                    *[ctypes.byref(o) for o in out]))
    return tuple(o.value for o in out)


# --- device entry points ---------------------------------------------------------

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Plan:
    """A planned GEMM (owns the native handle)."""

    def __init__(self, handle: int, M: int, N: int, K: int, dtype: int, epi: int):
        self._h = ctypes.c_void_p(handle)
        self.M, self.N, self.K, self.dtype, self.epi = M, N, K, dtype, epi

    @property
    def handle(self):
        return self._h

    @property
    def config(self) -> Config:
        c = Config()
        _check(lib().gemm_plan_config(self._h, ctypes.byref(c)))
        return c

    @property
    def launch_info(self) -> LaunchInfo:
        li = LaunchInfo()
        _check(lib().gemm_plan_launch_info(self._h, ctypes.byref(li)))
        return li

    def run(self, A, B, bias, C, stream=None) -> None:
        _check(lib().gemm_run(self._h, _ptr(A), _ptr(B), _ptr(bias), _ptr(C), _stream_handle(stream)))

    def set_scale(self, alpha: float) -> None:
        """C = act(alpha·(A·B) + bias) (+ R); for FP8 operands alpha = scale_A·scale_B."""
        _check(lib().gemm_plan_set_scale(self._h, float(alpha)))

    def set_independent_operands(self, operands: str = "AB") -> None:
        """Declare which operands ("A", "B", "AB" or "") the work queued before
        a launch never writes: their copies start while the previous kernel
        drains ("B" for a layer chain's weights, "AB" for independent GEMMs)."""
        bad = set(operands) - {"A", "B"}
        if bad:
            raise ValueError(f"unknown operands {sorted(bad)}")
        mask = (OPERAND_A if "A" in operands else 0) | (OPERAND_B if "B" in operands else 0)
        _check(lib().gemm_plan_set_independent_operands(self._h, mask))

    def run_ex(self, A, B, bias, R, C, stream=None) -> None:
        """C = act(A·B + bias) + R for the residual epilogues (R may be C)."""
        _check(lib().gemm_run_ex(self._h, _ptr(A), _ptr(B), _ptr(bias), _ptr(R), _ptr(C), _stream_handle(stream)))

    def run_mx(self, A, SA, B, SB, bias, C, R=None, stream=None) -> None:
        """Block-scaled FP8: SA and SB are A's and B's E8M0 scales packed by
        mx_pack_scales (R as in run_ex)."""
        _check(lib().gemm_run_mx(self._h, _ptr(A), _ptr(SA), _ptr(B), _ptr(SB), _ptr(bias), _ptr(R), _ptr(C),
                                 _stream_handle(stream)))

    def run_rc(self, A, B, bias, C, stream=None) -> int:
        return lib().gemm_run(self._h, _ptr(A), _ptr(B), _ptr(bias), _ptr(C), _stream_handle(stream))

    def run_host(self, A, B, bias, C, stream=None) -> None:
        _check(lib().gemm_run_host(self._h, _ptr(A), _ptr(B), _ptr(bias), _ptr(C), _stream_handle(stream)))

    def run_host_many(self, As, Bs, biases, Cs, stream=None) -> None:
        """gemm_run_host_many: len(As) GEMMs from host buffers, copies pipelined
        against the kernels; returns once every C is filled."""
        n = len(As)
        arr = ctypes.c_void_p * max(n, 1)
        a, b, c = arr(*[_ptr(x) for x in As]), arr(*[_ptr(x) for x in Bs]), arr(*[_ptr(x) for x in Cs])
        bb = None if biases is None else arr(*[_ptr(x) for x in biases])
        _check(lib().gemm_run_host_many(self._h, n, a, b, bb, c, _stream_handle(stream)))

    def status(self) -> int:
        return lib().gemm_plan_status(self._h)

    def close(self):
        if self._h is not None and self._h.value:
            lib().gemm_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def plan(M, N, K, dtype="bf16", epi="none") -> Plan:
    h = ctypes.c_void_p()
    _check(lib().gemm_plan(M, N, K, _dt(dtype), _ep(epi), ctypes.byref(h)))
    return Plan(h.value, M, N, K, _dt(dtype), _ep(epi))


def plan_tuned_on(M, N, K, dtype, epi, A, B, bias=None, SA=None, SB=None) -> Plan:
    """gemm_plan_tuned_on: like plan(), timing the candidates on copies of the
    given device operands on a cache miss."""
    h = ctypes.c_void_p()
    _check(lib().gemm_plan_tuned_on(M, N, K, _dt(dtype), _ep(epi), _ptr(A), _ptr(SA), _ptr(B), _ptr(SB), _ptr(bias),
                                    ctypes.byref(h)))
    return Plan(h.value, M, N, K, _dt(dtype), _ep(epi))


def plan_with_config(M, N, K, dtype, epi, cfg: Config) -> Plan:
    h = ctypes.c_void_p()
    _check(lib().gemm_plan_with_config(M, N, K, _dt(dtype), _ep(epi), ctypes.byref(cfg), ctypes.byref(h)))
    return Plan(h.value, M, N, K, _dt(dtype), _ep(epi))


def plan_with_config_rc(M, N, K, dtype, epi, cfg: Config):
    h = ctypes.c_void_p()
    rc = lib().gemm_plan_with_config(M, N, K, _dt(dtype), _ep(epi), ctypes.byref(cfg), ctypes.byref(h))
    return rc, (Plan(h.value, M, N, K, _dt(dtype), _ep(epi)) if rc == OK else None)


@dataclass
class TuneResult:
    rows: list
    stats: RankStats


def tune(M, N, K, dtype="bf16", epi="none", topk=0, cap=4096) -> TuneResult:
    rows = (TuneRow * cap)()
    n = ctypes.c_int32(0)
    s = RankStats()
    _check(lib().gemm_tune(M, N, K, _dt(dtype), _ep(epi), topk, rows, cap, ctypes.byref(n), ctypes.byref(s)))
    return TuneResult([rows[i] for i in range(n.value)], s)


def tune_on(M, N, K, dtype, epi, A, B, bias=None, SA=None, SB=None, topk=0, cap=4096) -> TuneResult:
    """gemm_tune_on: the ranked table, timed on copies of the given operands."""
    rows = (TuneRow * cap)()
    n = ctypes.c_int32(0)
    s = RankStats()
    _check(lib().gemm_tune_on(M, N, K, _dt(dtype), _ep(epi), _ptr(A), _ptr(SA), _ptr(B), _ptr(SB), _ptr(bias), topk,
                              rows, cap, ctypes.byref(n), ctypes.byref(s)))
    return TuneResult([rows[i] for i in range(n.value)], s)


SEARCH_EXHAUSTIVE, SEARCH_MODEL_TOPK, SEARCH_RANDOM_K = 0, 1, 2


def tune_search(M, N, K, dtype="bf16", epi="none", mode=SEARCH_MODEL_TOPK, k=24, seed=0, cap=4096) -> TuneResult:
    """Time candidates chosen by `mode` (exhaustive, model top-k, random-k)."""
    rows = (TuneRow * cap)()
    n = ctypes.c_int32(0)
    s = RankStats()
    _check(lib().gemm_tune_search(M, N, K, _dt(dtype), _ep(epi), mode, k, seed, rows, cap, ctypes.byref(n),
                                  ctypes.byref(s)))
    return TuneResult([rows[i] for i in range(n.value)], s)


def select_config_set(times, max_set):
    """Greedy shipped set from a measured table (rows: shapes, columns:
    configurations, <= 0: does not run).  Returns (chosen column indices,
    mean slowdown, worst slowdown)."""
    import numpy as np
    t = np.ascontiguousarray(np.asarray(times, dtype=np.float64))
    ns, nc = (t.shape if t.ndim == 2 else (0, 0))
    chosen = (ctypes.c_int32 * max(1, max_set))()
    n = ctypes.c_int32(0)
    mean, worst = ctypes.c_double(), ctypes.c_double()
    _check(lib().gemm_select_config_set(t.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), ns, nc, max_set, chosen,
                                        ctypes.byref(n), ctypes.byref(mean), ctypes.byref(worst)))
    return [chosen[i] for i in range(n.value)], mean.value, worst.value


def plan_from_list(M, N, K, dtype, epi, configs) -> Plan:
    """Plan by timing only the given configurations (a shipped set)."""
    arr = (Config * max(1, len(configs)))(*configs)
    h = ctypes.c_void_p()
    _check(lib().gemm_plan_from_list(M, N, K, _dt(dtype), _ep(epi), arr, len(configs), ctypes.byref(h)))
    return Plan(h.value, M, N, K, _dt(dtype), _ep(epi))


def tune_batch(shapes, dtype="bf16", epi="none", db_path=None) -> int:
    """Ahead-of-time tuning of (M, N, K) shapes into the cache; saves the cache
    to db_path when given.  Returns how many shapes were newly tuned."""
    flat = [int(v) for mnk in shapes for v in mnk]
    arr = (ctypes.c_int64 * max(1, len(flat)))(*flat)
    n = ctypes.c_int32(0)
    _check(lib().gemm_tune_batch(arr, len(shapes), _dt(dtype), _ep(epi),
                                 os.fsencode(db_path) if db_path else None, ctypes.byref(n)))
    return n.value


def cache_save(path: str) -> int:
    n = ctypes.c_int64(0)
    _check(lib().gemm_cache_save(os.fsencode(path), ctypes.byref(n)))
    return n.value


def cache_load(path: str) -> int:
    n = ctypes.c_int64(0)
    _check(lib().gemm_cache_load(os.fsencode(path), ctypes.byref(n)))
    return n.value


def cache_stats():
    t, h, e = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().gemm_cache_stats(ctypes.byref(t), ctypes.byref(h), ctypes.byref(e)))
    return {"tunes": t.value, "hits": h.value, "entries": e.value}


def cache_clear():
    lib().gemm_cache_clear()


def debug_set(what: int, value: int):
    _check(lib().gemm_debug_set(what, value))


def run_noalloc_rc(M, N, K, epi, cfg: Config, A, B, bias, C, stream=None) -> int:
    """bf16 GEMM through the allocation-free entry point (for callers that
    cannot allocate device memory); returns the status code."""
    return lib().gemm_run_noalloc(M, N, K, _ep(epi), ctypes.byref(cfg), _ptr(A), _ptr(B), _ptr(bias), _ptr(C),
                                  _stream_handle(stream))


def run_noalloc(M, N, K, epi, cfg: Config, A, B, bias, C, stream=None) -> None:
    _check(run_noalloc_rc(M, N, K, epi, cfg, A, B, bias, C, stream))


def mx_scales_bytes(rows: int, K: int) -> int:
    """Bytes of one operand's packed MX scales (rows = M for A, N for B)."""
    return int(lib().gemm_mx_scales_bytes(int(rows), int(K)))


def mx_pack_scales(scales, rows: int, K: int, b_side: bool, out=None, stream=None):
    """Pack E8M0 scales (a uint8 CUDA tensor: [rows, ceil(K/32)] for A, or
    [ceil(K/32), rows] for B) into the layout gemm_run_mx reads; returns the
    packed uint8 tensor (allocated when `out` is None)."""
    import torch
    n = mx_scales_bytes(rows, K)
    if out is None:
        out = torch.empty(max(n, 16), dtype=torch.uint8, device=scales.device)
    _check(lib().gemm_mx_pack_scales(_ptr(scales), int(rows), int(K), 1 if b_side else 0, _ptr(out),
                                     _stream_handle(stream)))
    return out


def gemm(A, B, bias=None, epi="none", out=None, stream=None):
    """C = act(A·B + bias) for CUDA tensors (bf16 or fp32), planned once per shape."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    dtype = BF16 if A.dtype == torch.bfloat16 else FP32_TF32
    key = (M, N, K, dtype, _ep(epi))
    p = _PLANS.get(key)
    if p is None:
        p = plan(M, N, K, dtype, epi)
        _PLANS[key] = p
    if out is None:
        out = torch.empty(M, N, dtype=A.dtype, device=A.device)
    p.run(A, B, bias, out, stream)
    return out


_PLANS: dict = {}
