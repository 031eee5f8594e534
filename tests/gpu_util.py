"""Helpers shared by the GPU test files: run the library through its C ABI and
compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import autotuning_tcgen05_tmem_gb300 as g
from autotuning_tcgen05_tmem_gb300 import inputs
from oracle import gemm as og

TOL = 2e-3   # max |C_gpu - C_ref| / (||a_i||·||b_j||), the bound the method states

EPI = {"none": og.EPI_NONE, "bias": og.EPI_BIAS, "relu": og.EPI_BIAS_RELU, "gelu": og.EPI_BIAS_GELU}


def device_tensors(A, B, bias, guard: int = 0):
    """Copy CPU operands to the device.  With guard > 0 the output sits inside a
    larger buffer filled with a sentinel so that writes outside C are caught."""
    dev = torch.device("cuda:0")
    Ad, Bd = A.to(dev), B.to(dev)
    bd = bias.to(dev) if bias is not None else None
    return Ad, Bd, bd


def alloc_out(M, N, dtype, guard: int = 0):
    """Output tensor (and the buffer holding it) with `guard` sentinel elements
    on each side; guard is a multiple of 64 so C stays 128-byte aligned."""
    td = torch.bfloat16 if dtype == g.BF16 else torch.float32
    total = M * N + 2 * guard
    buf = torch.full((max(total, 1),), 12345.0, dtype=td, device="cuda:0")
    C = buf[guard:guard + M * N].view(M, N)
    return C, buf


def guard_intact(buf, guard: int, M: int, N: int) -> bool:
    if guard == 0:
        return True
    head = buf[:guard]
    tail = buf[guard + M * N:]
    return bool((head == 12345.0).all().item() and (tail == 12345.0).all().item())


def run_config(A, B, bias, epi: str, cfg, guard: int = 64):
    """Plan with an explicit config, run once, return (C on CPU, guard ok)."""
    M, K = A.shape
    N = B.shape[1]
    dt = g.BF16 if A.dtype == torch.bfloat16 else g.FP32_TF32
    Ad, Bd, bd = device_tensors(A, B, bias)
    C, buf = alloc_out(M, N, dt, guard)
    with g.plan_with_config(M, N, K, dt, epi, cfg) as p:
        p.run(Ad, Bd, bd if epi != "none" else None, C)
        torch.cuda.synchronize()
        st = p.status()
    assert st == 0, g.last_error()
    return C.cpu(), guard_intact(buf, guard, M, N)


def oracle_rounded_bits(A, B, bias, epi: str, dtype: int) -> np.ndarray:
    """Oracle result rounded the way the output dtype stores it (bit patterns)."""
    ref = og.gemm(A, B, bias, EPI[epi])
    if dtype == g.BF16:
        return og.round_bf16_bits(ref)
    return og.round_f32(ref).view(np.uint32)


def device_bits(C) -> np.ndarray:
    if C.dtype == torch.bfloat16:
        return C.view(torch.int16).numpy().view(np.uint16)
    return C.numpy().view(np.uint32)


def normalised_error(C, A, B, bias, epi: str) -> float:
    ref = og.gemm(A, B, bias, EPI[epi])
    return og.normalised_error(C.float().numpy(), ref, A, B)


def sampled_error(C, A, B, bias, epi: str, n: int = 2048, seed: int = 0) -> float:
    """Normalised error over n sampled entries (full-size runs)."""
    M, N = C.shape
    rng = np.random.default_rng(seed)
    rows = np.concatenate([rng.integers(0, M, n - 4), [0, M - 1, 0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, n - 4), [0, N - 1, N - 1, 0]])
    ref = og.gemm_entries(A, B, bias, EPI[epi], rows, cols)
    got = C.float().numpy()[rows, cols].astype(np.float64)
    Af = A.float().numpy().astype(np.float64)
    Bf = B.float().numpy().astype(np.float64)
    ra = np.sqrt((Af[rows] ** 2).sum(axis=1))
    cb = np.sqrt((Bf[:, cols] ** 2).sum(axis=0))
    scale = ra * cb
    scale[scale == 0] = 1.0
    return float((np.abs(got - ref) / scale).max())


def operands(M, N, K, dtype: str, dist: str, seed: int = 0):
    return inputs.make_operands(M, N, K, dtype, dist, seed=seed)
