"""Seeded synthetic inputs shaped like the workloads the pages discuss.

This module holds no arithmetic of the method: it only draws random operands.
Both sides of every parity check (the CUDA path and the CPU oracle) take their
inputs from here, so that they see bit-identical values.

Recipe (per workload; seeds 0, 1, 2 for A, B and bias unless a caller passes
another base seed): draw in fp32 with torch's CPU generator (or a CUDA
generator for timing-only buffers), then round once, to bf16 with torch's
round-to-nearest-even conversion when the workload is bf16, or to FP8 E4M3
(round to nearest even; every value drawn stays inside the format's range)
when it is fp8, whose bias and C are bf16.

Block-scaled FP8 (mxfp8) workloads draw E4M3 elements of order one and E8M0
scale bytes separately (seeds +3 and +4 for A's and B's scales): for
"scaled_normal" the elements are N(0, 1) and each 32-element block's scale is
2^(e0 + u) with e0 = -round(log2(K) / 4) (so that C is of order one) and u
uniform in {-1, 0, 1}; for "decode", A's scales are 2^u and B's 2^(u - 6) (the
0.02 weight scale); for "int", elements are integers in [-2, 2] and scales
2^u, so every product and sum is exact in fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

BF16, FP32, FP8, MXFP8 = "bf16", "fp32", "fp8", "mxfp8"
EPI_CODES = {"none": 0, "bias": 1, "relu": 2, "gelu": 3}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str
    epi: str
    dist: str          # "uniform", "int", "scaled_normal", "decode"


# hidden 4096, FFN 14336: QKV (GQA, 4096 -> 6144), out, up, fused gate+up, down, KV
PROJECTIONS = [("qkv", 4096, 6144), ("out", 4096, 4096), ("up", 4096, 14336),
               ("gate_up", 4096, 28672), ("down", 14336, 4096), ("kv", 4096, 1024)]
TOKENS = (16, 128, 512, 2048, 8192)

WORKLOADS = {
    "fp32_relu_256": Workload("fp32_relu_256", 256, 256, 256, FP32, "relu", "uniform"),
    "fp32_relu_256_int": Workload("fp32_relu_256_int", 256, 256, 256, FP32, "relu", "int"),
    "bf16_gelu_1000x1000x8192": Workload("bf16_gelu_1000x1000x8192", 1000, 1000, 8192, BF16,
                                         "gelu", "scaled_normal"),
    "bf16_relu_8192": Workload("bf16_relu_8192", 8192, 8192, 8192, BF16, "relu", "scaled_normal"),
    "bf16_decode_16x8192x28672": Workload("bf16_decode_16x8192x28672", 16, 28672, 8192, BF16,
                                          "none", "decode"),
}
for _t in TOKENS:
    for _p, _k, _n in PROJECTIONS:
        _name = f"bf16_gelu_{_p}_t{_t}"
        WORKLOADS[_name] = Workload(_name, _t, _n, _k, BF16, "gelu", "scaled_normal")

SWEEP = [WORKLOADS[f"bf16_gelu_{p}_t{t}"] for t in TOKENS for (p, _k, _n) in PROJECTIONS]

# Gated projections over a fused gate+up weight (4096 -> 2 x 14336, C of
# 14336 columns): GeGLU and SwiGLU at 512 and 2048 tokens.
for _t in (512, 2048):
    for _act in ("geglu", "swiglu"):
        _name = f"bf16_{_act}_gate_up_t{_t}"
        WORKLOADS[_name] = Workload(_name, _t, 28672, 4096, BF16, _act, "scaled_normal")
GATED = ("reglu", "geglu", "swiglu")


def out_cols(w) -> int:
    """Columns of C: half the fused width for the gated epilogues."""
    return w.N // 2 if w.epi in GATED else w.N

# FP8 E4M3 operands (bf16 C) on the square, under-filled and decode shapes.
WORKLOADS["fp8_relu_8192"] = Workload("fp8_relu_8192", 8192, 8192, 8192, FP8, "relu", "scaled_normal")
WORKLOADS["fp8_gelu_1000x1000x8192"] = Workload("fp8_gelu_1000x1000x8192", 1000, 1000, 8192, FP8, "gelu",
                                                "scaled_normal")
WORKLOADS["fp8_decode_16x8192x28672"] = Workload("fp8_decode_16x8192x28672", 16, 28672, 8192, FP8, "none",
                                                 "decode")
# Block-scaled FP8 (MX: E8M0 scale per 32 elements of K) on the same shapes.
WORKLOADS["mxfp8_relu_8192"] = Workload("mxfp8_relu_8192", 8192, 8192, 8192, MXFP8, "relu", "scaled_normal")
WORKLOADS["mxfp8_gelu_1000x1000x8192"] = Workload("mxfp8_gelu_1000x1000x8192", 1000, 1000, 8192, MXFP8, "gelu",
                                                  "scaled_normal")
WORKLOADS["mxfp8_decode_16x8192x28672"] = Workload("mxfp8_decode_16x8192x28672", 16, 28672, 8192, MXFP8, "none",
                                                   "decode")


def torch_dtype(dtype: str):
    """Operand type: bf16, fp32, or FP8 E4M3 (plain or block-scaled)."""
    if dtype in (FP8, MXFP8):
        return torch.float8_e4m3fn
    return torch.bfloat16 if dtype == BF16 else torch.float32


def out_torch_dtype(dtype: str):
    """Type of C, bias and R: FP8 operands produce bf16."""
    return torch.bfloat16 if dtype in (BF16, FP8, MXFP8) else torch.float32


def _gen(seed: int, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_operands(M: int, N: int, K: int, dtype: str, dist: str, seed: int = 0,
                  device="cpu", with_bias: bool = True):
    """Return (A [M,K], B [K,N], bias [N] or None) in the workload dtype."""
    dev = torch.device(device)
    gA, gB, gb = _gen(seed, dev), _gen(seed + 1, dev), _gen(seed + 2, dev)
    f32 = torch.float32
    if dist == "uniform":
        A = torch.rand(M, K, generator=gA, device=dev, dtype=f32) * 2 - 1
        B = torch.rand(K, N, generator=gB, device=dev, dtype=f32) * 2 - 1
        bias = torch.rand(N, generator=gb, device=dev, dtype=f32) * 2 - 1
    elif dist == "int":
        A = torch.randint(-2, 3, (M, K), generator=gA, device=dev).to(f32)
        B = torch.randint(-2, 3, (K, N), generator=gB, device=dev).to(f32)
        bias = torch.randint(-2, 3, (N,), generator=gb, device=dev).to(f32)
    elif dist == "scaled_normal":
        s = 1.0 / math.sqrt(max(K, 1))
        A = torch.randn(M, K, generator=gA, device=dev, dtype=f32) * s
        B = torch.randn(K, N, generator=gB, device=dev, dtype=f32) * s
        bias = torch.randn(N, generator=gb, device=dev, dtype=f32) * 0.1
    elif dist == "decode":
        A = torch.randn(M, K, generator=gA, device=dev, dtype=f32)
        B = torch.randn(K, N, generator=gB, device=dev, dtype=f32) * 0.02
        bias = torch.randn(N, generator=gb, device=dev, dtype=f32) * 0.1
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    td = torch_dtype(dtype)
    tb = out_torch_dtype(dtype)
    return A.to(td).contiguous(), B.to(td).contiguous(), (bias.to(tb).contiguous() if with_bias else None)


def make_residual(M: int, N: int, dtype: str, dist: str, seed: int = 0, device="cpu"):
    """R [M, N] for the residual epilogues: small integers for the exact
    cases, otherwise N(0, 1) (a residual stream's scale)."""
    dev = torch.device(device)
    g = _gen(seed + 3, dev)
    if dist == "int":
        R = torch.randint(-4, 5, (M, N), generator=g, device=dev).to(torch.float32)
    else:
        R = torch.randn(M, N, generator=g, device=dev, dtype=torch.float32)
    return R.to(out_torch_dtype(dtype)).contiguous()


def make_mx_operands(M: int, N: int, K: int, dist: str, seed: int = 0, device="cpu", with_bias: bool = True):
    """Block-scaled FP8: (A [M,K] E4M3, SA [M, ceil(K/32)] uint8 E8M0,
    B [K,N] E4M3, SB [ceil(K/32), N] uint8 E8M0, bias [N] bf16 or None)."""
    dev = torch.device(device)
    gA, gB, gb, gsa, gsb = (_gen(seed + i, dev) for i in range(5))
    f32 = torch.float32
    kb = (K + 31) // 32

    def u(shape, g):
        return torch.randint(-1, 2, shape, generator=g, device=dev)

    if dist == "int":
        A = torch.randint(-2, 3, (M, K), generator=gA, device=dev).to(f32)
        B = torch.randint(-2, 3, (K, N), generator=gB, device=dev).to(f32)
        bias = torch.randint(-2, 3, (N,), generator=gb, device=dev).to(f32)
        ea, eb = u((M, kb), gsa), u((kb, N), gsb)
    elif dist in ("scaled_normal", "decode"):
        A = torch.randn(M, K, generator=gA, device=dev, dtype=f32)
        B = torch.randn(K, N, generator=gB, device=dev, dtype=f32)
        bias = torch.randn(N, generator=gb, device=dev, dtype=f32) * 0.1
        if dist == "scaled_normal":
            e0 = -round(math.log2(max(K, 1)) / 4)
            ea, eb = e0 + u((M, kb), gsa), e0 + u((kb, N), gsb)
        else:
            ea, eb = u((M, kb), gsa), u((kb, N), gsb) - 6
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    SA = (127 + ea).to(torch.uint8).contiguous()
    SB = (127 + eb).to(torch.uint8).contiguous()
    e4 = torch.float8_e4m3fn
    return (A.to(e4).contiguous(), SA, B.to(e4).contiguous(), SB,
            bias.to(torch.bfloat16).contiguous() if with_bias else None)


def make_workload(w: Workload, seed: int = 0, device="cpu"):
    """(A, B, bias) of a workload; for mxfp8 workloads use make_mx_workload."""
    if w.dtype == MXFP8:
        raise ValueError("block-scaled workloads have scales: use make_mx_workload")
    return make_operands(w.M, w.N, w.K, w.dtype, w.dist, seed=seed, device=device,
                         with_bias=(w.epi != "none"))


def make_mx_workload(w: Workload, seed: int = 0, device="cpu"):
    """(A, SA, B, SB, bias) of a block-scaled workload."""
    return make_mx_operands(w.M, w.N, w.K, w.dist, seed=seed, device=device, with_bias=(w.epi != "none"))
