"""numpy front end of the fp64 GEMM oracle (gemm_ref.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py.  The product package never imports it.

Citations (page title, section):
  * "Tile Selection: Cost Models Against Measurement", "The structure of the
    search space": C = AB, C is M x N, reduction depth K.
  * "Tiling the hierarchy", fusion section: bias + activation is an elementwise
    epilogue of the product.
Readings where the pages are silent: bias is a length-N vector added to every
row; GELU is the erf form 0.5·x·(1 + erf(x/√2)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_ref.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_gemm.so")

EPI_NONE, EPI_BIAS, EPI_BIAS_RELU, EPI_BIAS_GELU = 0, 1, 2, 3
# Residual variants: the epilogue above, then + R ([M, N], the residual connection).
EPI_BIAS_RESIDUAL, EPI_BIAS_RELU_RESIDUAL, EPI_BIAS_GELU_RESIDUAL = 4, 5, 6
# Gated (GLU-style dual-output) epilogues over a fused gate+up weight:
# C = act(A·B_gate + b_gate) ⊙ (A·B_up + b_up) with act ReLU, GELU or SiLU.
EPI_BIAS_REGLU, EPI_BIAS_GEGLU, EPI_BIAS_SWIGLU = 7, 8, 9
GLU_EPILOGUES = (EPI_BIAS_REGLU, EPI_BIAS_GEGLU, EPI_BIAS_SWIGLU)
# Fused weight layout: B is [K, N] with N a multiple of 64; its columns come in
# blocks of 32, gate and up alternating, so that output column o (of N/2) is
# gate column 64·(o // 32) + o % 32 and up column 32 more.
GLU_BLOCK = 32

_lib = None


def build(force: bool = False) -> str:
    """Compile gemm_ref.c with gcc into oracle/_build/liboracle_gemm.so."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-D_GNU_SOURCE",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_gemm.argtypes = [f32p, f32p, f32p, ctypes.c_int, ctypes.c_double, ctypes.c_int64,
                                    ctypes.c_int64, ctypes.c_int64, f64p, ctypes.c_int]
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm_entries.argtypes = [f32p, f32p, f32p, ctypes.c_int, ctypes.c_double, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, i64p, i64p,
                                            ctypes.c_int64, f64p]
        lib.oracle_gemm_entries.restype = ctypes.c_int
        lib.oracle_round_bf16.argtypes = [f64p, ctypes.c_int64,
                                          ctypes.POINTER(ctypes.c_uint16)]
        lib.oracle_round_bf16.restype = None
        _lib = lib
    return _lib


def _f32(x):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _as_f32_input(x):
    """Inputs may arrive as float32 arrays or torch tensors of bf16/fp32 (CPU),
    or FP8 E4M3 tensors, whose bytes are decoded here from the format's
    definition (oracle/fp8.py)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == getattr(torch, "float8_e4m3fn", None):
                from . import fp8
                return fp8.decode_codes(x.detach().cpu().contiguous().view(torch.uint8).numpy())
            return x.detach().to("cpu", torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float32)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def glu_columns(N: int):
    """(gate columns, up columns) of a fused [K, N] weight, in output-column order."""
    if N % (2 * GLU_BLOCK):
        raise ValueError("the fused gate+up width must be a multiple of 64")
    o = np.arange(N // 2)
    gate = 2 * GLU_BLOCK * (o // GLU_BLOCK) + o % GLU_BLOCK
    return gate, gate + GLU_BLOCK


def glu_act(x, epi: int):
    """The gate's activation in fp64: ReLU, GELU (erf form) or SiLU x·σ(x)."""
    x = np.asarray(x, dtype=np.float64)
    if epi == EPI_BIAS_REGLU:
        return np.maximum(x, 0.0)
    if epi == EPI_BIAS_GEGLU:
        from scipy.special import erf
        return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))
    if epi == EPI_BIAS_SWIGLU:
        from scipy.special import expit
        return x * expit(x)
    raise ValueError("not a gated epilogue")


def glu(A, B, bias, epi: int, threads: int | None = None, alpha: float = 1.0) -> np.ndarray:
    """fp64 C [M, N/2] = act(alpha·A·B_gate + b_gate) ⊙ (alpha·A·B_up + b_up) for
    the fused weight B [K, N] and bias [N] ("Tiling the hierarchy", fusion: the
    elementwise chain after the product is fused onto it; "CuTile Autotuning":
    dual-GEMM kernels such as Linear + GLU activation).  The two products come
    from the plain oracle on the de-interleaved columns."""
    Bf = _as_f32_input(B)
    gate, up = glu_columns(Bf.shape[1])
    bf = _as_f32_input(bias).reshape(-1)
    g = gemm(A, Bf[:, gate], bf[gate], EPI_BIAS, threads, alpha=alpha)
    u = gemm(A, Bf[:, up], bf[up], EPI_BIAS, threads, alpha=alpha)
    return glu_act(g, epi) * u


def gemm(A, B, bias=None, epi: int = EPI_NONE, threads: int | None = None, residual=None,
         alpha: float = 1.0) -> np.ndarray:
    """fp64 C = act(alpha·A·B + bias) for A [M,K], B [K,N], bias [N] (or None);
    for the residual epilogues (4, 5, 6) C = act(alpha·A·B + bias) + R with R
    [M, N] (its values exactly, in fp64); for the gated epilogues (7, 8, 9) the
    GLU-style product of glu() ([M, N/2])."""
    if epi in GLU_EPILOGUES:
        return glu(A, B, bias, epi, threads, alpha)
    if epi >= EPI_BIAS_RESIDUAL:
        if residual is None:
            raise ValueError("the residual epilogue needs R")
        base = gemm(A, B, bias, epi - 3, threads, alpha=alpha)
        R = _as_f32_input(residual).astype(np.float64)
        if R.shape != base.shape:
            raise ValueError("R must be [M, N]")
        return base + R
    lib = _load()
    A = _as_f32_input(A)
    B = _as_f32_input(B)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    a, ap = _f32(A)
    b, bp = _f32(B)
    if bias is not None:
        bb, biasp = _f32(_as_f32_input(bias).reshape(-1))
        if bb.shape[0] != N:
            raise ValueError("bias must have N entries")
    else:
        bb, biasp = None, ctypes.POINTER(ctypes.c_float)()
    C = np.empty((M, N), dtype=np.float64)
    rc = lib.oracle_gemm(ap, bp, biasp, int(epi), float(alpha), M, N, K,
                         C.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
                         int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return C


def gemm_entries(A, B, bias, epi: int, rows, cols, residual=None, alpha: float = 1.0) -> np.ndarray:
    """fp64 values of C at the listed (row, col) positions, one dot product each
    (plus R at those positions for the residual epilogues; the gated
    epilogues take output columns, of N/2)."""
    if epi in GLU_EPILOGUES:
        Bf = _as_f32_input(B)
        gate, up = glu_columns(Bf.shape[1])
        c = np.asarray(cols)
        g = gemm_entries(A, Bf, bias, EPI_BIAS, rows, gate[c], alpha=alpha)
        u = gemm_entries(A, Bf, bias, EPI_BIAS, rows, up[c], alpha=alpha)
        return glu_act(g, epi) * u
    if epi >= EPI_BIAS_RESIDUAL:
        if residual is None:
            raise ValueError("the residual epilogue needs R")
        base = gemm_entries(A, B, bias, epi - 3, rows, cols, alpha=alpha)
        R = _as_f32_input(residual)
        return base + R[np.asarray(rows), np.asarray(cols)].astype(np.float64)
    lib = _load()
    A = _as_f32_input(A)
    B = _as_f32_input(B)
    M, K = A.shape
    N = B.shape[1]
    a, ap = _f32(A)
    b, bp = _f32(B)
    if bias is not None:
        bb, biasp = _f32(_as_f32_input(bias).reshape(-1))
    else:
        bb, biasp = None, ctypes.POINTER(ctypes.c_float)()
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    out = np.empty(r.shape[0], dtype=np.float64)
    rc = lib.oracle_gemm_entries(ap, bp, biasp, int(epi), float(alpha), M, N, K,
                                 r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 c.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                 r.shape[0], out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return out


def round_bf16_bits(x) -> np.ndarray:
    """Round-to-nearest-even of fp64 values to bf16; returns the uint16 patterns."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_round_bf16(x.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), x.size,
                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)))
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (the pattern is the top half of a float)."""
    u = np.asarray(bits, dtype=np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def normalised_error(C_dev, C_ref, A, B) -> float:
    """max |C_dev - C_ref| / (||a_i||_2 · ||b_j||_2) over all (i, j).

    The error scale of entry (i, j) is the product of the norms of row i of A
    and column j of B (Cauchy–Schwarz bound of the dot product)."""
    A = _as_f32_input(A).astype(np.float64)
    B = _as_f32_input(B).astype(np.float64)
    ra = np.sqrt((A * A).sum(axis=1))
    cb = np.sqrt((B * B).sum(axis=0))
    scale = np.outer(ra, cb)
    scale[scale == 0] = 1.0
    d = np.abs(np.asarray(C_dev, dtype=np.float64) - np.asarray(C_ref, dtype=np.float64))
    return float((d / scale).max()) if d.size else 0.0


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
