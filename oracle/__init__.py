"""CPU oracle for NVFP4 block quantization -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or calls it, and this package
never imports the product path.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, one function per step
of the method, each citing the page and the part of the page it follows).
This module only marshals numpy arrays into it through ctypes.

Modes: 0 = max rule, 1 = FourOverSix, 2 = CJSO(T), 3 = decoupled CJSO(T).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "nvfp4_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libnvfp4_oracle.so")

MAX, FOUR_OVER_SIX, CJSO, CJSO_DECOUPLED = 0, 1, 2, 3
MODE_NAMES = {MAX: "max", FOUR_OVER_SIX: "four_over_six", CJSO: "cjso", CJSO_DECOUPLED: "cjso_decoupled"}


def compile_source(src: str, out: str) -> str:
    """Compiles an oracle C source into shared library `out` with gcc (no
    fused multiply-add contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-shared", "-fPIC", "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compiles the oracle (once; again when the source is newer)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC)):
        return LIB_PATH
    return compile_source(SRC, LIB_PATH)


_lib = None


def load_library(path: str) -> ctypes.CDLL:
    """Loads an oracle shared library and declares its functions."""
    L = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    ci = ctypes.c_int
    L.oracle_quantize.argtypes = [p, i64, i64, ci, ci, p, p, p, p, ci]
    L.oracle_quantize.restype = ci
    L.oracle_quantize_sampled.argtypes = [p, i64, i64, ci, ci, p, i64, p, p, p, ci]
    L.oracle_quantize_sampled.restype = ci
    L.oracle_dequantize.argtypes = [p, p, ctypes.c_float, i64, i64, p]
    L.oracle_dequantize.restype = ci
    L.oracle_mse.argtypes = [p, p, p, ctypes.c_float, i64]
    L.oracle_mse.restype = ctypes.c_double
    L.oracle_block_sse.argtypes = [p, p, p, ctypes.c_float, i64, p]
    L.oracle_block_sse.restype = None
    L.oracle_cjso_trace.argtypes = [p, i64, i64, ci, p, p]
    L.oracle_cjso_trace.restype = ci
    L.oracle_e2m1_encode.argtypes = [p, i64, p]
    L.oracle_e2m1_encode.restype = None
    L.oracle_e4m3_encode.argtypes = [p, i64, p]
    L.oracle_e4m3_encode.restype = None
    L.oracle_e4m3_floor_ceil.argtypes = [p, i64, p, p]
    L.oracle_e4m3_floor_ceil.restype = None
    L.oracle_e2m1_value.argtypes = [ci]
    L.oracle_e2m1_value.restype = ctypes.c_double
    L.oracle_e4m3_value.argtypes = [ci]
    L.oracle_e4m3_value.restype = ctypes.c_double
    L.oracle_u128_to_double.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    L.oracle_u128_to_double.restype = ctypes.c_double
    L.oracle_bf16_round.argtypes = [p, i64, p]
    L.oracle_bf16_round.restype = None
    L.oracle_block_sums.argtypes = [p, i64, ctypes.c_float, p, p, p, p]
    L.oracle_block_sums.restype = None
    L.oracle_gemv.argtypes = [p, p, ctypes.c_float, i64, i64, p, ci, p]
    L.oracle_gemv.restype = ci
    L.oracle_swizzled_size.argtypes = [i64, i64]
    L.oracle_swizzled_size.restype = i64
    L.oracle_swizzle_scales.argtypes = [p, i64, i64, p]
    L.oracle_swizzle_scales.restype = ci
    return L


def lib() -> ctypes.CDLL:
    """The oracle library: the one built from ``nvfp4_oracle.c``, or the one
    named by NVFP4_ORACLE_LIB (the mutation tests point it at copies of the
    oracle with a planted mistake)."""
    global _lib
    if _lib is None:
        path = os.environ.get("NVFP4_ORACLE_LIB") or build()
        _lib = load_library(path)
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits(w) -> np.ndarray:
    w = np.ascontiguousarray(w)
    if w.dtype != np.uint16:
        raise TypeError("weights must be bf16 bit patterns (uint16)")
    return w


def quantize(w_bits: np.ndarray, mode: int, iters: int = 0, threads: int = 1, m4_flags: bool = False):
    """Quantizes a [rows, cols] bf16 tensor given as uint16 bit patterns.

    Returns (codes uint8 [rows, cols/2], scales uint8 [rows, cols/16], alpha
    float) and, with m4_flags, a per-block uint8 array (FourOverSix only)."""
    w = _bits(w_bits)
    rows, cols = w.shape
    codes = np.zeros((rows, cols // 2), np.uint8)
    scales = np.zeros((rows, cols // 16), np.uint8)
    alpha = np.zeros(1, np.float32)
    flags = np.zeros(rows * cols // 16, np.uint8) if m4_flags else None
    rc = lib().oracle_quantize(_ptr(w), rows, cols, mode, iters, _ptr(codes), _ptr(scales),
                               _ptr(alpha), _ptr(flags) if flags is not None else None, threads)
    if rc != 0:
        raise ValueError(f"oracle_quantize failed with status {rc}")
    if m4_flags:
        return codes, scales, float(alpha[0]), flags
    return codes, scales, float(alpha[0])


def quantize_sampled(w_bits: np.ndarray, mode: int, iters: int, blocks: np.ndarray, threads: int = 1):
    """Quantizes the whole tensor's coupled state (alpha, CJSO iterations) but
    produces per-block outputs only for the listed flat block indices.
    Returns (codes uint8 [n, 8], scales uint8 [n], alpha)."""
    w = _bits(w_bits)
    rows, cols = w.shape
    blocks = np.ascontiguousarray(blocks, dtype=np.int64)
    codes = np.zeros((len(blocks), 8), np.uint8)
    scales = np.zeros(len(blocks), np.uint8)
    alpha = np.zeros(1, np.float32)
    rc = lib().oracle_quantize_sampled(_ptr(w), rows, cols, mode, iters, _ptr(blocks), len(blocks),
                                       _ptr(codes), _ptr(scales), _ptr(alpha), threads)
    if rc != 0:
        raise ValueError(f"oracle_quantize_sampled failed with status {rc}")
    return codes, scales, float(alpha[0])


def dequantize(codes: np.ndarray, scales: np.ndarray, alpha: float, rows: int, cols: int) -> np.ndarray:
    """Returns bf16 bit patterns (uint16 [rows, cols])."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    out = np.zeros((rows, cols), np.uint16)
    rc = lib().oracle_dequantize(_ptr(codes), _ptr(scales), ctypes.c_float(alpha), rows, cols, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_dequantize failed")
    return out


def mse(w_bits, codes, scales, alpha) -> float:
    w = _bits(w_bits)
    return lib().oracle_mse(_ptr(w), _ptr(np.ascontiguousarray(codes, np.uint8)),
                            _ptr(np.ascontiguousarray(scales, np.uint8)), ctypes.c_float(alpha), w.size)


def block_sse(w_bits, codes, scales, alpha) -> np.ndarray:
    w = _bits(w_bits)
    nb = w.size // 16
    out = np.zeros(nb, np.float64)
    lib().oracle_block_sse(_ptr(w), _ptr(np.ascontiguousarray(codes, np.uint8)),
                           _ptr(np.ascontiguousarray(scales, np.uint8)), ctypes.c_float(alpha), nb, _ptr(out))
    return out


def cjso_trace(w_bits, iters: int):
    """MSE (sum of squares, double) after the start and after each half-step of
    every CJSO iteration (4 per iteration), and alpha after each alpha step."""
    w = _bits(w_bits)
    rows, cols = w.shape
    trace = np.zeros(1 + 4 * iters, np.float64)
    alphas = np.zeros(1 + iters, np.float32)
    rc = lib().oracle_cjso_trace(_ptr(w), rows, cols, iters, _ptr(trace), _ptr(alphas))
    if rc != 0:
        raise ValueError("oracle_cjso_trace failed")
    return trace, alphas


def e2m1_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float32)
    out = np.zeros(v.shape, np.uint8)
    lib().oracle_e2m1_encode(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float32)
    out = np.zeros(v.shape, np.uint8)
    lib().oracle_e4m3_encode(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_floor_ceil(v):
    v = np.ascontiguousarray(v, np.float32)
    lo = np.zeros(v.shape, np.uint8)
    hi = np.zeros(v.shape, np.uint8)
    lib().oracle_e4m3_floor_ceil(_ptr(v), v.size, _ptr(lo), _ptr(hi))
    return lo, hi


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code))


def u128_to_double(v: int) -> float:
    """A nonnegative integer below 2^128 rounded to the nearest double (ties to even)."""
    return lib().oracle_u128_to_double((v >> 64) & (2**64 - 1), v & (2**64 - 1))


def bf16_round(v) -> np.ndarray:
    v = np.ascontiguousarray(v, np.float32)
    out = np.zeros(v.shape, np.uint16)
    lib().oracle_bf16_round(_ptr(v), v.size, _ptr(out))
    return out


def block_sums(w_bits, alpha: float, dcodes):
    """Per-block P (fp32), R (fp32) and the exact double sum of |x| q."""
    w = _bits(w_bits)
    nb = w.size // 16
    dcodes = np.ascontiguousarray(dcodes, np.uint8).reshape(-1)
    P = np.zeros(nb, np.float32)
    R = np.zeros(nb, np.float32)
    Pe = np.zeros(nb, np.float64)
    lib().oracle_block_sums(_ptr(w), nb, ctypes.c_float(alpha), _ptr(dcodes), _ptr(P), _ptr(R), _ptr(Pe))
    return P, R, Pe


def gemv(codes, scales, alpha: float, rows: int, cols: int, x_bits):
    """y [batch, rows] (float64) = dequantized bf16 weights times bf16
    activations x [batch, cols] (uint16 bit patterns), summed in double."""
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    x = np.ascontiguousarray(x_bits, np.uint16).reshape(-1, cols)
    y = np.zeros((x.shape[0], rows), np.float64)
    rc = lib().oracle_gemv(_ptr(codes), _ptr(scales), ctypes.c_float(alpha), rows, cols, _ptr(x), x.shape[0],
                           _ptr(y))
    if rc != 0:
        raise ValueError("oracle_gemv failed")
    return y


def swizzle_scales(scales, rows: int, kb: int) -> np.ndarray:
    """The [rows, kb] E4M3 scales in the tensor-core tile layout (flat uint8)."""
    sc = np.ascontiguousarray(scales, np.uint8)
    out = np.zeros(lib().oracle_swizzled_size(rows, kb), np.uint8)
    if lib().oracle_swizzle_scales(_ptr(sc), rows, kb, _ptr(out)) != 0:
        raise ValueError("oracle_swizzle_scales failed")
    return out
