"""Seeded synthetic weight tensors (bf16) for the tests and the benchmark.

This module holds no part of the quantization method: it only draws random
numbers and rounds them to bf16 with PyTorch's own cast.  Both the CPU
oracle's tests and the CUDA path's tests take their inputs from here, so the
two sides always see the same bytes.

Every generator returns a numpy uint16 array of bf16 bit patterns, shape
[rows, cols], row-major.  The recipes stand in for real LLM weights (the
method's pages measure on MiniCPM-SALA and Llama-2 weights, which are not
available here); see the workload table below.

  name        shape           distribution
  gauss_1k    1024 x 1024     N(0, 0.02), seed 0
  studentt_4k 4096 x 4096     Student-t df=4 scaled to std 0.02; 4 seeded
                              columns (0.1 % of 4096) multiplied by 20
  mlp_up      4096 x 14336    410 seeded rows (10 %) N(0, 0.05), rest N(0, 0.015)
  llama3_8b   32 layers x {q 4096^2, k/v 1024x4096, o 4096^2, gate/up 14336x4096,
              down 4096x14336}; Student-t df=5 scaled to std 0.02, one seed per tensor
  mlp_70b     8192 x 28672    N(0, 0.01) (row chunks from child streams of the
                              seed); 117,441 seeded entries (0.05 %) set to
                              +-U(0.3, 1.0) with random sign
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 numpy array -> bf16 bit patterns (round to nearest even, torch cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def sha256(b: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(b).tobytes()).hexdigest()


def gaussian(rows: int, cols: int, std: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return to_bf16_bits(rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(std))


def student_t(rows: int, cols: int, df: float, std: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    scale = std / np.sqrt(df / (df - 2.0))
    a = rng.standard_t(df, size=(rows, cols)).astype(np.float32) * np.float32(scale)
    return to_bf16_bits(a)


def gauss_1k(seed: int = 0) -> np.ndarray:
    """1024x1024, N(0, 0.02)."""
    return gaussian(1024, 1024, 0.02, seed)


def studentt_4k(seed: int = 1, rows: int = 4096, cols: int = 4096) -> np.ndarray:
    """Student-t df=4, std 0.02, with 0.1 % of the columns scaled by 20 (outlier channels)."""
    rng = np.random.default_rng(seed)
    scale = 0.02 / np.sqrt(2.0)
    a = rng.standard_t(4.0, size=(rows, cols)).astype(np.float32) * np.float32(scale)
    ncol = max(1, int(round(0.001 * cols)))
    cols_out = rng.choice(cols, size=ncol, replace=False)
    a[:, cols_out] *= np.float32(20.0)
    return to_bf16_bits(a)


def mlp_up(seed: int = 2, rows: int = 4096, cols: int = 14336) -> np.ndarray:
    """Row mixture: 10 % of rows N(0, 0.05), the rest N(0, 0.015)."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(0.015)
    nhot = int(round(0.1 * rows))
    hot = rng.choice(rows, size=nhot, replace=False)
    a[hot] = rng.standard_normal((nhot, cols), dtype=np.float32) * np.float32(0.05)
    return to_bf16_bits(a)


LLAMA3_8B_LAYER = (
    ("q_proj", 4096, 4096),
    ("k_proj", 1024, 4096),
    ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 14336, 4096),
    ("up_proj", 14336, 4096),
    ("down_proj", 4096, 14336),
)


def llama3_8b_shapes(layers: int = 32):
    """[(name, rows, cols)] of the 224-tensor Llama-3-8B-shaped stack."""
    return [(f"layer{l}.{n}", r, c) for l in range(layers) for (n, r, c) in LLAMA3_8B_LAYER]


def llama3_8b_tensor(index: int, seed_base: int = 1000, layers: int = 32) -> np.ndarray:
    """Tensor `index` of the stack: Student-t df=5, std 0.02, seed = base + index."""
    name, rows, cols = llama3_8b_shapes(layers)[index]
    return student_t(rows, cols, 5.0, 0.02, seed_base + index)


def _parallel_normal(rows: int, cols: int, std: float, seed: int, chunk_rows: int = 128) -> np.ndarray:
    """N(0, std) float32 [rows, cols], drawn in chunks of `chunk_rows` rows on
    host threads; chunk c uses its own PCG64 stream, the c-th child of
    SeedSequence(seed), so the result does not depend on the thread count."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    a = np.empty((rows, cols), np.float32)
    nch = (rows + chunk_rows - 1) // chunk_rows
    seqs = np.random.SeedSequence(seed).spawn(nch)

    def fill(c):
        part = a[c * chunk_rows:(c + 1) * chunk_rows]
        np.random.Generator(np.random.PCG64(seqs[c])).standard_normal(part.shape, dtype=np.float32, out=part)
        part *= np.float32(std)

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(nch)))
    return a


def gaussian_bf16_large(rows: int, cols: int, std: float, seed: int, chunk_rows: int = 256) -> np.ndarray:
    """N(0, std) as bf16 bits [rows, cols] for tensors too large to hold in
    float32 as well: chunk c (of `chunk_rows` rows) is drawn from the c-th child
    of SeedSequence(seed) on host threads and rounded to bf16 in place."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    out = np.empty((rows, cols), np.uint16)
    nch = (rows + chunk_rows - 1) // chunk_rows
    seqs = np.random.SeedSequence(seed).spawn(nch)

    def fill(c):
        lo, hi = c * chunk_rows, min(rows, (c + 1) * chunk_rows)
        a = np.random.Generator(np.random.PCG64(seqs[c])).standard_normal((hi - lo, cols), dtype=np.float32)
        a *= np.float32(std)
        out[lo:hi] = to_bf16_bits(a)

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(fill, range(nch)))
    return out


def mlp_70b(seed: int = 4, rows: int = 8192, cols: int = 28672) -> np.ndarray:
    """N(0, 0.01) with 0.05 % of entries set to +-U(0.3, 1.0).  The Gaussian
    part is drawn in row chunks from child streams of SeedSequence(seed)
    (host threads); the outlier positions, magnitudes and signs come from
    default_rng(seed)."""
    rng = np.random.default_rng(seed)
    a = _parallel_normal(rows, cols, 0.01, seed)
    n = rows * cols
    k = int(round(0.0005 * n))
    pos = rng.choice(n, size=k, replace=False)
    mag = rng.uniform(0.3, 1.0, size=k).astype(np.float32)
    sgn = np.where(rng.random(k) < 0.5, np.float32(-1.0), np.float32(1.0))
    a.reshape(-1)[pos] = mag * sgn
    return to_bf16_bits(a)


WORKLOADS = {
    "gauss_1k": dict(shape=(1024, 1024), make=gauss_1k,
                     recipe="1024x1024 bf16, N(0,0.02), seed 0"),
    "studentt_4k": dict(shape=(4096, 4096), make=studentt_4k,
                        recipe="4096x4096 bf16, Student-t df=4 std 0.02, 0.1% of columns x20, seed 1"),
    "mlp_up": dict(shape=(4096, 14336), make=mlp_up,
                   recipe="4096x14336 bf16, 10% rows N(0,0.05), 90% rows N(0,0.015), seed 2"),
    "mlp_70b": dict(shape=(8192, 28672), make=mlp_70b,
                    recipe="8192x28672 bf16, N(0,0.01), 0.05% entries +-U(0.3,1.0), seed 4"),
}
