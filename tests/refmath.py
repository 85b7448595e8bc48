"""Independent numpy restatements used by the tests to pin the oracle.

These are brute-force or closed-form definitions (nearest value on a table,
exact double-precision errors), written without looking at the oracle's
code paths; they share nothing with the oracle or the CUDA library.
"""
import numpy as np
import torch

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_MIDPOINTS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])

# E4M3FN values from PyTorch's float8 type (library definition of the format).
E4M3_VALUES = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def nearest_e2m1_mag(a):
    """Nearest E2M1 magnitude code of a >= 0 (float64 array), ties to even code."""
    a = np.asarray(a, np.float64)
    best = np.full(a.shape, np.inf)
    mag = np.zeros(a.shape, np.int64)
    for c, g in enumerate(E2M1_GRID):
        d = np.abs(a - g)
        take = (d < best) | ((d == best) & (c % 2 == 0))
        best = np.where(take, d, best)
        mag = np.where(take, c, mag)
    return mag


def near_e2m1_tie(a, rel=2.0 ** -21):
    """True where a lies within `rel` (relative) of an E2M1 decision midpoint."""
    a = np.asarray(a, np.float64)
    d = np.min(np.abs(a[..., None] - E2M1_MIDPOINTS) / E2M1_MIDPOINTS, axis=-1)
    return d <= rel


def nearest_e4m3(r):
    """Nearest non-negative E4M3FN code (ties to even code, 448 saturates)."""
    r = np.asarray(r, np.float64)
    d = np.abs(r[..., None] - E4M3_VALUES)
    dmin = d.min(axis=-1, keepdims=True)
    tied = d == dmin
    first = tied.argmax(axis=-1)
    ntied = tied.sum(axis=-1)
    return np.where((ntied > 1) & (first % 2 == 1), first + 1, first)


def near_e4m3_tie(r, rel=2.0 ** -21):
    mids = (E4M3_VALUES[1:] + E4M3_VALUES[:-1]) / 2
    r = np.asarray(r, np.float64)
    d = np.min(np.abs(r[..., None] - mids) / mids, axis=-1)
    return d <= rel


def unpack_codes(codes, n):
    """Packed bytes -> one 4-bit code per element (even element in the low nibble)."""
    c = np.asarray(codes, np.uint8).reshape(-1)
    out = np.empty(c.size * 2, np.uint8)
    out[0::2] = c & 0xF
    out[1::2] = c >> 4
    return out[:n]


def pack_codes(codes4):
    c = np.asarray(codes4, np.uint8).reshape(-1)
    return (c[0::2] | (c[1::2] << 4)).astype(np.uint8)


def code_values(codes4):
    c = np.asarray(codes4, np.int64)
    v = E2M1_GRID[c & 7]
    return np.where(c & 8, -v, v)


def block_view(w_bits):
    """[nblocks, 16] float64 view of a bf16 tensor."""
    return f32(w_bits).astype(np.float64).reshape(-1, 16)
