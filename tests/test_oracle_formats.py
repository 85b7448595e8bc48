"""Pins of the oracle's number formats against independent definitions.

E2M1 and E4M3 rounding are checked against brute-force nearest-value search
on the format's value table (ties to the even code), written here in numpy,
and E4M3 / bf16 rounding additionally against PyTorch's own casts.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_from_bits(bits):
    return np.asarray(bits, np.uint32).view(np.float32)


# ---------------------------------------------------------------- E2M1

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def brute_e2m1(v):
    """Nearest magnitude on the E2M1 grid, ties to the even code; sign bit copied."""
    v = np.asarray(v, np.float32)
    a = np.abs(v.astype(np.float64))
    best = np.full(a.shape, np.inf)
    mag = np.zeros(a.shape, np.uint8)
    for c, g in enumerate(E2M1_GRID):
        d = np.abs(a - g)
        # strictly nearer wins; an exact tie with the previous (odd) code goes to this even code
        take = (d < best) | ((d == best) & (c % 2 == 0))
        best = np.where(take, d, best)
        mag = np.where(take, np.uint8(c), mag)
    sign = np.signbit(v).astype(np.uint8)
    return (mag | (sign << 3)).astype(np.uint8)


def test_e2m1_value_set_is_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "e2m1_value_set.json")))
    vals = sorted(oracle.e2m1_value(c) for c in range(16))
    assert sorted(set(vals)) == sorted(set(float(v) for v in g["values"]))
    assert max(abs(v) for v in vals) == g["max_abs"]
    # magnitude codes are ordered by value; bit 3 is the sign
    mags = [oracle.e2m1_value(c) for c in range(8)]
    assert mags == sorted(mags)
    assert all(oracle.e2m1_value(c + 8) == -oracle.e2m1_value(c) for c in range(8))


def test_e2m1_exhaustive_0125_to_8():
    """Every fp32 value in [0.125, 8) (all 6 * 2^23 patterns), both signs."""
    lo = np.float32(0.125).view(np.uint32)
    hi = np.float32(8.0).view(np.uint32)
    step = 1 << 21
    for start in range(int(lo), int(hi), step):
        bits = np.arange(start, min(start + step, int(hi)), dtype=np.uint32)
        v = f32_from_bits(bits)
        assert np.array_equal(oracle.e2m1_encode(v), brute_e2m1(v)), hex(start)
    # negative side on a sample
    v = -f32_from_bits(np.arange(int(lo), int(hi), 997, dtype=np.uint32))
    assert np.array_equal(oracle.e2m1_encode(v), brute_e2m1(v))


def test_e2m1_midpoints_and_special_values():
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    # ties go to the even code: 0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0
    assert list(oracle.e2m1_encode(mids)) == [0, 2, 2, 4, 4, 6, 6]
    up = np.nextafter(mids, np.float32(np.inf))
    assert list(oracle.e2m1_encode(up)) == [1, 2, 3, 4, 5, 6, 7]
    dn = np.nextafter(mids, np.float32(0))
    assert list(oracle.e2m1_encode(dn)) == [0, 1, 2, 3, 4, 5, 6]
    special = np.array([0.0, -0.0, 1e-45, -1e-45, 6.0, 7.0, 7.0000005, 1e30, np.inf, -np.inf, -6.5],
                       np.float32)
    assert list(oracle.e2m1_encode(special)) == [0, 8, 0, 8, 7, 7, 7, 7, 7, 15, 15]
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(200000) * 4).astype(np.float32)
    assert np.array_equal(oracle.e2m1_encode(v), brute_e2m1(v))


# ---------------------------------------------------------------- E4M3

def e4m3_table():
    return np.array([oracle.e4m3_value(c) for c in range(0x7F)])


def brute_e4m3(v):
    """Nearest of the 127 non-negative E4M3FN values, ties to even code; values
    above 448 saturate (448 is then the nearest finite value)."""
    tab = e4m3_table()
    a = np.asarray(v, np.float64)
    out = np.empty(a.shape, np.uint8)
    for i0 in range(0, a.size, 200000):
        x = a[i0:i0 + 200000]
        d = np.abs(x[:, None] - tab[None, :])
        dmin = d.min(axis=1, keepdims=True)
        tied = d == dmin
        first = tied.argmax(axis=1)
        ntied = tied.sum(axis=1)
        out[i0:i0 + 200000] = np.where((ntied > 1) & (first % 2 == 1), first + 1, first)
    return out


def torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def structured_f32(e_lo, e_hi):
    """For every exponent in [e_lo, e_hi]: each top-5-bit mantissa prefix with
    low bits {0, 1, 2, half-1, half, half+1, max-1, max} (around every
    rounding decision of a 3-bit-mantissa format)."""
    lows = np.array([0, 1, 2, (1 << 17) - 1, 1 << 17, (1 << 17) + 1, (1 << 18) - 2, (1 << 18) - 1],
                    np.uint32)
    out = []
    for e in range(e_lo, e_hi + 1):
        for top in range(32):
            out.append(((e + 127) << 23) | (top << 18) | lows)
    return f32_from_bits(np.concatenate(out))


def test_e4m3_table_is_ocp_e4m3fn():
    tab = e4m3_table()
    assert tab[0x7E] == 448.0 and tab[1] == 2.0 ** -9 and tab[8] == 2.0 ** -6
    assert np.all(np.diff(tab) > 0)
    torch_vals = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(tab, torch_vals.astype(np.float64))


def test_e4m3_matches_torch_cast_and_brute_force():
    v = np.concatenate([structured_f32(-14, 8), np.float32(e4m3_table()),
                        np.random.default_rng(3).uniform(0, 460, 100000).astype(np.float32),
                        np.exp(np.random.default_rng(4).uniform(-12, 6, 100000)).astype(np.float32)])
    v = v[(v >= 0) & (v < 464)]
    ours = oracle.e4m3_encode(v)
    assert np.array_equal(ours, torch_e4m3(v))
    assert np.array_equal(ours, brute_e4m3(v))


def test_e4m3_exhaustive_subnormal_boundary():
    """Every fp32 in [2^-11, 2^-5): E4M3 subnormals, their midpoints and the
    first normal binade."""
    bits = np.arange(np.float32(2.0 ** -11).view(np.uint32), np.float32(2.0 ** -5).view(np.uint32),
                     dtype=np.uint32)
    v = f32_from_bits(bits)
    assert np.array_equal(oracle.e4m3_encode(v), torch_e4m3(v))


def test_e4m3_saturates_at_448():
    v = np.array([448.0, 463.9, 464.0, 500.0, 1e6, 3e38, np.inf], np.float32)
    assert list(oracle.e4m3_encode(v)) == [0x7E] * 7
    assert list(oracle.e4m3_encode(np.array([0.0, 1e-30, 2.0 ** -10], np.float32))) == [0, 0, 0]


def test_e4m3_floor_ceil_brute_force():
    tab = e4m3_table()
    rng = np.random.default_rng(7)
    v = np.concatenate([np.float32(tab), np.nextafter(np.float32(tab), np.float32(np.inf)),
                        np.exp(rng.uniform(-14, 7, 50000)).astype(np.float32),
                        np.array([0.0, 500.0, 1e-12], np.float32)]).astype(np.float32)
    lo, hi = oracle.e4m3_floor_ceil(v)
    x = v.astype(np.float64)
    for i in range(v.size):
        le = np.nonzero(tab <= x[i])[0]
        ge = np.nonzero(tab >= x[i])[0]
        assert lo[i] == (le[-1] if le.size else 0)
        assert hi[i] == (ge[0] if ge.size else 0x7E)


# ---------------------------------------------------------------- bf16

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(300000).astype(np.float32) * np.float32(3e-3),
                        f32_from_bits(rng.integers(0, 0x7F000000, 300000, dtype=np.uint32))])
    ours = oracle.bf16_round(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


@pytest.mark.parametrize("lo,hi", [(0.5, 2.0), (256.0, 464.0)])
def test_e4m3_exhaustive_normal_binades(lo, hi):
    """Every fp32 bit pattern of two normal binades and of the top binade up
    to the overflow point: the oracle's E4M3 rounding equals PyTorch's
    float8_e4m3fn cast (the subnormal range has its own exhaustive test; every
    binade's decision points are in the structured test)."""
    b_lo, b_hi = int(np.float32(lo).view(np.uint32)), int(np.float32(hi).view(np.uint32))
    step = 1 << 22
    for b0 in range(b_lo, b_hi, step):
        v = f32_from_bits(np.arange(b0, min(b0 + step, b_hi), dtype=np.uint32))
        assert np.array_equal(oracle.e4m3_encode(v), torch_e4m3(v)), hex(b0)
