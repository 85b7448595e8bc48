"""Pins of the oracle's quantization modes against what the pages and the
mathematics fix: round-trip exactness on representable tensors, hand-worked
FourOverSix blocks, the least-squares closed forms, monotone CJSO error,
brute-force searches on small inputs, and the decoupled search's guarantee.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic
from refmath import (E2M1_GRID, E4M3_VALUES, block_view, code_values, f32, near_e2m1_tie,
                     near_e4m3_tie, nearest_e2m1_mag, nearest_e4m3, pack_codes, unpack_codes)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ALPHA_EXACT = 2.0 ** -12  # 0.65625 / 2688


def bf16_bits(vals):
    a = np.asarray(vals, np.float32)
    b = synthetic.to_bf16_bits(a)
    assert np.array_equal(f32(b), a), "test tensor must be exactly representable in bf16"
    return b


def representable_tensor(rows, cols, seed, dcodes=None):
    """W = q * Delta * 2^-12 with a +-6 code in every block and the tensor max
    0.65625, so that alpha = 2^-12 and every code and scale is recoverable."""
    rng = np.random.default_rng(seed)
    nb = rows * cols // 16
    if dcodes is None:
        dcodes = rng.integers(1, 0x7F, nb)
    dcodes = np.asarray(dcodes)
    dcodes[0] = 0x7E
    mags = rng.integers(0, 8, (nb, 16))
    mags[np.arange(nb), rng.integers(0, 16, nb)] = 7
    signs = rng.integers(0, 2, (nb, 16))
    q = E2M1_GRID[mags] * np.where(signs == 1, -1.0, 1.0)
    w = q * E4M3_VALUES[dcodes][:, None] * ALPHA_EXACT
    codes4 = (mags | (signs << 3)).astype(np.uint8)
    return bf16_bits(w.reshape(rows, cols)), codes4.reshape(-1), dcodes.astype(np.uint8)


# ------------------------------------------------------------------- max rule

@pytest.mark.parametrize("seed", [0, 1])
def test_max_roundtrip_exact(seed):
    w, codes4, dcodes = representable_tensor(16, 256, seed)
    codes, scales, alpha = oracle.quantize(w, oracle.MAX)
    assert alpha == ALPHA_EXACT
    assert np.array_equal(scales.reshape(-1), dcodes)
    assert np.array_equal(unpack_codes(codes, w.size), codes4)
    out = oracle.dequantize(codes, scales, alpha, *w.shape)
    assert np.array_equal(out, w)


def test_max_rule_against_exact_division():
    """alpha, Delta and codes follow the pages' formulas evaluated exactly,
    except where the one fp32 rounding of the quotient (reading R4) moves a
    value that lies within half an ulp of a rounding midpoint onto it."""
    w = synthetic.gaussian(256, 512, 0.02, 21)
    codes, scales, alpha = oracle.quantize(w, oracle.MAX)
    x = block_view(w)
    amax = np.abs(f32(w)).max()
    assert alpha == float(np.float32(amax) / np.float32(2688.0))
    ratio = np.abs(x).max(axis=1) / (6.0 * alpha)
    ref_d = nearest_e4m3(ratio)
    got_d = scales.reshape(-1)
    bad = ref_d != got_d
    assert not np.any(bad & ~near_e4m3_tie(ratio, 2.0 ** -23)), np.nonzero(bad)[0][:5]
    s = np.float32(alpha) * E4M3_VALUES[got_d].astype(np.float32)  # fl(alpha*Delta)
    v = np.abs(x) / s.astype(np.float64)[:, None]
    ref_mag = nearest_e2m1_mag(v).reshape(-1)
    got = unpack_codes(codes, w.size)
    bad = (got & 7) != ref_mag
    assert not np.any(bad & ~near_e2m1_tie(v.reshape(-1), 2.0 ** -23)), np.nonzero(bad)[0][:5]
    # bf16 weights, E4M3 scales and 2688 are short numbers, so |x|/s often sits
    # exactly on a midpoint in real arithmetic; the rounded alpha moves such
    # values by an ulp, and the reference above (exact division by the rounded
    # s) then breaks the tie differently.  These are the only differences.
    assert bad.mean() < 1e-2
    assert np.array_equal(got >> 3, np.signbit(f32(w)).astype(np.uint8).reshape(-1))


def test_midpoint_quotients_resolve_to_even():
    """Reading R4 (the quotient is an IEEE division): elements that are exactly
    an E2M1 midpoint times the block's dequant scale give an exact quotient
    on the midpoint, which the even rule resolves.  Every E4M3 scale with a
    non-power-of-two significand is used, so that 1/s is inexact; a quotient
    taken as |x| * (1/s) leaves the midpoint for some of them."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    even = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    dcodes = [c for c in range(8, 0x7E) if c & 7]  # normal E4M3 values 1.m x 2^e, m != 0
    blocks, want = [np.r_[6.0 * 448.0, np.zeros(15)]], [np.r_[7, np.zeros(15, np.int64)]]
    for c in dcodes:
        d = E4M3_VALUES[c]
        blocks.append(np.r_[6.0, mids, mids[::-1], 0.0] * d)
        want.append(np.r_[7, [even[m] for m in mids], [even[m] for m in mids[::-1]], 0])
    w = bf16_bits((np.concatenate(blocks) * ALPHA_EXACT).reshape(1, -1))
    codes, scales, alpha = oracle.quantize(w, oracle.MAX)
    assert alpha == ALPHA_EXACT
    assert list(scales[0, 1:]) == dcodes
    assert np.array_equal(unpack_codes(codes, w.size), np.concatenate(want).astype(np.uint8))


def test_zero_and_tiny_blocks():
    w = np.zeros((2, 64), np.float32)
    w[0, 0] = 0.5
    w[0, 16] = 0.5 / 2688 * 6 * 2 ** -11  # block amax far below the smallest E4M3 scale
    w[1, 5] = -0.0
    b = synthetic.to_bf16_bits(w)
    for mode in (0, 1, 2, 3):
        codes, scales, alpha = oracle.quantize(b, mode, 2)
        sc = scales.reshape(-1)
        assert sc[1] == 0 and sc[2] == 0 and sc[5] == 0 and sc[7] == 0
        c4 = unpack_codes(codes, b.size)
        assert c4[16] == 0 and c4[64 + 5] == 8 and np.all(c4[32:64] == 0)
    z = synthetic.to_bf16_bits(np.zeros((1, 32), np.float32))
    codes, scales, alpha = oracle.quantize(z, 0)
    assert alpha == 0.0 and not codes.any() and not scales.any()


# ---------------------------------------------------------------- FourOverSix

def test_fos_worked_blocks():
    g = json.load(open(os.path.join(GOLDEN, "fos_worked_blocks.json")))
    u = 2.0 ** -8
    vals = np.concatenate([np.asarray(b["values_over_u"], np.float64) * u for b in g["blocks"]])
    w = bf16_bits(vals.reshape(1, -1))
    codes, scales, alpha, m4 = oracle.quantize(w, oracle.FOUR_OVER_SIX, m4_flags=True)
    assert alpha == g["alpha"]
    for i, b in enumerate(g["blocks"]):
        assert scales[0, i] == b["scale"], i
        assert m4[i] == b["m4"], i
        assert list(codes[0, 8 * i:8 * i + 8]) == b["code_bytes"], i


def test_fos_blocks_packed_in_2_to_4_choose_m4():
    """Blocks whose values are {2, 3, 4} * s4 with at least one 3*s4 are exact
    under M=4 and not under M=6, so M=4 must win; blocks of {3, 6} * s6 are
    exact under both, so the tie keeps M=6 (strict < of the rule)."""
    rng = np.random.default_rng(9)
    u = 2.0 ** -8
    blocks = [np.r_[168.0, np.zeros(15)] * u]
    kinds = []
    for _ in range(40):
        v = rng.choice([3.0, 4.5, 6.0], 16)
        v[0] = 6.0
        v[rng.integers(1, 16)] = 4.5
        blocks.append(v * u * np.where(rng.random(16) < 0.5, -1, 1))
        kinds.append(1)
        v = rng.choice([3.0, 6.0], 16)
        v[0] = 6.0
        blocks.append(v * u)
        kinds.append(0)
    w = bf16_bits(np.concatenate(blocks).reshape(1, -1))
    _, scales, alpha, m4 = oracle.quantize(w, oracle.FOUR_OVER_SIX, m4_flags=True)
    assert alpha == ALPHA_EXACT
    assert list(m4[1:]) == kinds
    assert np.all(scales[0, 1:][np.array(kinds) == 1] == 0x5C)
    assert np.all(scales[0, 1:][np.array(kinds) == 0] == 0x58)


def test_fos_picks_lower_exact_error():
    """Against exact double-precision errors of both candidates: FourOverSix
    never does worse than the max rule beyond fp32 rounding, and its choice
    agrees with the exact comparison except in near-ties."""
    w = synthetic.student_t(128, 1024, 4.0, 0.02, 31)
    c6, s6, a6 = oracle.quantize(w, oracle.MAX)
    cf, sf, af, m4 = oracle.quantize(w, oracle.FOUR_OVER_SIX, m4_flags=True)
    assert a6 == af
    x = block_view(w)
    sumsq = (x ** 2).sum(axis=1)
    sse6 = oracle.block_sse(w, c6, s6, a6)
    ssef = oracle.block_sse(w, cf, sf, af)
    assert np.all(ssef <= sse6 + 2.0 ** -20 * sumsq)
    d6 = s6.reshape(-1)
    d4 = nearest_e4m3(E4M3_VALUES[d6] * 1.5)
    got = sf.reshape(-1)
    assert np.all((got == d6) | (got == d4))
    assert np.array_equal(m4.astype(bool), (got == d4) & (d4 != d6))
    # exact error of the M=4 candidate, codes by exact division
    s4 = (np.float32(af) * E4M3_VALUES[d4].astype(np.float32)).astype(np.float64)
    q4 = E2M1_GRID[nearest_e2m1_mag(np.abs(x) / s4[:, None])]
    sse4 = ((np.abs(x) - q4 * s4[:, None]) ** 2).sum(axis=1)
    exact_m4 = sse4 < sse6
    disagree = exact_m4 != m4.astype(bool)
    assert np.all(np.abs(sse4 - sse6)[disagree] <= 2.0 ** -20 * sumsq[disagree])
    share = m4.mean()
    assert 0.1 < share < 0.9, share


# ------------------------------------------------------------------------ CJSO

def test_cjso_zero_iterations_is_max_rule():
    w = synthetic.gaussian(64, 256, 0.02, 5)
    a = oracle.quantize(w, oracle.MAX)
    b = oracle.quantize(w, oracle.CJSO, 0)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]


@pytest.mark.parametrize("make", [lambda: synthetic.gaussian(128, 512, 0.02, 6),
                                  lambda: synthetic.mlp_up(7, 128, 512),
                                  lambda: synthetic.student_t(128, 512, 4.0, 0.02, 8)])
def test_cjso_error_never_increases(make):
    """Each half-step is a least-squares or nearest-value step, so the error is
    non-increasing up to fp32 rounding of alpha and of the reciprocal."""
    w = make()
    trace, alphas = oracle.cjso_trace(w, 6)
    rel = np.diff(trace) / trace[:-1]
    assert np.all(rel <= 1e-6), rel
    assert trace[-1] < trace[0]


def alpha_closed_form(w, codes, scales):
    x = np.abs(block_view(w))
    q = np.abs(code_values(unpack_codes(codes, w.size))).reshape(-1, 16)
    d = E4M3_VALUES[scales.reshape(-1)]
    P = (x * q).sum(axis=1)
    R = (q * q).sum(axis=1)
    return (d * P).sum() / (d * d * R).sum(), x, q, d


@pytest.mark.parametrize("T", [0, 2])
def test_cjso_alpha_step_is_least_squares(T):
    w = synthetic.mlp_up(12, 128, 512)
    codes, scales, _ = oracle.quantize(w, oracle.CJSO, T)
    a_ref, x, q, d = alpha_closed_form(w, codes, scales)
    _, _, a_next = oracle.quantize(w, oracle.CJSO, T + 1)
    assert abs(a_next - a_ref) <= 1e-6 * a_ref
    f = lambda a: (((x - q * (a * d)[:, None])) ** 2).sum()
    for dl in (1e-4, 1e-3, 1e-2):
        assert f(a_ref) <= f(a_ref * (1 + dl)) and f(a_ref) <= f(a_ref * (1 - dl))


def test_cjso_one_iteration_brute_force():
    """CJSO(1) restated with exact division and a brute-force search of the
    block scale over all 127 E4M3 values.  The block error is a parabola in
    the scale with its vertex at P / (alpha R), so the nearest E4M3 value to
    the vertex is the best one; the two differ only where the vertex lies at
    an E4M3 midpoint up to the fp32 rounding of the quotient."""
    w = synthetic.student_t(64, 256, 5.0, 0.02, 13)
    c0, s0, a0 = oracle.quantize(w, oracle.MAX)
    a1 = np.float32(alpha_closed_form(w, c0, s0)[0])
    x = block_view(w)
    ax = np.abs(x)
    d0 = s0.reshape(-1)
    s = (a1 * E4M3_VALUES[d0].astype(np.float32)).astype(np.float64)
    vp = ax / s[:, None]
    qp = E2M1_GRID[nearest_e2m1_mag(vp)]  # re-quantized with the new alpha
    errs = ((ax[:, None, :] - qp[:, None, :] * (float(a1) * E4M3_VALUES)[None, :, None]) ** 2).sum(axis=2)
    Rp = (qp ** 2).sum(axis=1)
    d1 = np.where(Rp > 0, errs.argmin(axis=1), d0)
    vertex = (ax * qp).sum(axis=1) / (float(a1) * np.maximum(Rp, 1))
    s1 = (a1 * E4M3_VALUES[d1].astype(np.float32)).astype(np.float64)
    v1 = ax / s1[:, None]
    q1 = nearest_e2m1_mag(v1)
    codes, scales, alpha = oracle.quantize(w, oracle.CJSO, 1)
    assert alpha == float(a1)
    got_d = scales.reshape(-1)
    excused = near_e4m3_tie(vertex, 2.0 ** -20) | np.any(near_e2m1_tie(vp), axis=1)
    assert np.all((got_d == d1) | excused), np.nonzero((got_d != d1) & ~excused)[0][:5]
    assert excused.mean() < 0.01
    same = got_d == d1
    got_mag = (unpack_codes(codes, w.size) & 7).reshape(-1, 16)
    bad = (got_mag != q1) & same[:, None]
    assert not np.any(bad & ~near_e2m1_tie(v1))


def test_cjso_trace_ends_at_quantize_state():
    """The traced iteration and the quantizer reach the same final state: the
    last traced error equals the reconstruction error of CJSO(T)'s output."""
    w = synthetic.mlp_up(17, 64, 512)
    for T in (1, 3):
        trace, alphas = oracle.cjso_trace(w, T)
        codes, scales, alpha = oracle.quantize(w, oracle.CJSO, T)
        assert alphas[-1] == alpha
        assert abs(trace[-1] / w.size - oracle.mse(w, codes, scales, alpha)) <= 1e-6 * trace[-1] / w.size


# ----------------------------------------------------------- decoupled CJSO

def test_decoupled_never_worse_than_cjso_and_brute_force():
    w = synthetic.mlp_up(14, 32, 256)
    cc, sc, ac = oracle.quantize(w, oracle.CJSO, 3)
    cd, sd, ad = oracle.quantize(w, oracle.CJSO_DECOUPLED, 3)
    assert ac == ad
    x = block_view(w)
    ax = np.abs(x)
    sumsq = (x ** 2).sum(axis=1)
    sse_c = oracle.block_sse(w, cc, sc, ac)
    sse_d = oracle.block_sse(w, cd, sd, ad)
    assert np.all(sse_d <= sse_c + 2.0 ** -20 * sumsq)
    assert np.mean(sse_d < sse_c * (1 - 1e-6)) > 0.2
    # brute force over the 101 x 2 candidates with exact errors
    a = np.float32(ad)
    m = np.array([np.float32((50 + k) / 100.0) for k in range(101)])
    d0 = E4M3_VALUES[sc.reshape(-1)].astype(np.float32)
    best = np.full(len(d0), np.inf)
    for k in range(101):
        dq = d0 * m[k]
        sq = (a * dq).astype(np.float64)
        q = E2M1_GRID[nearest_e2m1_mag(ax / sq[:, None])]
        for side in (0, 1):
            lo = np.searchsorted(E4M3_VALUES, dq.astype(np.float64), side="right") - 1
            hi = np.minimum(np.searchsorted(E4M3_VALUES, dq.astype(np.float64), side="left"), 0x7E)
            dd = np.maximum(lo, 0) if side == 0 else hi
            sdv = (a * E4M3_VALUES[dd].astype(np.float32)).astype(np.float64)
            err = ((ax - q * sdv[:, None]) ** 2).sum(axis=1)
            best = np.minimum(best, err)
    assert np.all(sse_d <= best * (1 + 1e-6) + 2.0 ** -22 * sumsq)


# ------------------------------------------------------------------ dequant

def test_dequantize_matches_torch_rounding():
    w = synthetic.gaussian(64, 256, 0.02, 15)
    codes, scales, alpha = oracle.quantize(w, oracle.FOUR_OVER_SIX)
    out = oracle.dequantize(codes, scales, alpha, *w.shape)
    q = code_values(unpack_codes(codes, w.size)).astype(np.float32)
    s = np.repeat(np.float32(alpha) * E4M3_VALUES[scales.reshape(-1)].astype(np.float32), 16)
    ref = torch.from_numpy(q * s).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out.reshape(-1), ref)


# ---------------------------------------------------------- oracle plumbing

@pytest.mark.parametrize("mode,iters", [(0, 0), (1, 0), (2, 3), (3, 2)])
def test_threads_and_sampling_do_not_change_results(mode, iters):
    w = synthetic.gaussian(48, 256, 0.02, 16)
    a = oracle.quantize(w, mode, iters, threads=1)
    b = oracle.quantize(w, mode, iters, threads=5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]
    blocks = np.array([0, 7, 100, 767, 5, 300])
    c, s, al = oracle.quantize_sampled(w, mode, iters, blocks, threads=3)
    assert al == a[2]
    assert np.array_equal(s, a[1].reshape(-1)[blocks])
    assert np.array_equal(c, a[0].reshape(-1, 8)[blocks])


@pytest.mark.parametrize("make", [lambda: synthetic.gaussian(256, 512, 0.02, 40),
                                  lambda: synthetic.studentt_4k(41, 256, 1024),
                                  lambda: synthetic.mlp_70b(42, 64, 4096)])
def test_block_sums_exact(make):
    """Reading R5: the fp32 block sums P = sum |x| q equal their exact values,
    for max-rule scales, for 1.5x and for 0.5x of them (codes up to 12x)."""
    w = make()
    _, scales, alpha = oracle.quantize(w, oracle.MAX)
    d = scales.reshape(-1).astype(np.int64)
    for dc in (d, nearest_e4m3(E4M3_VALUES[d] * 1.5), np.maximum(d - 8, 0)):
        P, R, Pe = oracle.block_sums(w, alpha, dc.astype(np.uint8))
        assert np.array_equal(P.astype(np.float64), Pe)
        assert np.all(R * 4 == np.round(R * 4)) and np.all(R <= 576)


# ------------------------------------------------------- W4A16 product (consumer)

def _acts(batch, cols, seed):
    rng = np.random.default_rng(seed)
    return synthetic.to_bf16_bits(rng.standard_normal((batch, cols)).astype(np.float32))


def test_gemv_on_representable_weights_is_the_plain_product():
    """Round-trip-exact weights: the product equals W x of the original
    weights, computed here in float64 from W itself."""
    w, _, _ = representable_tensor(24, 256, 3)
    codes, scales, alpha = oracle.quantize(w, oracle.MAX)
    x = _acts(3, 256, 4)
    y = oracle.gemv(codes, scales, alpha, 24, 256, x)
    ref = f32(x).astype(np.float64) @ f32(w).astype(np.float64).T
    bound = 1e-13 * (np.abs(f32(x)).astype(np.float64) @ np.abs(f32(w)).astype(np.float64).T)
    assert np.all(np.abs(y - ref) <= bound)


@pytest.mark.parametrize("mode,iters", [(0, 0), (1, 0), (2, 2), (3, 1)])
def test_gemv_consumes_the_dequantized_bf16_weights(mode, iters):
    """Every scale rule feeds the same product: y = dequantize(codes) x."""
    w = synthetic.student_t(20, 320, 4.0, 0.02, 60 + mode)
    codes, scales, alpha = oracle.quantize(w, mode, iters)
    x = _acts(2, 320, 61)
    y = oracle.gemv(codes, scales, alpha, 20, 320, x)
    deq = f32(oracle.dequantize(codes, scales, alpha, 20, 320)).astype(np.float64)
    ref = f32(x).astype(np.float64) @ deq.T
    assert np.all(np.abs(y - ref) <= 1e-13 * (np.abs(f32(x)).astype(np.float64) @ np.abs(deq).T))


def test_gemv_single_block_by_hand():
    """1 x 16 weights [6, -3, 0.5, 0...] * 2^-12 (alpha exact, scale 448 for
    the block maximum 6 * 448 * 2^-12... here a block of its own): y = sum w x."""
    vals = np.zeros(16, np.float64)
    vals[:3] = [6.0, -3.0, 0.5]
    w = bf16_bits((vals * 448.0 * ALPHA_EXACT).reshape(1, 16))
    codes, scales, alpha = oracle.quantize(w, oracle.MAX)
    x = bf16_bits(np.r_[1.0, 2.0, 4.0, np.full(13, 3.0)].reshape(1, 16))
    y = oracle.gemv(codes, scales, alpha, 1, 16, x)
    assert y[0, 0] == (6.0 * 1 - 3.0 * 2 + 0.5 * 4) * 448.0 * ALPHA_EXACT


# ------------------------------------------------ tensor-core scale layout (R13)

def test_swizzle_hand_worked_positions():
    """Scales of a 300 x 10 (kb) matrix: tiles of 128 x 4, column tiles
    fastest (3 per row of tiles), byte (r%32)*16 + (r//32)*4 + c inside."""
    rows, kb = 300, 10
    sc = (np.arange(rows * kb) % 251 + 1).astype(np.uint8).reshape(rows, kb)
    out = oracle.swizzle_scales(sc, rows, kb)
    assert out.size == 384 * 12
    assert out[0] == sc[0, 0] and out[1] == sc[0, 1] and out[4] == sc[32, 0] and out[16] == sc[1, 0]
    assert out[22 + 0] == sc[33, 2]                      # r = 33: 1*16 + 1*4 + 2
    assert out[512 + 0] == sc[0, 4]                      # second column tile of the first row tile
    assert out[3 * 512 + 5 * 16 + 3 * 4 + 1] == sc[128 + 96 + 5, 1]
    assert out[8 * 512 + (299 % 32) * 16 + ((299 % 128) // 32) * 4 + 1] == sc[299, 9]


def test_swizzle_is_a_padded_permutation():
    rows, kb = 131, 7
    sc = np.arange(1, rows * kb + 1, dtype=np.int64)
    lo = (sc % 256).astype(np.uint8).reshape(rows, kb)
    hi = (sc // 256).astype(np.uint8).reshape(rows, kb)
    a, b = oracle.swizzle_scales(lo, rows, kb), oracle.swizzle_scales(hi, rows, kb)
    ids = a.astype(np.int64) + 256 * b.astype(np.int64)
    nz = ids[ids != 0]
    assert np.array_equal(np.sort(nz), np.arange(1, rows * kb + 1))
    assert ids.size == 256 * 8 and (ids == 0).sum() == 256 * 8 - rows * kb


# ------------------------------------------------------ exact alpha step

def test_u128_to_double_rounds_to_nearest_even():
    """The conversion of the exact sums against Python's int -> float, which
    rounds to nearest with ties to even: random magnitudes, exact ties,
    values one unit either side of a tie, and carries into the next binade."""
    rng = np.random.default_rng(21)
    vals = [0, 1, 2**53 - 1, 2**53, 2**53 + 1, 2**53 + 3, 2**54 + 2, 2**54 + 6, 2**64 - 1, 2**64, 2**128 - 1,
            (2**53 - 1) * 2**60 + 2**59, (2**53 - 1) * 2**60 + 2**59 - 1, (2**53 - 1) * 2**60 + 2**59 + 1]
    for _ in range(2000):
        bits = int(rng.integers(1, 129))
        v = int(rng.integers(0, 2**63)) | (int(rng.integers(0, 2**63)) << 63) | (int(rng.integers(0, 4)) << 126)
        vals.append(v & (2**bits - 1))
        h = int(rng.integers(53, 127))  # an exact tie at bit h - 53
        t = (int(rng.integers(2**52, 2**53)) << (h - 52)) | (1 << (h - 53))
        vals += [t, t - 1, t + 1]
    for v in vals:
        assert oracle.u128_to_double(v) == float(v), v


def exact_alpha(w, codes, scales):
    """alpha* of the closed form from the exact rationals: sum Delta P and
    sum Delta^2 R as Python fractions (no rounding), each rounded once to
    double, the quotient in double, rounded to fp32."""
    from fractions import Fraction
    x = np.abs(block_view(w))
    q = np.abs(code_values(unpack_codes(codes, w.size))).reshape(-1, 16)
    d = E4M3_VALUES[scales.reshape(-1)]
    num, den = Fraction(0), Fraction(0)
    for xb, qb, db in zip(x, q, d):
        if db == 0.0:
            continue
        P = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xb, qb))
        R = sum(Fraction(float(b)) ** 2 for b in qb)
        num += Fraction(float(db)) * P
        den += Fraction(float(db)) ** 2 * R
    return float(np.float32(float(num) / float(den)))


def wide_range_tensor():
    """N(0, 1e-5) with one element 1.0: most block scales are E4M3 subnormals
    and most terms Delta P lie ~2^-30 below alpha, so any loss of low bits in
    the sums shows in alpha."""
    a = synthetic.bits_to_f32(synthetic.gaussian(16, 512, 1e-5, 35)).copy()
    a[3, 77] = 1.0
    return synthetic.to_bf16_bits(a)


@pytest.mark.parametrize("make", [lambda: synthetic.mlp_up(31, 16, 512), lambda: synthetic.student_t(8, 1024, 4.0, 0.02, 32),
                                  lambda: synthetic.mlp_70b(33, 16, 512), wide_range_tensor])
def test_cjso_alpha_is_the_exact_closed_form(make):
    """alpha after each CJSO iteration equals the closed form evaluated on
    exact sums (Python fractions), whatever the block order."""
    w = make()
    for T in (0, 1, 2):
        codes, scales, _ = oracle.quantize(w, oracle.CJSO, T)
        _, _, a_next = oracle.quantize(w, oracle.CJSO, T + 1)
        assert a_next == exact_alpha(w, codes, scales)
    # the blocks in another order (rows reversed): the same alpha
    _, _, a = oracle.quantize(w, oracle.CJSO, 2)
    _, _, b = oracle.quantize(np.ascontiguousarray(w[::-1]), oracle.CJSO, 2)
    assert a == b


def tie_tensor(extra_half_codes: int):
    """A tensor whose first CJSO alpha step lands exactly on an fp32 midpoint
    (extra_half_codes = 0), or one quarter of R below or above it (+1 / -1).

    alpha0 = 2^-12 (global max 0.65625 = 2688 * 2^-12).  Every block is
    exactly representable on its max-rule scale (x = q * Delta * alpha0, so
    Delta P = alpha0 Delta^2 R) except block B = [y, 0, ...]: y = 1.5078125 *
    2^-4 has scale Delta = 64 and code 6, and 6y exceeds 36 alpha0 Delta by
    eps = 3 * 2^-10.  Hence alpha1 = alpha0 + Delta eps / den with den =
    sum Delta^2 R; filler blocks of scale 64 make den = 3 * 2^32 exactly, and
    alpha1 = 2^-12 + 2^-36: halfway between 2^-12 and 2^-12 + 2^-35.  One more
    (one fewer) element of code 0.5 raises (lowers) den by 1024 and moves
    alpha1 just below (above) the midpoint."""
    u = 2.0 ** -6  # alpha0 * 64
    blocks = [[0.65625] + [0.0] * 15, [1.5078125 * 2.0 ** -4] + [0.0] * 15]
    blocks += [[6 * u] * 16] * 5458
    special = [6 * u] * 3 + [3 * u, 1.5 * u] + [0.5 * u] * (3 + extra_half_codes)
    blocks.append(special + [0.0] * (16 - len(special)))
    blocks += [[0.0] * 16] * (5504 - len(blocks))
    a = np.array(blocks, np.float32).reshape(128, 688)
    sign = np.where(np.random.default_rng(34).random(a.shape) < 0.5, -1.0, 1.0).astype(np.float32)
    return synthetic.to_bf16_bits(a * sign)


@pytest.mark.parametrize("extra,expect", [(0, 2.0 ** -12), (1, 2.0 ** -12), (-1, 2.0 ** -12 + 2.0 ** -35)])
def test_cjso_alpha_on_an_fp32_midpoint(extra, expect):
    """The first alpha step of the constructed tensors: exactly on a midpoint
    (ties to the even neighbour 2^-12), a hair below, a hair above."""
    w = tie_tensor(extra)
    _, _, a0 = oracle.quantize(w, oracle.MAX)
    assert a0 == 2.0 ** -12
    _, _, a1 = oracle.quantize(w, oracle.CJSO, 1)
    assert a1 == expect
