"""Parity of the CUDA path (through the C ABI) with the CPU oracle on seeded
inputs small enough for the whole oracle: several tiles, ragged tails, edge
cases.  Max rule, FourOverSix and dequantize must be bit-exact; CJSO modes
must give the same alpha, differ in at most 1e-6 of the blocks, and agree on
the reconstruction MSE to 1e-6 relative."""
import numpy as np
import pytest
import torch

import nvfp4_block_scale_gb300 as nv
import oracle
import synthetic
from gpu_util import block_mismatch, gpu_dequantize, gpu_quantize, to_device

pytestmark = pytest.mark.gpu

MODES = [(oracle.MAX, 0), (oracle.FOUR_OVER_SIX, 0), (oracle.CJSO, 0), (oracle.CJSO, 1), (oracle.CJSO, 5),
         (oracle.CJSO_DECOUPLED, 0), (oracle.CJSO_DECOUPLED, 3)]


def check(w, mode, iters, threads=8):
    gc, gs, ga = gpu_quantize(w, mode, iters)
    oc, os_, oa = oracle.quantize(w, mode, iters, threads=threads)
    if mode in (oracle.MAX, oracle.FOUR_OVER_SIX):
        assert ga == oa
        assert np.array_equal(gs, os_), "scales differ"
        assert np.array_equal(gc, oc), "codes differ"
    else:
        assert ga == oa, (ga, oa)
        bad = block_mismatch(gc, gs, oc, os_)
        assert bad.sum() <= int(1e-6 * bad.size), (bad.sum(), bad.size)
        mg = oracle.mse(w, gc, gs, ga)
        mo = oracle.mse(w, oc, os_, oa)
        assert abs(mg - mo) <= 1e-6 * max(mo, 1e-300)
    return gc, gs, ga


SHAPES = [(1, 16), (1, 32), (3, 48), (2, 4096), (37, 1040), (129, 272), (256, 512)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("mode,iters", MODES)
def test_parity_small_shapes(shape, mode, iters):
    rows, cols = shape
    w = synthetic.student_t(rows, cols, 4.0, 0.02, 1000 + rows * 7 + cols)
    check(w, mode, iters)


@pytest.mark.parametrize("mode,iters", MODES)
def test_parity_gauss_1k(mode, iters):
    """1024x1024 N(0, 0.02), seed 0: all four modes and the dequant round trip."""
    w = synthetic.gauss_1k()
    gc, gs, ga = check(w, mode, iters)
    od = oracle.dequantize(gc, gs, ga, *w.shape)
    assert np.array_equal(gpu_dequantize(gc, gs, ga, *w.shape), od)


@pytest.mark.parametrize("mode,iters", MODES)
def test_parity_mixtures(mode, iters):
    check(synthetic.mlp_up(50, 256, 1024), mode, iters)
    check(synthetic.studentt_4k(51, 512, 1024), mode, iters)
    check(synthetic.mlp_70b(52, 128, 2048), mode, iters)


def test_representable_roundtrip_and_edge_values():
    """Exactly representable tensors come back exactly; zeros, -0.0, tiny
    blocks (scale 0), E4M3-saturating outliers."""
    rng = np.random.default_rng(3)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    nb = 512
    d = rng.integers(1, 0x7F, nb)
    d[0] = 0x7E
    e4 = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    mags = rng.integers(0, 8, (nb, 16))
    mags[:, 3] = 7
    sg = rng.integers(0, 2, (nb, 16))
    w = grid[mags] * np.where(sg == 1, -1.0, 1.0) * e4[d][:, None] * 2.0 ** -12
    w = w.reshape(8, 1024).astype(np.float32)
    w[1, 0:16] = 0.0
    w[1, 16:32] = -0.0
    w[2, 0:16] = 1e-12
    bits = synthetic.to_bf16_bits(w)
    for mode, iters in MODES:
        check(bits, mode, iters)
    gc, gs, ga = gpu_quantize(bits, oracle.MAX)
    back = gpu_dequantize(gc, gs, ga, *bits.shape)
    keep = np.ones(bits.shape, bool)
    keep[1:3, 0:32] = False
    assert np.array_equal(back[keep], bits[keep])


def test_all_zero_and_empty():
    z = synthetic.to_bf16_bits(np.zeros((4, 64), np.float32))
    for mode, iters in MODES:
        gc, gs, ga = check(z, mode, iters)
        assert ga == 0.0 and not gc.any() and not gs.any()
    W = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    alpha = torch.full((1,), 7.0, device="cuda")
    st = nv.nvfp4_quantize(W.data_ptr(), 0, 64, 0, 0, None, None, alpha.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and alpha.item() == 0.0


def test_deterministic_and_stream_ordered():
    """Same bits on repeated runs, on a side stream, with the input written
    just before on that stream (catches races and missing stream ordering)."""
    w = synthetic.mlp_up(60, 512, 2048)
    ref = [gpu_quantize(w, m, i) for m, i in MODES]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        W = torch.empty((512, 2048), dtype=torch.bfloat16, device="cuda")
        W.copy_(to_device(w))
        for (m, i), r in zip(MODES, ref):
            for _ in range(2):
                c, sc, a = nv.quantize(W, m, i, stream=s)
                s.synchronize()
                assert np.array_equal(c.cpu().numpy(), r[0]) and np.array_equal(sc.cpu().numpy(), r[1])
                assert a.item() == r[2]


def test_dequant_of_every_code_and_scale():
    """Every (code, scale) pair once: 16 codes x 256 scale bytes."""
    rows, cols = 256, 256  # 4096 blocks
    codes = np.zeros((rows, cols // 2), np.uint8)
    c = np.arange(16, dtype=np.uint8)
    codes[:] = np.tile(c[0::2] | (c[1::2] << 4), cols // 16)
    scales = np.repeat(np.arange(256, dtype=np.uint8), 16).reshape(rows, cols // 16)
    scales[scales == 0x7F] = 0x7E
    scales[scales == 0xFF] = 0xFE
    for a in (2.0 ** -12, 1.2345e-5, 0.0):
        od = oracle.dequantize(codes, scales, a, rows, cols)
        assert np.array_equal(gpu_dequantize(codes, scales, a, rows, cols), od)


@pytest.mark.parametrize("extra,expect", [(0, 2.0 ** -12), (1, 2.0 ** -12), (-1, 2.0 ** -12 + 2.0 ** -35)])
def test_cjso_alpha_on_an_fp32_midpoint(extra, expect):
    """Tensors whose first CJSO alpha step lands exactly on an fp32 midpoint,
    a hair below it and a hair above it (constructed in the oracle's pins):
    the device's exact 128-bit sums give the same alpha as the oracle and as
    the arithmetic, and every block agrees, for CJSO(1) and CJSO(3)."""
    from test_oracle_method import tie_tensor
    w = tie_tensor(extra)
    gc, gs, ga = gpu_quantize(w, oracle.CJSO, 1)
    assert ga == expect
    for iters in (1, 3):
        gc, gs, ga = gpu_quantize(w, oracle.CJSO, iters)
        oc, os_, oa = oracle.quantize(w, oracle.CJSO, iters)
        assert ga == oa
        assert np.array_equal(gc, oc) and np.array_equal(gs, os_)


def test_decoupled_deferred_blocks_beyond_the_list():
    """On exactly representable tensors the decoupled search's crossings land
    exactly on integer k, so nearly every block goes to the plain search:
    524,288 blocks are more than the list of deferred blocks holds (2^18), so
    some are searched by the second kernel and the rest inline by the first.
    Every block compared on a seeded sample (both kinds), and the first rows
    in full."""
    rng = np.random.default_rng(44)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rows, cols = 2048, 4096
    nb = rows * cols // 16
    e4 = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    d = rng.integers(0x30, 0x70, nb)
    d[0] = 0x7E
    mags = rng.integers(0, 8, (nb, 16))
    mags[:, 5] = 7
    w = grid[mags] * np.where(rng.integers(0, 2, (nb, 16)) == 1, -1.0, 1.0) * e4[d][:, None] * 2.0 ** -12
    bits = synthetic.to_bf16_bits(w.reshape(rows, cols).astype(np.float32))
    gc, gs, ga = gpu_quantize(bits, oracle.CJSO_DECOUPLED, 0)
    blocks = np.unique(np.concatenate([np.arange(0, 2048), rng.choice(nb, 20000, replace=False)])).astype(np.int64)
    oc, os_, oa = oracle.quantize_sampled(bits, oracle.CJSO_DECOUPLED, 0, blocks, threads=8)
    assert ga == oa
    bad = block_mismatch(gc.reshape(-1, 8)[blocks], gs.reshape(-1)[blocks], oc, os_)
    assert not bad.any(), bad.sum()
