"""A tensor of more than 2^31 elements (65,600 x 32,768 = 2,149,580,800; 4.3 GB
of bf16), so that every flat element, code-byte and block index the kernels
form crosses 32 bits somewhere: max rule, FourOverSix and decoupled CJSO(1)
against the oracle on blocks at both ends, on both sides of element 2^31 and
on a seeded sample; dequantize on the rows around element 2^31 and the last
rows."""
import os

import numpy as np
import pytest

import oracle
import synthetic
from gpu_util import block_mismatch, gpu_dequantize, gpu_quantize

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 8
ROWS, COLS = 65600, 32768


@pytest.fixture(scope="module")
def big():
    w = synthetic.gaussian_bf16_large(ROWS, COLS, 0.02, 2031)
    w[ROWS - 1, COLS - 5] = 0x3F00  # the tensor's maximum, 0.5, in its last block
    return w


def probe_blocks(nb):
    edge = 1 << 27  # block of element 2^31
    rng = np.random.default_rng(31)
    parts = [np.arange(0, 1000), np.arange(nb - 1000, nb), np.arange(edge - 500, edge + 500),
             rng.choice(nb, 20000, replace=False)]
    return np.unique(np.concatenate(parts)).astype(np.int64)


@pytest.mark.parametrize("mode,iters", [(oracle.MAX, 0), (oracle.FOUR_OVER_SIX, 0), (oracle.CJSO_DECOUPLED, 1)])
def test_quantize_beyond_2_31_elements(big, mode, iters):
    assert big.size > (1 << 31)
    gc, gs, ga = gpu_quantize(big, mode, iters)
    nb = big.size // 16
    blocks = probe_blocks(nb)
    oc, os_, oa = oracle.quantize_sampled(big, mode, iters, blocks, threads=THREADS)
    assert ga == oa
    assert ga == np.float32(0.5) / np.float32(2688.0) or mode == oracle.CJSO_DECOUPLED
    bad = block_mismatch(gc.reshape(-1, 8)[blocks], gs.reshape(-1)[blocks], oc, os_)
    assert not bad.any(), (bad.sum(), len(blocks))
    if mode == oracle.MAX:
        dq = gpu_dequantize(gc, gs, ga, ROWS, COLS)
        for r0 in ((1 << 31) // COLS - 2, ROWS - 3):  # the rows around element 2^31, the last rows
            r1 = r0 + 3
            od = oracle.dequantize(gc[r0:r1], gs[r0:r1], ga, r1 - r0, COLS)
            assert np.array_equal(dq[r0:r1], od), r0
