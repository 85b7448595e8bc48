"""Parity at the benchmark workloads' full sizes, in the same launch
configuration the benchmark times.  The oracle computes alpha and every CJSO
iteration on the whole tensor and, except for the decoupled search, every
block; the decoupled search's final pass (about 100x the oracle's cost of the
other rules) is compared on whole row slabs, or on a seeded sample of blocks
of the stack's tensors."""
import os

import numpy as np
import pytest

import oracle
import synthetic
from gpu_util import block_mismatch, gpu_dequantize, gpu_quantize

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 8


def sample_blocks(nblocks, n=20000, seed=0):
    rng = np.random.default_rng(seed)
    s = rng.choice(nblocks, size=min(n, nblocks), replace=False)
    return np.unique(np.concatenate([s, [0, nblocks - 1]])).astype(np.int64)


def check_full(w, mode, iters):
    gc, gs, ga = gpu_quantize(w, mode, iters)
    oc, os_, oa = oracle.quantize(w, mode, iters, threads=THREADS)
    assert ga == oa
    bad = block_mismatch(gc, gs, oc, os_)
    if mode in (oracle.MAX, oracle.FOUR_OVER_SIX):
        assert not bad.any(), bad.sum()
    else:
        assert bad.sum() <= int(1e-6 * bad.size), (bad.sum(), bad.size)
        mg, mo = oracle.mse(w, gc, gs, ga), oracle.mse(w, oc, os_, oa)
        assert abs(mg - mo) <= 1e-6 * mo
    return gc, gs, ga


def check_sampled(w, mode, iters, nsample=20000):
    gc, gs, ga = gpu_quantize(w, mode, iters)
    nb = w.size // 16
    blocks = sample_blocks(nb, nsample, seed=mode * 100 + iters)
    oc, os_, oa = oracle.quantize_sampled(w, mode, iters, blocks, threads=THREADS)
    assert ga == oa
    g8 = gc.reshape(-1, 8)[blocks]
    gsc = gs.reshape(-1)[blocks]
    bad = block_mismatch(g8, gsc, oc, os_)
    assert bad.sum() <= int(1e-6 * nb), (bad.sum(), len(blocks))
    return gc, gs, ga


@pytest.fixture(scope="module")
def studentt_4k():
    return synthetic.studentt_4k()


@pytest.fixture(scope="module")
def mlp_up():
    return synthetic.mlp_up()


@pytest.mark.parametrize("mode", [oracle.MAX, oracle.FOUR_OVER_SIX])
def test_studentt_4k_full(studentt_4k, mode):
    """4096x4096 Student-t df=4 with outlier columns: max rule and FourOverSix."""
    check_full(studentt_4k, mode, 0)


@pytest.mark.parametrize("mode,iters", [(oracle.MAX, 0), (oracle.FOUR_OVER_SIX, 0), (oracle.CJSO, 5)])
def test_mlp_up_full(mlp_up, mode, iters):
    """4096x14336 row mixture: every block compared."""
    gc, gs, ga = check_full(mlp_up, mode, iters)
    if mode == oracle.MAX:
        od = oracle.dequantize(gc, gs, ga, *mlp_up.shape)
        assert np.array_equal(gpu_dequantize(gc, gs, ga, *mlp_up.shape), od)


def test_mlp_up_decoupled_row_slab(mlp_up):
    """Decoupled CJSO(5) on the 4096x14336 tensor: rows 0..511 in full (the
    10 % of hot rows are spread over them), plus a seeded sample elsewhere."""
    check_rows(mlp_up, oracle.CJSO_DECOUPLED, 5, np.arange(512))
    check_sampled(mlp_up, oracle.CJSO_DECOUPLED, 5)


def check_rows(w, mode, iters, rows):
    """Every block of the listed rows, against the oracle's final pass on them
    (alpha and the CJSO iterations over the whole tensor)."""
    gc, gs, ga = gpu_quantize(w, mode, iters)
    kb = w.shape[1] // 16
    blocks = (np.asarray(rows)[:, None] * kb + np.arange(kb)[None, :]).reshape(-1).astype(np.int64)
    oc, os_, oa = oracle.quantize_sampled(w, mode, iters, blocks, threads=THREADS)
    assert ga == oa
    bad = block_mismatch(gc.reshape(-1, 8)[blocks], gs.reshape(-1)[blocks], oc, os_)
    assert bad.sum() <= int(1e-6 * (w.size // 16)), (bad.sum(), len(blocks))
    return gc, gs, ga


@pytest.fixture(scope="module")
def mlp_70b():
    return synthetic.mlp_70b()


@pytest.mark.parametrize("mode,iters", [(oracle.MAX, 0), (oracle.FOUR_OVER_SIX, 0), (oracle.CJSO, 5)])
def test_mlp_70b_full(mlp_70b, mode, iters):
    """8192x28672 N(0, 0.01) with +-U(0.3, 1) spikes (larger than L2): every
    block compared; the max-rule output dequantized in full."""
    gc, gs, ga = check_full(mlp_70b, mode, iters)
    if mode == oracle.MAX:
        od = oracle.dequantize(gc, gs, ga, *mlp_70b.shape)
        assert np.array_equal(gpu_dequantize(gc, gs, ga, *mlp_70b.shape), od)


def test_mlp_70b_decoupled_row_slabs(mlp_70b):
    """Decoupled CJSO(5) on the 8192x28672 tensor: 512 whole rows (the first
    and last 256), every block of them."""
    rows = np.r_[0:256, mlp_70b.shape[0] - 256:mlp_70b.shape[0]]
    check_rows(mlp_70b, oracle.CJSO_DECOUPLED, 5, rows)


@pytest.mark.parametrize("index", [0, 1, 4, 6, 223])
def test_llama3_8b_tensors(index):
    """Tensors of the 224-tensor Llama-3-8B-shaped stack (each its own alpha):
    FourOverSix in full, decoupled CJSO on sampled blocks."""
    w = synthetic.llama3_8b_tensor(index)
    check_full(w, oracle.FOUR_OVER_SIX, 0)
    check_sampled(w, oracle.CJSO_DECOUPLED, 5, nsample=3000)


@pytest.mark.parametrize("mode,iters", [(oracle.MAX, 0), (oracle.FOUR_OVER_SIX, 0), (oracle.CJSO, 2)])
def test_beyond_half_l2_with_a_partial_last_chunk(mode, iters):
    """4099 x 9232 (72 MiB of bf16, more than half of L2): the amax pass streams
    W through shared memory in 32 KiB bulk copies, the last one partial."""
    w = synthetic.student_t(4099, 9232, 4.0, 0.02, 4242)
    assert (w.nbytes % 32768) != 0
    if mode == oracle.CJSO:
        check_sampled(w, mode, iters)
    else:
        check_full(w, mode, iters)
