"""nvfp4_gemv, the W4A16 consumer of the quantized weights, against the
oracle's product of the dequantized bf16 weights (summed in double): within
the fp32 accumulation bound cols * 2^-24 * sum |w x| (every product is exact),
for every scale rule, 1..8 vectors, ragged rows and column chunks, both
kernel forms (activations resident in shared memory, or staged chunk by
chunk when they exceed 112 KiB), and the full-size tensors on sampled rows;
reproducible bit for bit."""
import numpy as np
import pytest
import torch

import nvfp4_block_scale_gb300 as nv
import oracle
import synthetic
from gpu_util import to_device

pytestmark = pytest.mark.gpu


def _acts(batch, cols, seed):
    rng = np.random.default_rng(seed)
    return synthetic.to_bf16_bits(rng.standard_normal((batch, cols)).astype(np.float32))


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _check(codes, scales, alpha, rows, cols, x_bits, y_gpu):
    y = oracle.gemv(codes, scales, alpha, rows, cols, x_bits)
    deq = _f32(oracle.dequantize(codes, scales, alpha, rows, cols)).astype(np.float64)
    mag = np.abs(_f32(x_bits).astype(np.float64)) @ np.abs(deq).T
    bound = cols * 2.0 ** -24 * mag + 1e-30
    err = np.abs(y_gpu.astype(np.float64) - y)
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("rows,cols,batch", [(1, 16, 1), (3, 48, 2), (37, 1040, 3), (129, 2064, 8),
                                             (256, 4096, 1), (256, 4096, 4), (17, 3072, 5), (64, 512, 7),
                                             (37, 8192, 8), (20, 28688, 2)])  # the last two: x beyond 112 KiB
@pytest.mark.parametrize("mode,iters", [(0, 0), (1, 0), (2, 2), (3, 1)])
def test_gemv_matches_oracle(rows, cols, batch, mode, iters):
    w = synthetic.student_t(rows, cols, 4.0, 0.02, 7000 + rows + cols + mode)
    codes, scales, alpha = nv.quantize(to_device(w), mode, iters)
    x_bits = _acts(batch, cols, rows * 3 + batch)
    y = nv.gemv(codes, scales, alpha, rows, cols, to_device(x_bits))
    torch.cuda.synchronize()
    _check(codes.cpu().numpy(), scales.cpu().numpy(), alpha.item(), rows, cols, x_bits, y.cpu().numpy())


def test_gemv_reproducible_and_empty():
    w = synthetic.mlp_up(80, 300, 2064)
    codes, scales, alpha = nv.quantize(to_device(w), nv.FOUR_OVER_SIX)
    x = to_device(_acts(4, 2064, 81))
    a = nv.gemv(codes, scales, alpha, 300, 2064, x)
    b = nv.gemv(codes, scales, alpha, 300, 2064, x)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    y = torch.full((2, 5), 7.0, device="cuda")
    z = torch.zeros((5, 0), dtype=torch.uint8, device="cuda")
    nv.gemv(z, z, alpha, 5, 0, torch.zeros((2, 0), dtype=torch.bfloat16, device="cuda"), out=y)
    torch.cuda.synchronize()
    assert not y.any()


@pytest.mark.parametrize("make,batch", [(lambda: synthetic.mlp_70b(4), 1), (lambda: synthetic.mlp_up(2), 8)])
def test_gemv_full_size_sampled_rows(make, batch):
    w = make()
    rows, cols = w.shape
    codes, scales, alpha = nv.quantize(to_device(w), nv.FOUR_OVER_SIX)
    x_bits = _acts(batch, cols, 90 + batch)
    y = nv.gemv(codes, scales, alpha, rows, cols, to_device(x_bits)).cpu().numpy()
    c, s, a = codes.cpu().numpy(), scales.cpu().numpy(), alpha.item()
    for r0 in (0, rows // 2 + 3, rows - 40):  # blocks of 40 rows: rows are contiguous in every layout
        _check(c[r0:r0 + 40], s[r0:r0 + 40], a, 40, cols, x_bits, y[:, r0:r0 + 40])
