"""nvfp4_gemm, the W4A16 product on the tensor cores (tcgen05, accumulator in
tensor memory), against the oracle's product of the dequantized bf16 weights
summed in double.  Every product is exact; the tensor cores accumulate in
fp32 in an order of their own, so the bar is 2 * (cols + 2) * 2^-24 *
sum |w x| per output (twice the bound of any order of fp32 additions plus
the additions of the partial sums of CTAs that share a tile).  Ragged rows
and K steps, every tile width (16..256 vectors), CTAs whose step ranges
cover one step, part of a tile or several whole tiles (so the double-buffered
accumulator is reused), code and scale arrays that are not 16-byte aligned,
all four scale rules, and the benchmark's 8192x28672 tensor on sampled
rows."""
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
    bound = 2 * (cols + 2) * 2.0 ** -24 * mag + 1e-30
    err = np.abs(y_gpu.astype(np.float64) - y)
    assert np.all(np.isfinite(y_gpu))
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("rows,cols,batch", [(128, 64, 16), (1, 16, 1), (300, 1040, 20), (1024, 4096, 64),
                                             (200, 2064, 256), (5000, 512, 3), (130, 28688, 40)])
def test_gemm_matches_oracle(rows, cols, batch):
    w = synthetic.student_t(rows, cols, 4.0, 0.02, 9000 + rows + cols)
    codes, scales, alpha = nv.quantize(to_device(w), nv.FOUR_OVER_SIX)
    x_bits = _acts(batch, cols, rows + batch)
    y = nv.gemm(codes, scales, alpha, rows, cols, to_device(x_bits))
    torch.cuda.synchronize()
    _check(codes.cpu().numpy(), scales.cpu().numpy(), alpha.item(), rows, cols, x_bits, y.cpu().numpy())


@pytest.mark.parametrize("mode,iters", [(0, 0), (2, 2), (3, 1)])
def test_gemm_every_rule_and_repeatable(mode, iters):
    w = synthetic.mlp_up(9100 + mode, 256, 1024)
    codes, scales, alpha = nv.quantize(to_device(w), mode, iters)
    x = to_device(_acts(24, 1024, 9101))
    a = nv.gemm(codes, scales, alpha, 256, 1024, x)
    b = nv.gemm(codes, scales, alpha, 256, 1024, x)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    _check(codes.cpu().numpy(), scales.cpu().numpy(), alpha.item(), 256, 1024, x.view(torch.int16).cpu().numpy()
           .view(np.uint16), a.cpu().numpy())


def test_gemm_full_size_sampled_rows():
    w = synthetic.mlp_70b(4)
    rows, cols = w.shape
    codes, scales, alpha = nv.quantize(to_device(w), nv.FOUR_OVER_SIX)
    x_bits = _acts(64, cols, 9200)
    y = nv.gemm(codes, scales, alpha, rows, cols, to_device(x_bits)).cpu().numpy()
    c, s, a = codes.cpu().numpy(), scales.cpu().numpy(), alpha.item()
    for r0 in (0, rows // 2 + 5, rows - 24):
        _check(c[r0:r0 + 24], s[r0:r0 + 24], a, 24, cols, x_bits, y[:, r0:r0 + 24])


@pytest.mark.parametrize("rows,cols,batch", [(51200, 128, 16), (40000, 64, 200), (30000, 192, 33), (1, 4096, 5)])
def test_gemm_ctas_spanning_several_tiles(rows, cols, batch):
    # 128-column steps: K = 1 or 2 per tile, so one CTA's range covers 2-3 tiles
    # (three or more accumulators in a row); the last case gives every CTA one step
    w = synthetic.gaussian(rows, cols, 0.02, 9300 + rows)
    codes, scales, alpha = nv.quantize(to_device(w), nv.MAX)
    x_bits = _acts(batch, cols, 9301 + batch)
    y = nv.gemm(codes, scales, alpha, rows, cols, to_device(x_bits))
    torch.cuda.synchronize()
    _check(codes.cpu().numpy(), scales.cpu().numpy(), alpha.item(), rows, cols, x_bits, y.cpu().numpy())


def test_gemm_unaligned_codes_and_scales():
    # codes 8 bytes and scales 1 byte past a 16-byte boundary: the per-block load path
    rows, cols, batch = 384, 2048, 12
    w = synthetic.student_t(rows, cols, 4.0, 0.02, 9400)
    codes, scales, alpha = nv.quantize(to_device(w), nv.FOUR_OVER_SIX)
    cbuf = torch.zeros(codes.numel() + 16, dtype=torch.uint8, device="cuda")
    sbuf = torch.zeros(scales.numel() + 16, dtype=torch.uint8, device="cuda")
    c8 = cbuf[8:8 + codes.numel()]
    s1 = sbuf[1:1 + scales.numel()]
    c8.copy_(codes.reshape(-1))
    s1.copy_(scales.reshape(-1))
    x_bits = _acts(batch, cols, 9401)
    x = to_device(x_bits)
    y = nv.gemm(c8, s1, alpha, rows, cols, x)
    ref = nv.gemm(codes, scales, alpha, rows, cols, x)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)  # same steps, same order: only the load path differs
    _check(codes.cpu().numpy(), scales.cpu().numpy(), alpha.item(), rows, cols, x_bits, y.cpu().numpy())
