"""Hardware E2M1 / E4M3 rounding (the cvt instructions the kernels use),
checked bit for bit against the oracle's definitions through the C ABI's
element-wise encode entry points."""
import numpy as np
import pytest
import torch

import nvfp4_block_scale_gb300 as nv
import oracle

pytestmark = pytest.mark.gpu


def f32_from_bits(bits):
    return np.asarray(bits, np.uint32).view(np.float32)


def gpu_e2m1(v):
    out = nv.encode_e2m1(torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda())
    return out.cpu().numpy()


def gpu_e4m3(v):
    out = nv.encode_e4m3(torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda())
    return out.cpu().numpy()


def test_e2m1_every_fp32_in_0125_to_8_both_signs():
    lo = int(np.float32(0.125).view(np.uint32))
    hi = int(np.float32(8.0).view(np.uint32))
    step = 1 << 23
    for start in range(lo, hi, step):
        v = f32_from_bits(np.arange(start, min(start + step, hi), dtype=np.uint32))
        assert np.array_equal(gpu_e2m1(v), oracle.e2m1_encode(v)), hex(start)
        assert np.array_equal(gpu_e2m1(-v), oracle.e2m1_encode(-v)), hex(start)


def test_e2m1_special_values():
    v = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-30, 0.124, 6.0, 7.0, 7.0000005, 1e30, np.inf, -np.inf, -6.5,
                  3.4e38], np.float32)
    assert np.array_equal(gpu_e2m1(v), oracle.e2m1_encode(v))


def test_e4m3_every_fp32_in_range():
    """Every fp32 pattern in [2^-12, 448] (the range block scales take), plus
    saturation above 448."""
    lo = int(np.float32(2.0 ** -12).view(np.uint32))
    hi = int(np.float32(448.0).view(np.uint32)) + 1
    step = 1 << 24
    for start in range(lo, hi, step):
        v = f32_from_bits(np.arange(start, min(start + step, hi), dtype=np.uint32))
        assert np.array_equal(gpu_e4m3(v), oracle.e4m3_encode(v)), hex(start)
    v = np.array([0.0, 1e-30, 2.0 ** -10, 448.5, 463.9, 464.0, 1e6, 3e38, np.inf], np.float32)
    assert np.array_equal(gpu_e4m3(v), oracle.e4m3_encode(v))
