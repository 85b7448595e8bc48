"""nvfp4_swizzle_scales: the tensor-core scale layout, bit-exact against the
oracle's layout on ragged and full-size shapes; and the quantized codes with
swizzled scales consumed by a block-scaled NVFP4 x NVFP4 tensor-core matrix
multiply (PyTorch's _scaled_mm over cuBLASLt), an independent reader of the
layout, against the exact product of the decoded operands."""
import numpy as np
import pytest
import torch

import nvfp4_block_scale_gb300 as nv
import oracle
import synthetic
from gpu_util import to_device

pytestmark = pytest.mark.gpu

E2M1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (128, 64), (300, 160), (129, 2064), (4096, 4096),
                                       (8192, 28672)])  # the last: the benchmark's 8192x28672 tensor
def test_swizzle_matches_oracle(rows, cols):
    rng = np.random.default_rng(rows * 31 + cols)
    sc = rng.integers(0, 127, (rows, cols // 16)).astype(np.uint8)
    got = nv.swizzle_scales(torch.from_numpy(sc).cuda(), rows, cols)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.swizzle_scales(sc, rows, cols // 16))


def _decode(codes, scales, rows, cols):
    c = codes.reshape(rows, cols // 2)
    nib = np.empty((rows, cols), np.uint8)
    nib[:, 0::2] = c & 0xF
    nib[:, 1::2] = c >> 4
    q = E2M1[nib & 7] * np.where(nib & 8, -1.0, 1.0)
    d = np.array([oracle.e4m3_value(int(v)) for v in range(256)])[scales.reshape(rows, cols // 16)]
    return q * np.repeat(d, 16, axis=1)  # q * Delta (alpha applied outside the product)


def test_tensor_core_gemm_reads_the_layout():
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this PyTorch has no float4_e2m1fn_x2 type")
    M, N, K = 256, 128, 1024
    wa = synthetic.student_t(M, K, 4.0, 0.02, 901)
    wb = synthetic.gaussian(N, K, 0.02, 902)
    ca, sa, aa = nv.quantize(to_device(wa), nv.FOUR_OVER_SIX)
    cb, sb, ab = nv.quantize(to_device(wb), nv.MAX)
    za = nv.swizzle_scales(sa, M, K)
    zb = nv.swizzle_scales(sb, N, K)
    try:
        out = torch._scaled_mm(ca.view(torch.float4_e2m1fn_x2), cb.view(torch.float4_e2m1fn_x2).t(),
                               za.view(torch.float8_e4m3fn), zb.view(torch.float8_e4m3fn),
                               out_dtype=torch.bfloat16)
    except (RuntimeError, TypeError, ValueError, NotImplementedError) as e:
        pytest.skip(f"block-scaled NVFP4 matrix multiply not available in this PyTorch: {e}")
    torch.cuda.synchronize()
    A = _decode(ca.cpu().numpy(), sa.cpu().numpy(), M, K)
    B = _decode(cb.cpu().numpy(), sb.cpu().numpy(), N, K)
    ref = A @ B.T
    mag = np.abs(A) @ np.abs(B).T
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -23 * mag + 1e-30)
    # the layout matters: the same product with linear scales is wrong somewhere
    try:
        bad = torch._scaled_mm(ca.view(torch.float4_e2m1fn_x2), cb.view(torch.float4_e2m1fn_x2).t(),
                               sa.reshape(-1).view(torch.float8_e4m3fn), sb.reshape(-1).view(torch.float8_e4m3fn),
                               out_dtype=torch.bfloat16).float().cpu().numpy()
        assert not np.allclose(bad, ref, rtol=2.0 ** -6, atol=0)
    except RuntimeError:
        pass  # a size check rejected the unpadded scales: also fine
