"""Failure paths, driven through the C ABI's test hooks without faulting
anything: a scratch allocation that fails (the call returns
NVFP4_ERR_OUT_OF_MEMORY and enqueues nothing), and a bounded device wait that
gives up (alpha, or the product's outputs, come out NaN; every copy and MMA
already issued completes, and the context stays usable)."""
import math

import pytest
import torch

import nvfp4_block_scale_gb300 as nv
import synthetic
from gpu_util import to_device

pytestmark = pytest.mark.gpu

OOM = 5


def _sentinel(shape, dtype, value):
    return torch.full(shape, value, dtype=dtype, device="cuda")


def test_allocation_failure_returns_out_of_memory_and_enqueues_nothing():
    stream = torch.cuda.current_stream().cuda_stream
    w = to_device(synthetic.mlp_up(80, 256, 1024))
    rows, cols = w.shape
    ref = nv.quantize(w, nv.FOUR_OVER_SIX)
    x = to_device(synthetic.gaussian(16, cols, 1.0, 81))
    try:
        for mode, iters in ((nv.FOUR_OVER_SIX, 0), (nv.CJSO, 2), (nv.CJSO_DECOUPLED, 1)):
            codes = _sentinel((rows, cols // 2), torch.uint8, 0xAB)
            scales = _sentinel((rows, cols // 16), torch.uint8, 0xCD)
            alpha = _sentinel((1,), torch.float32, -1.0)
            assert nv.nvfp4_test_fail_allocations(1) == 0
            st = nv.nvfp4_quantize(w.data_ptr(), rows, cols, mode, iters, codes.data_ptr(), scales.data_ptr(),
                                   alpha.data_ptr(), stream)
            torch.cuda.synchronize()
            assert st == OOM
            assert bool((codes == 0xAB).all()) and bool((scales == 0xCD).all()) and alpha.item() == -1.0
        # the hook is used up: the next call succeeds
        got = nv.quantize(w, nv.FOUR_OVER_SIX)
        assert all(torch.equal(a, b) for a, b in zip(got, ref))
        # a grouped call: its one scratch allocation fails before anything is enqueued
        outs = [(_sentinel((rows, cols // 2), torch.uint8, 0xAB), _sentinel((rows, cols // 16), torch.uint8, 0xCD),
                 _sentinel((1,), torch.float32, -1.0)) for _ in range(2)]
        nv.nvfp4_test_fail_allocations(1)
        with pytest.raises(nv.Nvfp4Error) as ei:
            nv.quantize_grouped([w, w], nv.MAX, outs=outs)
        torch.cuda.synchronize()
        assert ei.value.status == OOM
        for c, s, a in outs:
            assert bool((c == 0xAB).all()) and bool((s == 0xCD).all()) and a.item() == -1.0
        # the tensor-core product
        y = _sentinel((16, rows), torch.float32, 7.0)
        nv.nvfp4_test_fail_allocations(1)
        with pytest.raises(nv.Nvfp4Error) as ei:
            nv.gemm(*ref, rows, cols, x, out=y)
        torch.cuda.synchronize()
        assert ei.value.status == OOM and bool((y == 7.0).all())
    finally:
        nv.nvfp4_test_fail_allocations(0)


def test_amax_pass_wait_that_gives_up_makes_alpha_nan():
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    cols = 4096
    rows = l2 // 4 // cols + 64  # bf16 bytes > L2 / 2: the bulk-copy max|W| pass
    w = to_device(synthetic.gaussian(rows, cols, 0.02, 82))
    ref = nv.quantize(w, nv.MAX)
    torch.cuda.synchronize()
    try:
        assert nv.nvfp4_test_first_wait_tries(0) == 0
        _, _, a = nv.quantize(w, nv.MAX)
        torch.cuda.synchronize()
        assert math.isnan(a.item())
    finally:
        nv.nvfp4_test_first_wait_tries(-1)
    got = nv.quantize(w, nv.MAX)  # the context is still usable
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(got, ref))


def test_tensor_core_product_wait_that_gives_up_makes_outputs_nan():
    rows, cols, batch = 512, 2048, 16
    w = to_device(synthetic.mlp_up(83, rows, cols))
    q = nv.quantize(w, nv.FOUR_OVER_SIX)
    x = to_device(synthetic.gaussian(batch, cols, 1.0, 84))
    ref = nv.gemm(*q, rows, cols, x)
    torch.cuda.synchronize()
    try:
        assert nv.nvfp4_test_first_wait_tries(0) == 0
        y = nv.gemm(*q, rows, cols, x)
        torch.cuda.synchronize()
        assert bool(torch.isnan(y).all())
    finally:
        nv.nvfp4_test_first_wait_tries(-1)
    y = nv.gemm(*q, rows, cols, x)  # the context is still usable
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
