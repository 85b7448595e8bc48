"""nvfp4_quantize_noalloc: the allocation-free quantize entry point.

Some callers cannot let a library allocate device memory: serving engines
that reserve nearly all HBM up front and account for every byte, threads that
must never enter an allocator because it can block, and embedders whose own
allocator must stay the only one.  For them the library offers
nvfp4_quantize_noalloc, which keeps its scratch in a fixed 16 KiB static
device array.  These tests check, through the C ABI, that it returns exactly
what nvfp4_quantize returns, on two consecutive calls (the second call finds
the first call's leftovers in the shared array), and that it rejects tensors
larger than its scratch can serve.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

import nvfp4_block_scale_gb300 as nv
import synthetic

A16 = 0x10000  # fake aligned address: the size check happens before any device access


def test_noalloc_rejects_tensors_beyond_its_scratch():
    too_many = (1 << 28) + 16  # NVFP4_NOALLOC_MAX_ELEMS + one block
    assert nv.nvfp4_quantize_noalloc(A16, 1, too_many, 0, A16, A16, A16, None) == 1
    assert nv.nvfp4_quantize_noalloc(A16, 16384, 16385 + 15, 1, A16, A16, A16, None) == 1
    assert nv.nvfp4_quantize_noalloc(A16, 4, 16, 2, A16, A16, A16, None) == 1  # CJSO modes not offered


@pytest.mark.gpu
def test_noalloc_matches_quantize_on_two_calls_in_a_row():
    import torch

    from gpu_util import to_device

    stream = torch.cuda.current_stream()
    cases = [(synthetic.studentt_4k(71, 1024, 4096), nv.FOUR_OVER_SIX),
             (synthetic.mlp_up(72, 300, 2064), nv.MAX)]
    for w_bits, mode in cases:  # two calls in a row, different tensors and modes
        W = to_device(w_bits)
        rows, cols = w_bits.shape
        ref = nv.quantize(W, mode)
        codes = torch.full((rows, cols // 2), 0xAB, dtype=torch.uint8, device="cuda")
        scales = torch.full((rows, cols // 16), 0xCD, dtype=torch.uint8, device="cuda")
        alpha = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        st = nv.nvfp4_quantize_noalloc(W.data_ptr(), rows, cols, mode, codes.data_ptr(), scales.data_ptr(),
                                       alpha.data_ptr(), stream.cuda_stream)
        assert st == 0, nv.nvfp4_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(codes, ref[0])
        assert torch.equal(scales, ref[1])
        assert alpha.item() == ref[2].item()


@pytest.mark.gpu
def test_noalloc_at_its_size_limit_then_on_a_smaller_tensor():
    """Exactly NVFP4_NOALLOC_MAX_ELEMS = 2^28 elements (512 MiB of bf16: every
    scratch slot in use, the last one read), then a smaller tensor whose
    max|W| is far below the first one's: its call uses fewer slots, so a
    leftover slot of the first call, if read, would change its alpha.  Both
    compared with nvfp4_quantize."""
    import torch

    stream = torch.cuda.current_stream()
    g = torch.Generator(device="cuda").manual_seed(90)
    big = (torch.randn((16384, 16384), generator=g, device="cuda") * 3.0).to(torch.bfloat16)  # 2^28 elements
    small = (torch.randn((1024, 4096), generator=g, device="cuda") * 0.01).to(torch.bfloat16)
    for W, mode in ((big, nv.MAX), (small, nv.FOUR_OVER_SIX)):
        rows, cols = W.shape
        ref = nv.quantize(W, mode)
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device="cuda")
        alpha = torch.empty((1,), dtype=torch.float32, device="cuda")
        st = nv.nvfp4_quantize_noalloc(W.data_ptr(), rows, cols, mode, codes.data_ptr(), scales.data_ptr(),
                                       alpha.data_ptr(), stream.cuda_stream)
        assert st == 0, nv.nvfp4_status_string(st)
        torch.cuda.synchronize()
        assert alpha.item() == ref[2].item()
        assert torch.equal(codes, ref[0]) and torch.equal(scales, ref[1])
