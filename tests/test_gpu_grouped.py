"""nvfp4_quantize_grouped: every tensor of a group comes out exactly as the
single-tensor call (and the oracle) gives it, whatever its size, position in
the group or neighbours: tiny and ragged tensors, all-zero and empty ones,
tensors of several tiles, groups longer than one slice of NVFP4_GROUP_MAX
tensors, and groups large enough to be cut into parts that alternate between
two streams (also under CUDA-graph capture)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scale_gb300 as nv
import oracle
import synthetic
from gpu_util import to_device

pytestmark = pytest.mark.gpu


def _mixed_group(seed):
    rng = np.random.default_rng(seed)
    ws = [synthetic.student_t(1, 16, 4.0, 0.02, seed + 1),        # one block
          synthetic.gaussian(3, 32, 0.02, seed + 2),
          np.zeros((4, 64), np.uint16),                           # all zero: alpha 0
          np.zeros((0, 16), np.uint16),                           # empty
          synthetic.mlp_up(seed + 3, 300, 2064),                  # ragged last tile
          synthetic.student_t(17, 4112, 5.0, 0.02, seed + 4),
          synthetic.studentt_4k(seed + 5, 1024, 4096),            # many tiles
          np.zeros((0, 0), np.uint16)]
    for k in range(6):  # small tensors of random shapes between the others
        ws.insert(int(rng.integers(0, len(ws))),
                  synthetic.gaussian(int(rng.integers(1, 40)), 16 * int(rng.integers(1, 70)), 0.01 * (k + 1),
                                     seed + 10 + k))
    return ws


def _run_group(ws, mode, iters=0):
    Wd = [to_device(w) if w.size else torch.empty(w.shape, dtype=torch.bfloat16, device="cuda") for w in ws]
    outs = []
    for W in Wd:  # garbage in every output, so that a skipped block shows
        r, c = W.shape
        outs.append((torch.full((r, c // 2), 0xA5, dtype=torch.uint8, device="cuda"),
                     torch.full((r, c // 16), 0x5A, dtype=torch.uint8, device="cuda"),
                     torch.full((1,), -7.0, dtype=torch.float32, device="cuda")))
    nv.quantize_grouped(Wd, mode, iters, outs=outs)
    torch.cuda.synchronize()
    return Wd, outs


@pytest.mark.parametrize("mode", [nv.MAX, nv.FOUR_OVER_SIX])
def test_grouped_matches_single_calls_and_oracle(mode):
    ws = _mixed_group(300 + mode)
    Wd, outs = _run_group(ws, mode)
    for w, W, (c, s, a) in zip(ws, Wd, outs):
        if w.size == 0:
            assert a.item() == 0.0
            continue
        rc, rs, ra = nv.quantize(W, mode)
        assert torch.equal(c, rc) and torch.equal(s, rs) and a.item() == ra.item()
        if w.size <= 1 << 16:
            oc, os_, oa = oracle.quantize(w, mode)
            assert np.array_equal(c.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy(), os_)
            assert a.item() == oa


def test_grouped_longer_than_one_slice():
    rng = np.random.default_rng(77)
    ws = [synthetic.gaussian(int(rng.integers(1, 9)), 16 * int(rng.integers(1, 20)), 0.02, 1000 + i)
          for i in range(nv.NVFP4_GROUP_MAX + 45)]
    Wd, outs = _run_group(ws, nv.FOUR_OVER_SIX)
    for W, (c, s, a) in zip(Wd, outs):
        rc, rs, ra = nv.quantize(W, nv.FOUR_OVER_SIX)
        assert torch.equal(c, rc) and torch.equal(s, rs) and a.item() == ra.item()


@pytest.mark.parametrize("mode,iters", [(nv.CJSO, 2), (nv.CJSO_DECOUPLED, 1)])
def test_grouped_cjso_modes_match_single_calls(mode, iters):
    ws = [synthetic.gaussian(8, 256, 0.02, 500), synthetic.mlp_up(501, 40, 512), np.zeros((0, 32), np.uint16)]
    Wd, outs = _run_group(ws, mode, iters)
    for w, W, (c, s, a) in zip(ws, Wd, outs):
        if w.size == 0:
            assert a.item() == 0.0
            continue
        rc, rs, ra = nv.quantize(W, mode, iters)
        assert torch.equal(c, rc) and torch.equal(s, rs) and a.item() == ra.item()


def test_grouped_one_large_tensor_beyond_l2():
    """A single 8192x28672 tensor (448 MiB, larger than L2) as a group of one."""
    w = synthetic.mlp_70b(4)
    W = to_device(w)
    (c, s, a), = nv.quantize_grouped([W], nv.FOUR_OVER_SIX)
    rc, rs, ra = nv.quantize(W, nv.FOUR_OVER_SIX)
    torch.cuda.synchronize()
    assert torch.equal(c, rc) and torch.equal(s, rs) and a.item() == ra.item()


def test_grouped_all_empty_and_zero_count():
    Wd = [torch.empty((0, 16), dtype=torch.bfloat16, device="cuda"),
          torch.empty((3, 0), dtype=torch.bfloat16, device="cuda")]
    outs = nv.quantize_grouped(Wd, nv.FOUR_OVER_SIX)
    torch.cuda.synchronize()
    assert all(a.item() == 0.0 for _, _, a in outs)
    assert nv.nvfp4_quantize_grouped(None, 0, 0, 0, torch.cuda.current_stream().cuda_stream) == 0


def test_grouped_full_llama3_stack_matches_single_calls():
    """The benchmark's launch configuration: all 224 tensors of the
    Llama-3-8B-shaped stack (13 GiB, generated on the device as the benchmark
    does) in one grouped FourOverSix call, every tensor bit-identical to its
    single-tensor call (which the other tests check against the oracle)."""
    import bench
    shapes, Ws = bench.model_tensors(torch.device("cuda"))
    outs = nv.quantize_grouped(Ws, nv.FOUR_OVER_SIX)
    for W, (c, s, a) in zip(Ws, outs):
        rc, rs, ra = nv.quantize(W, nv.FOUR_OVER_SIX)
        assert torch.equal(c, rc) and torch.equal(s, rs) and a.item() == ra.item()
        del rc, rs, ra


def _large_group():
    """112 tensors, 2.2 GiB of bf16 (beyond 16 x L2): the grouped call cuts it into
    parts that alternate between two streams."""
    g = torch.Generator(device="cuda").manual_seed(77)
    shapes = [(4096, 4096), (1024, 4096), (3000, 2064), (14336, 1024)] * 28
    return [(torch.randn(r, c, generator=g, device="cuda") * (0.01 + 0.001 * (i % 7))).to(torch.bfloat16)
            for i, (r, c) in enumerate(shapes)]


@pytest.mark.parametrize("mode", [nv.MAX, nv.FOUR_OVER_SIX])
def test_grouped_two_stream_parts_match_single_calls(mode):
    Ws = _large_group()
    assert sum(W.numel() for W in Ws) * 2 >= 16 * torch.cuda.get_device_properties(0).L2_cache_size
    outs = nv.quantize_grouped(Ws, mode)
    torch.cuda.synchronize()
    for W, (c, s, a) in zip(Ws, outs):
        rc, rs, ra = nv.quantize(W, mode)
        assert torch.equal(c, rc) and torch.equal(s, rs) and a.item() == ra.item()


def test_grouped_two_stream_parts_under_graph_capture():
    Ws = _large_group()
    outs = nv.quantize_grouped(Ws, nv.FOUR_OVER_SIX)  # first call outside any capture
    torch.cuda.synchronize()
    ref = [(c.clone(), s.clone(), a.clone()) for c, s, a in outs]
    for c, s, a in outs:
        c.fill_(0xA5)
        s.fill_(0xA5)
        a.fill_(-1.0)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):  # the fork to the library's second stream joins back inside the capture
        nv.quantize_grouped(Ws, nv.FOUR_OVER_SIX, outs=outs)
    gr.replay()
    torch.cuda.synchronize()
    for (c, s, a), (rc, rs, ra) in zip(outs, ref):
        assert torch.equal(c, rc) and torch.equal(s, rs) and torch.equal(a, ra)
