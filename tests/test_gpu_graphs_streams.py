"""The library under CUDA-graph capture and on concurrent streams: every entry
point captured into one graph (after a first, uncaptured call per device)
and replayed on fresh inputs gives what eager calls give; calls on four
streams at once give what the same calls give one after another."""
import pytest
import torch

import nvfp4_block_scale_gb300 as nv
import synthetic
from gpu_util import to_device

pytestmark = pytest.mark.gpu


def _pipeline(W, X, outs):
    """quantize (every rule) -> dequantize, gemv, gemm, scale layout; grouped quantize."""
    res = []
    for mode, iters in ((nv.MAX, 0), (nv.FOUR_OVER_SIX, 0), (nv.CJSO, 2), (nv.CJSO_DECOUPLED, 1)):
        c, s, a = nv.quantize(W, mode, iters, out=outs[mode])
        res += [c, s, a]
    c, s, a = outs[nv.FOUR_OVER_SIX]
    rows, cols = W.shape
    res.append(nv.dequantize(c, s, a, rows, cols, out=outs["deq"]))
    res.append(nv.gemv(c, s, a, rows, cols, X[:4], out=outs["gemv"]))
    res.append(nv.gemm(c, s, a, rows, cols, X, out=outs["gemm"]))
    res.append(outs["swz"].copy_(nv.swizzle_scales(s, rows, cols)))
    for (gc, gs, ga) in nv.quantize_grouped([W, W[: rows // 2]], nv.MAX, outs=outs["grp"]):
        res += [gc, gs, ga]
    # CJSO groups alternate tensors between the caller's stream and the library's second one
    for (gc, gs, ga) in nv.quantize_grouped([W, W[: rows // 2], W[rows // 2:]], nv.CJSO_DECOUPLED, 1,
                                            outs=outs["grp3"]):
        res += [gc, gs, ga]
    return res


def _outs(rows, cols, batch):
    d = "cuda"
    q = lambda r: (torch.empty((r, cols // 2), dtype=torch.uint8, device=d),
                   torch.empty((r, cols // 16), dtype=torch.uint8, device=d),
                   torch.empty(1, dtype=torch.float32, device=d))
    o = {m: q(rows) for m in (nv.MAX, nv.FOUR_OVER_SIX, nv.CJSO, nv.CJSO_DECOUPLED)}
    o["deq"] = torch.empty((rows, cols), dtype=torch.bfloat16, device=d)
    o["gemv"] = torch.empty((4, rows), dtype=torch.float32, device=d)
    o["gemm"] = torch.empty((batch, rows), dtype=torch.float32, device=d)
    o["swz"] = torch.empty(nv.nvfp4_swizzled_scales_bytes(rows, cols), dtype=torch.uint8, device=d)
    o["grp"] = [q(rows), q(rows // 2)]
    o["grp3"] = [q(rows), q(rows // 2), q(rows - rows // 2)]
    return o


def test_every_entry_point_under_graph_capture():
    rows, cols, batch = 256, 2064, 24
    W = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    X = torch.empty((batch, cols), dtype=torch.bfloat16, device="cuda")
    outs = _outs(rows, cols, batch)
    W.copy_(to_device(synthetic.mlp_up(700, rows, cols)))
    X.copy_(to_device(synthetic.gaussian(batch, cols, 1.0, 701)))
    _pipeline(W, X, outs)  # the first calls: one-time set-up outside any capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        captured = _pipeline(W, X, outs)
    for seed in (702, 703):  # replay on fresh inputs, compare with eager calls on the same inputs
        w = to_device(synthetic.student_t(rows, cols, 4.0, 0.02, seed))
        x = to_device(synthetic.gaussian(batch, cols, 1.0, seed + 10))
        W.copy_(w)
        X.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in captured]
        ref = _pipeline(w, x, _outs(rows, cols, batch))
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(got, ref)):
            assert torch.equal(a, b), i


def test_concurrent_streams_match_sequential_calls():
    tensors = [to_device(synthetic.studentt_4k(800 + i, 1024, 4096)) for i in range(4)]
    seq = [nv.quantize(W, nv.FOUR_OVER_SIX) for W in tensors]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in tensors]
    conc = []
    for W, s in zip(tensors, streams):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            conc.append(nv.quantize(W, nv.FOUR_OVER_SIX, stream=s))
    torch.cuda.synchronize()
    for (a, b, c), (d, e, f) in zip(seq, conc):
        assert torch.equal(a, d) and torch.equal(b, e) and torch.equal(c, f)


def test_grouped_calls_captured_in_one_thread_while_another_thread_calls():
    """One thread captures grouped calls into a CUDA graph (the CJSO tensor
    alternation and the two-stream FourOverSix parts both use a second stream)
    and, before it ends the capture, another thread makes the same kinds of
    grouped calls uncaptured.  Both must succeed: the uncaptured calls must
    not land on a second stream that still belongs to the open capture.  The
    graph's replay and the other thread's results equal eager calls."""
    import threading

    small = [to_device(synthetic.mlp_up(900 + i, 256, 1024)) for i in range(3)]
    small_o = [to_device(synthetic.mlp_up(910 + i, 256, 1024)) for i in range(3)]
    big = [to_device(synthetic.studentt_4k(920 + i, 8192, 12288)) for i in range(3)]  # 576 MiB: two parts
    big_o = [to_device(synthetic.studentt_4k(930 + i, 8192, 12288)) for i in range(3)]
    runs = [(small, nv.CJSO, 2), (big, nv.FOUR_OVER_SIX, 0)]
    runs_o = [(small_o, nv.CJSO, 2), (big_o, nv.FOUR_OVER_SIX, 0)]
    ref = [nv.quantize_grouped(ws, m, it) for ws, m, it in runs]  # eager; also the one-time set-up
    ref_o = [nv.quantize_grouped(ws, m, it) for ws, m, it in runs_o]
    torch.cuda.synchronize()
    outs = [[tuple(torch.empty_like(t) for t in o) for o in r] for r in ref]
    outs_o = [[tuple(torch.empty_like(t) for t in o) for o in r] for r in ref_o]
    captured, done, errors = threading.Event(), threading.Event(), []

    def other_thread():
        try:
            assert captured.wait(120)
            s = torch.cuda.Stream()
            for (ws, m, it), o in zip(runs_o, outs_o):
                nv.quantize_grouped(ws, m, it, outs=o, stream=s)
            s.synchronize()
        except Exception as e:  # reported below
            errors.append(e)
        finally:
            done.set()

    th = threading.Thread(target=other_thread)
    th.start()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=torch.cuda.Stream(), capture_error_mode="thread_local"):
            for (ws, m, it), o in zip(runs, outs):
                nv.quantize_grouped(ws, m, it, outs=o)
            captured.set()
            assert done.wait(300)
    finally:
        captured.set()
        th.join()
    assert not errors, errors
    g.replay()
    torch.cuda.synchronize()
    for got, exp in ((outs, ref), (outs_o, ref_o)):
        for r_got, r_exp in zip(got, exp):
            for a, b in zip(r_got, r_exp):
                for x, y in zip(a, b):
                    assert torch.equal(x, y)
