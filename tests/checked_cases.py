"""Runs a fixed set of calls through one build of the library and prints, as
one JSON line, a digest of every output and the sites of failed checks the
build recorded.  `python tests/checked_cases.py normal|checked`: the
bounds-checked build (-DNVFP4_CHECKED) must give the normal build's outputs
bit for bit and record no failed check.  Inputs are seeded on the device, so
both runs see the same tensors; the cases reach every instrumented kernel:
ragged and tiny shapes, the bulk-copy max|W| pass (W larger than half of L2),
the decoupled search's deferred list and its overflow, the grouped kernels on
one part and on the two-stream parts, and dequantize."""
import hashlib
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import nvfp4_block_scale_gb300 as nv  # noqa: E402

SHAPES = [(1, 16), (3, 48), (37, 160), (64, 1024), (257, 4112), (4096, 8704)]
MODES = [(nv.MAX, 0), (nv.FOUR_OVER_SIX, 0), (nv.CJSO, 3), (nv.CJSO_DECOUPLED, 2)]


def digest(*ts) -> str:
    h = hashlib.sha256()
    for t in ts:
        h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())
    return h.hexdigest()[:32]


def weights(rows: int, cols: int, seed: int) -> torch.Tensor:
    """N(0, 0.02) with 0.05 % of the entries raised to +-U(0.3, 1)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, device="cuda") * 0.02
    n = rows * cols
    k = max(1, n // 2000)
    step = n // k  # one spike in each of k equal ranges: distinct positions, so the writes do not race
    idx = torch.arange(k, device="cuda") * step + torch.randint(0, step, (k,), generator=g, device="cuda")
    v = (torch.rand(k, generator=g, device="cuda") * 0.7 + 0.3) * torch.sign(torch.randn(k, generator=g, device="cuda"))
    x.view(-1)[idx] = v
    return x.to(torch.bfloat16)


def representable(rows: int, cols: int, seed: int) -> torch.Tensor:
    """Blocks of E2M1 values times an E4M3 scale times 2^-12: the decoupled
    search's crossings fall on integer k, so nearly every block is deferred,
    more than the list holds."""
    rng = np.random.default_rng(seed)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    nb = rows * cols // 16
    e4 = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    d = rng.integers(0x30, 0x70, nb)
    mags = rng.integers(0, 8, (nb, 16))
    mags[:, 5] = 7
    w = grid[mags] * np.where(rng.integers(0, 2, (nb, 16)) == 1, -1.0, 1.0) * e4[d][:, None] * 2.0 ** -12
    return torch.from_numpy(w.reshape(rows, cols).astype(np.float32)).cuda().to(torch.bfloat16)


def main(which: str) -> None:
    nv.load(nv.checked_library_path(build=False) if which == "checked" else nv.library_path())
    out = {"checked_build": nv.nvfp4_checked_build(), "digests": {}, "sites": {}}
    dg, sites = out["digests"], out["sites"]
    sites["start"] = nv.check_take()
    Ws = [weights(r, c, 100 + i) for i, (r, c) in enumerate(SHAPES)]
    for (r, c), W in zip(SHAPES, Ws):
        for mode, iters in MODES:
            codes, scales, alpha = nv.quantize(W, mode, iters)
            dg[f"q{mode}_{r}x{c}"] = digest(codes, scales, alpha)
            if mode == nv.FOUR_OVER_SIX:
                dg[f"dq_{r}x{c}"] = digest(nv.dequantize(codes, scales, alpha, r, c))
    sites["single"] = nv.check_take()
    Wr = representable(2048, 4096, 44)
    dg["deferred_overflow"] = digest(*nv.quantize(Wr, nv.CJSO_DECOUPLED, 0))
    sites["deferred"] = nv.check_take()
    for mode in (nv.MAX, nv.FOUR_OVER_SIX):
        res = nv.quantize_grouped(Ws, mode)
        dg[f"group{mode}"] = digest(*[t for o in res for t in o])
    big = [weights(4096, 14336, 200 + i) for i in range(5)]  # 587 MB of bf16: the two-stream parts
    res = nv.quantize_grouped(big, nv.FOUR_OVER_SIX)
    dg["group_parts"] = digest(*[t for o in res for t in o])
    sites["grouped"] = nv.check_take()
    dg["inputs"] = digest(*Ws, Wr, *big)
    # the mechanism itself: an index outside [0, n) is recorded (checked build only)
    nv.nvfp4_check_selftest(5, 4, None)
    sites["selftest_outside"] = nv.check_take()
    nv.nvfp4_check_selftest(3, 4, None)
    sites["selftest_inside"] = nv.check_take()
    torch.cuda.synchronize()
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main(sys.argv[1])
