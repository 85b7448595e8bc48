"""The C ABI from plain C: tests/c_abi_client.c (CUDA runtime only, no
PyTorch) is compiled with gcc against include/nvfp4.h, linked with the
library, run, and its results (alpha bits and hashes of codes, scales and the
dequantized tensor, per scale rule) must equal those of the same calls made
through the Python binding on the same tensor."""
import os
import subprocess

import numpy as np
import pytest
import torch

import nvfp4_block_scale_gb300 as nv

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _fnv1a(b: bytes) -> int:
    h = 1469598103934665603
    for x in np.frombuffer(b, np.uint8):
        h ^= int(x)
        h = (h * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h


def _weights(rows, cols):
    i = np.arange(rows * cols, dtype=np.uint64)
    with np.errstate(over="ignore"):
        x = i * np.uint64(0x9E3779B97F4A7C15) + np.uint64(12345)
        x ^= x >> np.uint64(33)
        x *= np.uint64(0xFF51AFD7ED558CCD)
        x ^= x >> np.uint64(33)
    sign = ((x >> np.uint64(8)) & np.uint64(0x8000)).astype(np.uint16)
    exp = (np.uint64(113) + x % np.uint64(11)).astype(np.uint16)
    man = ((x >> np.uint64(20)) & np.uint64(0x7F)).astype(np.uint16)
    return (sign | (exp << 7) | man).reshape(rows, cols)


def test_plain_c_client_matches_the_binding(tmp_path):
    lib = nv.load()._name
    exe = os.path.join(str(tmp_path), "c_abi_client")
    cmd = ["gcc", "-std=c11", "-O2", "-o", exe, os.path.join(HERE, "c_abi_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           lib, "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.dirname(lib)}",
           f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    subprocess.run(cmd, check=True)
    rows, cols = 96, 1040
    r = subprocess.run([exe, str(rows), str(cols)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.strip().splitlines()
    assert lines[-1] == nv.nvfp4_status_string(2)
    W = torch.from_numpy(_weights(rows, cols).view(np.int16)).view(torch.bfloat16).cuda()
    for line in lines[:-1]:
        mode, abits, hc, hs, hd = line.split()
        mode = int(mode)
        c, s, a = nv.quantize(W, mode, 3 if mode >= 2 else 0)
        d = nv.dequantize(c, s, a, rows, cols)
        torch.cuda.synchronize()
        assert int(abits, 16) == int(a.cpu().numpy().view(np.uint32)[0])
        assert int(hc, 16) == _fnv1a(c.cpu().numpy().tobytes())
        assert int(hs, 16) == _fnv1a(s.cpu().numpy().tobytes())
        assert int(hd, 16) == _fnv1a(d.view(torch.int16).cpu().numpy().tobytes())
