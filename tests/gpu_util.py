"""Helpers for the GPU parity tests: move seeded bf16 inputs to the device and
run the library through its C ABI (via the thin binding)."""
import numpy as np
import torch

import nvfp4_block_scale_gb300 as nv


def to_device(w_bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(w_bits).view(np.int16)).view(torch.bfloat16).cuda()


def gpu_quantize(w_bits: np.ndarray, mode: int, iters: int = 0):
    W = to_device(w_bits)
    codes, scales, alpha = nv.quantize(W, mode, iters)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), float(alpha.item())


def gpu_dequantize(codes: np.ndarray, scales: np.ndarray, alpha: float, rows: int, cols: int) -> np.ndarray:
    c = torch.from_numpy(np.ascontiguousarray(codes)).cuda()
    s = torch.from_numpy(np.ascontiguousarray(scales)).cuda()
    a = torch.tensor([alpha], dtype=torch.float32).cuda()
    out = nv.dequantize(c, s, a, rows, cols)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def block_mismatch(codes_a, scales_a, codes_b, scales_b) -> np.ndarray:
    """Per-block flag: codes or scale differ."""
    ca = np.asarray(codes_a).reshape(-1, 8)
    cb = np.asarray(codes_b).reshape(-1, 8)
    return np.any(ca != cb, axis=1) | (np.asarray(scales_a).reshape(-1) != np.asarray(scales_b).reshape(-1))
