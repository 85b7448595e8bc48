"""GB300-native NVFP4 block quantization: Python binding of libnvfp4_gb300.so.

The functions named like the C ABI (``nvfp4_quantize``, ``nvfp4_dequantize``,
``nvfp4_encode_e2m1``, ``nvfp4_encode_e4m3``, ``nvfp4_status_string``) take
raw device pointers and sizes and return the C status code, exactly as
declared in include/nvfp4.h.  ``quantize`` / ``dequantize`` / ``encode_*``
are conveniences over them that take torch tensors (torch supplies device
memory and the current stream; every step of the computation runs in the
library's CUDA kernels).  There is no fallback: if the library is missing or
fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import CHECKED_LIB_PATH, LIB_PATH, build as _build

MAX, FOUR_OVER_SIX, CJSO, CJSO_DECOUPLED = 0, 1, 2, 3
MODES = {"max": MAX, "four_over_six": FOUR_OVER_SIX, "cjso": CJSO, "cjso_decoupled": CJSO_DECOUPLED}

NVFP4_OK = 0
NVFP4_GROUP_MAX = 256

_lib = None


class nvfp4_tensor(ctypes.Structure):
    """One descriptor of nvfp4_quantize_grouped (include/nvfp4.h)."""
    _fields_ = [("W", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("alpha", ctypes.c_void_p)]


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({nvfp4_status_string(status)})")
        self.status = status


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads the CUDA library (building it first if it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = _build()
    if not os.path.exists(path):
        raise ImportError(f"NVFP4 CUDA library not found at {path}")
    L = ctypes.CDLL(path)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.nvfp4_quantize.argtypes = [vp, i64, i64, ci, ci, vp, vp, vp, vp]
    L.nvfp4_quantize.restype = ci
    L.nvfp4_dequantize.argtypes = [vp, vp, vp, i64, i64, vp, vp]
    L.nvfp4_dequantize.restype = ci
    L.nvfp4_encode_e2m1.argtypes = [vp, i64, vp, vp]
    L.nvfp4_encode_e2m1.restype = ci
    L.nvfp4_encode_e4m3.argtypes = [vp, i64, vp, vp]
    L.nvfp4_encode_e4m3.restype = ci
    L.nvfp4_quantize_grouped.argtypes = [ctypes.POINTER(nvfp4_tensor), ci, ci, ci, vp]
    L.nvfp4_quantize_grouped.restype = ci
    L.nvfp4_gemv.argtypes = [vp, vp, vp, i64, i64, vp, ci, vp, vp]
    L.nvfp4_gemv.restype = ci
    L.nvfp4_gemm.argtypes = [vp, vp, vp, i64, i64, vp, ci, vp, vp]
    L.nvfp4_gemm.restype = ci
    L.nvfp4_swizzled_scales_bytes.argtypes = [i64, i64]
    L.nvfp4_swizzled_scales_bytes.restype = i64
    L.nvfp4_swizzle_scales.argtypes = [vp, i64, i64, vp, vp]
    L.nvfp4_swizzle_scales.restype = ci
    L.nvfp4_quantize_noalloc.argtypes = [vp, i64, i64, ci, vp, vp, vp, vp]
    L.nvfp4_quantize_noalloc.restype = ci
    L.nvfp4_profiler_enable.argtypes = [ci]
    L.nvfp4_profiler_enable.restype = ci
    L.nvfp4_profiler_reset.argtypes = []
    L.nvfp4_profiler_reset.restype = ci
    L.nvfp4_profiler_kinds.argtypes = []
    L.nvfp4_profiler_kinds.restype = ci
    L.nvfp4_profiler_get.argtypes = [ci, ctypes.c_char_p, ci, ctypes.POINTER(ctypes.c_int64),
                                     ctypes.POINTER(ctypes.c_double)]
    L.nvfp4_profiler_get.restype = ci
    L.nvfp4_ffma_probe.argtypes = [ci, i64, vp, i64, ctypes.POINTER(ctypes.c_int64), vp]
    L.nvfp4_ffma_probe.restype = ci
    L.nvfp4_test_fail_allocations.argtypes = [ci]
    L.nvfp4_test_fail_allocations.restype = ci
    L.nvfp4_test_first_wait_tries.argtypes = [i64]
    L.nvfp4_test_first_wait_tries.restype = ci
    L.nvfp4_checked_build.argtypes = []
    L.nvfp4_checked_build.restype = ci
    L.nvfp4_check_take.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.nvfp4_check_take.restype = ci
    L.nvfp4_check_selftest.argtypes = [i64, i64, vp]
    L.nvfp4_check_selftest.restype = ci
    L.nvfp4_status_string.argtypes = [ci]
    L.nvfp4_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def library_path() -> str:
    return LIB_PATH


def checked_library_path(build: bool = True) -> str:
    """The bounds-checked build (-DNVFP4_CHECKED), built first if asked; load
    it with load(path) before any other call of the process."""
    return _build(checked=True) if build else CHECKED_LIB_PATH


# ---------------------------------------------------------------- C ABI mirror

def nvfp4_quantize(W, rows, cols, mode, iters, codes, scales, alpha, stream) -> int:
    return load().nvfp4_quantize(W, rows, cols, mode, iters, codes, scales, alpha, stream)


def nvfp4_quantize_noalloc(W, rows, cols, mode, codes, scales, alpha, stream) -> int:
    """Allocation-free max-rule / FourOverSix quantize (see include/nvfp4.h):
    for callers that must not let the library allocate device memory."""
    return load().nvfp4_quantize_noalloc(W, rows, cols, mode, codes, scales, alpha, stream)


def nvfp4_quantize_grouped(tensors, count, mode, iters, stream) -> int:
    """`tensors`: a ctypes array of nvfp4_tensor (or None with count 0)."""
    return load().nvfp4_quantize_grouped(tensors, count, mode, iters, stream)


def nvfp4_dequantize(codes, scales, alpha, rows, cols, out, stream) -> int:
    return load().nvfp4_dequantize(codes, scales, alpha, rows, cols, out, stream)


def nvfp4_gemv(codes, scales, alpha, rows, cols, x, batch, y, stream) -> int:
    return load().nvfp4_gemv(codes, scales, alpha, rows, cols, x, batch, y, stream)


def nvfp4_gemm(codes, scales, alpha, rows, cols, x, batch, y, stream) -> int:
    return load().nvfp4_gemm(codes, scales, alpha, rows, cols, x, batch, y, stream)


def nvfp4_swizzled_scales_bytes(rows, cols) -> int:
    return load().nvfp4_swizzled_scales_bytes(rows, cols)


def nvfp4_swizzle_scales(scales, rows, cols, out, stream) -> int:
    return load().nvfp4_swizzle_scales(scales, rows, cols, out, stream)


def nvfp4_encode_e2m1(v, n, out, stream) -> int:
    return load().nvfp4_encode_e2m1(v, n, out, stream)


def nvfp4_encode_e4m3(v, n, out, stream) -> int:
    return load().nvfp4_encode_e4m3(v, n, out, stream)


def nvfp4_ffma_probe(packed, rounds, sink, sink_floats, fmas, stream) -> int:
    """fp32 FMA throughput probe (instrumentation); `fmas` is a ctypes int64 pointer."""
    return load().nvfp4_ffma_probe(packed, rounds, sink, sink_floats, fmas, stream)


def nvfp4_test_fail_allocations(count) -> int:
    """Test hook: the next `count` scratch allocations fail (out of memory)."""
    return load().nvfp4_test_fail_allocations(int(count))


def nvfp4_test_first_wait_tries(tries) -> int:
    """Test hook: the first bounded device wait gives up after `tries` polls (< 0: normal)."""
    return load().nvfp4_test_first_wait_tries(int(tries))


def nvfp4_checked_build() -> int:
    return load().nvfp4_checked_build()


def nvfp4_check_take(site) -> int:
    """`site`: a ctypes.c_uint32 (byref'd here)."""
    return load().nvfp4_check_take(ctypes.byref(site))


def nvfp4_check_selftest(i, n, stream) -> int:
    return load().nvfp4_check_selftest(int(i), int(n), stream)


def check_take() -> int:
    """The first failed check's site recorded since the last take (0: none);
    waits for the device to be idle.  Always 0 in the normal build."""
    site = ctypes.c_uint32(0)
    st = nvfp4_check_take(site)
    if st != NVFP4_OK:
        raise Nvfp4Error(st, "nvfp4_check_take")
    return int(site.value)


def nvfp4_status_string(status: int) -> str:
    return load().nvfp4_status_string(int(status)).decode()


def nvfp4_profiler_enable(on: int) -> int:
    return load().nvfp4_profiler_enable(int(on))


def nvfp4_profiler_reset() -> int:
    return load().nvfp4_profiler_reset()


def nvfp4_profiler_kinds() -> int:
    return load().nvfp4_profiler_kinds()


def nvfp4_profiler_get(index, name, name_len, launches, total_ms) -> int:
    return load().nvfp4_profiler_get(index, name, name_len, launches, total_ms)


def profiler_report() -> dict:
    """{kernel name: (launches, total device ms)} of the traced launches."""
    n = nvfp4_profiler_kinds()
    if n < 0:
        raise Nvfp4Error(-n, "nvfp4_profiler_kinds")
    out = {}
    for i in range(n):
        buf = ctypes.create_string_buffer(64)
        cnt = ctypes.c_int64()
        ms = ctypes.c_double()
        _check(nvfp4_profiler_get(i, buf, 64, ctypes.byref(cnt), ctypes.byref(ms)), "nvfp4_profiler_get")
        out[buf.value.decode()] = (int(cnt.value), float(ms.value))
    return out


# ------------------------------------------------------------ torch helpers

def fp32_peak_tflops(seconds: float = 0.05, stream=None) -> dict:
    """Measured fp32 FMA peak of the current device (TFLOP/s): the probe
    kernel, scalar and packed, each timed with CUDA events after a warm-up
    launch; the larger of the two is the peak."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    sink = torch.empty(2048 * sms, dtype=torch.float32, device="cuda")
    res = {}
    for packed in (0, 1):
        fmas = ctypes.c_int64()
        rounds = 1 << 12
        for _ in range(12):  # grow until one launch takes about `seconds`
            _check(nvfp4_ffma_probe(packed, rounds, sink.data_ptr(), sink.numel(), ctypes.byref(fmas), s.cuda_stream),
                   "nvfp4_ffma_probe")
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            _check(nvfp4_ffma_probe(packed, rounds, sink.data_ptr(), sink.numel(), ctypes.byref(fmas), s.cuda_stream),
                   "nvfp4_ffma_probe")
            e1.record(s)
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            if ms >= seconds * 1e3 or rounds >= (1 << 30):
                break
            rounds = min(1 << 30, rounds * max(2, int(seconds * 1e3 / max(ms, 1e-3))))
        res["packed" if packed else "scalar"] = 2.0 * fmas.value / (ms / 1e3) / 1e12
    res["tflops"] = max(res["scalar"], res["packed"])
    return res


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(status: int, what: str):
    if status != NVFP4_OK:
        raise Nvfp4Error(status, what)


def quantize(W, mode=MAX, iters: int = 0, out=None, stream=None):
    """Quantizes a contiguous bf16 CUDA tensor [rows, cols] (cols % 16 == 0).

    Returns (codes uint8 [rows, cols/2], scales uint8 [rows, cols/16] holding
    E4M3 bit patterns, alpha float32 [1]), all on W's device.  `out` may pass
    preallocated (codes, scales, alpha) tensors."""
    import torch
    if isinstance(mode, str):
        mode = MODES[mode]
    if W.dtype != torch.bfloat16 or not W.is_cuda or W.dim() != 2 or not W.is_contiguous():
        raise ValueError("W must be a contiguous 2-D bf16 CUDA tensor")
    rows, cols = W.shape
    if out is None:
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=W.device)
        scales = torch.empty((rows, cols // 16), dtype=torch.uint8, device=W.device)
        alpha = torch.empty(1, dtype=torch.float32, device=W.device)
    else:
        codes, scales, alpha = out
    st = nvfp4_quantize(W.data_ptr(), rows, cols, int(mode), int(iters), codes.data_ptr(), scales.data_ptr(),
                        alpha.data_ptr(), _stream_ptr(stream))
    _check(st, "nvfp4_quantize")
    return codes, scales, alpha


def quantize_grouped(Ws, mode=MAX, iters: int = 0, outs=None, stream=None):
    """Quantizes a list of contiguous 2-D bf16 CUDA tensors with one grouped
    call; returns a list of (codes, scales, alpha) as `quantize` does."""
    import torch
    if isinstance(mode, str):
        mode = MODES[mode]
    res = []
    arr = (nvfp4_tensor * max(1, len(Ws)))()
    for i, W in enumerate(Ws):
        if W.dtype != torch.bfloat16 or not W.is_cuda or W.dim() != 2 or not W.is_contiguous():
            raise ValueError("every W must be a contiguous 2-D bf16 CUDA tensor")
        rows, cols = W.shape
        if outs is None:
            o = (torch.empty((rows, cols // 2), dtype=torch.uint8, device=W.device),
                 torch.empty((rows, cols // 16), dtype=torch.uint8, device=W.device),
                 torch.empty(1, dtype=torch.float32, device=W.device))
        else:
            o = outs[i]
        arr[i] = nvfp4_tensor(W.data_ptr(), rows, cols, o[0].data_ptr(), o[1].data_ptr(), o[2].data_ptr())
        res.append(o)
    _check(nvfp4_quantize_grouped(arr, len(Ws), int(mode), int(iters), _stream_ptr(stream)),
           "nvfp4_quantize_grouped")
    return res


def dequantize(codes, scales, alpha, rows: int, cols: int, out=None, stream=None):
    """Returns the bf16 CUDA tensor [rows, cols] that the NVFP4 tensor encodes."""
    import torch
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.bfloat16, device=codes.device)
    st = nvfp4_dequantize(codes.data_ptr(), scales.data_ptr(), alpha.data_ptr(), rows, cols, out.data_ptr(),
                          _stream_ptr(stream))
    _check(st, "nvfp4_dequantize")
    return out


def gemv(codes, scales, alpha, rows: int, cols: int, x, out=None, stream=None):
    """y [batch, rows] fp32 = dequantized weights [rows, cols] times the bf16
    activations x [batch, cols] (batch 1..8), on x's device."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.shape[1] != cols:
        raise ValueError("x must be a contiguous bf16 CUDA tensor [batch, cols]")
    batch = x.shape[0]
    y = out if out is not None else torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(nvfp4_gemv(codes.data_ptr(), scales.data_ptr(), alpha.data_ptr(), rows, cols, x.data_ptr(), batch,
                      y.data_ptr(), _stream_ptr(stream)), "nvfp4_gemv")
    return y


def gemm(codes, scales, alpha, rows: int, cols: int, x, out=None, stream=None):
    """As gemv, on the tensor cores, for x [batch, cols] with batch 1..256."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous() or x.shape[1] != cols:
        raise ValueError("x must be a contiguous bf16 CUDA tensor [batch, cols]")
    batch = x.shape[0]
    y = out if out is not None else torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    _check(nvfp4_gemm(codes.data_ptr(), scales.data_ptr(), alpha.data_ptr(), rows, cols, x.data_ptr(), batch,
                      y.data_ptr(), _stream_ptr(stream)), "nvfp4_gemm")
    return y


def swizzle_scales(scales, rows: int, cols: int, stream=None):
    """The [rows, cols/16] scales in the tensor-core tile layout (flat uint8)."""
    import torch
    out = torch.empty(nvfp4_swizzled_scales_bytes(rows, cols), dtype=torch.uint8, device=scales.device)
    _check(nvfp4_swizzle_scales(scales.data_ptr(), rows, cols, out.data_ptr(), _stream_ptr(stream)),
           "nvfp4_swizzle_scales")
    return out


def encode_e2m1(v, stream=None):
    import torch
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check(nvfp4_encode_e2m1(v.data_ptr(), v.numel(), out.data_ptr(), _stream_ptr(stream)), "nvfp4_encode_e2m1")
    return out


def encode_e4m3(v, stream=None):
    import torch
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check(nvfp4_encode_e4m3(v.data_ptr(), v.numel(), out.data_ptr(), _stream_ptr(stream)), "nvfp4_encode_e4m3")
    return out
