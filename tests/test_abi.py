"""The C ABI on the host: the library loads without a GPU, exports every
function include/nvfp4.h declares, and rejects bad arguments with the
documented status before touching the device."""
import ctypes
import os
import re

import pytest

import nvfp4_block_scale_gb300 as nv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")

OK, INVALID, MISALIGNED = 0, 1, 2
A16 = 0x10000  # fake, suitably aligned device addresses: never dereferenced on these paths


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function():
    lib = nv.load()
    names = declared_functions()
    assert "nvfp4_quantize" in names and "nvfp4_dequantize" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    assert nv.nvfp4_status_string(0) == "ok"
    for s in range(1, 6):
        assert nv.nvfp4_status_string(s) not in ("ok", "unknown status")
    assert nv.nvfp4_status_string(99) == "unknown status"


@pytest.mark.parametrize("rows,cols,mode,iters,expect", [
    (4, 17, 0, 0, INVALID),      # cols % 16 != 0
    (-1, 16, 0, 0, INVALID),     # negative rows
    (4, -16, 0, 0, INVALID),
    (4, 16, 4, 0, INVALID),      # unknown mode
    (4, 16, -1, 0, INVALID),
    (4, 16, 2, -1, INVALID),     # CJSO iterations out of range
    (4, 16, 3, 65, INVALID),
    (1 << 25, 1 << 16, 0, 0, INVALID),  # 2^41 elements: too large
])
def test_quantize_rejects_bad_arguments(rows, cols, mode, iters, expect):
    assert nv.nvfp4_quantize(A16, rows, cols, mode, iters, A16, A16, A16, None) == expect


def test_quantize_rejects_null_and_misaligned():
    assert nv.nvfp4_quantize(None, 4, 16, 0, 0, A16, A16, A16, None) == INVALID
    assert nv.nvfp4_quantize(A16, 4, 16, 0, 0, None, A16, A16, None) == INVALID
    assert nv.nvfp4_quantize(A16, 4, 16, 0, 0, A16, None, A16, None) == INVALID
    assert nv.nvfp4_quantize(A16, 4, 16, 0, 0, A16, A16, None, None) == INVALID
    assert nv.nvfp4_quantize(A16 + 8, 4, 16, 0, 0, A16, A16, A16, None) == MISALIGNED
    assert nv.nvfp4_quantize(A16, 4, 16, 0, 0, A16 + 2, A16, A16, None) == MISALIGNED
    assert nv.nvfp4_quantize(A16, 4, 16, 0, 0, A16, A16, A16 + 1, None) == MISALIGNED


def test_dequantize_and_encode_reject_bad_arguments():
    assert nv.nvfp4_dequantize(A16, A16, A16, 4, 24, A16, None) == INVALID
    assert nv.nvfp4_dequantize(None, A16, A16, 4, 16, A16, None) == INVALID
    assert nv.nvfp4_dequantize(A16, A16, None, 4, 16, A16, None) == INVALID
    assert nv.nvfp4_dequantize(A16, A16, A16, 4, 16, A16 + 4, None) == MISALIGNED
    assert nv.nvfp4_dequantize(A16 + 1, A16, A16, 4, 16, A16, None) == MISALIGNED
    assert nv.nvfp4_encode_e2m1(None, 5, A16, None) == INVALID
    assert nv.nvfp4_encode_e4m3(A16, -1, A16, None) == INVALID
    assert nv.nvfp4_encode_e4m3(A16 + 1, 3, A16, None) == MISALIGNED


def test_binding_names_mirror_the_header():
    for n in declared_functions():
        assert callable(getattr(nv, n)), n


def _descs(*specs):
    arr = (nv.nvfp4_tensor * max(1, len(specs)))()
    for i, (w, rows, cols, c, s, a) in enumerate(specs):
        arr[i] = nv.nvfp4_tensor(w, rows, cols, c, s, a)
    return arr


def test_grouped_rejects_bad_descriptors_before_anything():
    good = (A16, 4, 16, A16, A16, A16)
    assert nv.nvfp4_quantize_grouped(None, 3, 0, 0, None) == INVALID         # null list
    assert nv.nvfp4_quantize_grouped(_descs(good), -1, 0, 0, None) == INVALID  # negative count
    assert nv.nvfp4_quantize_grouped(_descs(good), 1, 5, 0, None) == INVALID   # unknown mode
    assert nv.nvfp4_quantize_grouped(_descs(good), 1, 2, 65, None) == INVALID  # CJSO iterations
    # the bad descriptor sits after a good one: nothing may have been enqueued for the first
    assert nv.nvfp4_quantize_grouped(_descs(good, (A16, 4, 17, A16, A16, A16)), 2, 1, 0, None) == INVALID
    assert nv.nvfp4_quantize_grouped(_descs(good, (A16, 4, 16, A16, A16, None)), 2, 0, 0, None) == INVALID
    assert nv.nvfp4_quantize_grouped(_descs(good, (None, 4, 16, A16, A16, A16)), 2, 0, 0, None) == INVALID
    assert nv.nvfp4_quantize_grouped(_descs(good, (A16 + 8, 4, 16, A16, A16, A16)), 2, 0, 0, None) == MISALIGNED
    assert nv.nvfp4_quantize_grouped(_descs(good, (A16, 4, 16, A16 + 1, A16, A16)), 2, 1, 0, None) == MISALIGNED
    assert nv.nvfp4_quantize_grouped(_descs(good, (A16, 4, 16, A16, A16, A16 + 2)), 2, 0, 0, None) == MISALIGNED


def test_grouped_descriptor_layout_matches_header():
    text = open(HEADER).read()
    body = re.search(r"typedef struct nvfp4_tensor \{(.*?)\} nvfp4_tensor;", text, re.S).group(1)
    names = re.findall(r"\b(\w+);", body)
    assert names == [f[0] for f in nv.nvfp4_tensor._fields_]
    assert ctypes.sizeof(nv.nvfp4_tensor) == 48
    m = re.search(r"#define NVFP4_GROUP_MAX (\d+)", text)
    assert int(m.group(1)) == nv.NVFP4_GROUP_MAX


@pytest.mark.parametrize("rows,cols,batch,expect", [
    (4, 17, 1, INVALID), (-1, 16, 1, INVALID), (4, 16, 0, INVALID), (4, 16, 9, INVALID)])
def test_gemv_rejects_bad_arguments(rows, cols, batch, expect):
    assert nv.nvfp4_gemv(A16, A16, A16, rows, cols, A16, batch, A16, None) == expect


def test_gemv_rejects_null_and_misaligned():
    assert nv.nvfp4_gemv(None, A16, A16, 4, 16, A16, 1, A16, None) == INVALID
    assert nv.nvfp4_gemv(A16, A16, None, 4, 16, A16, 1, A16, None) == INVALID
    assert nv.nvfp4_gemv(A16, A16, A16, 4, 16, None, 1, A16, None) == INVALID
    assert nv.nvfp4_gemv(A16 + 4, A16, A16, 4, 16, A16, 1, A16, None) == MISALIGNED  # codes: 8 bytes
    assert nv.nvfp4_gemv(A16, A16, A16, 4, 16, A16 + 8, 1, A16, None) == MISALIGNED  # x: 16 bytes
    assert nv.nvfp4_gemv(A16, A16, A16, 4, 16, A16, 1, A16 + 2, None) == MISALIGNED


def test_swizzled_size_and_checks():
    assert nv.nvfp4_swizzled_scales_bytes(300, 160) == 384 * 12
    assert nv.nvfp4_swizzled_scales_bytes(128, 64) == 512
    assert nv.nvfp4_swizzled_scales_bytes(4, 17) == -1
    assert nv.nvfp4_swizzle_scales(A16, 4, 17, A16, None) == INVALID
    assert nv.nvfp4_swizzle_scales(None, 4, 16, A16, None) == INVALID
    assert nv.nvfp4_swizzle_scales(A16, 4, 16, A16 + 2, None) == MISALIGNED


def test_profiler_api_without_launches():
    assert nv.nvfp4_profiler_reset() == OK
    assert nv.nvfp4_profiler_enable(1) == OK
    assert nv.nvfp4_profiler_enable(0) == OK
    assert nv.nvfp4_profiler_kinds() == 0
    name = ctypes.create_string_buffer(64)
    launches, total = ctypes.c_int64(), ctypes.c_double()
    assert nv.nvfp4_profiler_get(0, name, 64, ctypes.byref(launches), ctypes.byref(total)) == INVALID
    assert nv.profiler_report() == {}


def test_gemm_rejects_bad_arguments():
    assert nv.nvfp4_gemm(A16, A16, A16, 4, 17, A16, 1, A16, None) == INVALID
    assert nv.nvfp4_gemm(A16, A16, A16, 4, 16, A16, 0, A16, None) == INVALID
    assert nv.nvfp4_gemm(A16, A16, A16, 4, 16, A16, 257, A16, None) == INVALID
    assert nv.nvfp4_gemm(A16 + 4, A16, A16, 4, 16, A16, 1, A16, None) == MISALIGNED
    assert nv.nvfp4_gemm(A16, A16, A16, 4, 16, A16 + 8, 1, A16, None) == MISALIGNED


def test_checked_build_exports_the_same_functions():
    """The bounds-checked variant exports every declared function and says
    which build it is (no device needed); take rejects a null pointer."""
    lib = ctypes.CDLL(nv.checked_library_path(build=True))
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert lib.nvfp4_checked_build() == 1
    assert nv.load().nvfp4_checked_build() == 0
    lib.nvfp4_check_take.argtypes = [ctypes.c_void_p]
    assert lib.nvfp4_check_take(None) == INVALID
