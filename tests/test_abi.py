"""The C ABI on the host: the library and the header agree, helpers compute the
documented sizes, and argument errors return codes before any device work."""
import ctypes
import os
import re

import pytest

from moe_grouped_gemm_wgrad_gb300 import build, mgw

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return mgw.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "mgw.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mgw_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    declared = _declared_functions()
    assert set(declared) == set(mgw.EXPORTS), declared
    for name in declared:
        assert hasattr(lib, name), name


def test_host_helpers(lib):
    assert lib.mgw_version() >= 100
    assert lib.mgw_mxfp8_token_capacity(256, 2) == 512
    assert lib.mgw_mxfp8_token_capacity(8192, 8) == 9216
    assert lib.mgw_mxfp8_token_capacity(65536, 64) == 73728
    assert lib.mgw_mxfp8_token_capacity(-1, 2) == 0
    assert lib.mgw_mxfp8_scale_bytes(256, 512) == 256 * 512 // 32
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.mgw_status_string(code)


def test_argument_errors_before_device_work(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: validation fails first
    # null pointers
    assert lib.mgw_mxfp8_quantize(fake, 4, 128, None, 1, fake, fake, 256, 0, None, None) == -1
    # C not a multiple of 128
    assert lib.mgw_mxfp8_quantize(fake, 4, 96, fake, 1, fake, fake, 256, 0, None, None) == -2
    # Mcap too small / not a multiple of 128
    assert lib.mgw_mxfp8_quantize(fake, 300, 128, fake, 2, fake, fake, 384, 0, None, None) == -3
    assert lib.mgw_mxfp8_quantize(fake, 4, 128, fake, 1, fake, fake, 200, 0, None, None) == -3
    # unknown scale rule
    assert lib.mgw_mxfp8_quantize(fake, 4, 128, fake, 1, fake, fake, 256, 7, None, None) == -1
    # E out of range
    assert lib.mgw_mxfp8_quantize(fake, 4, 128, fake, 0, fake, fake, 256, 0, None, None) == -1
    assert lib.mgw_mxfp8_quantize(fake, 4, 128, fake, 1025, fake, fake, 1 << 20, 0, None, None) == -1
    # gather: missing row index / source, bad scale rule, C not a multiple of 128
    assert lib.mgw_mxfp8_quantize_gather(fake, 10, None, 4, 128, fake, 1, fake, fake, 256, 0, None, None) == -1
    assert lib.mgw_mxfp8_quantize_gather(fake, 0, fake, 4, 128, fake, 1, fake, fake, 256, 0, None, None) == -1
    assert lib.mgw_mxfp8_quantize_gather(fake, 10, fake, 4, 128, fake, 1, fake, fake, 256, 3, None, None) == -1
    assert lib.mgw_mxfp8_quantize_gather(fake, 10, fake, 4, 64, fake, 1, fake, fake, 256, 0, None, None) == -2
    # wgrad: K not a multiple of 256, N not a multiple of 128
    assert lib.mgw_grouped_wgrad_mxfp8(fake, fake, fake, fake, fake, 1, 4, 128, 128, 256, fake, None, None) == -2
    assert lib.mgw_grouped_wgrad_mxfp8(fake, fake, fake, fake, fake, 1, 4, 64, 256, 256, fake, None, None) == -2
    assert lib.mgw_grouped_wgrad_mxfp8(None, fake, fake, fake, fake, 1, 4, 128, 256, 256, fake, None, None) == -1
    # misaligned pointer
    assert lib.mgw_grouped_wgrad_mxfp8(P(0x1001), fake, fake, fake, fake, 1, 4, 128, 256, 256, fake, None, None) == -1
    # dgrad: in_f not a multiple of 256, out_f not a multiple of 32
    assert lib.mgw_grouped_dgrad_f32(fake, fake, fake, 1, 4, 32, 128, fake, None, None) == -2
    assert lib.mgw_grouped_dgrad_f32(fake, fake, fake, 1, 4, 48, 256, fake, None, None) == -2
    assert lib.mgw_grouped_dgrad_f32(fake, None, fake, 1, 4, 32, 256, fake, None, None) == -1
    # stacked weight rows E * out_f must stay below 2^31
    assert lib.mgw_grouped_dgrad_f32(fake, fake, fake, 1024, 4, 1 << 21, 256, fake, None, None) == -2


def test_argument_errors_forward_and_mx_dgrad(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # row-wise quantize: null offsets, C not a multiple of 128, small Mcap, bad rule,
    # row index without a source row count, misaligned output
    assert lib.mgw_mxfp8_quantize_rows(fake, 4, None, 4, 128, None, 1, fake, fake, 256, 0, None, None) == -1
    assert lib.mgw_mxfp8_quantize_rows(fake, 4, None, 4, 96, fake, 1, fake, fake, 256, 0, None, None) == -2
    assert lib.mgw_mxfp8_quantize_rows(fake, 300, None, 300, 128, fake, 2, fake, fake, 384, 0, None, None) == -3
    assert lib.mgw_mxfp8_quantize_rows(fake, 4, None, 4, 128, fake, 1, fake, fake, 256, 2, None, None) == -1
    assert lib.mgw_mxfp8_quantize_rows(fake, 0, fake, 4, 128, fake, 1, fake, fake, 256, 0, None, None) == -1
    assert lib.mgw_mxfp8_quantize_rows(fake, 4, None, 4, 128, fake, 1, P(0x1008), fake, 256, 0, None, None) == -1
    # forward: N not a multiple of 256, K not a multiple of 128, Mw too small, Mcap too small
    assert lib.mgw_grouped_fprop_mxfp8(fake, fake, fake, fake, fake, 1, 4, 128, 128, 256, 256, fake, None, None) == -2
    assert lib.mgw_grouped_fprop_mxfp8(fake, fake, fake, fake, fake, 1, 4, 256, 64, 256, 256, fake, None, None) == -2
    assert lib.mgw_grouped_fprop_mxfp8(fake, fake, fake, fake, fake, 2, 4, 256, 128, 384, 384, fake, None, None) == -3
    assert lib.mgw_grouped_fprop_mxfp8(fake, fake, fake, fake, fake, 2, 300, 256, 128, 384, 512, fake, None, None) == -3
    assert lib.mgw_grouped_fprop_mxfp8(fake, fake, None, fake, fake, 1, 4, 256, 128, 256, 256, fake, None, None) == -1
    # MXFP8 data gradient: N not a multiple of 128, K not a multiple of 256, misaligned
    assert lib.mgw_grouped_dgrad_mxfp8(fake, fake, fake, fake, fake, 1, 4, 64, 256, 256, 256, fake, None, None) == -2
    assert lib.mgw_grouped_dgrad_mxfp8(fake, fake, fake, fake, fake, 1, 4, 128, 128, 256, 256, fake, None, None) == -2
    assert lib.mgw_grouped_dgrad_mxfp8(fake, fake, P(0x1004), fake, fake, 1, 4, 128, 256, 256, 256, fake, None, None) == -1
    # Mw below E*N, or not a multiple of 128
    assert lib.mgw_grouped_dgrad_mxfp8(fake, fake, fake, fake, fake, 2, 4, 128, 256, 384, 128, fake, None, None) == -3
    assert lib.mgw_grouped_fprop_mxfp8(fake, fake, fake, fake, fake, 1, 4, 256, 128, 256, 320, fake, None, None) == -3
    # no rows: the output may be null only then
    assert lib.mgw_grouped_fprop_mxfp8(fake, fake, fake, fake, fake, 1, 4, 256, 128, 256, 256, None, None, None) == -1


def test_wgrad_32bit_size_limits(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    # E*N above 2^31 output rows
    assert lib.mgw_grouped_wgrad_mxfp8(fake, fake, fake, fake, fake, 1024, 4, (1 << 21) + 128, 256,
                                       1 << 17, fake, None, None) == -2
    # E*N = 2^31 is allowed, but 1024 x 16384 x 128 = 2^31 output tiles is not
    assert lib.mgw_grouped_wgrad_mxfp8(fake, fake, fake, fake, fake, 1024, 4, 1 << 21, 1 << 15,
                                       1 << 17, fake, None, None) == -2


def test_argument_errors_balanced_wgrad(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    ws = P(0x10000)  # 256-byte aligned
    args = [fake, fake, fake, fake, fake, 1, 4, 128, 256, 256, fake]
    # missing or misaligned workspace
    assert lib.mgw_grouped_wgrad_mxfp8_balanced(*args, None, 1 << 20, None, None) == -1
    assert lib.mgw_grouped_wgrad_mxfp8_balanced(*args, P(0x10010), 1 << 20, None, None) == -1
    # workspace smaller than its 256-byte header
    assert lib.mgw_grouped_wgrad_mxfp8_balanced(*args, ws, 255, None, None) == -3
    # more experts than the balanced kernel's tables hold
    big = [fake, fake, fake, fake, fake, 513, 4, 128, 256, 1 << 17, fake]
    assert lib.mgw_grouped_wgrad_mxfp8_balanced(*big, ws, 1 << 20, None, None) == -2
    # the static kernel's checks apply too
    bad_k = [fake, fake, fake, fake, fake, 1, 4, 128, 128, 256, fake]
    assert lib.mgw_grouped_wgrad_mxfp8_balanced(*bad_k, ws, 1 << 20, None, None) == -2


def test_argument_errors_noalloc_wgrad(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)
    assert lib.mgw_grouped_wgrad_mxfp8_balanced_noalloc(
        None, fake, fake, fake, fake, 1, 4, 128, 256, 256, fake, None, None) == -1
    assert lib.mgw_grouped_wgrad_mxfp8_balanced_noalloc(
        fake, fake, fake, fake, fake, 513, 4, 128, 256, 1 << 17, fake, None, None) == -2


def test_workspace_size_helper(lib):
    import torch

    n = lib.mgw_grouped_wgrad_workspace_bytes(8, 256, 256)
    if torch.cuda.is_available():
        # header + tile counters (padded to 256 bytes) + 2 x SM count partial tiles of 128 KB
        slots = 2 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        assert n == 256 + (4 * slots + 255) // 256 * 256 + slots * 128 * 256 * 4
    else:
        assert n == 0


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_is_self_contained_c_and_cxx(lang, std):
    """include/mgw.h compiles on its own as strict C99 and as C++17, and every entry point's
    address can be taken with the declared type (the header is the whole contract)."""
    import shutil
    import subprocess

    compiler = "gcc" if lang == "c" else "g++"
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not available")
    uses = "\n".join(f"  (void)&{name};" for name in _declared_functions())
    src = f'#include "mgw.h"\nint main(void) {{\n{uses}\n  return MGW_OK;\n}}\n'
    out = subprocess.run([compiler, "-x", lang, f"-std={std}", "-Wall", "-Wextra", "-Werror",
                          "-pedantic", "-fsyntax-only", "-I", os.path.join(ROOT, "include"), "-"],
                         input=src, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr


def _diag_declared_functions():
    text = open(os.path.join(ROOT, "include", "mgw_diag.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mgw_[a-z0-9_]+)\s*\(", text)))


def test_diagnostic_library_exports_and_the_product_does_not(lib):
    """libmgw_diag.so exports every function of mgw.h and mgw_diag.h; libmgw.so exports
    none of mgw_diag.h's (the diagnostics are not in the product library)."""
    diag = _diag_declared_functions()
    assert set(diag) == set(mgw.DIAG_EXPORTS), diag
    dlib = ctypes.CDLL(build.LIB_DIAG)
    for name in _declared_functions() + diag:
        assert hasattr(dlib, name), name
    for name in diag:
        assert not hasattr(lib, name), name


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_diag_header_is_self_contained(lang, std):
    import shutil
    import subprocess

    compiler = "gcc" if lang == "c" else "g++"
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not available")
    uses = "\n".join(f"  (void)&{name};" for name in _diag_declared_functions())
    src = (f'#include "mgw_diag.h"\nint main(void) {{\n{uses}\n'
           f'  mgw_diag_record r; (void)r;\n  return MGW_DEV_BOUNDS == 8 ? MGW_OK : 1;\n}}\n')
    out = subprocess.run([compiler, "-x", lang, f"-std={std}", "-Wall", "-Wextra", "-Werror",
                          "-pedantic", "-fsyntax-only", "-I", os.path.join(ROOT, "include"), "-"],
                         input=src, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr


def test_diag_record_layout_matches_header():
    assert ctypes.sizeof(mgw.DiagRecord) == 40
    assert mgw.DiagRecord.item.offset == 16 and mgw.DiagRecord.t_done_ns.offset == 32
