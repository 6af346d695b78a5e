"""Builds libmgw.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit compiles in parallel to an object under ``_build/``;
the objects link into ``libmgw.so`` next to this file.  Run as
``python -m moe_grouped_gemm_wgrad_gb300.build`` or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmgw.so")
# Test build: the same objects, except the C ABI compiled with MGW_TEST_HOOKS, which lets
# the device time-limit test make a pipeline stage that never fills (MGW_TEST_DROP_LOAD=1).
# libmgw.so itself has no such switch.
LIB_TESTHOOKS = os.path.join(HERE, "libmgw_testhooks.so")
# Diagnostic build (include/mgw_diag.h): the wgrad and fp32 dgrad kernels and the C ABI
# compiled with MGW_DIAG -- a work-item timeline and device bounds checks that report
# MGW_DEV_BOUNDS.  The other objects are shared with libmgw.so.
LIB_DIAG = os.path.join(HERE, "libmgw_diag.so")
DIAG_SOURCES = ["api.cu", "wgrad.cu", "dgrad.cu", "dgrad_pair.cu"]
SOURCES = ["api.cu", "quantize.cu", "quantize_rows.cu", "wgrad.cu", "wgrad_balanced.cu", "wgrad_noalloc.cu", "grouped_mm.cu", "dgrad.cu", "dgrad_pair.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libmgw.so")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "mgw.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _compile(job: tuple[str, tuple[str, ...]]) -> tuple[str, str]:
    src, defines = job
    suffix = {(): "", ("-DMGW_TEST_HOOKS",): "_hooks", ("-DMGW_DIAG",): "_diag"}[tuple(defines)]
    stem = os.path.splitext(src)[0] + suffix
    obj = os.path.join(BUILD, stem + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + list(defines) + ["-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def _link(out: str, objs: list[str]) -> None:
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, out)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libmgw.so (and its test build) if any source is newer; returns its path."""
    newest = _deps_mtime()
    if (not force and all(os.path.exists(p) and os.path.getmtime(p) >= newest
                          for p in (LIB, LIB_TESTHOOKS, LIB_DIAG))):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    jobs = ([(src, ()) for src in SOURCES] + [("api.cu", ("-DMGW_TEST_HOOKS",))] +
            [(src, ("-DMGW_DIAG",)) for src in DIAG_SOURCES])
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(_compile, jobs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results[:len(SOURCES)]]
    _link(LIB, objs)
    hook_api = results[len(SOURCES)][0]
    _link(LIB_TESTHOOKS, [hook_api if os.path.basename(o) == "api.o" else o for o in objs])
    diag = {os.path.basename(o).replace("_diag.o", ".o"): o for o, _ in results[len(SOURCES) + 1:]}
    _link(LIB_DIAG, [diag.get(os.path.basename(o), o) for o in objs])
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
