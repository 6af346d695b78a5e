"""Thin ctypes binding of libmgw.so (C ABI in include/mgw.h).

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.  If the
library is missing or fails to load, every call raises :class:`MgwError`;
there is no fallback implementation.

The C ABI sees only pointers, so the binding checks what the tensors know and the
library cannot: dtype, contiguity, one device for all operands, and that every
caller-supplied buffer holds at least the elements the call reads or writes.  A
failed check raises :class:`MgwError` before anything is launched.  Each call runs
with the operands' device current.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmgw.so")
# The diagnostic build (include/mgw_diag.h): same results, plus a work-item timeline and
# device bounds checks.  Only diagnostic_library() switches the binding to it.
LIB_DIAG_PATH = os.path.join(HERE, "libmgw_diag.so")

MGW_OK = 0
MGW_DEV_BAD_OFFSETS = 1
MGW_DEV_TIMEOUT = 2
MGW_DEV_BAD_INDEX = 4
MGW_DEV_BOUNDS = 8   # diagnostic library only
DIAG_KERNELS = {1: "grouped_wgrad_pair_kernel", 2: "grouped_dgrad_kernel", 3: "grouped_dgrad_pair_kernel"}
MAX_EXPERTS = 1024
SCALE_FLOOR = 0      # OCP MX rule 2^(floor(log2 amax) - 8)
SCALE_CEIL_448 = 1   # the post-attn page's RoundUp rule ceil_pow2(amax / 448)

EXPORTS = (
    "mgw_status_string", "mgw_version", "mgw_mxfp8_token_capacity", "mgw_mxfp8_scale_bytes",
    "mgw_mxfp8_quantize", "mgw_mxfp8_quantize_gather", "mgw_grouped_wgrad_mxfp8",
    "mgw_grouped_dgrad_f32", "mgw_mxfp8_quantize_rows", "mgw_grouped_fprop_mxfp8",
    "mgw_grouped_dgrad_mxfp8", "mgw_grouped_wgrad_mxfp8_balanced",
    "mgw_grouped_wgrad_workspace_bytes", "mgw_grouped_wgrad_mxfp8_balanced_noalloc",
)


DIAG_EXPORTS = ("mgw_diag_timeline", "mgw_diag_timeline_reset")


class MgwError(RuntimeError):
    pass


class DiagRecord(ctypes.Structure):
    """mgw_diag_record of include/mgw_diag.h."""
    _fields_ = [("kernel", ctypes.c_uint32), ("sm", ctypes.c_uint32), ("cta", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32), ("item", ctypes.c_int64),
                ("t_wait_ns", ctypes.c_uint64), ("t_done_ns", ctypes.c_uint64)]


_lock = threading.Lock()
_lib = None


def bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declares the C ABI's argument and return types on a loaded build of the library."""
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.mgw_status_string.argtypes = [I]
    lib.mgw_status_string.restype = ctypes.c_char_p
    lib.mgw_version.argtypes = []
    lib.mgw_version.restype = I
    lib.mgw_mxfp8_token_capacity.argtypes = [I, I]
    lib.mgw_mxfp8_token_capacity.restype = SZ
    lib.mgw_mxfp8_scale_bytes.argtypes = [I, SZ]
    lib.mgw_mxfp8_scale_bytes.restype = SZ
    lib.mgw_mxfp8_quantize.argtypes = [P, I, I, P, I, P, P, SZ, I, P, P]
    lib.mgw_mxfp8_quantize.restype = I
    lib.mgw_mxfp8_quantize_gather.argtypes = [P, I, P, I, I, P, I, P, P, SZ, I, P, P]
    lib.mgw_mxfp8_quantize_gather.restype = I
    lib.mgw_grouped_wgrad_mxfp8.argtypes = [P, P, P, P, P, I, I, I, I, SZ, P, P, P]
    lib.mgw_grouped_wgrad_mxfp8.restype = I
    lib.mgw_grouped_dgrad_f32.argtypes = [P, P, P, I, I, I, I, P, P, P]
    lib.mgw_grouped_dgrad_f32.restype = I
    lib.mgw_mxfp8_quantize_rows.argtypes = [P, I, P, I, I, P, I, P, P, SZ, I, P, P]
    lib.mgw_mxfp8_quantize_rows.restype = I
    lib.mgw_grouped_fprop_mxfp8.argtypes = [P, P, P, P, P, I, I, I, I, SZ, SZ, P, P, P]
    lib.mgw_grouped_fprop_mxfp8.restype = I
    lib.mgw_grouped_dgrad_mxfp8.argtypes = [P, P, P, P, P, I, I, I, I, SZ, SZ, P, P, P]
    lib.mgw_grouped_dgrad_mxfp8.restype = I
    lib.mgw_grouped_wgrad_mxfp8_balanced.argtypes = [P, P, P, P, P, I, I, I, I, SZ, P, P, SZ, P, P]
    lib.mgw_grouped_wgrad_mxfp8_balanced.restype = I
    lib.mgw_grouped_wgrad_workspace_bytes.argtypes = [I, I, I]
    lib.mgw_grouped_wgrad_workspace_bytes.restype = SZ
    lib.mgw_grouped_wgrad_mxfp8_balanced_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, SZ, P, P, P]
    lib.mgw_grouped_wgrad_mxfp8_balanced_noalloc.restype = I
    return lib


def bind_diag(lib: ctypes.CDLL) -> ctypes.CDLL:
    """bind() plus the two entry points only the diagnostic library exports."""
    bind(lib)
    lib.mgw_diag_timeline.argtypes = [ctypes.POINTER(DiagRecord), ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_int)]
    lib.mgw_diag_timeline.restype = ctypes.c_int
    lib.mgw_diag_timeline_reset.argtypes = []
    lib.mgw_diag_timeline_reset.restype = ctypes.c_int
    return lib


_diag_lib = None


@contextlib.contextmanager
def diagnostic_library():
    """Runs the calls made inside the block through libmgw_diag.so (built beside libmgw.so):
    the same results, a work-item timeline (diag_timeline) and device bounds checks that set
    MGW_DEV_BOUNDS in a call's status word.  Not thread-safe against concurrent calls made
    outside the block."""
    global _lib, _diag_lib
    with _lock:
        if _diag_lib is None:
            if not os.path.exists(LIB_DIAG_PATH):
                raise MgwError(f"{LIB_DIAG_PATH} is not built; run `python -m moe_grouped_gemm_wgrad_gb300.build`")
            _diag_lib = bind_diag(ctypes.CDLL(LIB_DIAG_PATH))
        prev, _lib = _lib, _diag_lib
    try:
        yield _diag_lib
    finally:
        with _lock:
            _lib = prev


def diag_timeline(cap: int = 3 * 65536) -> list[dict]:
    """The work-item timeline recorded by the diagnostic library since the last
    diag_timeline_reset(), one dict per (CTA, item); synchronises with the device."""
    if _diag_lib is None:
        raise MgwError("diag_timeline needs diagnostic_library() to have been entered")
    buf = (DiagRecord * cap)()
    total = ctypes.c_int(0)
    _check(_diag_lib.mgw_diag_timeline(buf, cap, ctypes.byref(total)), "mgw_diag_timeline")
    out = []
    for r in buf[:min(cap, total.value)]:
        out.append({"kernel": DIAG_KERNELS.get(r.kernel, str(r.kernel)), "sm": r.sm, "cta": r.cta,
                    "item": r.item, "t_wait_ns": r.t_wait_ns, "t_done_ns": r.t_done_ns})
    return out


def diag_timeline_reset() -> None:
    if _diag_lib is None:
        raise MgwError("diag_timeline_reset needs diagnostic_library() to have been entered")
    _check(_diag_lib.mgw_diag_timeline_reset(), "mgw_diag_timeline_reset")


def load() -> ctypes.CDLL:
    """Load libmgw.so (built in-tree by ``moe_grouped_gemm_wgrad_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise MgwError(f"{LIB_PATH} is not built; run `python -m moe_grouped_gemm_wgrad_gb300.build`")
        _lib = bind(ctypes.CDLL(LIB_PATH))
        return _lib


def _check(st: int, what: str) -> None:
    if st != MGW_OK:
        msg = load().mgw_status_string(st).decode()
        raise MgwError(f"{what}: {msg} (status {st})")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _on_cuda(t: torch.Tensor) -> bool:
    return t.is_cuda


def _dev_tensor(t: torch.Tensor, dtype, name: str, ndim: int | None = None) -> None:
    if not isinstance(t, torch.Tensor) or not _on_cuda(t):
        raise MgwError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MgwError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MgwError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise MgwError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")


def _need(t: torch.Tensor, n: int, name: str) -> None:
    """``t`` holds at least the ``n`` elements the call touches."""
    if t.numel() < n:
        raise MgwError(f"{name} holds {t.numel()} elements; the call needs {n}")


def _offsets(expert_off: torch.Tensor, E: int | None = None) -> int:
    """Checks expert_off (int32, E+1 >= 2 entries) and returns E."""
    _dev_tensor(expert_off, torch.int32, "expert_off", 1)
    n = expert_off.numel()
    if n < 2:
        raise MgwError("expert_off needs E+1 >= 2 entries")
    if E is not None and n != E + 1:
        raise MgwError(f"expert_off has {n} entries; {E} experts need {E + 1}")
    return n - 1


def _status(status: torch.Tensor | None) -> None:
    if status is not None:
        _dev_tensor(status, torch.int32, "status")
        _need(status, 1, "status")


def _one_device(*ts) -> torch.device:
    devs = {t.device for t in ts if t is not None}
    if len(devs) != 1:
        raise MgwError(f"all tensors must be on one CUDA device, got {sorted(str(d) for d in devs)}")
    return next(iter(devs))


def _out(t: torch.Tensor | None, shape, dtype, dev, name: str) -> torch.Tensor:
    """The caller's output buffer after checks, or a new one of ``shape``."""
    n = 1
    for d in shape:
        n *= int(d)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=dev)
    _dev_tensor(t, dtype, name)
    _need(t, n, name)
    return t


def _device(dev: torch.device):
    """Makes ``dev`` the current CUDA device for the call (the library launches on, and
    sizes its grids for, the current device)."""
    return torch.cuda.device(dev)


def token_capacity(M: int, E: int) -> int:
    """Padded token axis length that fits any split of M tokens over E experts."""
    return int(load().mgw_mxfp8_token_capacity(int(M), int(E)))


def scale_bytes(C: int, Mcap: int) -> int:
    return int(load().mgw_mxfp8_scale_bytes(int(C), int(Mcap)))


def mxfp8_quantize(src: torch.Tensor, expert_off: torch.Tensor, Mcap: int | None = None,
                   q: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                   status: torch.Tensor | None = None, stream=None, scale_rule: int = SCALE_FLOOR):
    """MXFP8-quantize bf16 ``src`` [M, C] along tokens -> (q uint8 [C, Mcap], scales uint8)."""
    _dev_tensor(src, torch.bfloat16, "src", 2)
    E = _offsets(expert_off)
    _status(status)
    M, C = src.shape
    Mcap = token_capacity(M, E) if Mcap is None else int(Mcap)
    dev = _one_device(src, expert_off, q, scales, status)
    q = _out(q, (C, Mcap), torch.uint8, dev, "q")
    scales = _out(scales, (scale_bytes(C, Mcap),), torch.uint8, dev, "scales")
    with _device(dev):
        st = load().mgw_mxfp8_quantize(_ptr(src), M, C, _ptr(expert_off), E, _ptr(q), _ptr(scales),
                                       Mcap, int(scale_rule), _ptr(status), _stream(stream))
    _check(st, "mgw_mxfp8_quantize")
    return q, scales


def mxfp8_quantize_gather(src: torch.Tensor, row_index: torch.Tensor, expert_off: torch.Tensor,
                          Mcap: int | None = None, q: torch.Tensor | None = None,
                          scales: torch.Tensor | None = None, status: torch.Tensor | None = None,
                          stream=None, scale_rule: int = SCALE_FLOOR):
    """MXFP8-quantize the routed rows src[row_index] (src bf16 [rows, C], row_index int32 [M])
    without materialising them -> (q uint8 [C, Mcap], scales uint8)."""
    _dev_tensor(src, torch.bfloat16, "src", 2)
    _dev_tensor(row_index, torch.int32, "row_index", 1)
    E = _offsets(expert_off)
    _status(status)
    src_rows, C = src.shape
    M = row_index.numel()
    Mcap = token_capacity(M, E) if Mcap is None else int(Mcap)
    dev = _one_device(src, row_index, expert_off, q, scales, status)
    q = _out(q, (C, Mcap), torch.uint8, dev, "q")
    scales = _out(scales, (scale_bytes(C, Mcap),), torch.uint8, dev, "scales")
    with _device(dev):
        st = load().mgw_mxfp8_quantize_gather(_ptr(src), src_rows, _ptr(row_index), M, C,
                                              _ptr(expert_off), E, _ptr(q), _ptr(scales), Mcap,
                                              int(scale_rule), _ptr(status), _stream(stream))
    _check(st, "mgw_mxfp8_quantize_gather")
    return q, scales


def _wgrad_operands(gq, gs, xq, xs, expert_off, status, *others):
    """Checks the quantized wgrad operands; returns (E, N, K, Mcap, device)."""
    for t, n in ((gq, "gq"), (xq, "xq")):
        _dev_tensor(t, torch.uint8, n, 2)
    for t, n in ((gs, "gs"), (xs, "xs")):
        _dev_tensor(t, torch.uint8, n)
    E = _offsets(expert_off)
    _status(status)
    N, Mcap = gq.shape
    K, Mcap_x = xq.shape
    if Mcap_x != Mcap:
        raise MgwError(f"gq [N, {Mcap}] and xq [K, {Mcap_x}] must share one padded token axis")
    _need(gs, scale_bytes(N, Mcap), "gs")
    _need(xs, scale_bytes(K, Mcap), "xs")
    dev = _one_device(gq, gs, xq, xs, expert_off, status, *others)
    return E, N, K, Mcap, dev


def grouped_wgrad_mxfp8(gq: torch.Tensor, gs: torch.Tensor, xq: torch.Tensor, xs: torch.Tensor,
                        expert_off: torch.Tensor, M: int, out: torch.Tensor | None = None,
                        status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """grad_w [E*N, K] bf16 from quantized g^T (N rows) and x^T (K rows)."""
    E, N, K, Mcap, dev = _wgrad_operands(gq, gs, xq, xs, expert_off, status, out)
    out = _out(out, (E * N, K), torch.bfloat16, dev, "out")
    with _device(dev):
        st = load().mgw_grouped_wgrad_mxfp8(_ptr(gq), _ptr(gs), _ptr(xq), _ptr(xs),
                                            _ptr(expert_off), E, int(M), N, K, Mcap, _ptr(out),
                                            _ptr(status), _stream(stream))
    _check(st, "mgw_grouped_wgrad_mxfp8")
    return out


def wgrad_workspace(E: int, N: int, K: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for :func:`grouped_wgrad_mxfp8_balanced` on ``device``."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        nbytes = int(load().mgw_grouped_wgrad_workspace_bytes(int(E), int(N), int(K)))
    if nbytes == 0:
        raise MgwError("mgw_grouped_wgrad_workspace_bytes: no usable device")
    return torch.zeros(nbytes, dtype=torch.uint8, device=dev)


def grouped_wgrad_mxfp8_balanced(gq: torch.Tensor, gs: torch.Tensor, xq: torch.Tensor,
                                 xs: torch.Tensor, expert_off: torch.Tensor, M: int,
                                 workspace: torch.Tensor, out: torch.Tensor | None = None,
                                 status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """grad_w [E*N, K] bf16, as :func:`grouped_wgrad_mxfp8`, with split-K and dynamic
    scheduling for skewed routings.  ``workspace``: uint8, zero-filled before first use
    (see :func:`wgrad_workspace`); calls sharing it must not overlap."""
    _dev_tensor(workspace, torch.uint8, "workspace")
    E, N, K, Mcap, dev = _wgrad_operands(gq, gs, xq, xs, expert_off, status, out, workspace)
    out = _out(out, (E * N, K), torch.bfloat16, dev, "out")
    with _device(dev):
        st = load().mgw_grouped_wgrad_mxfp8_balanced(
            _ptr(gq), _ptr(gs), _ptr(xq), _ptr(xs), _ptr(expert_off), E, int(M), N, K, Mcap,
            _ptr(out), _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _check(st, "mgw_grouped_wgrad_mxfp8_balanced")
    return out


def grouped_wgrad_mxfp8_balanced_noalloc(gq: torch.Tensor, gs: torch.Tensor, xq: torch.Tensor,
                                         xs: torch.Tensor, expert_off: torch.Tensor, M: int,
                                         out: torch.Tensor | None = None,
                                         status: torch.Tensor | None = None,
                                         stream=None) -> torch.Tensor:
    """As :func:`grouped_wgrad_mxfp8_balanced` on the library's own workspace (a device array
    in the library; nothing is allocated, calls must not overlap)."""
    E, N, K, Mcap, dev = _wgrad_operands(gq, gs, xq, xs, expert_off, status, out)
    out = _out(out, (E * N, K), torch.bfloat16, dev, "out")
    with _device(dev):
        st = load().mgw_grouped_wgrad_mxfp8_balanced_noalloc(
            _ptr(gq), _ptr(gs), _ptr(xq), _ptr(xs), _ptr(expert_off), E, int(M), N, K, Mcap,
            _ptr(out), _ptr(status), _stream(stream))
    _check(st, "mgw_grouped_wgrad_mxfp8_balanced_noalloc")
    return out


def grouped_dgrad_f32(dy: torch.Tensor, W: torch.Tensor, expert_off: torch.Tensor,
                      out: torch.Tensor | None = None, status: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """dx [rows, in_f] fp32 = dy[r] . W[e(r)] per row's expert."""
    _dev_tensor(dy, torch.float32, "dy", 2)
    _dev_tensor(W, torch.float32, "W", 3)
    rows, out_f = dy.shape
    E, out_w, in_f = W.shape
    if out_w != out_f:
        raise MgwError(f"W [E, {out_w}, in_f] does not match dy [rows, {out_f}]")
    _offsets(expert_off, E)
    _status(status)
    dev = _one_device(dy, W, expert_off, out, status)
    out = _out(out, (rows, in_f), torch.float32, dev, "out")
    with _device(dev):
        st = load().mgw_grouped_dgrad_f32(_ptr(dy), _ptr(W), _ptr(expert_off), E, rows, out_f,
                                          in_f, _ptr(out), _ptr(status), _stream(stream))
    _check(st, "mgw_grouped_dgrad_f32")
    return out


def mxfp8_quantize_rows(src: torch.Tensor, expert_off: torch.Tensor, Mcap: int | None = None,
                        q: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                        status: torch.Tensor | None = None, stream=None,
                        scale_rule: int = SCALE_FLOOR, row_index: torch.Tensor | None = None):
    """Row-wise MXFP8 quantization (one scale per 32 columns of a row) of the routed rows:
    ``src[row_index]`` when ``row_index`` (int32 [M]) is given, else ``src`` [M, C].
    -> (q uint8 [Mcap, C] on the padded row axis, scale atoms uint8)."""
    _dev_tensor(src, torch.bfloat16, "src", 2)
    E = _offsets(expert_off)
    _status(status)
    src_rows, C = src.shape
    if row_index is not None:
        _dev_tensor(row_index, torch.int32, "row_index", 1)
        M = row_index.numel()
    else:
        M = src_rows
    Mcap = token_capacity(M, E) if Mcap is None else int(Mcap)
    dev = _one_device(src, expert_off, row_index, q, scales, status)
    q = _out(q, (Mcap, C), torch.uint8, dev, "q")
    scales = _out(scales, (scale_bytes(C, Mcap),), torch.uint8, dev, "scales")
    with _device(dev):
        st = load().mgw_mxfp8_quantize_rows(_ptr(src), src_rows, _ptr(row_index), M, C,
                                            _ptr(expert_off), E, _ptr(q), _ptr(scales), Mcap,
                                            int(scale_rule), _ptr(status), _stream(stream))
    _check(st, "mgw_mxfp8_quantize_rows")
    return q, scales


def grouped_fprop_mxfp8(xq: torch.Tensor, xs: torch.Tensor, wq: torch.Tensor, ws: torch.Tensor,
                        expert_off: torch.Tensor, M: int, N: int, out: torch.Tensor | None = None,
                        status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y [M, N] bf16 = x[r] . W[e(r)]^T from row-wise quantized x [Mcap, K] and W [Mw, K]
    (W [E, N, K] quantized with offsets {0, N, ..., E*N})."""
    for t, n in ((xq, "xq"), (wq, "wq")):
        _dev_tensor(t, torch.uint8, n, 2)
    for t, n in ((xs, "xs"), (ws, "ws")):
        _dev_tensor(t, torch.uint8, n)
    E = _offsets(expert_off)
    _status(status)
    Mcap, K = xq.shape
    Mw, K_w = wq.shape
    if K_w != K:
        raise MgwError(f"wq [Mw, {K_w}] and xq [Mcap, {K}] must share the contraction width")
    _need(xs, scale_bytes(K, Mcap), "xs")
    _need(ws, scale_bytes(K, Mw), "ws")
    dev = _one_device(xq, xs, wq, ws, expert_off, out, status)
    out = _out(out, (int(M), int(N)), torch.bfloat16, dev, "out")
    with _device(dev):
        st = load().mgw_grouped_fprop_mxfp8(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws),
                                            _ptr(expert_off), E, int(M), int(N), K, Mcap, Mw,
                                            _ptr(out), _ptr(status), _stream(stream))
    _check(st, "mgw_grouped_fprop_mxfp8")
    return out


def grouped_dgrad_mxfp8(dyq: torch.Tensor, dys: torch.Tensor, wtq: torch.Tensor,
                        wts: torch.Tensor, expert_off: torch.Tensor, M: int,
                        out: torch.Tensor | None = None, status: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """dx [M, K] bf16 = dy[r] . W[e(r)] from row-wise quantized dy [Mcap, N] and W quantized
    along n per expert by :func:`mxfp8_quantize` (wtq [K, Mw])."""
    for t, n in ((dyq, "dyq"), (wtq, "wtq")):
        _dev_tensor(t, torch.uint8, n, 2)
    for t, n in ((dys, "dys"), (wts, "wts")):
        _dev_tensor(t, torch.uint8, n)
    E = _offsets(expert_off)
    _status(status)
    Mcap, N = dyq.shape
    K, Mw = wtq.shape
    _need(dys, scale_bytes(N, Mcap), "dys")
    _need(wts, scale_bytes(K, Mw), "wts")
    dev = _one_device(dyq, dys, wtq, wts, expert_off, out, status)
    out = _out(out, (int(M), K), torch.bfloat16, dev, "out")
    with _device(dev):
        st = load().mgw_grouped_dgrad_mxfp8(_ptr(dyq), _ptr(dys), _ptr(wtq), _ptr(wts),
                                            _ptr(expert_off), E, int(M), N, K, Mcap, Mw,
                                            _ptr(out), _ptr(status), _stream(stream))
    _check(st, "mgw_grouped_dgrad_mxfp8")
    return out
