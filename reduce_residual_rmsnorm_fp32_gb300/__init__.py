"""Fused reduce + residual add + RMSNorm (+ per-group dynamic FP8) for GB300.

Thin Python binding of ``libfrn.so`` (C ABI in ``include/frn.h``).  This module
only marshals arguments -- tensor pointers, sizes, the stream -- and allocates
outputs with torch when the caller does not pass them; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback: if
the library is missing, the first call raises.

Entry points (same names as the C ABI):

* ``fused_reduce_rmsnorm(partials, residual, gamma, eps)`` -> ``(y, residual_out)``
  -- the pair the replaced all_reduce -> rms_norm subgraph returns
  ("ROCm AITER fused all-reduce + RMSNorm", vLLM PR 37646 summary).
* ``fused_reduce_rmsnorm_quant_per_group(..., group_size=128, emit_bf16=False)``
  -> ``((q, scales), residual_out)`` or, with ``emit_bf16``,
  ``((y, q, scales), residual_out)`` -- the output contract of the fused quant
  path ("AMD fused AllReduce-RMSNorm quant kernel", SGLang PR 24651 summary).

``partials`` is a bf16 CUDA tensor ``[R, T, H]`` or a sequence of ``R`` bf16
``[T, H]`` tensors (they need not be one allocation).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Sequence

import torch

__all__ = [
    "FrnError", "fused_reduce_rmsnorm", "fused_reduce_rmsnorm_quant_per_group", "library",
    "set_pdl", "set_kernel", "set_ctas_per_row", "set_stream_groups", "query_launch", "device_status", "set_test_hooks",
    "status_string", "version", "KERNEL_AUTO", "KERNEL_ROWS", "KERNEL_STREAM",
    "fused_reduce_rmsnorm_mxfp4", "fused_add_rmsnorm", "rmsnorm", "unfused_workspace_bytes", "unfused_reduce_rmsnorm", "unfused_reduce_rmsnorm_noalloc",
    "STATIC_WORKSPACE_BYTES",
    "FRN_OK", "FRN_ERR_INVALID_ARG", "FRN_ERR_UNSUPPORTED", "FRN_ERR_MISALIGNED", "FRN_ERR_CUDA",
    "FRN_ERR_TIMEOUT", "MAX_PARTIALS", "MAX_HIDDEN", "QUANT_GROUP",
]

FRN_OK, FRN_ERR_INVALID_ARG, FRN_ERR_UNSUPPORTED, FRN_ERR_MISALIGNED, FRN_ERR_CUDA, FRN_ERR_TIMEOUT = range(6)
KERNEL_AUTO, KERNEL_ROWS, KERNEL_STREAM = 0, 1, 2
MAX_PARTIALS = 16
MAX_HIDDEN = 16384
QUANT_GROUP = 128
STATIC_WORKSPACE_BYTES = 16 << 20

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfrn.so")
_lib = None
_lock = threading.Lock()


class FrnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"{status_string(status)}: {detail}")


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.fused_reduce_rmsnorm.argtypes = [ctypes.POINTER(vp), i32, vp, vp, vp, vp, i64, i32, f32, vp]
    lib.fused_reduce_rmsnorm.restype = i32
    lib.fused_reduce_rmsnorm_quant_per_group.argtypes = [ctypes.POINTER(vp), i32, vp, vp, vp, vp, vp, vp,
                                                         i64, i32, f32, i32, vp]
    lib.fused_reduce_rmsnorm_quant_per_group.restype = i32
    lib.frn_status_string.argtypes = [i32]
    lib.frn_status_string.restype = ctypes.c_char_p
    lib.frn_last_error_detail.argtypes = []
    lib.frn_last_error_detail.restype = ctypes.c_char_p
    lib.frn_version.argtypes = []
    lib.frn_version.restype = i32
    lib.frn_set_pdl.argtypes = [i32]
    lib.frn_set_pdl.restype = i32
    lib.frn_set_l2_prefetch.argtypes = [i32]
    lib.frn_set_l2_prefetch.restype = i32
    lib.frn_set_ctas_per_row.argtypes = [i32]
    lib.frn_set_ctas_per_row.restype = i32
    lib.frn_set_kernel.argtypes = [i32]
    lib.frn_set_kernel.restype = i32
    lib.frn_set_stream_groups.argtypes = [i32]
    lib.frn_set_stream_groups.restype = i32
    lib.frn_plan_launch.argtypes = [i64, i32, i32, i32, i32, i32, vp]
    lib.frn_plan_launch.restype = i32
    lib.frn_query_launch.argtypes = [i64, i32, i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                     ctypes.POINTER(i32), ctypes.POINTER(i64)]
    lib.frn_query_launch.restype = i32
    lib.frn_device_status.argtypes = [i32]
    lib.frn_device_status.restype = i32
    lib.frn_set_test_hooks.argtypes = [i32, i64]
    lib.frn_set_test_hooks.restype = i32
    lib.fused_reduce_rmsnorm_mxfp4.argtypes = [ctypes.POINTER(vp), i32, vp, vp, vp, vp, vp, vp, i64, i32, f32, vp]
    lib.fused_reduce_rmsnorm_mxfp4.restype = i32
    lib.frn_fused_add_rmsnorm.argtypes = [vp, vp, vp, vp, vp, i64, i32, f32, vp]
    lib.frn_fused_add_rmsnorm.restype = i32
    lib.frn_rmsnorm.argtypes = [vp, vp, vp, i64, i32, f32, vp]
    lib.frn_rmsnorm.restype = i32
    lib.frn_unfused_workspace_bytes.argtypes = [i64, i32, i32, i32, i32]
    lib.frn_unfused_workspace_bytes.restype = i64
    lib.frn_unfused_reduce_rmsnorm.argtypes = [ctypes.POINTER(vp), i32, vp, vp, vp, vp, vp, vp, i64, i32, f32, i32,
                                               i32, vp, i64, vp]
    lib.frn_unfused_reduce_rmsnorm.restype = i32
    lib.frn_unfused_reduce_rmsnorm_noalloc.argtypes = [ctypes.POINTER(vp), i32, vp, vp, vp, vp, vp, vp, i64, i32,
                                                       f32, i32, i32, vp]
    lib.frn_unfused_reduce_rmsnorm_noalloc.restype = i32
    lib.frn_floor_launch.argtypes = [i32, ctypes.POINTER(vp), i32, vp, vp, i64, i32, i64, i32, vp]
    lib.frn_floor_launch.restype = i32
    return lib


def library() -> ctypes.CDLL:
    """The loaded libfrn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"libfrn.so not found at {LIB_PATH}; build it with "
                        "`python -m reduce_residual_rmsnorm_fp32_gb300._build` (needs nvcc)")
                _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(status: int) -> str:
    return library().frn_status_string(int(status)).decode()


def version() -> int:
    return int(library().frn_version())


def _check(status: int) -> None:
    if status != FRN_OK:
        raise FrnError(status, library().frn_last_error_detail().decode())


def set_pdl(enable: bool) -> None:
    _check(library().frn_set_pdl(1 if enable else 0))


def set_l2_prefetch(mode: int) -> None:
    """Row kernel: 0 decide from the launch shape, 1 never, 2 always prefetch the row into L2."""
    _check(library().frn_set_l2_prefetch(int(mode)))


def set_ctas_per_row(n: int) -> None:
    _check(library().frn_set_ctas_per_row(int(n)))


def set_kernel(kind: int) -> None:
    """KERNEL_AUTO (default), KERNEL_ROWS or KERNEL_STREAM."""
    _check(library().frn_set_kernel(int(kind)))


def set_stream_groups(groups: int) -> None:
    """Stream kernel consumer groups: 0 = automatic, 1..4 forced."""
    _check(library().frn_set_stream_groups(int(groups)))


class _LaunchPlan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("ctas_per_row", ctypes.c_int), ("rows_per_cta", ctypes.c_int),
                ("tiles_per_cta", ctypes.c_int), ("tiles_per_warp", ctypes.c_int), ("threads", ctypes.c_int),
                ("grid", ctypes.c_int64), ("groups", ctypes.c_int), ("consumer_warps", ctypes.c_int),
                ("slots", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("staged", ctypes.c_int)]


def plan_launch(T: int, H: int, R: int, quant: int = 0, residual: bool = True, num_sms: int = 152) -> dict:
    """The launch the library plans for these sizes on a device with num_sms SMs
    (host code only: no device is touched).  See frn_plan_launch in frn.h."""
    out = _LaunchPlan()
    _check(library().frn_plan_launch(int(T), int(H), int(R), int(quant), 1 if residual else 0, int(num_sms),
                                     ctypes.byref(out)))
    return {name: getattr(out, name) for name, _ in _LaunchPlan._fields_}


def query_launch(T: int, H: int, R: int, quant: int = 0, residual: bool = True) -> tuple[int, int, int, int]:
    """(kernel, ctas_per_row, threads_per_cta, grid_ctas) a call would use on the current device.
    quant: 0 none, 1 / 2 FP8 without / with y, 3 / 4 MXFP4 without / with y; residual: whether the
    call passes one."""
    k, c, t, g = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    _check(library().frn_query_launch(int(T), int(H), int(R), int(quant), 1 if residual else 0, ctypes.byref(k),
                                      ctypes.byref(c), ctypes.byref(t), ctypes.byref(g)))
    return k.value, c.value, t.value, g.value


def device_status(clear: bool = False) -> int:
    """FRN_OK, or FRN_ERR_TIMEOUT if a bounded device-side wait ran out (synchronous read)."""
    return int(library().frn_device_status(1 if clear else 0))


def set_test_hooks(inject_stall: bool = False, wait_limit_ns: int = 0) -> None:
    _check(library().frn_set_test_hooks(1 if inject_stall else 0, int(wait_limit_ns)))


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check_tensor(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple, device: torch.device,
                  out: bool = False) -> None:
    """Inputs must be on the call's CUDA device; an output (out=True) may also be
    a pinned host tensor, which the kernel writes over the host link."""
    # the common case, without building device objects; anything else takes the
    # detailed checks below
    if (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.get_device() == device.index
            and t.shape == shape and t.is_contiguous()):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device or device.type != "cuda":
        if not (out and device.type == "cuda" and t.device.type == "cpu" and t.is_pinned()):
            raise ValueError(f"{name} must be on {device}" + (" or in pinned host memory" if out else "") +
                             f" (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if t.shape != shape:
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_tls = threading.local()


def _pointer_array(ptrs: list[int]):
    """The partial pointers as a C array of void* for the call.  One array per
    thread, reused: the library copies the pointers during the call."""
    buf = getattr(_tls, "ptrs", None)
    if buf is None:
        buf = _tls.ptrs = (ctypes.c_void_p * MAX_PARTIALS)()
    if len(ptrs) > MAX_PARTIALS:
        return (ctypes.c_void_p * len(ptrs))(*ptrs)   # the library rejects R > MAX_PARTIALS
    buf[:len(ptrs)] = ptrs
    return buf


def _partials(partials) -> tuple[list[int], int, int, int, torch.device]:
    if isinstance(partials, torch.Tensor):
        if partials.dim() != 3:
            raise ValueError("stacked partials must be [R, T, H]")
        R, T, H = partials.shape
        dev = partials.device
        _check_tensor(partials, "partials", torch.bfloat16, (R, T, H), dev)
        base, step = partials.data_ptr(), T * H * 2
        return list(range(base, base + R * step, step)) if step else [base] * R, R, T, H, dev
    parts = list(partials)
    if not parts:
        raise ValueError("partials is empty")
    T, H = parts[0].shape
    dev = parts[0].device
    for i, p in enumerate(parts):
        _check_tensor(p, f"partials[{i}]", torch.bfloat16, (T, H), dev)
    return [p.data_ptr() for p in parts], len(parts), T, H, dev


# The current stream's raw handle without building a Stream object (a few
# microseconds less per call); the public route where torch lacks it.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_SAME_DEVICE = contextlib.nullcontext()


def _stream(stream, device) -> int | None:
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(device.index)
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _on(device):
    """The call's device as the current one (a no-op when it already is)."""
    return _SAME_DEVICE if torch.cuda.current_device() == device.index else torch.cuda.device(device)


def fused_reduce_rmsnorm(partials: torch.Tensor | Sequence[torch.Tensor], residual: torch.Tensor | None,
                         gamma: torch.Tensor, eps: float = 1e-6, *, residual_out: torch.Tensor | None = None,
                         y: torch.Tensor | None = None, stream=None):
    """Returns ``(y, residual_out)``.  ``residual_out`` may be ``residual`` (in place)."""
    ptrs, R, T, H, dev = _partials(partials)
    if residual is not None:
        _check_tensor(residual, "residual", torch.bfloat16, (T, H), dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (H,), dev)
    if residual_out is None:
        residual_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    _check_tensor(residual_out, "residual_out", torch.bfloat16, (T, H), dev, out=True)
    _check_tensor(y, "y", torch.bfloat16, (T, H), dev, out=True)
    arr = _pointer_array(ptrs)
    with _on(dev):
        st = library().fused_reduce_rmsnorm(arr, R, _ptr(residual), _ptr(gamma), _ptr(residual_out), _ptr(y),
                                            T, H, float(eps), _stream(stream, dev))
    _check(st)
    return y, residual_out


def fused_reduce_rmsnorm_quant_per_group(partials, residual: torch.Tensor | None, gamma: torch.Tensor,
                                         eps: float = 1e-6, group_size: int = QUANT_GROUP,
                                         emit_bf16: bool = False, *, residual_out: torch.Tensor | None = None,
                                         y: torch.Tensor | None = None, q: torch.Tensor | None = None,
                                         scales: torch.Tensor | None = None, stream=None):
    """Returns ``((q, scales), residual_out)``, or ``((y, q, scales), residual_out)`` when
    ``emit_bf16`` (or when ``y`` is given).  ``q`` is float8_e4m3fn ``[T, H]``, ``scales``
    float32 ``[T, H // group_size]``."""
    ptrs, R, T, H, dev = _partials(partials)
    if residual is not None:
        _check_tensor(residual, "residual", torch.bfloat16, (T, H), dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (H,), dev)
    if group_size < 1 or H % group_size:
        raise ValueError(f"group_size={group_size} must divide H={H}")
    emit_bf16 = emit_bf16 or y is not None
    if residual_out is None:
        residual_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if emit_bf16 and y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if q is None:
        q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=dev)
    if scales is None:
        scales = torch.empty((T, H // group_size), dtype=torch.float32, device=dev)
    _check_tensor(residual_out, "residual_out", torch.bfloat16, (T, H), dev, out=True)
    if y is not None:
        _check_tensor(y, "y", torch.bfloat16, (T, H), dev, out=True)
    if q.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError("q must be float8_e4m3fn or uint8")
    _check_tensor(q, "q", q.dtype, (T, H), dev, out=True)
    _check_tensor(scales, "scales", torch.float32, (T, H // group_size), dev, out=True)
    arr = _pointer_array(ptrs)
    with _on(dev):
        st = library().fused_reduce_rmsnorm_quant_per_group(
            arr, R, _ptr(residual), _ptr(gamma), _ptr(residual_out), _ptr(y), _ptr(q), _ptr(scales),
            T, H, float(eps), int(group_size), _stream(stream, dev))
    _check(st)
    if emit_bf16:
        return (y, q, scales), residual_out
    return (q, scales), residual_out


def unfused_workspace_bytes(T: int, H: int, stages: int, quant: bool, emit_y: bool) -> int:
    return int(library().frn_unfused_workspace_bytes(int(T), int(H), int(stages), int(bool(quant)),
                                                     int(bool(emit_y))))


def _check_unfused_outputs(T, H, dev, quant, group_size, residual_out, y, q, scales) -> None:
    """The unfused paths' outputs: the C side sees only pointers, so every
    tensor's device, dtype, shape and layout is checked here, before anything is
    launched."""
    _check_tensor(residual_out, "residual_out", torch.bfloat16, (T, H), dev, out=True)
    if y is not None:
        _check_tensor(y, "y", torch.bfloat16, (T, H), dev, out=True)
    if quant:
        if group_size < 1 or H % group_size:
            raise ValueError(f"group_size={group_size} must divide H={H}")
        if q is None or scales is None:
            raise ValueError("quant needs both q and scales")
        if q.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError("q must be float8_e4m3fn or uint8")
        _check_tensor(q, "q", q.dtype, (T, H), dev, out=True)
        _check_tensor(scales, "scales", torch.float32, (T, H // group_size), dev, out=True)
    elif y is None:
        raise ValueError("without quant, y is the output and must be given")


def unfused_reduce_rmsnorm(partials, residual: torch.Tensor | None, gamma: torch.Tensor, eps: float = 1e-6, *,
                           stages: int = 2, quant: bool = False, emit_bf16: bool = True,
                           group_size: int = QUANT_GROUP, workspace: torch.Tensor | None = None,
                           residual_out: torch.Tensor | None = None, y: torch.Tensor | None = None,
                           q: torch.Tensor | None = None, scales: torch.Tensor | None = None, stream=None):
    """The unfused comparison paths (same bits as the fused entry points).

    Without quant returns ``(y, residual_out)``; with quant returns like
    ``fused_reduce_rmsnorm_quant_per_group``.  ``workspace`` is a CUDA uint8
    tensor of at least ``unfused_workspace_bytes(...)`` bytes (allocated here
    when not given)."""
    ptrs, R, T, H, dev = _partials(partials)
    if residual is not None:
        _check_tensor(residual, "residual", torch.bfloat16, (T, H), dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (H,), dev)
    emit_y = (not quant) or emit_bf16 or y is not None
    need = unfused_workspace_bytes(T, H, stages, quant, emit_y)
    if need < 0:
        raise ValueError(f"stages={stages} needs quant" if stages == 3 else f"stages={stages} must be 2 or 3")
    if workspace is None:
        workspace = torch.empty((max(need, 16),), dtype=torch.uint8, device=dev)
    if residual_out is None:
        residual_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if emit_y and y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if quant:
        if q is None:
            q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=dev)
        if scales is None:
            scales = torch.empty((T, H // group_size), dtype=torch.float32, device=dev)
    _check_unfused_outputs(T, H, dev, quant, group_size, residual_out, y, q, scales)
    if workspace.device != dev:
        raise ValueError(f"workspace must be on {dev} (got {workspace.device})")
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    arr = _pointer_array(ptrs)
    with _on(dev):
        st = library().frn_unfused_reduce_rmsnorm(
            arr, R, _ptr(residual), _ptr(gamma), _ptr(residual_out), _ptr(y), _ptr(q) if quant else None,
            _ptr(scales) if quant else None, T, H, float(eps), int(group_size), int(stages), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(st)
    if not quant:
        return y, residual_out
    if emit_y:
        return (y, q, scales), residual_out
    return (q, scales), residual_out


def unfused_reduce_rmsnorm_noalloc(partials, residual: torch.Tensor | None, gamma: torch.Tensor,
                                   eps: float = 1e-6, *, stages: int = 2, residual_out: torch.Tensor,
                                   y: torch.Tensor | None = None, q: torch.Tensor | None = None,
                                   scales: torch.Tensor | None = None, group_size: int = QUANT_GROUP, stream=None):
    """The unfused paths with the library's fixed static scratch instead of a
    workspace, for callers that cannot allocate device memory.  The caller passes
    every output (nothing is allocated here either); results as
    ``unfused_reduce_rmsnorm``.  The first call on a device should come before
    any stream capture, and calls that can overlap on the GPU race on the shared
    scratch."""
    ptrs, R, T, H, dev = _partials(partials)
    if residual is not None:
        _check_tensor(residual, "residual", torch.bfloat16, (T, H), dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (H,), dev)
    if (q is None) != (scales is None):
        raise ValueError("pass both q and scales (quant) or neither")
    _check_unfused_outputs(T, H, dev, q is not None, group_size, residual_out, y, q, scales)
    arr = _pointer_array(ptrs)
    with _on(dev):
        st = library().frn_unfused_reduce_rmsnorm_noalloc(
            arr, R, _ptr(residual), _ptr(gamma), _ptr(residual_out), _ptr(y), _ptr(q), _ptr(scales), T, H,
            float(eps), int(group_size), int(stages), _stream(stream, dev))
    _check(st)


FLOOR_EMPTY, FLOOR_READ, FLOOR_COPY = 0, 1, 2


def floor_launch(kind: int, sources: Sequence[torch.Tensor] = (), dst0: torch.Tensor | None = None,
                 dst1: torch.Tensor | None = None, threads: int = 128, grid: int = 1, pdl: bool = True,
                 stream=None) -> None:
    """Launch one of the measurement reference kernels (frn_floor_launch in frn.h):
    FLOOR_EMPTY (``grid`` CTAs of ``threads``), FLOOR_READ (one 16-byte load per
    thread of every source) or FLOOR_COPY (the same loads, stores into dst0 and
    dst1).  Sources and destinations are contiguous CUDA tensors of one size."""
    srcs = list(sources)
    nbytes = 0
    dev = torch.device("cuda", torch.cuda.current_device())
    if srcs:
        nbytes = srcs[0].numel() * srcs[0].element_size()
        dev = srcs[0].device
        for t in srcs + [t for t in (dst0, dst1) if t is not None]:
            if t.device != dev or not t.is_contiguous() or t.numel() * t.element_size() != nbytes:
                raise ValueError("floor_launch buffers must be contiguous, on one device, of one size")
    arr = (ctypes.c_void_p * max(1, len(srcs)))(*[t.data_ptr() for t in srcs])
    st = library().frn_floor_launch(int(kind), arr if srcs else None, len(srcs), _ptr(dst0), _ptr(dst1), nbytes,
                                    int(threads), int(grid), 1 if pdl else 0, _stream(stream, dev))
    if st != FRN_OK:
        raise FrnError(st, "frn_floor_launch")


def fused_add_rmsnorm(x: torch.Tensor, residual: torch.Tensor | None, gamma: torch.Tensor, eps: float = 1e-6, *,
                      residual_out: torch.Tensor | None = None, y: torch.Tensor | None = None, stream=None):
    """residual_out = x + residual (fp32, one rounding), y = RMSNorm(residual_out); returns (y, residual_out)."""
    T, H = x.shape
    dev = x.device
    _check_tensor(x, "x", torch.bfloat16, (T, H), dev)
    if residual is not None:
        _check_tensor(residual, "residual", torch.bfloat16, (T, H), dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (H,), dev)
    residual_out = torch.empty_like(x) if residual_out is None else residual_out
    y = torch.empty_like(x) if y is None else y
    _check_tensor(residual_out, "residual_out", torch.bfloat16, (T, H), dev, out=True)
    _check_tensor(y, "y", torch.bfloat16, (T, H), dev, out=True)
    with _on(dev):
        st = library().frn_fused_add_rmsnorm(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(residual_out), _ptr(y), T,
                                             H, float(eps), _stream(stream, dev))
    _check(st)
    return y, residual_out


def rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, *, y: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """y = RMSNorm(x) with weight gamma (bf16 in and out, fp32 arithmetic)."""
    T, H = x.shape
    dev = x.device
    _check_tensor(x, "x", torch.bfloat16, (T, H), dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (H,), dev)
    y = torch.empty_like(x) if y is None else y
    _check_tensor(y, "y", torch.bfloat16, (T, H), dev, out=True)
    with _on(dev):
        st = library().frn_rmsnorm(_ptr(x), _ptr(gamma), _ptr(y), T, H, float(eps), _stream(stream, dev))
    _check(st)
    return y


def fused_reduce_rmsnorm_mxfp4(partials, residual: torch.Tensor | None, gamma: torch.Tensor, eps: float = 1e-6,
                               emit_bf16: bool = False, *, residual_out: torch.Tensor | None = None,
                               y: torch.Tensor | None = None, q: torch.Tensor | None = None,
                               scales: torch.Tensor | None = None, stream=None):
    """Fused epilogue with MXFP4 output (OCP MX: 32-blocks, E8M0 scale, E2M1).

    Returns ``((q, scales), residual_out)`` or, with ``emit_bf16``,
    ``((y, q, scales), residual_out)``; ``q`` is uint8 ``[T, H/2]`` (element 2i in
    the low nibble), ``scales`` uint8 ``[T, H/32]`` E8M0 codes."""
    ptrs, R, T, H, dev = _partials(partials)
    if residual is not None:
        _check_tensor(residual, "residual", torch.bfloat16, (T, H), dev)
    _check_tensor(gamma, "gamma", torch.bfloat16, (H,), dev)
    if H % 32:
        raise ValueError(f"H={H} must be a multiple of 32")
    emit_bf16 = emit_bf16 or y is not None
    residual_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if residual_out is None else residual_out
    if emit_bf16 and y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    q = torch.empty((T, H // 2), dtype=torch.uint8, device=dev) if q is None else q
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device=dev) if scales is None else scales
    _check_tensor(residual_out, "residual_out", torch.bfloat16, (T, H), dev, out=True)
    if y is not None:
        _check_tensor(y, "y", torch.bfloat16, (T, H), dev, out=True)
    _check_tensor(q, "q", torch.uint8, (T, H // 2), dev, out=True)
    _check_tensor(scales, "scales", torch.uint8, (T, H // 32), dev, out=True)
    arr = _pointer_array(ptrs)
    with _on(dev):
        st = library().fused_reduce_rmsnorm_mxfp4(arr, R, _ptr(residual), _ptr(gamma), _ptr(residual_out), _ptr(y),
                                                  _ptr(q), _ptr(scales), T, H, float(eps), _stream(stream, dev))
    _check(st)
    if emit_bf16:
        return (y, q, scales), residual_out
    return (q, scales), residual_out
