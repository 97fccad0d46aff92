"""CPU oracle for the fused reduce + residual-add + RMSNorm (+ per-group FP8) epilogue.

TEST INFRASTRUCTURE ONLY.  The only callers allowed are the test-suite, the
smoke check in ``__graft_entry__`` and the benchmark's CPU-baseline / reference
leg.  The product library never imports, links or executes anything here, and
this package imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain C, one row at a time, fp32 sum in
rank order, fp64 norm, bf16 / e4m3 rounding written from the format
definitions).  This module only compiles it with gcc and marshals numpy arrays.

Every output is pinned by the CPU tests against closed forms, brute force and
library special cases; no function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fexcess-precision=standard",
          "-fopenmp", "-shared", "-fPIC", "-Wall"]

_lib = None
_lock = threading.Lock()


def build(out_path: str | None = None, src: str | None = None) -> str:
    """Compile oracle.c (or, for the mutation tests, a deliberately broken copy of
    it given as ``src``) into a shared library and return its path."""
    out = out_path or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, "-o", out, src or _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    u16p = ctypes.c_void_p
    lib.oracle_reduce_rmsnorm.argtypes = [u16p, ctypes.c_int, u16p, u16p, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_float, u16p, u16p, ctypes.c_int]
    lib.oracle_reduce_rmsnorm.restype = ctypes.c_int
    lib.oracle_quant_per_group.argtypes = [u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_quant_per_group.restype = ctypes.c_int
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_from_double.argtypes = [ctypes.c_double]
    lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
    lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_to_double.restype = ctypes.c_double
    lib.oracle_e2m1_from_double.argtypes = [ctypes.c_double]
    lib.oracle_e2m1_from_double.restype = ctypes.c_uint8
    lib.oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0_to_double.restype = ctypes.c_double
    lib.oracle_mxfp4.argtypes = [u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_mxfp4.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if it is missing)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


class Oracle:
    """numpy front end over one compiled oracle library (the real one or a mutant)."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    @staticmethod
    def _ptr(a: np.ndarray | None):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    def reduce_rmsnorm(self, partials: np.ndarray, residual: np.ndarray | None, gamma: np.ndarray,
                       eps: float, want_y: bool = True, threads: int = 1):
        """partials uint16 [R,T,H] (bf16 bits), residual uint16 [T,H] or None, gamma uint16 [H].

        Returns (residual_out uint16 [T,H], y uint16 [T,H] or None).
        """
        partials = np.ascontiguousarray(partials, dtype=np.uint16)
        R, T, H = partials.shape
        if residual is not None:
            residual = np.ascontiguousarray(residual, dtype=np.uint16)
            assert residual.shape == (T, H)
        gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
        assert gamma.shape == (H,)
        ro = np.empty((T, H), dtype=np.uint16)
        y = np.empty((T, H), dtype=np.uint16) if want_y else None
        rc = self.lib.oracle_reduce_rmsnorm(self._ptr(partials), R, self._ptr(residual), self._ptr(gamma),
                                            T, H, float(eps), self._ptr(ro), self._ptr(y), int(threads))
        if rc != 0:
            raise ValueError("oracle_reduce_rmsnorm rejected its arguments")
        return ro, y

    def quant_per_group(self, y: np.ndarray, group_size: int = 128, threads: int = 1):
        """y uint16 [T,H] bf16 bits -> (q uint8 [T,H] e4m3fn codes, scales float32 [T,H/group])."""
        y = np.ascontiguousarray(y, dtype=np.uint16)
        T, H = y.shape
        q = np.empty((T, H), dtype=np.uint8)
        scales = np.empty((T, H // group_size), dtype=np.float32)
        rc = self.lib.oracle_quant_per_group(self._ptr(y), T, H, int(group_size), self._ptr(q),
                                             self._ptr(scales), int(threads))
        if rc != 0:
            raise ValueError("oracle_quant_per_group rejected its arguments")
        return q, scales

    def reduce_rmsnorm_quant(self, partials, residual, gamma, eps, group_size=128, threads=1):
        """Full quant epilogue: returns (residual_out, y, q, scales)."""
        ro, y = self.reduce_rmsnorm(partials, residual, gamma, eps, True, threads)
        q, s = self.quant_per_group(y, group_size, threads)
        return ro, y, q, s

    def mxfp4(self, y: np.ndarray, threads: int = 1):
        """y uint16 [T,H] bf16 bits -> (q uint8 [T,H/2] packed E2M1, scales uint8 [T,H/32] E8M0)."""
        y = np.ascontiguousarray(y, dtype=np.uint16)
        T, H = y.shape
        q = np.empty((T, H // 2), dtype=np.uint8)
        scales = np.empty((T, H // 32), dtype=np.uint8)
        rc = self.lib.oracle_mxfp4(self._ptr(y), T, H, self._ptr(q), self._ptr(scales), int(threads))
        if rc != 0:
            raise ValueError("oracle_mxfp4 rejected its arguments")
        return q, scales

    def reduce_rmsnorm_mxfp4(self, partials, residual, gamma, eps, threads=1):
        """MXFP4 epilogue: returns (residual_out, y, q, scales)."""
        ro, y = self.reduce_rmsnorm(partials, residual, gamma, eps, True, threads)
        q, s = self.mxfp4(y, threads)
        return ro, y, q, s

    def e2m1_to_double(self, c: int) -> float:
        return self.lib.oracle_e2m1_to_double(int(c) & 0xF)

    def e2m1_from_double(self, v: float) -> int:
        return int(self.lib.oracle_e2m1_from_double(float(v)))

    def e8m0_to_double(self, c: int) -> float:
        return self.lib.oracle_e8m0_to_double(int(c) & 0xFF)

    # scalar format helpers (used by the pins)
    def bf16_to_double(self, b: int) -> float:
        return self.lib.oracle_bf16_to_double(int(b) & 0xFFFF)

    def bf16_from_double(self, v: float) -> int:
        return int(self.lib.oracle_bf16_from_double(float(v)))

    def e4m3_to_double(self, c: int) -> float:
        return self.lib.oracle_e4m3_to_double(int(c) & 0xFF)

    def e4m3_from_double(self, v: float) -> int:
        return int(self.lib.oracle_e4m3_from_double(float(v)))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())
