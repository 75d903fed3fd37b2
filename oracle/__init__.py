"""CPU oracle for the dense GEMM ``C = A @ B.T`` (bf16 / fp16 in and out).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never loads it, and it imports nothing from the
CUDA package: the two sides share only the seeded input generators.

The arithmetic lives in ``oracle.c`` (plain C, fp64): each input is widened
exactly to double, products are summed in double in plain order
``k = 0 .. K-1``, and the sum is rounded once to the output format with
round-to-nearest-even.  This module only compiles it and marshals numpy
arrays of raw 16-bit patterns through ctypes.

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(identity, permutation, rank-1 closed forms, brute force in exact rational
arithmetic, hand-derived rounding fixtures, and an fp64 numpy cross-check).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

DTYPES = {"bf16": 0, "fp16": 1}

_lock = threading.Lock()
_default = None


def _dtype_code(dtype) -> int:
    if isinstance(dtype, str):
        if dtype not in DTYPES:
            raise ValueError(f"unknown dtype {dtype!r}")
        return DTYPES[dtype]
    code = int(dtype)
    if code not in (0, 1):
        raise ValueError(f"unknown dtype code {dtype!r}")
    return code


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (OpenMP if gcc has it)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_decode.argtypes = [ctypes.c_uint16, ctypes.c_int]
    lib.oracle_decode.restype = ctypes.c_double
    lib.oracle_round.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.oracle_round.restype = ctypes.c_uint16
    lib.oracle_decode_array.argtypes = [u16p, f64p, i64, ctypes.c_int]
    lib.oracle_decode_array.restype = None
    lib.oracle_round_array.argtypes = [f64p, u16p, i64, ctypes.c_int]
    lib.oracle_round_array.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [u16p, u16p, u16p, f64p, i64, i64, i64, i64, i64,
                                ctypes.c_int, i64p, i64, i64p, i64, ctypes.c_int]
    lib.oracle_gemm.restype = ctypes.c_int
    return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_rows(x: np.ndarray, name: str):
    x = np.asarray(x)
    if x.dtype != np.uint16 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D uint16 array of bit patterns")
    if x.shape[0] > 0 and x.shape[1] > 0 and x.strides[1] != 2:
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // 2 if x.shape[0] > 1 else max(x.shape[1], 1)
    return x, ld


class Oracle:
    """ctypes view of one compiled copy of ``oracle.c``.

    The default instance (module-level functions) uses ``_build/liboracle.so``;
    the pin tests also load deliberately broken copies to show that the pins
    catch a planted mistake.
    """

    def __init__(self, lib_path: str):
        self.lib = _bind(ctypes.CDLL(lib_path))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def decode(self, bits, dtype) -> np.ndarray:
        """Exact values (float64) of an array of 16-bit patterns."""
        b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_decode_array(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double),
                                     b.size, _dtype_code(dtype))
        return out

    def round_to(self, x, dtype) -> np.ndarray:
        """Round float64 values to bf16 / fp16 (nearest, ties to even): bit patterns."""
        a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_round_array(_ptr(a, ctypes.c_double), _ptr(out, ctypes.c_uint16),
                                    a.size, _dtype_code(dtype))
        return out

    def gemm(self, A_bits, B_bits, dtype, rows=None, cols=None, with_acc: bool = False,
             threads: int = 0):
        """Reference ``round(A @ B.T)`` for the chosen rows x cols block of C.

        ``A_bits`` (M x K) and ``B_bits`` (N x K) are uint16 arrays of bf16/fp16
        bit patterns.  ``rows`` / ``cols`` select C's rows / columns (default
        all).  Returns the uint16 block, and with ``with_acc`` also the
        unrounded float64 sums.
        """
        A, lda = _as_rows(A_bits, "A")
        B, ldb = _as_rows(B_bits, "B")
        M, K = A.shape
        N, Kb = B.shape
        if Kb != K:
            raise ValueError(f"K mismatch: A has {K}, B has {Kb}")
        code = _dtype_code(dtype)
        r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        c = None if cols is None else np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        nr = M if r is None else r.size
        nc = N if c is None else c.size
        out = np.empty((nr, nc), dtype=np.uint16)
        acc = np.empty((nr, nc), dtype=np.float64) if with_acc else None
        i64p = ctypes.POINTER(ctypes.c_int64)
        # empty arrays still need a valid pointer for ctypes
        a_keep = A if A.size else np.zeros(1, np.uint16)
        b_keep = B if B.size else np.zeros(1, np.uint16)
        rc = self.lib.oracle_gemm(
            _ptr(a_keep, ctypes.c_uint16), _ptr(b_keep, ctypes.c_uint16),
            _ptr(out, ctypes.c_uint16) if out.size else None,
            _ptr(acc, ctypes.c_double) if (acc is not None and acc.size) else None,
            M, N, K, max(lda, K), max(ldb, K), code,
            _ptr(r, ctypes.c_int64) if r is not None else ctypes.cast(None, i64p), nr,
            _ptr(c, ctypes.c_int64) if c is not None else ctypes.cast(None, i64p), nc,
            int(threads))
        if rc != 0:
            raise ValueError("oracle_gemm rejected its arguments")
        return (out, acc) if with_acc else out


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def max_threads() -> int:
    return default().max_threads()


def decode(bits, dtype) -> np.ndarray:
    return default().decode(bits, dtype)


def round_to(x, dtype) -> np.ndarray:
    return default().round_to(x, dtype)


def gemm(A_bits, B_bits, dtype, rows=None, cols=None, with_acc: bool = False, threads: int = 0):
    return default().gemm(A_bits, B_bits, dtype, rows=rows, cols=cols, with_acc=with_acc,
                          threads=threads)
