"""CPU oracle for the GEMV library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library
(``memory_bound_gemv_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``gemv_oracle.c`` (plain C, double precision, one row
at a time in ascending column order); this module compiles it with gcc on
first use and wraps it for numpy arrays.  Each function states the passage of
the pages it follows in the C file's header:

* GEMV definition and row-major layout -- "Making GEMV Fast", sections
  "Row-major indexing refresher" and "Algorithm"; "llama.cpp GEMV CUDA",
  kernel-equation paragraph.
* dequantised weight q * s with one FP16 scale per row per 128 columns and
  int4 stored two per byte -- "membound", section "The kernel decode actually
  runs: dequant GEMV" (group width and nibble order are fixed by the
  workload definition, the page leaves the order open).
* FLOP and byte counts -- "Making GEMV Fast", sections "Memory Access" and
  "Computation".
* row softmax -- "membound", section "Bonus kernel: online softmax" (the
  oracle is the plain definition; the page's online update reaches the same
  value up to rounding).
* symmetric INT8 / INT4 weight quantisation and its squared error --
  "membound", section "The kernel decode actually runs: dequant GEMV" (scale
  max|w|/127 per row or per 128 columns, max|w|/7 per 128 columns for INT4;
  FP32 arithmetic, FP16 scales rounded to nearest even).

Every function is pinned by ``tests/test_oracle.py`` against values fixed by
the pages or by mathematics (worked example, identity, unit vectors, all-ones
sums, exact rational brute force, library FP16 decoding); no function is
"parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

KIND = {"f32": 0, "f16": 1, "q8": 2, "q4": 3, "f16x32": 4, "q8row": 5}

_lock = threading.Lock()
_cache = {}


def lib_path(mutant: int = 0, build_dir: Optional[str] = None) -> str:
    d = build_dir or _BUILD
    name = "libgemv_oracle.so" if mutant == 0 else f"libgemv_oracle_mutant{mutant}.so"
    return os.path.join(d, name)


def build(mutant: int = 0, build_dir: Optional[str] = None, force: bool = False) -> str:
    """Compile the oracle (or one deliberately broken variant) with gcc."""
    out = lib_path(mutant, build_dir)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
           f"-DORACLE_MUTANT={int(mutant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes wrapper around one build of ``gemv_oracle.c``."""

    def __init__(self, path: str):
        self.path = path
        L = ctypes.CDLL(path)
        i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        L.oracle_dec16.restype = ctypes.c_double
        L.oracle_dec16.argtypes = [ctypes.c_uint16]
        L.oracle_dec16_array.restype = None
        L.oracle_dec16_array.argtypes = [vp, vp, i64]
        for name in ("oracle_gemv_f32", "oracle_gemv_f16", "oracle_gemv_f16_xf32"):
            f = getattr(L, name)
            f.restype = i32
            f.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp, i32]
        for name in ("oracle_gemv_q8", "oracle_gemv_q4", "oracle_gemv_q8_rowscale"):
            f = getattr(L, name)
            f.restype = i32
            f.argtypes = [vp, vp, vp, i64, i64, vp, i64, vp, vp, i32]
        for name in ("oracle_dequant_q8", "oracle_dequant_q4"):
            f = getattr(L, name)
            f.restype = i32
            f.argtypes = [vp, vp, i64, i64, vp]
        L.oracle_flops.restype = ctypes.c_double
        L.oracle_flops.argtypes = [i64, i64]
        L.oracle_bytes.restype = ctypes.c_double
        L.oracle_bytes.argtypes = [i32, i64, i64]
        L.oracle_mutant_id.restype = i32
        L.oracle_softmax_f16.restype = i32
        L.oracle_softmax_f16.argtypes = [vp, i64, i64, vp, i64, vp, i32]
        L.oracle_enc16.restype = ctypes.c_uint16
        L.oracle_enc16.argtypes = [ctypes.c_float]
        L.oracle_enc16_array.restype = None
        L.oracle_enc16_array.argtypes = [vp, vp, i64]
        L.oracle_quantize.restype = i32
        L.oracle_quantize.argtypes = [i32, i32, i32, vp, i64, i64, vp, vp, vp]
        self._L = L

    # -- binary16 --------------------------------------------------------
    def dec16(self, bits) -> np.ndarray:
        """IEEE binary16 bit patterns -> float64 (own decoder, not numpy's)."""
        b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
        out = np.empty(b.shape, dtype=np.float64)
        self._L.oracle_dec16_array(b.ctypes.data, out.ctypes.data, b.size)
        return out

    def enc16(self, values) -> np.ndarray:
        """float32 values -> IEEE binary16 bit patterns, nearest even (own encoder)."""
        f = np.ascontiguousarray(np.asarray(values, dtype=np.float32))
        out = np.empty(f.shape, dtype=np.uint16)
        self._L.oracle_enc16_array(f.ctypes.data, out.ctypes.data, f.size)
        return out

    # -- quantiser ---------------------------------------------------------
    def quantize(self, dtype: str, W, M: int, N: int):
        """Symmetric quantisation of W [M, N] for 'q8', 'q8row' or 'q4'.

        W: float32 values, or uint16 binary16 bit patterns.  Returns (codes,
        scales, sq_err): int8 [M, N] or packed uint8 [M, N/2]; FP16 bits
        [M, groups] ([M, 1] for 'q8row'); sum of squared errors (double).
        """
        W = np.ascontiguousarray(W)
        w_kind = 1 if W.dtype == np.uint16 else 0
        if w_kind == 0 and W.dtype != np.float32:
            raise ValueError("W must be float32 or binary16 bits")
        bits = 4 if dtype == "q4" else 8
        per_row = 1 if dtype == "q8row" else 0
        groups = 0 if N == 0 else (1 if per_row else (N + 127) // 128)
        A = np.zeros((M, N // 2 if bits == 4 else N), dtype=np.uint8 if bits == 4 else np.int8)
        S = np.zeros((M, groups), dtype=np.uint16)
        err = ctypes.c_double(0.0)
        rc = self._L.oracle_quantize(bits, per_row, w_kind, W.ctypes.data, M, N, A.ctypes.data,
                                     S.ctypes.data, ctypes.addressof(err))
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments of {dtype} quantize")
        return A, S, err.value

    # -- GEMV --------------------------------------------------------------
    def gemv(self, dtype: str, A, x, M: int, N: int, scales=None,
             rows: Optional[Sequence[int]] = None, threads: int = 1):
        """Reference y and normaliser den for all rows, or for ``rows``.

        Storage formats: f32 -> float32 A [M, N], x [N]; f16 -> uint16 bits;
        q8 -> int8 A [M, N]; q4 -> uint8 A [M, N/2]; x FP16 bits for q8/q4;
        scales FP16 bits [M, ceil(N/128)]; f16x32 -> uint16 bits A, float32
        x; q8row -> int8 A, FP16 bits scales [M] (one per row).  Returns
        (y, den) as float64.
        """
        A = np.ascontiguousarray(A)
        x = np.ascontiguousarray(x)
        if rows is None:
            r_ptr, nrows = None, M
        else:
            r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            r_ptr, nrows = r.ctypes.data, r.size
        y = np.empty(max(nrows, 0), dtype=np.float64)
        den = np.empty(max(nrows, 0), dtype=np.float64)
        if dtype in ("f32", "f16", "f16x32"):
            fn = {"f32": self._L.oracle_gemv_f32, "f16": self._L.oracle_gemv_f16,
                  "f16x32": self._L.oracle_gemv_f16_xf32}[dtype]
            rc = fn(A.ctypes.data, x.ctypes.data, M, N, r_ptr, nrows,
                    y.ctypes.data, den.ctypes.data, threads)
        elif dtype in ("q8", "q4", "q8row"):
            s = np.ascontiguousarray(scales)
            fn = {"q8": self._L.oracle_gemv_q8, "q4": self._L.oracle_gemv_q4,
                  "q8row": self._L.oracle_gemv_q8_rowscale}[dtype]
            rc = fn(A.ctypes.data, x.ctypes.data, s.ctypes.data, M, N, r_ptr, nrows,
                    y.ctypes.data, den.ctypes.data, threads)
        else:
            raise ValueError(dtype)
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments of {dtype} gemv")
        return y, den

    def dequant(self, dtype: str, A, scales, M: int, N: int) -> np.ndarray:
        """Dequantised weights q * s as float64 [M, N] (q8 or q4)."""
        A = np.ascontiguousarray(A)
        s = np.ascontiguousarray(scales)
        W = np.empty((M, N), dtype=np.float64)
        fn = self._L.oracle_dequant_q8 if dtype == "q8" else self._L.oracle_dequant_q4
        if fn(A.ctypes.data, s.ctypes.data, M, N, W.ctypes.data) != 0:
            raise ValueError(f"oracle rejected the arguments of {dtype} dequant")
        return W

    # -- row softmax ---------------------------------------------------------
    def softmax(self, x_bits, M: int, N: int, rows: Optional[Sequence[int]] = None,
                threads: int = 1) -> np.ndarray:
        """Row softmax of binary16 bits [M, N] in double: [nrows, N]."""
        x = np.ascontiguousarray(np.asarray(x_bits, dtype=np.uint16))
        if rows is None:
            r_ptr, nrows = None, M
        else:
            r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            r_ptr, nrows = r.ctypes.data, r.size
        y = np.empty((max(nrows, 0), N), dtype=np.float64)
        if self._L.oracle_softmax_f16(x.ctypes.data, M, N, r_ptr, nrows, y.ctypes.data, threads) != 0:
            raise ValueError("oracle rejected the arguments of softmax")
        return y

    # -- counting model ------------------------------------------------------
    def flops(self, M: int, N: int) -> float:
        return self._L.oracle_flops(M, N)

    def bytes(self, dtype: str, M: int, N: int) -> float:
        return self._L.oracle_bytes(KIND[dtype], M, N)

    @property
    def mutant(self) -> int:
        return self._L.oracle_mutant_id()


def load(mutant: int = 0, build_dir: Optional[str] = None) -> Oracle:
    """Build (if stale) and load the oracle; cached per (mutant, dir)."""
    key = (mutant, build_dir)
    with _lock:
        if key not in _cache:
            _cache[key] = Oracle(build(mutant, build_dir))
        return _cache[key]


def max_normalised_error(y_gpu, y_ref, den) -> float:
    """max_i |y_gpu[i] - y_ref[i]| / den[i]; rows with den == 0 must be exactly 0.

    A row whose normaliser is zero has the exact answer 0 and any non-zero
    output there counts as an infinite error.
    """
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    den = np.asarray(den, dtype=np.float64)
    if y_gpu.size == 0:
        return 0.0
    if not np.all(np.isfinite(y_gpu)):
        return float("inf")
    err = np.abs(y_gpu - y_ref)
    zero = den == 0
    out = np.zeros_like(err)
    out[~zero] = err[~zero] / den[~zero]
    out[zero & (err != 0)] = np.inf
    return float(out.max())
