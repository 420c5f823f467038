"""Seeded synthetic inputs for the GEMV library and its oracle.

This module is the only code shared by the CUDA path's tests/bench and the
CPU oracle.  It draws random numbers and lays them out in the storage formats
the library consumes (FP32, IEEE binary16 bits, int8, packed int4, FP16 group
scales).  It contains none of the GEMV arithmetic: no dot products, no
dequantisation, no FP16 decoding.

Random numbers
--------------
SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) used as a counter-based generator: a stream with
initial state ``s`` produces output ``k`` (0-based) as ``mix(s + (k+1)*GAMMA)``,
where ``mix`` is the published SplitMix64 finaliser.  Every tensor of a
workload gets its own stream, with state ``mix(seed + tag*GAMMA)`` where
``tag`` is 1 for the weights A, 2 for x and 3 for the scales.  Because output
``k`` depends only on ``(seed, tag, k)``, any row of a matrix can be
regenerated on its own, which lets parity tests at full size rebuild sampled
rows on the host without holding the whole matrix twice.

Distributions
-------------
* uniform double on [0, 1): ``(u >> 11) * 2**-53``; U[lo, hi) is
  ``lo + (hi - lo) * that``.
* normal(0, sigma): Box-Muller, element k uses outputs 2k and 2k+1:
  ``sigma * sqrt(-2 ln(1 - U0)) * cos(2 pi U1)``.
* integers uniform on [lo, hi] with n = hi - lo + 1 values:
  ``lo + (((u >> 32) * n) >> 32)`` (exact for n a power of two; for n = 255
  the bias is below 255 / 2**32).
* FP32 / FP16 values are drawn in double and rounded to nearest-even by
  numpy's conversions; the FP16 bit patterns are what both sides consume.

Int4 packing: element j of a row is stored in byte j // 2 of that row, in the
low nibble when j is even and the high nibble when j is odd, as the 4-bit
two's-complement code of a value in [-8, 7].
"""

from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Dict, Optional, Tuple

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

TAG_A = 1
TAG_X = 2
TAG_SCALES = 3

GROUP = 128  # columns per FP16 scale in the quantised formats

_CHUNK = 1 << 22  # elements generated per numpy pass (bounds temporaries)


def _mix_int(z: int) -> int:
    """SplitMix64 finaliser on a Python int (used for stream keys)."""
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = z ^ (z >> np.uint64(30))
    z = z * _C1
    z = z ^ (z >> np.uint64(27))
    z = z * _C2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tag: int) -> int:
    """Initial state of the stream for tensor ``tag`` of workload ``seed``."""
    return _mix_int((seed + tag * GAMMA) & _M64)


def raw_u64(seed: int, tag: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of the (seed, tag) stream."""
    key = np.uint64(stream_key(seed, tag))
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + k * np.uint64(GAMMA))


def _unit(u: np.ndarray) -> np.ndarray:
    return (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform(seed: int, tag: int, start: int, count: int, lo: float, hi: float) -> np.ndarray:
    """``count`` doubles from U[lo, hi), stream positions start.."""
    out = np.empty(count, dtype=np.float64)
    for off in range(0, count, _CHUNK):
        n = min(_CHUNK, count - off)
        out[off:off + n] = lo + (hi - lo) * _unit(raw_u64(seed, tag, start + off, n))
    return out


def normal(seed: int, tag: int, start: int, count: int, sigma: float) -> np.ndarray:
    """``count`` doubles from normal(0, sigma); element k uses outputs 2k, 2k+1."""
    out = np.empty(count, dtype=np.float64)
    for off in range(0, count, _CHUNK):
        n = min(_CHUNK, count - off)
        u = raw_u64(seed, tag, 2 * (start + off), 2 * n)
        u0 = 1.0 - _unit(u[0::2])  # (0, 1]
        u1 = _unit(u[1::2])
        out[off:off + n] = sigma * np.sqrt(-2.0 * np.log(u0)) * np.cos(2.0 * math.pi * u1)
    return out


def integers(seed: int, tag: int, start: int, count: int, lo: int, hi: int) -> np.ndarray:
    """``count`` int64 values uniform on [lo, hi]."""
    n_vals = np.uint64(hi - lo + 1)
    out = np.empty(count, dtype=np.int64)
    for off in range(0, count, _CHUNK):
        n = min(_CHUNK, count - off)
        u = raw_u64(seed, tag, start + off, n) >> np.uint64(32)
        with np.errstate(over="ignore"):
            out[off:off + n] = ((u * n_vals) >> np.uint64(32)).astype(np.int64) + lo
    return out


def to_f16_bits(v: np.ndarray) -> np.ndarray:
    """Round doubles to binary16 (nearest-even) and return the raw bits."""
    return v.astype(np.float16).view(np.uint16)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Pack an int array [M, N] (N even, values in [-8, 7]) into [M, N/2] bytes.

    Even column -> low nibble, odd column -> high nibble, two's complement.
    """
    q = np.asarray(q, dtype=np.int64)
    if q.ndim != 2 or q.shape[1] % 2:
        raise ValueError("pack_int4 wants a 2-D array with an even column count")
    if q.size and (q.min() < -8 or q.max() > 7):
        raise ValueError("int4 values must lie in [-8, 7]")
    lo = (q[:, 0::2] & 0xF).astype(np.uint8)
    hi = (q[:, 1::2] & 0xF).astype(np.uint8)
    return (lo | (hi << 4)).astype(np.uint8)


def n_groups(N: int) -> int:
    return (N + GROUP - 1) // GROUP


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMV problem: dtype, shape, seed and value distributions."""

    name: str
    dtype: str          # "f32" | "f16" | "q8" | "q4" | "f16x32" | "q8row"
    M: int
    N: int
    seed: int
    a_dist: Tuple       # ("uniform", lo, hi) | ("normal", sigma) | ("int", lo, hi)
    x_dist: Tuple
    s_dist: Optional[Tuple] = None  # scales, quantised dtypes only

    @property
    def quantised(self) -> bool:
        return self.dtype in ("q8", "q4", "q8row")

    @property
    def scale_groups(self) -> int:
        """FP16 scales per row: one per 128 columns, or one for "q8row"."""
        return 1 if self.dtype == "q8row" else n_groups(self.N)


def _wl(name, dtype, M, N, seed, a, x, s=None) -> Workload:
    return Workload(name, dtype, M, N, seed, a, x, s)


U11 = ("uniform", -1.0, 1.0)
N002 = ("normal", 0.02)
N1 = ("normal", 1.0)
Q8D = ("int", -127, 127)
Q4D = ("int", -8, 7)
SCD = ("uniform", 0.001, 0.01)


def _sweep():
    out = {}
    for n in (2048, 4096, 8192, 16384):
        seed = 40 + int(math.log2(n))
        out[f"sweep_f32_{n}"] = _wl(f"sweep_f32_{n}", "f32", n, n, seed, U11, U11)
        out[f"sweep_f16_{n}"] = _wl(f"sweep_f16_{n}", "f16", n, n, seed + 100, U11, U11)
    return out


#: The five workload families the library is measured on.  Names say what
#: each is; seeds are fixed so every run sees the same bits.
WORKLOADS: Dict[str, Workload] = {
    # FP32 1024x1024, A and x uniform[-1, 1]
    "f32_1024": _wl("f32_1024", "f32", 1024, 1024, 1, U11, U11),
    # FP16 4096x4096, normal(0, 0.02)
    "f16_4096": _wl("f16_4096", "f16", 4096, 4096, 2, N002, N002),
    # FP16 decode-MLP up-projection (x length 4096) and down-projection (x length 14336)
    "f16_up_14336x4096": _wl("f16_up_14336x4096", "f16", 14336, 4096, 3, N002, N002),
    "f16_down_4096x14336": _wl("f16_down_4096x14336", "f16", 4096, 14336, 31, N002, N002),
    **_sweep(),
    # weight-only quantised, FP16 scale per row per 128 columns
    "q8_4096x14336": _wl("q8_4096x14336", "q8", 4096, 14336, 5, Q8D, N1, SCD),
    "q8_14336x4096": _wl("q8_14336x4096", "q8", 14336, 4096, 51, Q8D, N1, SCD),
    "q4_4096x14336": _wl("q4_4096x14336", "q4", 4096, 14336, 52, Q4D, N1, SCD),
    "q4_14336x4096": _wl("q4_14336x4096", "q4", 14336, 4096, 53, Q4D, N1, SCD),
    # format options: FP16 weights with an FP32 hidden state; INT8 with one
    # FP16 scale per row
    "f16x32_down_4096x14336": _wl("f16x32_down_4096x14336", "f16x32", 4096, 14336, 61, N002, N1),
    "q8row_4096x14336": _wl("q8row_4096x14336", "q8row", 4096, 14336, 62, Q8D, N1, SCD),
}


#: Row-softmax inputs of the same decode workloads ("membound", "Bonus kernel":
#: 8192x8192, 4096x32768 and 1024x131072 FP16).  The page gives no value
#: distribution; logits are drawn from normal(0, 2) and rounded to FP16.
SOFTMAX_WORKLOADS: Dict[str, Workload] = {
    "softmax_8192x8192": _wl("softmax_8192x8192", "f16", 8192, 8192, 81, ("normal", 2.0), ("normal", 2.0)),
    "softmax_4096x32768": _wl("softmax_4096x32768", "f16", 4096, 32768, 82, ("normal", 2.0), ("normal", 2.0)),
    "softmax_1024x131072": _wl("softmax_1024x131072", "f16", 1024, 131072, 83, ("normal", 2.0),
                               ("normal", 2.0)),
}


def _draw_serial(dist: Tuple, seed: int, tag: int, start: int, count: int) -> np.ndarray:
    kind = dist[0]
    if kind == "uniform":
        return uniform(seed, tag, start, count, dist[1], dist[2])
    if kind == "normal":
        return normal(seed, tag, start, count, dist[1])
    if kind == "int":
        return integers(seed, tag, start, count, dist[1], dist[2])
    raise ValueError(f"unknown distribution {dist!r}")


_PARALLEL_MIN = 1 << 23  # elements; smaller draws stay on one thread


def _host_threads() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(32, n))


def _draw(dist: Tuple, seed: int, tag: int, start: int, count: int,
          parallel: bool = True) -> np.ndarray:
    """``count`` values of ``dist`` from stream positions ``start..``.

    Every output depends only on (seed, tag, position), so large draws are
    split into position ranges filled by several threads (numpy releases the
    interpreter lock inside its array loops); the values are the same as on
    one thread."""
    nthreads = _host_threads()
    if not parallel or count < _PARALLEL_MIN or nthreads == 1:
        return _draw_serial(dist, seed, tag, start, count)
    first = _draw_serial(dist, seed, tag, start, min(count, _CHUNK))
    out = np.empty(count, dtype=first.dtype)
    out[:first.size] = first
    pieces = [(off, min(_CHUNK, count - off)) for off in range(first.size, count, _CHUNK)]

    def fill(piece):
        off, n = piece
        out[off:off + n] = _draw_serial(dist, seed, tag, start + off, n)

    with concurrent.futures.ThreadPoolExecutor(max_workers=nthreads) as ex:
        list(ex.map(fill, pieces))
    return out


def _encode_rows(dtype: str, vals: np.ndarray, nrows: int, N: int) -> np.ndarray:
    if dtype == "f32":
        return vals.astype(np.float32).reshape(nrows, N)
    if dtype in ("f16", "f16x32"):
        return to_f16_bits(vals).reshape(nrows, N)
    if dtype in ("q8", "q8row"):
        return vals.astype(np.int8).reshape(nrows, N)
    if dtype == "q4":
        return pack_int4(vals.reshape(nrows, N))
    raise ValueError(dtype)


def weight_rows(w: Workload, row0: int, nrows: int, parallel: bool = True) -> np.ndarray:
    """Rows ``row0 .. row0+nrows-1`` of A in storage format.

    f32 -> float32 [n, N]; f16 -> uint16 bits [n, N]; q8 -> int8 [n, N];
    q4 -> uint8 [n, N/2]; f16x32 as f16; q8row as q8.
    """
    if w.dtype == "q4" and w.N % 2:
        raise ValueError("int4 rows need an even column count")
    if parallel and nrows > 1 and nrows * w.N >= _PARALLEL_MIN and _host_threads() > 1:
        # row blocks drawn and encoded on several threads (same values)
        nt = _host_threads()
        step = max(1, -(-nrows // (4 * nt)))
        blocks = [(r, min(step, nrows - r)) for r in range(0, nrows, step)]
        parts = [None] * len(blocks)

        def fill(k):
            r, n = blocks[k]
            parts[k] = weight_rows(w, row0 + r, n, parallel=False)

        with concurrent.futures.ThreadPoolExecutor(max_workers=nt) as ex:
            list(ex.map(fill, range(len(blocks))))
        return np.concatenate(parts, axis=0)
    vals = _draw(w.a_dist, w.seed, TAG_A, row0 * w.N, nrows * w.N, parallel=parallel)
    return _encode_rows(w.dtype, vals, nrows, w.N)


def x_vector(w: Workload) -> np.ndarray:
    """x in storage format: float32 [N] for f32 and f16x32, FP16 bits uint16 [N] otherwise."""
    vals = _draw(w.x_dist, w.seed, TAG_X, 0, w.N)
    return vals.astype(np.float32) if w.dtype in ("f32", "f16x32") else to_f16_bits(vals)


def scale_rows(w: Workload, row0: int, nrows: int) -> np.ndarray:
    """FP16 bits [nrows, groups] of the scales (groups = ceil(N/128), or 1 for q8row)."""
    if not w.quantised:
        raise ValueError("scales exist only for q8/q4/q8row")
    g = w.scale_groups
    vals = _draw(w.s_dist, w.seed, TAG_SCALES, row0 * g, nrows * g)
    return to_f16_bits(vals).reshape(nrows, g)


def make(w: Workload):
    """All inputs of a workload: dict with 'A', 'x' and (quantised) 'scales'."""
    out = {"A": weight_rows(w, 0, w.M), "x": x_vector(w)}
    if w.quantised:
        out["scales"] = scale_rows(w, 0, w.M)
    return out


def random_case(dtype: str, M: int, N: int, seed: int) -> Workload:
    """A workload of arbitrary shape with the distributions of the named families.

    f32 uses uniform[-1, 1]; f16 normal(0, 0.02); q8/q4 the quantised recipe.
    """
    if dtype == "f32":
        return _wl(f"case_f32_{M}x{N}", "f32", M, N, seed, U11, U11)
    if dtype == "f16":
        return _wl(f"case_f16_{M}x{N}", "f16", M, N, seed, N002, N002)
    if dtype == "q8":
        return _wl(f"case_q8_{M}x{N}", "q8", M, N, seed, Q8D, N1, SCD)
    if dtype == "q4":
        return _wl(f"case_q4_{M}x{N}", "q4", M, N, seed, Q4D, N1, SCD)
    if dtype == "f16x32":
        return _wl(f"case_f16x32_{M}x{N}", "f16x32", M, N, seed, N002, N1)
    if dtype == "q8row":
        return _wl(f"case_q8row_{M}x{N}", "q8row", M, N, seed, Q8D, N1, SCD)
    raise ValueError(dtype)
