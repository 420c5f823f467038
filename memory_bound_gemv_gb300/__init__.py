"""Python binding of the GB300 GEMV library (``include/gemv.h``).

Argument marshalling only: every call checks tensor dtypes, shapes, devices
and contiguity, then passes raw device pointers, sizes and the current CUDA
stream to the C ABI of ``_build/libmbgemv.so``.  All arithmetic runs in that
library's CUDA kernels.  There is no CPU fallback: if the library cannot be
built or loaded, every call raises.

Function names match the C entry points: ``gemv_f32``, ``gemv_f16``,
``gemv_q8``, ``gemv_q4``, ``gemv_f16_xf32``, ``gemv_q8_rowscale``, ``gemv_probe_read``, ``gemv_dequant_q8``,
``gemv_dequant_q4``, ``gemv_run_variant`` ...  ``lib()`` returns the raw
ctypes handle for callers that want to pass pointers themselves.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import List, Optional

F32, F16, Q8, Q4, F16X32 = 0, 1, 2, 3, 4
DTYPES = {"f32": F32, "f16": F16, "q8": Q8, "q4": Q4, "f16x32": F16X32}
GROUP = 128

STATUS = {0: "GEMV_OK", 1: "GEMV_ERR_INVALID_VALUE", 2: "GEMV_ERR_MISALIGNED",
          3: "GEMV_ERR_UNSUPPORTED", 4: "GEMV_ERR_LAUNCH", 5: "GEMV_ERR_TIMEOUT",
          6: "GEMV_ERR_CUDA", 7: "GEMV_ERR_TIMEOUT_UNDRAINED"}
(OK, ERR_INVALID_VALUE, ERR_MISALIGNED, ERR_UNSUPPORTED, ERR_LAUNCH, ERR_TIMEOUT, ERR_CUDA,
 ERR_TIMEOUT_UNDRAINED) = range(8)

# test hooks (gemv_debug_skip_copies)
SKIP_X, SKIP_STAGE, SKIP_SEGMENT, SKIP_PROBE = 1, 2, 4, 8

XMODES = {0: "bulk", 1: "vec", 2: "l1", 3: "elem", 4: "reg"}


class GemvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


KINDS = {0: "vec", 1: "tile", 2: "elem", 3: "bulk", 4: "band", 5: "sband", 6: "mma", 7: "smma"}


class VariantInfo(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("kind", ctypes.c_int), ("threads_per_row", ctypes.c_int),
                ("rows_per_group", ctypes.c_int), ("unroll", ctypes.c_int),
                ("warps", ctypes.c_int), ("math", ctypes.c_int), ("xmode", ctypes.c_int),
                ("name", ctypes.c_char * 48)]


_lock = threading.Lock()
_lib = None


def _declare(L):
    i64, vp, i32, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    sig = {
        "gemv_f32": [vp, vp, vp, i64, i64, vp],
        "gemv_f16": [vp, vp, vp, i64, i64, vp],
        "gemv_q8": [vp, vp, vp, i64, i64, vp, vp],
        "gemv_q4": [vp, vp, vp, i64, i64, vp, vp],
        "gemv_f16_xf32": [vp, vp, vp, i64, i64, vp],
        "gemv_q8_rowscale": [vp, vp, vp, i64, i64, vp, vp],
        "gemv_q8_rowscale_run_variant": [i32, vp, vp, vp, i64, i64, vp, vp],
        "gemv_q8_rowscale_ex": [vp, vp, vp, i64, i64, vp, ctypes.c_uint, vp],
        "gemv_probe_read": [vp, ctypes.c_size_t, vp, i32, vp],
        "gemv_dequant_q8": [vp, vp, vp, i64, i64, vp],
        "gemv_quantize_q8": [vp, i32, vp, vp, i64, i64, i32, vp, vp],
        "gemv_quantize_q4": [vp, i32, vp, vp, i64, i64, vp, vp],
        "gemv_dequant_q4": [vp, vp, vp, i64, i64, vp],
        "gemv_variant_info": [i32, i32, ctypes.POINTER(VariantInfo)],
        "gemv_run_variant": [i32, i32, vp, vp, vp, i64, i64, vp, vp],
        "gemv_run_variant_ex": [i32, i32, vp, vp, vp, i64, i64, vp, ctypes.c_uint, vp],
        "gemv_get_device_error": [vp],
        "gemv_ex": [i32, vp, vp, vp, i64, i64, vp, ctypes.c_uint, vp],
        "gemv_ex_host": [i32, vp, vp, vp, vp, i64, i64, vp, ctypes.c_uint, vp],
        "gemv_ex_host_noalloc": [i32, vp, vp, vp, i64, i64, vp, ctypes.c_uint, vp],
        "gemv_softmax_f16": [vp, vp, i64, i64, vp],
        "gemv_softmax_run_variant": [i32, vp, vp, i64, i64, vp],
        "gemv_probe_copy": [vp, vp, ctypes.c_size_t, i32, vp],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = st
    L.gemv_probe_variant_count.argtypes = []
    L.gemv_probe_variant_count.restype = i32
    L.gemv_probe_variant_name.argtypes = [i32]
    L.gemv_probe_variant_name.restype = ctypes.c_char_p
    L.gemv_variant_count.argtypes = [i32]
    L.gemv_variant_count.restype = i32
    L.gemv_select_variant.argtypes = [i32, vp, vp, i64, i64]
    L.gemv_select_variant.restype = i32
    L.gemv_q8_rowscale_select_variant.argtypes = [vp, vp, i64, i64]
    L.gemv_q8_rowscale_select_variant.restype = i32
    for name in ("gemv_softmax_variant_count", "gemv_probe_copy_variant_count"):
        getattr(L, name).argtypes = []
        getattr(L, name).restype = i32
    for name in ("gemv_softmax_variant_name", "gemv_probe_copy_variant_name"):
        getattr(L, name).argtypes = [i32]
        getattr(L, name).restype = ctypes.c_char_p
    L.gemv_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.gemv_debug_set_wait_limit_ns.restype = None
    L.gemv_debug_skip_x_copy.argtypes = [i32]
    L.gemv_debug_skip_x_copy.restype = None
    L.gemv_debug_skip_copies.argtypes = [ctypes.c_uint]
    L.gemv_debug_skip_copies.restype = None
    L.gemv_debug_late_fill.argtypes = [vp, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64, vp]
    L.gemv_debug_late_fill.restype = st
    L.gemv_status_string.argtypes = [st]
    L.gemv_status_string.restype = ctypes.c_char_p
    L.gemv_last_cuda_error.argtypes = []
    L.gemv_last_cuda_error.restype = i32
    L.gemv_build_info.argtypes = []
    L.gemv_build_info.restype = ctypes.c_char_p
    return L


def library_path() -> str:
    from . import build as _b
    return _b.LIB


def lib(build_if_stale: bool = True):
    """The ctypes handle of libmbgemv.so (built in-tree on first use if stale)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            from . import build as _b
            path = _b.LIB
            if build_if_stale and not _b.up_to_date():
                path = _b.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library missing: {path} (run memory_bound_gemv_gb300.build)")
            _lib = _declare(ctypes.CDLL(path))
        return _lib


# ---------------------------------------------------------------------------
# tensor marshalling
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_ptr(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        # the current stream's handle without building a Stream object (this
        # runs once per call, on the host's critical path in a decode loop)
        try:
            return torch._C._cuda_getCurrentRawStream(torch._C._cuda_getDevice())
        except AttributeError:  # pragma: no cover - other torch builds
            stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(t, name, dtypes, shape, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must live on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _raise(status, what):
    if status != OK:
        raise GemvError(status, what)


def _f16_types():
    torch = _torch()
    return (torch.float16, torch.int16, torch.uint16)


def _out(y, M, device):
    torch = _torch()
    if y is None:
        return torch.empty(M, dtype=torch.float32, device=device)
    _check(y, "y", (torch.float32,), (M,), device)
    return y


def _mn(A, dtype):
    if A.dim() != 2:
        raise ValueError("A must be 2-D")
    M, W = A.shape
    return M, (2 * W if dtype == Q4 else W)


def gemv_f32(A, x, y=None, stream=None):
    """y = A x with FP32 A [M, N] and x [N]; returns y (float32 [M])."""
    torch = _torch()
    M, N = _mn(A, F32)
    _check(A, "A", (torch.float32,), (M, N))
    _check(x, "x", (torch.float32,), (N,), A.device)
    y = _out(y, M, A.device)
    _raise(lib().gemv_f32(A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, _stream_ptr(stream)), "gemv_f32")
    return y


def gemv_f16(A, x, y=None, stream=None):
    """y = A x with FP16 A [M, N] and x [N], FP32 accumulation and output."""
    M, N = _mn(A, F16)
    _check(A, "A", _f16_types(), (M, N))
    _check(x, "x", _f16_types(), (N,), A.device)
    y = _out(y, M, A.device)
    _raise(lib().gemv_f16(A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, _stream_ptr(stream)), "gemv_f16")
    return y


def gemv_f16_xf32(A, x, y=None, stream=None):
    """y = A x with FP16 A [M, N] and an FP32 x [N]; FP32 arithmetic and output."""
    torch = _torch()
    M, N = _mn(A, F16X32)
    _check(A, "A", _f16_types(), (M, N))
    _check(x, "x", (torch.float32,), (N,), A.device)
    y = _out(y, M, A.device)
    _raise(lib().gemv_f16_xf32(A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, _stream_ptr(stream)),
           "gemv_f16_xf32")
    return y


def gemv_q8_rowscale(A, x, row_scales, y=None, stream=None, flags: int = 0):
    """INT8 weights A [M, N] with one FP16 scale per row (row_scales [M]), FP16 x [N].

    ``flags`` as for ``gemv_ex``."""
    torch = _torch()
    M, N = _mn(A, Q8)
    _check(A, "A", (torch.int8,), (M, N))
    _check(x, "x", _f16_types(), (N,), A.device)
    _check(row_scales, "row_scales", _f16_types(), (M,), A.device)
    y = _out(y, M, A.device)
    if flags:
        st = lib().gemv_q8_rowscale_ex(A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N,
                                       row_scales.data_ptr(), flags, _stream_ptr(stream))
    else:
        st = lib().gemv_q8_rowscale(A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N,
                                    row_scales.data_ptr(), _stream_ptr(stream))
    _raise(st, "gemv_q8_rowscale")
    return y


def _quant(fn_name, dtype, A, x, scales, y, stream):
    torch = _torch()
    M, N = _mn(A, dtype)
    _check(A, "A", (torch.int8,) if dtype == Q8 else (torch.uint8,), tuple(A.shape))
    _check(x, "x", _f16_types(), (N,), A.device)
    _check(scales, "scales", _f16_types(), (M, (N + GROUP - 1) // GROUP), A.device)
    y = _out(y, M, A.device)
    fn = getattr(lib(), fn_name)
    _raise(fn(A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, scales.data_ptr(), _stream_ptr(stream)), fn_name)
    return y


def gemv_q8(A, x, scales, y=None, stream=None):
    """INT8 weights A [M, N], FP16 scales [M, ceil(N/128)], FP16 x [N]."""
    return _quant("gemv_q8", Q8, A, x, scales, y, stream)


def gemv_q4(A, x, scales, y=None, stream=None):
    """Packed INT4 weights A uint8 [M, N/2] (low nibble = even column)."""
    return _quant("gemv_q4", Q4, A, x, scales, y, stream)


FLAG_OVERLAP_PRECEDING = 1


def gemv_ex(dtype: str, A, x, scales=None, y=None, stream=None, flags: int = 0):
    """Any GEMV with launch flags (``FLAG_OVERLAP_PRECEDING``: A and scales are
    not written by the kernel just before this call on the stream)."""
    torch = _torch()
    dt = DTYPES[dtype]
    M, N = _mn(A, dt)
    a_types = {F32: (torch.float32,), F16: _f16_types(), Q8: (torch.int8,), Q4: (torch.uint8,),
               F16X32: _f16_types()}[dt]
    _check(A, "A", a_types, tuple(A.shape))
    _check(x, "x", (torch.float32,) if dt in (F32, F16X32) else _f16_types(), (N,), A.device)
    s_ptr = None
    if dt in (Q8, Q4):
        _check(scales, "scales", _f16_types(), (M, (N + GROUP - 1) // GROUP), A.device)
        s_ptr = scales.data_ptr()
    y = _out(y, M, A.device)
    _raise(lib().gemv_ex(dt, A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N, s_ptr, flags,
                         _stream_ptr(stream)), "gemv_ex")
    return y


def gemv_host(dtype: str, A, x_host, x_dev, scales=None, y_host=None, stream=None,
              overlap: bool = False):
    """GEMV with x and y in page-locked host memory (``gemv_ex_host``).

    x_host: pinned CPU tensor [N]; x_dev: CUDA tensor like it that receives
    x; y_host: pinned CPU float32 [M] (allocated pinned when None), written
    by the kernel -- synchronise the stream before reading it.  ``overlap``:
    the kernel before this call on the stream writes neither A, scales nor
    x_host (a previous gemv_host call qualifies)."""
    torch = _torch()
    dt = DTYPES[dtype]
    M, N = _mn(A, dt)
    a_types = {F32: (torch.float32,), F16: _f16_types(), Q8: (torch.int8,), Q4: (torch.uint8,),
               F16X32: _f16_types()}[dt]
    x_types = (torch.float32,) if dt in (F32, F16X32) else _f16_types()
    _check(A, "A", a_types, tuple(A.shape))
    _check(x_dev, "x_dev", x_types, (N,), A.device)
    # page-locking is checked by the library (GEMV_ERR_INVALID_VALUE otherwise)
    if not isinstance(x_host, torch.Tensor) or x_host.device.type != "cpu":
        raise ValueError("x_host must be a pinned CPU tensor")
    if x_host.dtype not in x_types or tuple(x_host.shape) != (N,) or not x_host.is_contiguous():
        raise ValueError(f"x_host must be a contiguous [{N}] tensor of {x_types}")
    if y_host is None:
        y_host = torch.empty(M, dtype=torch.float32).pin_memory()
    elif (not isinstance(y_host, torch.Tensor) or y_host.device.type != "cpu"
          or y_host.dtype != torch.float32 or tuple(y_host.shape) != (M,) or not y_host.is_contiguous()):
        raise ValueError(f"y_host must be a pinned contiguous float32 [{M}] CPU tensor")
    s_ptr = None
    if dt in (Q8, Q4):
        _check(scales, "scales", _f16_types(), (M, (N + GROUP - 1) // GROUP), A.device)
        s_ptr = scales.data_ptr()
    flags = FLAG_OVERLAP_PRECEDING if overlap else 0
    _raise(lib().gemv_ex_host(dt, A.data_ptr(), x_host.data_ptr(), x_dev.data_ptr(), y_host.data_ptr(),
                              M, N, s_ptr, flags, _stream_ptr(stream)), "gemv_ex_host")
    return y_host


def gemv(dtype: str, A, x, scales=None, y=None, stream=None, overlap: bool = False):
    """Dispatch on the storage type name: 'f32', 'f16', 'q8', 'q4', 'f16x32', 'q8row'.

    'q8row' takes one scale per row (``scales`` of shape [M])."""
    if dtype == "q8row":
        return gemv_q8_rowscale(A, x, scales, y, stream,
                                FLAG_OVERLAP_PRECEDING if overlap else 0)
    if overlap:
        return gemv_ex(dtype, A, x, scales, y, stream, FLAG_OVERLAP_PRECEDING)
    if dtype == "f32":
        return gemv_f32(A, x, y, stream)
    if dtype == "f16":
        return gemv_f16(A, x, y, stream)
    if dtype == "q8":
        return gemv_q8(A, x, scales, y, stream)
    if dtype == "q4":
        return gemv_q4(A, x, scales, y, stream)
    if dtype == "f16x32":
        return gemv_f16_xf32(A, x, y, stream)
    raise ValueError(dtype)


def gemv_run_variant(dtype: str, variant: int, A, x, scales=None, y=None, stream=None,
                     overlap: bool = False):
    """Run one compiled kernel variant (see ``variants``) on tensors.

    'q8row' (one scale per row) runs a variant of the INT8 table.  ``overlap``:
    launch flag GEMV_FLAG_OVERLAP_PRECEDING (as for ``gemv_ex``)."""
    dt = _table_dtype(dtype)
    M, N = _mn(A, dt)
    y = _out(y, M, A.device)
    s_ptr = scales.data_ptr() if scales is not None else None
    if dtype == "q8row":
        if overlap:
            raise ValueError("the row-scale variant runner takes no launch flags")
        st = lib().gemv_q8_rowscale_run_variant(variant, A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N,
                                                s_ptr, _stream_ptr(stream))
    elif overlap:
        st = lib().gemv_run_variant_ex(dt, variant, A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N,
                                       s_ptr, FLAG_OVERLAP_PRECEDING, _stream_ptr(stream))
    else:
        st = lib().gemv_run_variant(dt, variant, A.data_ptr(), x.data_ptr(), y.data_ptr(), M, N,
                                    s_ptr, _stream_ptr(stream))
    _raise(st, f"gemv_run_variant({dtype}, {variant})")
    return y


def _table_dtype(dtype: str) -> int:
    """Variant table of a storage type name ('q8row' shares the INT8 table)."""
    return Q8 if dtype == "q8row" else DTYPES[dtype]


def variants(dtype: str) -> List[dict]:
    L = lib()
    dt = _table_dtype(dtype)
    out = []
    for k in range(L.gemv_variant_count(dt)):
        info = VariantInfo()
        _raise(L.gemv_variant_info(dt, k, ctypes.byref(info)), "gemv_variant_info")
        out.append({"id": k, "name": info.name.decode(), "kind": KINDS[info.kind],
                    "threads_per_row": info.threads_per_row,
                    "rows_per_group": info.rows_per_group, "unroll": info.unroll,
                    "warps": info.warps, "math": "mixed" if info.math else "f32",
                    "xmode": XMODES[info.xmode]})
    return out


def select_variant(dtype: str, A, x) -> int:
    dt = _table_dtype(dtype)
    M, N = _mn(A, dt)
    if dtype == "q8row":
        return lib().gemv_q8_rowscale_select_variant(A.data_ptr(), x.data_ptr(), M, N)
    return lib().gemv_select_variant(dt, A.data_ptr(), x.data_ptr(), M, N)


def quantize(W, dtype: str, sq_err=None, stream=None):
    """Symmetric quantisation of W (float32 or float16 [M, N]) on the GPU.

    dtype 'q8' (one scale per 128 columns), 'q8row' (one per row) or 'q4'.
    Returns (A, scales) in the layouts gemv_q8 / gemv_q8_rowscale / gemv_q4
    take.  ``sq_err``: optional float64 CUDA tensor of one element to which the
    sum of squared quantisation errors is added."""
    torch = _torch()
    if W.dim() != 2:
        raise ValueError("W must be 2-D")
    M, N = W.shape
    _check(W, "W", (torch.float32, torch.float16), (M, N))
    w_dt = F32 if W.dtype == torch.float32 else F16
    e_ptr = None
    if sq_err is not None:
        _check(sq_err, "sq_err", (torch.float64,), (1,), W.device)
        e_ptr = sq_err.data_ptr()
    if dtype == "q4":
        A = torch.empty(M, N // 2, dtype=torch.uint8, device=W.device)
        S = torch.empty(M, (N + GROUP - 1) // GROUP, dtype=torch.float16, device=W.device)
        st = lib().gemv_quantize_q4(W.data_ptr(), w_dt, A.data_ptr(), S.data_ptr(), M, N, e_ptr,
                                    _stream_ptr(stream))
    elif dtype in ("q8", "q8row"):
        per_row = dtype == "q8row"
        A = torch.empty(M, N, dtype=torch.int8, device=W.device)
        S = torch.empty((M,) if per_row else (M, (N + GROUP - 1) // GROUP), dtype=torch.float16,
                        device=W.device)
        st = lib().gemv_quantize_q8(W.data_ptr(), w_dt, A.data_ptr(), S.data_ptr(), M, N,
                                    1 if per_row else 0, e_ptr, _stream_ptr(stream))
    else:
        raise ValueError(dtype)
    _raise(st, f"quantize({dtype})")
    return A, S


def gemv_dequant_q8(A, scales, W=None, stream=None):
    torch = _torch()
    M, N = _mn(A, Q8)
    if W is None:
        W = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _raise(lib().gemv_dequant_q8(A.data_ptr(), scales.data_ptr(), W.data_ptr(), M, N,
                                 _stream_ptr(stream)), "gemv_dequant_q8")
    return W


def gemv_dequant_q4(A, scales, W=None, stream=None):
    torch = _torch()
    M, N = _mn(A, Q4)
    if W is None:
        W = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _raise(lib().gemv_dequant_q4(A.data_ptr(), scales.data_ptr(), W.data_ptr(), M, N,
                                 _stream_ptr(stream)), "gemv_dequant_q4")
    return W


def probe_variants() -> List[str]:
    L = lib()
    return [L.gemv_probe_variant_name(k).decode() for k in range(L.gemv_probe_variant_count())]


def gemv_probe_read(buf, sink, variant: int = 0, stream=None):
    """Stream ``buf`` (any dtype, contiguous, 16-byte multiple) once; XOR into sink (int64 [1])."""
    nbytes = buf.numel() * buf.element_size()
    _raise(lib().gemv_probe_read(buf.data_ptr(), nbytes, sink.data_ptr(), variant, _stream_ptr(stream)),
           "gemv_probe_read")


def gemv_softmax_f16(x, y=None, stream=None, variant: Optional[int] = None):
    """Row softmax of an FP16 matrix x [M, N] -> FP16 y (may be x itself)."""
    torch = _torch()
    if x.dim() != 2:
        raise ValueError("x must be 2-D")
    M, N = x.shape
    _check(x, "x", _f16_types(), (M, N))
    if y is None:
        y = torch.empty_like(x)
    _check(y, "y", _f16_types(), (M, N), x.device)
    L = lib()
    if variant is None:
        st = L.gemv_softmax_f16(x.data_ptr(), y.data_ptr(), M, N, _stream_ptr(stream))
    else:
        st = L.gemv_softmax_run_variant(variant, x.data_ptr(), y.data_ptr(), M, N, _stream_ptr(stream))
    _raise(st, "gemv_softmax_f16")
    return y


def softmax_variants() -> List[str]:
    L = lib()
    return [L.gemv_softmax_variant_name(k).decode() for k in range(L.gemv_softmax_variant_count())]


def gemv_probe_copy(src, dst, variant: int = 0, stream=None):
    """Copy src to dst (same byte size, 16-byte multiple) with the probe kernel."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("src and dst differ in size")
    _raise(lib().gemv_probe_copy(src.data_ptr(), dst.data_ptr(), nbytes, variant, _stream_ptr(stream)),
           "gemv_probe_copy")


def copy_probe_variants() -> List[str]:
    L = lib()
    return [L.gemv_probe_copy_variant_name(k).decode() for k in range(L.gemv_probe_copy_variant_count())]


def gemv_get_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device status (OK or ERR_TIMEOUT)."""
    return lib().gemv_get_device_error(_stream_ptr(stream))


def debug_set_wait_limit_ns(ns: int):
    lib().gemv_debug_set_wait_limit_ns(ns)


def debug_skip_x_copy(on: bool):
    lib().gemv_debug_skip_x_copy(1 if on else 0)


def debug_skip_copies(mask: int):
    """Test hook: SKIP_X | SKIP_STAGE | SKIP_SEGMENT | SKIP_PROBE (0 clears all)."""
    lib().gemv_debug_skip_copies(mask)


def debug_late_fill(dst, word: int, delay_ns: int, stream=None):
    """Test hook: fill dst (a CUDA tensor) with a 32-bit pattern after delay_ns,
    letting the next kernel on the stream start at once."""
    nbytes = dst.numel() * dst.element_size()
    _raise(lib().gemv_debug_late_fill(dst.data_ptr(), nbytes, word, delay_ns, _stream_ptr(stream)),
           "gemv_debug_late_fill")


def status_string(status: int) -> str:
    return lib().gemv_status_string(status).decode()


def build_info() -> str:
    return lib().gemv_build_info().decode()
