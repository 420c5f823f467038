"""The C-ABI library builds for sm_103a, loads, and exports what gemv.h declares.

Runs without a GPU: only calls that return before touching the device
(argument validation, tables, strings) are made.
"""

import ctypes
import os
import re

import pytest

import memory_bound_gemv_gb300 as mbg
from memory_bound_gemv_gb300 import build as mbg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(gemv_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_four_gemv_entry_points():
    names = declared_functions()
    for n in ("gemv_f32", "gemv_f16", "gemv_q8", "gemv_q4", "gemv_probe_read",
              "gemv_f16_xf32", "gemv_q8_rowscale"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = mbg.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def test_library_is_built_for_sm_103a_only():
    assert os.path.exists(mbg_build.LIB)
    assert "arch=compute_103a,code=sm_103a" in " ".join(mbg_build.ARCH)
    assert "sm_103a" in mbg.build_info()


def test_status_strings():
    for code, name in mbg.STATUS.items():
        assert mbg.status_string(code) == name


def test_variant_tables():
    for dt in ("f32", "f16", "q8", "q4", "f16x32"):
        vs = mbg.variants(dt)
        assert len(vs) >= 2
        assert any(v["xmode"] == "elem" for v in vs)
        assert any(v["kind"] == "tile" for v in vs)
        for v in vs:
            g = v["threads_per_row"]
            assert (32 % g == 0 if g <= 32 else g % 32 == 0) and v["warps"] >= 1
    assert len(mbg.probe_variants()) >= 2


FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("fn,extra", [("gemv_f32", []), ("gemv_f16", []),
                                      ("gemv_q8", [FAKE]), ("gemv_q4", [FAKE]),
                                      ("gemv_f16_xf32", []), ("gemv_q8_rowscale", [FAKE])])
def test_validation_errors_without_device(fn, extra):
    L = mbg.lib()
    f = getattr(L, fn)
    # negative sizes
    assert f(FAKE, FAKE, FAKE, -1, 4, *extra, None) == mbg.ERR_INVALID_VALUE
    assert f(FAKE, FAKE, FAKE, 4, -1, *extra, None) == mbg.ERR_INVALID_VALUE
    # M == 0 is a no-op that touches nothing
    assert f(None, None, None, 0, 8, *([None] if extra else []), None) == mbg.OK
    # NULL pointers
    assert f(None, FAKE, FAKE, 4, 8, *extra, None) == mbg.ERR_INVALID_VALUE
    assert f(FAKE, None, FAKE, 4, 8, *extra, None) == mbg.ERR_INVALID_VALUE
    assert f(FAKE, FAKE, None, 4, 8, *extra, None) == mbg.ERR_INVALID_VALUE
    # y not 4-byte aligned
    assert f(FAKE, FAKE, FAKE + 2, 4, 8, *extra, None) == mbg.ERR_MISALIGNED
    # x not aligned to its element size
    assert f(FAKE, FAKE + 1, FAKE, 4, 8, *extra, None) == mbg.ERR_MISALIGNED
    if fn == "gemv_f16_xf32":
        assert f(FAKE, FAKE + 2, FAKE, 4, 8, None) == mbg.ERR_MISALIGNED  # FP32 x
    if fn in ("gemv_f32", "gemv_f16", "gemv_f16_xf32"):
        assert f(FAKE + 1, FAKE, FAKE, 4, 8, None) == mbg.ERR_MISALIGNED
    else:
        assert f(FAKE, FAKE, FAKE, 4, 8, None, None) == mbg.ERR_INVALID_VALUE  # scales NULL
        assert f(FAKE, FAKE, FAKE, 4, 8, FAKE + 1, None) == mbg.ERR_MISALIGNED


def test_q4_odd_n_unsupported():
    L = mbg.lib()
    assert L.gemv_q4(FAKE, FAKE, FAKE, 4, 7, FAKE, None) == mbg.ERR_UNSUPPORTED
    assert L.gemv_dequant_q4(FAKE, FAKE, FAKE, 4, 7, None) == mbg.ERR_UNSUPPORTED


def test_probe_validation():
    L = mbg.lib()
    sink = FAKE
    assert L.gemv_probe_read(FAKE, 4096, sink, -1, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_probe_read(FAKE, 4096, None, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_probe_read(FAKE, 4097, sink, 0, None) == mbg.ERR_MISALIGNED
    assert L.gemv_probe_read(FAKE + 8, 4096, sink, 0, None) == mbg.ERR_MISALIGNED
    assert L.gemv_probe_read(FAKE, 0, sink, 0, None) == mbg.OK


def test_variant_id_out_of_range():
    L = mbg.lib()
    assert L.gemv_run_variant(mbg.F16, 10_000, FAKE, FAKE, FAKE, 4, 8, None, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_run_variant(mbg.F16, -1, FAKE, FAKE, FAKE, 4, 8, None, None) == mbg.ERR_INVALID_VALUE
    info = mbg.VariantInfo()
    assert L.gemv_variant_info(mbg.F16, 10_000, ctypes.byref(info)) == mbg.ERR_INVALID_VALUE
    # the flagged runner checks the variant id and the flags before anything else
    assert L.gemv_run_variant_ex(mbg.F16, -1, FAKE, FAKE, FAKE, 4, 8, None, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_run_variant_ex(mbg.F16, 0, FAKE, FAKE, FAKE, 4, 8, None, 2, None) == mbg.ERR_INVALID_VALUE


def test_debug_hook_arguments():
    """The late-writing test kernel rejects bad arguments before any launch;
    the skip switches take only the documented bits."""
    L = mbg.lib()
    assert L.gemv_debug_late_fill(None, 16, 0, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_debug_late_fill(FAKE, 6, 0, 0, None) == mbg.ERR_MISALIGNED
    assert L.gemv_debug_late_fill(FAKE + 2, 16, 0, 0, None) == mbg.ERR_MISALIGNED
    assert L.gemv_debug_late_fill(FAKE, 0, 0, 0, None) == mbg.OK
    L.gemv_debug_skip_copies(0)
    L.gemv_debug_skip_x_copy(0)


def test_status_codes_match_the_header():
    header = open(os.path.join(ROOT, "include", "gemv.h")).read()
    for code, name in mbg.STATUS.items():
        assert f"{name} = {code}" in header, name


def test_binding_rejects_cpu_tensors():
    torch = pytest.importorskip("torch")
    A = torch.zeros(4, 8, dtype=torch.float16)
    with pytest.raises(ValueError):
        mbg.gemv_f16(A, torch.zeros(8, dtype=torch.float16))


def test_product_package_does_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "memory_bound_gemv_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "gemv_oracle" not in text, f


def test_gemv_ex_rejects_unknown_flags():
    L = mbg.lib()
    assert L.gemv_ex(mbg.F16, FAKE, FAKE, FAKE, 4, 8, None, 2, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex(mbg.F16, FAKE, FAKE, FAKE, -1, 8, None, 1, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex(9, FAKE, FAKE, FAKE, 4, 8, None, 0, None) == mbg.ERR_INVALID_VALUE


def test_host_buffer_and_option_validation():
    L = mbg.lib()
    # gemv_ex_host(dtype, A, x_host, x_dev, y_host, M, N, scales, flags, stream):
    # argument checks come before any device call
    assert L.gemv_ex_host(mbg.F16, FAKE, FAKE, FAKE, FAKE, 4, 8, None, 2, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex_host(mbg.F16, FAKE, FAKE, FAKE, FAKE, -1, 8, None, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex_host(9, FAKE, FAKE, FAKE, FAKE, 4, 8, None, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex_host(mbg.F16, FAKE, FAKE, None, FAKE, 4, 8, None, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex_host(mbg.F16, FAKE, FAKE, FAKE + 1, FAKE, 4, 8, None, 0, None) == mbg.ERR_MISALIGNED
    assert L.gemv_ex_host(mbg.F16, FAKE, FAKE, FAKE, FAKE + 2, 4, 8, None, 0, None) == mbg.ERR_MISALIGNED
    assert L.gemv_ex_host(mbg.Q4, FAKE, FAKE, FAKE, FAKE, 4, 7, FAKE, 0, None) == mbg.ERR_UNSUPPORTED
    assert L.gemv_ex_host(mbg.F16, None, None, None, None, 0, 8, None, 0, None) == mbg.OK
    # the no-allocation variant refuses x beyond its array before anything else
    assert L.gemv_ex_host_noalloc(mbg.F32, FAKE, FAKE, FAKE, 4, 1 << 20, None, 0, None) == mbg.ERR_UNSUPPORTED
    # per-row INT8 with flags, FP16 weights with FP32 x
    assert L.gemv_q8_rowscale_ex(FAKE, FAKE, FAKE, 4, 8, FAKE, 2, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_q8_rowscale_ex(FAKE, FAKE, FAKE, 4, 8, None, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_q8_rowscale_run_variant(-1, FAKE, FAKE, FAKE, 4, 8, FAKE, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex(mbg.F16X32, FAKE, FAKE + 2, FAKE, 4, 8, None, 0, None) == mbg.ERR_MISALIGNED


def test_softmax_and_copy_validation():
    L = mbg.lib()
    assert L.gemv_softmax_f16(FAKE, FAKE, -1, 8, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_softmax_f16(None, None, 0, 8, None) == mbg.OK
    assert L.gemv_softmax_f16(None, FAKE, 2, 8, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_softmax_f16(FAKE + 1, FAKE, 2, 8, None) == mbg.ERR_MISALIGNED
    assert L.gemv_softmax_run_variant(10_000, FAKE, FAKE, 2, 8, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_probe_copy(FAKE, FAKE, 4096, -1, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_probe_copy(FAKE, FAKE + 8, 4096, 0, None) == mbg.ERR_MISALIGNED
    assert len(mbg.softmax_variants()) >= 2 and len(mbg.copy_probe_variants()) >= 1


def test_quantize_validation():
    L = mbg.lib()
    E = FAKE
    # (W, w_dtype, A, scales, M, N, [per_row], sq_err, stream)
    q8 = lambda *a: L.gemv_quantize_q8(*a)
    assert q8(E, mbg.F32, E, E, -1, 4, 0, None, None) == mbg.ERR_INVALID_VALUE
    assert q8(E, mbg.Q8, E, E, 4, 4, 0, None, None) == mbg.ERR_INVALID_VALUE  # weights must be F32/F16
    assert q8(None, mbg.F32, None, None, 0, 4, 0, None, None) == mbg.OK
    assert q8(None, mbg.F32, E, E, 4, 4, 0, None, None) == mbg.ERR_INVALID_VALUE
    assert q8(E, mbg.F32, E, None, 4, 4, 0, None, None) == mbg.ERR_INVALID_VALUE
    assert q8(E + 2, mbg.F32, E, E, 4, 4, 0, None, None) == mbg.ERR_MISALIGNED
    assert q8(E + 1, mbg.F16, E, E, 4, 4, 0, None, None) == mbg.ERR_MISALIGNED
    assert q8(E, mbg.F32, E, E + 1, 4, 4, 1, None, None) == mbg.ERR_MISALIGNED
    assert q8(E, mbg.F32, E, E, 4, 4, 0, E + 4, None) == mbg.ERR_MISALIGNED
    assert L.gemv_quantize_q4(E, mbg.F32, E, E, 4, 7, None, None) == mbg.ERR_UNSUPPORTED
    assert L.gemv_quantize_q4(E, mbg.F32, E, E, -4, 8, None, None) == mbg.ERR_INVALID_VALUE
