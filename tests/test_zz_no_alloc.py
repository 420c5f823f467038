"""gemv_ex_host_noalloc, the entry point for callers that cannot allocate
device memory (a loop that may not allocate after start-up, a plug-in whose
host program owns the allocator, a caller with only the C ABI).  It keeps the
device copy of x in a fixed array inside the library; its results must match
gemv_ex_host, which takes that buffer from the caller.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""

import numpy as np
import pytest

import memory_bound_gemv_gb300 as mbg
import oracle
import synth

from gpu_util import assert_close, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _second_x(dtype, N, seed):
    v = synth.normal(seed, 9, 0, N, 1.0)
    return v.astype(np.float32) if dtype in ("f32", "f16x32") else synth.to_f16_bits(v)


@pytest.mark.parametrize("dtype,M,N", [("f16", 512, 14336), ("q4", 300, 4160), ("f32", 129, 1000),
                                       ("f16", 7, 131072)])
def test_noalloc_matches_gemv_ex_host_on_two_calls(dtype, M, N):
    L = mbg.lib()
    orc = oracle.load()
    inp = synth.make(synth.random_case(dtype, M, N, 900 + N))
    t = upload(dtype, inp)
    dt = mbg.DTYPES[dtype]
    s_ptr = t["scales"].data_ptr() if "scales" in t else None
    x_dev = torch.empty_like(t["x"])
    for call, x_np in enumerate((inp["x"], _second_x(dtype, N, 31))):
        x_view = x_np if x_np.dtype == np.float32 else x_np.view(np.float16)
        x_host = torch.from_numpy(np.ascontiguousarray(x_view)).pin_memory()
        y_noalloc = torch.full((M,), np.nan, dtype=torch.float32).pin_memory()
        y_host = torch.full((M,), np.nan, dtype=torch.float32).pin_memory()
        st = L.gemv_ex_host_noalloc(dt, t["A"].data_ptr(), x_host.data_ptr(), y_noalloc.data_ptr(),
                                    M, N, s_ptr, 0, None)
        assert st == mbg.OK, mbg.status_string(st)
        st = L.gemv_ex_host(dt, t["A"].data_ptr(), x_host.data_ptr(), x_dev.data_ptr(), y_host.data_ptr(),
                            M, N, s_ptr, 0, None)
        assert st == mbg.OK, mbg.status_string(st)
        torch.cuda.synchronize()
        # against the oracle's y on the same inputs
        y_ref, den = orc.gemv(dtype, inp["A"], x_np, M, N, scales=inp.get("scales"))
        assert_close(dtype, y_noalloc.numpy(), y_ref, den, f"noalloc {dtype} call {call}")
        assert_close(dtype, y_host.numpy(), y_ref, den, f"gemv_ex_host {dtype} call {call}")
        # the same kernel on the same x: bit for bit the result of gemv_ex_host
        assert np.array_equal(y_noalloc.numpy(), y_host.numpy()), (dtype, call)
    assert mbg.gemv_get_device_error() == mbg.OK


def test_noalloc_rejects_x_beyond_its_limit():
    L = mbg.lib()
    fake = 0x10000  # never dereferenced: the size check comes first
    assert L.gemv_ex_host_noalloc(mbg.F16, fake, fake, fake, 4, 131073, None, 0, None) == mbg.ERR_UNSUPPORTED
    assert L.gemv_ex_host_noalloc(mbg.F32, fake, fake, fake, 4, 65537, None, 0, None) == mbg.ERR_UNSUPPORTED
