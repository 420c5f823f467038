"""gemv_ex_host: x and y in page-locked host memory, bit-identical to the
device-resident call, also in a chain of overlapped calls sharing x_dev."""

import ctypes

import numpy as np
import pytest

import memory_bound_gemv_gb300 as mbg
import synth

from gpu_util import upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

CASES = [("f32", 300, 4160), ("f16", 300, 4160), ("q8", 257, 4096), ("q4", 129, 4160),
         ("f16x32", 77, 1000), ("f16", 4096, 14336), ("f16", 5, 3)]


@pytest.mark.parametrize("overlap", (False, True), ids=("plain", "overlap"))
@pytest.mark.parametrize("dtype,M,N", CASES)
def test_host_buffers_match_device_call(dtype, M, N, overlap):
    inp = synth.make(synth.random_case(dtype, M, N, 600 + M + N))
    t = upload(dtype, inp)
    y_dev = mbg.gemv(dtype, t["A"], t["x"], t.get("scales"))
    x_host = t["x"].cpu().pin_memory()
    x_dev = torch.empty_like(t["x"])
    y_host = mbg.gemv_host(dtype, t["A"], x_host, x_dev, t.get("scales"), overlap=overlap)
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu()), dtype
    assert torch.equal(x_dev, t["x"])


@pytest.mark.parametrize("overlap", (False, True), ids=("plain", "overlap"))
def test_chain_of_calls_sharing_x_dev(overlap):
    """Each call's copy of x must not overwrite x_dev before the previous GEMV is done."""
    dtype, M, N, steps = "f16", 2048, 14336, 24
    inp = synth.make(synth.random_case(dtype, M, N, 77))
    t = upload(dtype, inp)
    xs = [torch.from_numpy(synth.to_f16_bits(synth.normal(500 + k, 1, 0, N, 1.0)).view(np.float16))
          for k in range(steps)]
    x_hosts = [x.pin_memory() for x in xs]
    y_hosts = [torch.empty(M, dtype=torch.float32).pin_memory() for _ in range(steps)]
    x_dev = torch.empty(N, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for k in range(steps):
            mbg.gemv_host(dtype, t["A"], x_hosts[k], x_dev, y_host=y_hosts[k], overlap=overlap)
    s.synchronize()
    for k in range(steps):
        y_ref = mbg.gemv(dtype, t["A"], xs[k].cuda())
        torch.cuda.synchronize()
        assert torch.equal(y_hosts[k], y_ref.cpu()), k


def test_host_x_alignment_and_rejections():
    dtype, M, N = "f16", 64, 1000
    inp = synth.make(synth.random_case(dtype, M, N, 5))
    t = upload(dtype, inp)
    y_dev = mbg.gemv(dtype, t["A"], t["x"])
    # x_host at an odd 2-byte offset inside a pinned buffer: the copy goes element-wise
    big = torch.empty(N + 1, dtype=torch.float16).pin_memory()
    big[1:].copy_(t["x"].cpu())
    x_dev = torch.empty_like(t["x"])
    y_host = torch.empty(M, dtype=torch.float32).pin_memory()
    L = mbg.lib()
    st = L.gemv_ex_host(mbg.F16, t["A"].data_ptr(), big.data_ptr() + 2, x_dev.data_ptr(), y_host.data_ptr(),
                        M, N, None, 0, None)
    assert st == mbg.OK
    torch.cuda.synchronize()
    assert torch.equal(y_host, y_dev.cpu())
    # pageable host memory is refused; so is a misaligned x_host and an unknown flag
    pageable = t["x"].cpu()
    assert L.gemv_ex_host(mbg.F16, t["A"].data_ptr(), pageable.data_ptr(), x_dev.data_ptr(),
                          y_host.data_ptr(), M, N, None, 0, None) == mbg.ERR_INVALID_VALUE
    y_pageable = torch.empty(M, dtype=torch.float32)
    assert L.gemv_ex_host(mbg.F16, t["A"].data_ptr(), big.data_ptr() + 2, x_dev.data_ptr(),
                          y_pageable.data_ptr(), M, N, None, 0, None) == mbg.ERR_INVALID_VALUE
    assert L.gemv_ex_host(mbg.F16, t["A"].data_ptr(), big.data_ptr() + 1, x_dev.data_ptr(),
                          y_host.data_ptr(), M, N, None, 0, None) == mbg.ERR_MISALIGNED
    assert L.gemv_ex_host(mbg.F16, t["A"].data_ptr(), big.data_ptr() + 2, x_dev.data_ptr(),
                          y_host.data_ptr(), M, N, None, 4, None) == mbg.ERR_INVALID_VALUE
    with pytest.raises(mbg.GemvError):
        mbg.gemv_host(dtype, t["A"], pageable, x_dev)
    with pytest.raises(ValueError):
        mbg.gemv_host(dtype, t["A"], t["x"], x_dev)  # a CUDA tensor is not host memory
    # N == 0 fills y_host with zeros
    y_host.fill_(3.0)
    assert L.gemv_ex_host(mbg.F16, None, None, None, y_host.data_ptr(), M, 0, None, 0, None) == mbg.OK
    torch.cuda.synchronize()
    assert torch.all(y_host == 0)
    assert mbg.gemv_get_device_error() == mbg.OK
