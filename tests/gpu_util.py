"""Helpers for the GPU tests: upload synthetic inputs, compare with the oracle."""

import numpy as np

import oracle
import synth

# FP32 arithmetic (f32, and f16 weights with an FP32 x) at 1e-5; the FP16 and
# quantised formats at 2e-3, both normalised by sum_j |w_ij| |x_j|.
TOL = {"f32": 1e-5, "f16": 2e-3, "q8": 2e-3, "q4": 2e-3, "f16x32": 1e-5, "q8row": 2e-3}


def torch_mod():
    import torch
    return torch


def upload(dtype, inp, device="cuda"):
    """numpy storage arrays -> CUDA tensors the binding accepts."""
    torch = torch_mod()
    A, x = inp["A"], inp["x"]
    if dtype in ("f32", "f16x32"):
        tx = torch.from_numpy(np.ascontiguousarray(x))
    else:
        tx = torch.from_numpy(np.ascontiguousarray(x).view(np.float16))
    if dtype in ("f16", "f16x32"):
        tA = torch.from_numpy(np.ascontiguousarray(A).view(np.float16))
    else:
        tA = torch.from_numpy(np.ascontiguousarray(A))
    out = {"A": tA.to(device), "x": tx.to(device)}
    if "scales" in inp:
        s = torch.from_numpy(np.ascontiguousarray(inp["scales"]).view(np.float16))
        if dtype == "q8row":
            s = s.reshape(-1)  # one scale per row: [M]
        out["scales"] = s.to(device)
    return out


def reference(dtype, inp, M, N, rows=None, threads=8):
    orc = oracle.load()
    return orc.gemv(dtype, inp["A"], inp["x"], M, N, scales=inp.get("scales"), rows=rows,
                    threads=threads)


def assert_close(dtype, y_gpu, y_ref, den, what=""):
    err = oracle.max_normalised_error(y_gpu, y_ref, den)
    assert err <= TOL[dtype], f"{what}: max normalised error {err:.3e} > {TOL[dtype]:.0e}"
    return err
