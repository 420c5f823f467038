"""Helpers for the GPU tests: upload synthetic inputs, compare with the oracle."""

import numpy as np

import oracle
import synth

TOL = {"f32": 1e-5, "f16": 2e-3, "q8": 2e-3, "q4": 2e-3}


def torch_mod():
    import torch
    return torch


def upload(dtype, inp, device="cuda"):
    """numpy storage arrays -> CUDA tensors the binding accepts."""
    torch = torch_mod()
    A, x = inp["A"], inp["x"]
    if dtype == "f32":
        tA = torch.from_numpy(np.ascontiguousarray(A))
        tx = torch.from_numpy(np.ascontiguousarray(x))
    else:
        tx = torch.from_numpy(np.ascontiguousarray(x).view(np.float16))
        if dtype == "f16":
            tA = torch.from_numpy(np.ascontiguousarray(A).view(np.float16))
        else:
            tA = torch.from_numpy(np.ascontiguousarray(A))
    out = {"A": tA.to(device), "x": tx.to(device)}
    if "scales" in inp:
        out["scales"] = torch.from_numpy(np.ascontiguousarray(inp["scales"]).view(np.float16)).to(device)
    return out


def reference(dtype, inp, M, N, rows=None, threads=8):
    orc = oracle.load()
    return orc.gemv(dtype, inp["A"], inp["x"], M, N, scales=inp.get("scales"), rows=rows,
                    threads=threads)


def assert_close(dtype, y_gpu, y_ref, den, what=""):
    err = oracle.max_normalised_error(y_gpu, y_ref, den)
    assert err <= TOL[dtype], f"{what}: max normalised error {err:.3e} > {TOL[dtype]:.0e}"
    return err
