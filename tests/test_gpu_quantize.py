"""GPU quantiser against the oracle: codes and scales bit for bit, the squared
error to rounding, and the page's RMSE figures at full decode size."""

import json
import os

import numpy as np
import pytest

import memory_bound_gemv_gb300 as mbg
import oracle
import synth

from gpu_util import assert_close, reference

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
QDTYPES = ("q8", "q8row", "q4")
SHAPES = [(1, 2), (3, 6), (2, 126), (5, 128), (4, 130), (7, 300), (33, 1000), (9, 4160), (64, 4096)]


def _weights(M, N, seed, f16):
    W = synth.uniform(seed, 1, 0, M * N, -1.0, 1.0).reshape(M, N)
    # a zero group, a row with one huge value, exact ties on a coarse grid
    if N >= 256:
        W[0, 128:256] = 0.0
    if M > 2:
        W[2, :] = np.round(W[2, :] * 14) / 14
    if M > 3:
        W[3, N // 2] = 30.0
    W = W.astype(np.float32)
    if f16:
        return W.astype(np.float16)
    return W


def _gpu(dtype, W):
    t = torch.from_numpy(np.ascontiguousarray(W)).cuda()
    err = torch.zeros(1, dtype=torch.float64, device="cuda")
    A, S = mbg.quantize(t, dtype, sq_err=err)
    torch.cuda.synchronize()
    return A.cpu().numpy(), S.cpu().numpy().view(np.uint16), float(err.item())


@pytest.mark.parametrize("f16", (False, True), ids=("fp32_in", "fp16_in"))
@pytest.mark.parametrize("dtype", QDTYPES)
def test_codes_and_scales_bit_exact(dtype, f16):
    orc = oracle.load()
    for (M, N) in SHAPES:
        W = _weights(M, N, 100 + M + N, f16)
        A, S, e = _gpu(dtype, W)
        Wo = W.view(np.uint16) if f16 else W
        A_ref, S_ref, e_ref = orc.quantize(dtype, Wo, M, N)
        assert np.array_equal(A, A_ref.reshape(A.shape)), (dtype, M, N)
        assert np.array_equal(S.reshape(S_ref.shape), S_ref), (dtype, M, N)
        # a sum of M*N non-negative doubles in another order: |difference| <= M*N*2^-52 * sum
        assert abs(e - e_ref) <= M * N * 2.0 ** -52 * e_ref, (dtype, M, N, e, e_ref)


def test_special_values():
    orc = oracle.load()
    M, N = 4, 256
    W = _weights(M, N, 7, False)
    W[0, 5] = np.inf
    W[1, 200] = -np.inf
    W[2, 17] = np.nan
    W[3, :] = 1e-30  # scale underflows to zero in binary16
    for dtype in QDTYPES:
        t = torch.from_numpy(W).cuda()
        A, S = mbg.quantize(t, dtype)
        torch.cuda.synchronize()
        A_ref, S_ref, _ = orc.quantize(dtype, W, M, N)
        assert np.array_equal(A.cpu().numpy(), A_ref), dtype
        assert np.array_equal(S.cpu().numpy().view(np.uint16).reshape(S_ref.shape), S_ref), dtype


def test_page_rmse_and_round_trip_at_decode_size():
    g = json.load(open(os.path.join(GOLDEN, "quantization_rmse.json")))
    M, N = 4096, 14336
    W = torch.from_numpy(synth.uniform(31, 1, 0, M * N, -1.0, 1.0).astype(np.float32).reshape(M, N)).cuda()
    rmse = {}
    out = {}
    for dtype in ("q8row", "q4"):
        err = torch.zeros(1, dtype=torch.float64, device="cuda")
        out[dtype] = mbg.quantize(W, dtype, sq_err=err)
        torch.cuda.synchronize()
        rmse[dtype] = (err.item() / (M * N)) ** 0.5
    assert float(f"{rmse['q8row']:.1e}") == g["q8_per_row_rmse"]
    assert float(f"{rmse['q4']:.1e}") == g["q4_group128_rmse"]
    # sampled rows bit-exact against the oracle, then the GEMV on the result
    rows = [0, 1, 777, 2048, M - 1]
    orc = oracle.load()
    Wr = W[rows].cpu().numpy()
    for dtype in ("q8row", "q4"):
        A, S = out[dtype]
        A_ref, S_ref, _ = orc.quantize(dtype, Wr, len(rows), N)
        assert np.array_equal(A[rows].cpu().numpy(), A_ref), dtype
        assert np.array_equal(S[rows].cpu().numpy().view(np.uint16).reshape(S_ref.shape), S_ref), dtype
    x_bits = synth.to_f16_bits(synth.normal(32, 1, 0, N, 1.0))
    x = torch.from_numpy(x_bits.view(np.float16)).cuda()
    A, S = out["q4"]
    y = mbg.gemv_q4(A, x, S)
    torch.cuda.synchronize()
    inp = {"A": A[rows].cpu().numpy(), "x": x_bits, "scales": S[rows].cpu().numpy().view(np.uint16)}
    y_ref, den = reference("q4", inp, len(rows), N)
    assert_close("q4", y.cpu().numpy()[rows], y_ref, den, "q4 after quantize")
    A, S = out["q8row"]
    y = mbg.gemv_q8_rowscale(A, x, S)
    torch.cuda.synchronize()
    inp = {"A": A[rows].cpu().numpy(), "x": x_bits, "scales": S[rows].cpu().numpy().view(np.uint16).reshape(-1, 1)}
    y_ref, den = reference("q8row", inp, len(rows), N)
    assert_close("q8row", y.cpu().numpy()[rows], y_ref, den, "q8row after quantize")


@pytest.mark.parametrize("f16", (False, True), ids=("fp32_in", "fp16_in"))
@pytest.mark.parametrize("dtype", QDTYPES)
def test_layout_paths_agree(dtype, f16):
    """The same weights through the 16-byte path (aligned, whole groups) and through the general
    path (the weights 2 or 4 bytes past a 16-byte boundary), each with and without the error sum:
    codes and scales bit-exact with the oracle, the error sum within the reordering bound.  FP32
    input adds a row of values around 1e9, whose residual w - s q is not exact in FP32 (the scale
    saturates at 65504), so the error sum takes its double-precision branch."""
    M, N = 48, 4096
    W = _weights(M, N, 211, f16)
    if not f16:
        W[5, :] *= np.float32(1e9)
    orc = oracle.load()
    A_ref, S_ref, e_ref = orc.quantize(dtype, W.view(np.uint16) if f16 else W, M, N)
    t = torch.from_numpy(np.ascontiguousarray(W)).cuda()
    big = torch.empty(M * N + 8, dtype=t.dtype, device="cuda")
    off = big[1:1 + M * N].view(M, N)
    off.copy_(t)
    assert off.data_ptr() % 16 != 0
    for src in (t, off):
        for want_err in (True, False):
            err = torch.zeros(1, dtype=torch.float64, device="cuda") if want_err else None
            A, S = mbg.quantize(src, dtype, sq_err=err)
            torch.cuda.synchronize()
            assert np.array_equal(A.cpu().numpy(), A_ref.reshape(A.shape)), (dtype, src is t, want_err)
            assert np.array_equal(S.cpu().numpy().view(np.uint16).reshape(S_ref.shape), S_ref)
            if want_err:
                e = float(err.item())
                assert abs(e - e_ref) <= M * N * 2.0 ** -52 * e_ref, (dtype, src is t, e, e_ref)
