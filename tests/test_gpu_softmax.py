"""GPU parity of the row softmax against the oracle, through the C ABI.

Metric ("membound", section "Bonus kernel: online softmax"): relative error
against max(y_ref, 1e-4), so that binary16 subnormal outputs do not raise
false alarms.  Tolerance 1e-3: twice the binary16 rounding of the output
(2^-11 = 4.9e-4); the FP32 arithmetic adds about 1e-6.
"""

import numpy as np
import pytest

import memory_bound_gemv_gb300 as mbg
import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TOL = 1e-3


def _err(y_gpu_bits, y_ref):
    y = np.asarray(y_gpu_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    return float(np.max(np.abs(y - y_ref) / np.maximum(y_ref, 1e-4)))


def _case(M, N, seed, sigma=2.0):
    w = synth.Workload(f"sm_{M}x{N}", "f16", M, N, seed, ("normal", sigma), ("normal", sigma))
    return synth.weight_rows(w, 0, M)


def _run(bits, variant=None, inplace=False):
    x = torch.from_numpy(bits.view(np.float16)).cuda()
    if inplace:
        mbg.gemv_softmax_f16(x, y=x, variant=variant)
        y = x
    else:
        y = mbg.gemv_softmax_f16(x, variant=variant)
    torch.cuda.synchronize()
    return y.cpu().numpy().view(np.uint16)


SHAPES = [(1, 1), (3, 7), (5, 8), (2, 64), (7, 1000), (9, 1024), (4, 1032), (3, 4096),
          (2, 8192), (2, 9000), (2, 16384), (2, 24576), (2, 32768), (1, 65536), (1, 131072),
          (1, 131080)]


def test_every_variant_against_the_oracle():
    orc = oracle.load()
    nvar = len(mbg.softmax_variants())
    checked = 0
    for (M, N) in SHAPES:
        bits = _case(M, N, 7 + N)
        ref = orc.softmax(bits, M, N, threads=8)
        assert _err(_run(bits), ref) <= TOL, (M, N, "auto")
        for v in range(nvar):
            try:
                y = _run(bits, variant=v)
            except mbg.GemvError as e:
                assert e.status == mbg.ERR_UNSUPPORTED
                continue
            assert _err(y, ref) <= TOL, (M, N, mbg.softmax_variants()[v])
            checked += 1
    assert checked > len(SHAPES)


@pytest.mark.parametrize("name", sorted(synth.SOFTMAX_WORKLOADS))
def test_softmax_workloads_sampled_rows(name):
    w = synth.SOFTMAX_WORKLOADS[name]
    bits = synth.weight_rows(w, 0, w.M)
    y = _run(bits)
    rows = sorted(set([0, w.M // 2, w.M - 1]) | set(np.random.default_rng(w.seed).integers(0, w.M, 13).tolist()))
    ref = oracle.load().softmax(bits, w.M, w.N, rows=rows, threads=8)
    assert _err(y[rows], ref) <= TOL
    # every row sums to one within the binary16 rounding of its entries
    sums = y.view(np.float16).astype(np.float64).sum(axis=1)
    assert np.all(np.abs(sums - 1.0) < 1e-2)


def test_in_place_and_large_values():
    orc = oracle.load()
    for (M, N) in ((4, 8192), (3, 1000), (2, 65536)):
        bits = _case(M, N, 31, sigma=2.0)
        ref = orc.softmax(bits, M, N)
        assert _err(_run(bits, inplace=True), ref) <= TOL
    big = synth.to_f16_bits(np.array([[65504.0, 65472.0, 60000.0, -65504.0] * 256]))
    ref = orc.softmax(big, 1, 1024)
    assert _err(_run(big), ref) <= TOL


def test_degenerate_rows():
    # one column: y = 1; a constant row: 1/N
    assert np.all(_run(synth.to_f16_bits(np.array([[3.0], [-2.0]]))).view(np.float16) == 1.0)
    bits = synth.to_f16_bits(np.full((2, 4096), 1.5))
    y = _run(bits).view(np.float16).astype(np.float64)
    assert np.all(np.abs(y - 1.0 / 4096) <= 1.0 / 4096 * 2.0 ** -11)


def test_copy_probe_copies():
    src = torch.randint(-2 ** 31, 2 ** 31 - 1, ((4 << 20) // 4,), dtype=torch.int32, device="cuda")
    for v in range(len(mbg.copy_probe_variants())):
        dst = torch.zeros_like(src)
        mbg.gemv_probe_copy(src, dst, v)
        torch.cuda.synchronize()
        assert torch.equal(src, dst), mbg.copy_probe_variants()[v]
