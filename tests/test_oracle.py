"""Pins for the CPU oracle (no GPU).

Each ``pin_*`` function checks the oracle against something other than
itself: values the pages print (``tests/golden``), closed forms, exact
rational brute force, numpy's own binary16 decoding, and hand-built int4
byte tables.  ``test_mutants_are_caught`` builds the oracle with one planted
mistake at a time and requires at least one pin to fail for each.
"""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ONE_F16 = 0x3C00


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f16_value(bits):
    """Independent FP16 decode (numpy's), used only as a check on the oracle."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def _scales_ones(M, N):
    return np.full((M, synth.n_groups(N)), ONE_F16, dtype=np.uint16)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_dec16_all_patterns(orc):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = orc.dec16(bits)
    ref = _f16_value(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    named = {0x3C00: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24,
             0x0400: 2.0 ** -14, 0x7BFF: 65504.0, 0x7C00: np.inf, 0xFC00: -np.inf}
    for b, v in named.items():
        assert orc.dec16([b])[0] == v, hex(b)


def pin_rowmajor_worked_example(orc):
    g = _golden("rowmajor_worked_example.json")
    M, N = g["M"], g["N"]
    flat = np.arange(M * N)
    assert flat.reshape(M, N)[g["probe_row"], g["probe_col"]] == flat[g["probe_offset"]]
    expect = np.array([flat[i * N + g["probe_col"]] for i in range(M)], dtype=np.float64)
    assert list(expect) == [2.0, 6.0, 10.0]
    e = np.zeros(N)
    e[g["probe_col"]] = 1.0
    cases = {
        "f32": (flat.astype(np.float32), e.astype(np.float32), None),
        "f16": (synth.to_f16_bits(flat.astype(np.float64)), synth.to_f16_bits(e), None),
        "q8": (flat.astype(np.int8), synth.to_f16_bits(e), _scales_ones(M, N)),
    }
    for dt, (A, x, s) in cases.items():
        y, den = orc.gemv(dt, A.reshape(M, N), x, M, N, scales=s)
        assert np.array_equal(y, expect), dt
        assert y[g["probe_row"]] == flat[g["probe_offset"]], dt
        assert np.array_equal(den, np.abs(expect)), dt


def pin_identity(orc):
    for n in (1, 6, 130):
        eye = np.eye(n)
        xf = synth.uniform(7, 2, 0, n, -1, 1).astype(np.float32)
        y, _ = orc.gemv("f32", eye.astype(np.float32), xf, n, n)
        assert np.array_equal(y, xf.astype(np.float64))
        xb = synth.to_f16_bits(synth.normal(7, 2, 0, n, 1.0))
        xv = _f16_value(xb)
        y, _ = orc.gemv("f16", synth.to_f16_bits(eye), xb, n, n)
        assert np.array_equal(y, xv)
        y, _ = orc.gemv("q8", eye.astype(np.int8), xb, n, n, scales=_scales_ones(n, n))
        assert np.array_equal(y, xv)
        if n % 2 == 0:
            Aq = synth.pack_int4(eye.astype(np.int64))
            y, _ = orc.gemv("q4", Aq, xb, n, n, scales=_scales_ones(n, n))
            assert np.array_equal(y, xv)


def _grouped_quant_case(dtype, M=3, N=300):
    """Random codes and per-(row, group) power-of-two scales, all exact in FP16."""
    lo, hi = (-127, 127) if dtype == "q8" else (-8, 7)
    q = synth.integers(11, 1, 0, M * N, lo, hi).reshape(M, N)
    g = synth.n_groups(N)
    expo = np.arange(M * g).reshape(M, g) - 6
    s_val = np.ldexp(1.0, expo)
    s_bits = synth.to_f16_bits(s_val)
    A = q.astype(np.int8) if dtype == "q8" else synth.pack_int4(q)
    return q, A, s_val, s_bits


def pin_unit_vectors(orc):
    M, N = 3, 300
    for dt in ("f32", "f16"):
        w = synth.random_case(dt, M, N, 5)
        A = synth.weight_rows(w, 0, M)
        Av = A.astype(np.float64) if dt == "f32" else _f16_value(A)
        for k in (0, 1, 127, 128, 299):
            e = np.zeros(N)
            e[k] = 1.0
            x = e.astype(np.float32) if dt == "f32" else synth.to_f16_bits(e)
            y, _ = orc.gemv(dt, A, x, M, N)
            assert np.array_equal(y, Av[:, k]), (dt, k)
    for dt in ("q8", "q4"):
        q, A, s_val, s_bits = _grouped_quant_case(dt, M, N)
        expect_w = s_val[:, np.arange(N) // 128] * q
        assert np.array_equal(orc.dequant(dt, A, s_bits, M, N), expect_w), dt
        for k in (0, 1, 63, 64, 127, 128, 255, 256, 299):
            e = np.zeros(N)
            e[k] = 1.0
            y, _ = orc.gemv(dt, A, synth.to_f16_bits(e), M, N, scales=s_bits)
            assert np.array_equal(y, expect_w[:, k]), (dt, k)


def pin_format_options_unit_vectors(orc):
    # f16 weights with FP32 x: e_k picks column k exactly, and an FP32 x that
    # is not a binary16 value (1 + 2^-20) scales it exactly
    M, N = 4, 200
    w = synth.random_case("f16x32", M, N, 8)
    A = synth.weight_rows(w, 0, M)
    Av = _f16_value(A)
    for k in (0, 1, 100, 199):
        e = np.zeros(N, dtype=np.float32)
        e[k] = 1.0 + 2.0 ** -20
        y, _ = orc.gemv("f16x32", A, e, M, N)
        assert np.array_equal(y, Av[:, k] * (1.0 + 2.0 ** -20)), k
    # one scale per row: row i's weights are s_i * q, whatever the column
    q = synth.integers(9, 1, 0, M * N, -127, 127).reshape(M, N)
    s_val = np.ldexp(1.0, np.arange(M) - 3)
    for k in (0, 127, 128, 199):
        e = np.zeros(N)
        e[k] = 1.0
        y, _ = orc.gemv("q8row", q.astype(np.int8), synth.to_f16_bits(e), M, N,
                        scales=synth.to_f16_bits(s_val))
        assert np.array_equal(y, s_val * q[:, k]), k


def pin_int4_byte_table(orc):
    # one row, hand-built bytes: low nibble = even column, two's complement
    row = np.array([[0x21, 0x43, 0x8F, 0x7E, 0x09]], dtype=np.uint8)
    codes = [1, 2, 3, 4, -1, -8, -2, 7, -7, 0]
    N = 10
    s = _scales_ones(1, N)
    W = orc.dequant("q4", row, s, 1, N)
    assert list(W[0]) == codes
    for k in range(N):
        e = np.zeros(N)
        e[k] = 1.0
        y, _ = orc.gemv("q4", row, synth.to_f16_bits(e), 1, N, scales=s)
        assert y[0] == codes[k], k


def pin_all_ones(orc):
    for (M, N) in ((1, 1), (4, 37), (3, 258)):
        x = synth.integers(13, 2, 0, N, -4, 4).astype(np.float64)
        total = float(x.sum())
        ones = np.ones((M, N))
        y, den = orc.gemv("f32", ones.astype(np.float32), x.astype(np.float32), M, N)
        assert np.all(y == total) and np.all(den == np.abs(x).sum())
        xb = synth.to_f16_bits(x)
        y, _ = orc.gemv("f16", synth.to_f16_bits(ones), xb, M, N)
        assert np.all(y == total)
        y, _ = orc.gemv("q8", ones.astype(np.int8), xb, M, N, scales=_scales_ones(M, N))
        assert np.all(y == total)
        if N % 2 == 0:
            y, _ = orc.gemv("q4", synth.pack_int4(ones.astype(np.int64)), xb, M, N,
                            scales=_scales_ones(M, N))
            assert np.all(y == total)


def _exact_weights(dt, A, s_bits, M, N):
    """Exact rational weights, decoded independently of the oracle."""
    W = [[None] * N for _ in range(M)]
    for i in range(M):
        for j in range(N):
            if dt == "f32":
                W[i][j] = Fraction(float(A[i, j]))
            elif dt in ("f16", "f16x32"):
                W[i][j] = Fraction(float(np.uint16(A[i, j]).view(np.float16)))
            else:
                col = 0 if dt == "q8row" else j // 128
                sc = Fraction(float(np.uint16(s_bits[i, col]).view(np.float16)))
                if dt in ("q8", "q8row"):
                    code = int(A[i, j])
                else:
                    byte = int(A[i, j // 2])
                    nib = (byte >> (4 * (j % 2))) & 0xF
                    code = nib - 16 if nib > 7 else nib
                W[i][j] = sc * code
    return W


def pin_bruteforce_exact(orc):
    shapes = [(1, 1), (2, 3), (4, 8), (9, 33), (5, 130), (3, 257), (2, 64)]
    for dt in ("f32", "f16", "q8", "q4", "f16x32", "q8row"):
        for (M, N) in shapes:
            if dt == "q4" and N % 2:
                continue
            w = synth.random_case(dt, M, N, 1000 + M * 7 + N)
            inp = synth.make(w)
            A, x, s = inp["A"], inp["x"], inp.get("scales")
            W = _exact_weights(dt, A, s, M, N)
            xv = [Fraction(float(v)) for v in (x if x.dtype == np.float32 else x.view(np.float16))]
            y, den = orc.gemv(dt, A, x, M, N, scales=s)
            for i in range(M):
                ex = sum((W[i][j] * xv[j] for j in range(N)), Fraction(0))
                ed = sum((abs(W[i][j]) * abs(xv[j]) for j in range(N)), Fraction(0))
                # double accumulation over N terms: |error| <= N * 2^-53 * den
                bound = float(ed) * N * 2.0 ** -52
                assert abs(y[i] - float(ex)) <= bound, (dt, M, N, i)
                assert abs(den[i] - float(ed)) <= bound, (dt, M, N, i)


def pin_counts(orc):
    M = N = 1024
    assert orc.flops(M, N) == 2 * M * N - M == 2096128
    assert orc.bytes("f32", M, N) == 4 * (M * N + N + M) == 4202496
    g = _golden("published_bandwidth.json")
    # both printed numbers are rounded (ms to 4 places, GB/s to 1): the byte
    # count must make the two intervals overlap
    b = orc.bytes("f16", g["fp16_M"], g["fp16_N"])
    lo = b / ((g["fp16_ms"] + 0.00005) * 1e-3) / 1e9
    hi = b / ((g["fp16_ms"] - 0.00005) * 1e-3) / 1e9
    assert lo <= g["fp16_gbs"] + 0.05 and hi >= g["fp16_gbs"] - 0.05
    # FP16 : INT4 byte ratio at the decode shape approaches 2 / (0.5 + 2/128)
    ratio = orc.bytes("f16", 4096, 14336) / orc.bytes("q4", 4096, 14336)
    assert abs(ratio - g["int4_cap_printed"]) < 0.01
    assert int(2 / (0.5 + 2 / 128) * 100) / 100 == g["int4_cap_printed"]
    assert orc.bytes("q8", 4096, 14336) == 4096 * 14336 + 2 * 4096 * 112 + 2 * 14336 + 4 * 4096
    assert orc.flops(0, 5) == 0 and orc.flops(5, 0) == 0
    # FP32 x: 4 bytes per element of x; one scale per row: 2 bytes per row
    assert orc.bytes("f16x32", 4096, 14336) == 2 * 4096 * 14336 + 4 * 14336 + 4 * 4096
    assert orc.bytes("q8row", 4096, 14336) == 4096 * 14336 + 2 * 4096 + 2 * 14336 + 4 * 4096


def _f16(vals):
    return synth.to_f16_bits(np.asarray(vals, dtype=np.float64))


def pin_softmax_closed_forms(orc):
    import math
    # a constant row gives 1/N everywhere
    for N in (1, 3, 1000):
        y = orc.softmax(_f16(np.full((2, N), 0.75)), 2, N)
        assert np.allclose(y, 1.0 / N, rtol=1e-14, atol=0)
    # two elements: y0 = 1 / (1 + e^(x1 - x0))
    for a, b in ((0.0, 1.0), (-3.5, 2.25), (7.0, 7.0)):
        y = orc.softmax(_f16([[a, b]]), 1, 2)[0]
        assert abs(y[0] - 1.0 / (1.0 + math.exp(b - a))) < 1e-15
        assert abs(y[1] - 1.0 / (1.0 + math.exp(a - b))) < 1e-15
    # large inputs: the maximum is subtracted, so nothing overflows
    y = orc.softmax(_f16([[60000.0, 60000.0, 59968.0]]), 1, 3)[0]
    assert np.all(np.isfinite(y)) and abs(y[0] - y[1]) == 0.0
    # shifting a row by a constant leaves the result unchanged (integer inputs stay exact)
    xi = synth.integers(3, 2, 0, 64, -8, 8).astype(np.float64)
    y1 = orc.softmax(_f16([xi]), 1, 64)[0]
    y2 = orc.softmax(_f16([xi + 5.0]), 1, 64)[0]
    assert np.allclose(y1, y2, rtol=1e-14, atol=0)


def pin_softmax_sums_and_brute_force(orc):
    import math
    w = synth.random_case("f16", 5, 37, 91)
    bits = synth.weight_rows(synth.Workload("sm", "f16", 5, 37, 91, ("normal", 2.0), ("normal", 2.0)), 0, 5)
    y = orc.softmax(bits, 5, 37)
    assert np.allclose(y.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    vals = bits.view(np.float16).astype(np.float64)
    for i in range(5):
        m = max(vals[i])
        e = [math.exp(v - m) for v in vals[i]]
        s = math.fsum(e)
        for j in range(37):
            assert abs(y[i, j] - e[j] / s) <= 1e-15 * max(1.0, e[j] / s)
    del w


# ---------------------------------------------------------------------------
# quantiser pins
# ---------------------------------------------------------------------------

def _f32(v):
    return np.asarray(v, dtype=np.float32)


def pin_enc16_against_numpy(orc):
    # every binary16 value, the midpoints between neighbours (ties), one
    # float32 ulp either side of each midpoint, the overflow edge and a random
    # spread from the subnormal range up
    h = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    vals = h.view(np.float16).astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2.0
    m32 = _f32(mids)
    around = np.concatenate([m32, np.nextafter(m32, np.float32(np.inf)),
                             np.nextafter(m32, np.float32(0))])
    rnd = _f32(np.ldexp(synth.uniform(4, 1, 0, 20000, 1.0, 2.0), synth.integers(4, 2, 0, 20000, -30, 16)))
    edge = _f32([65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                 2.0 ** -26, 0.0, -0.0, np.inf, -np.inf])
    f = np.concatenate([_f32(vals), around, rnd, edge])
    f = np.concatenate([f, -f])
    ours = orc.enc16(f)
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    assert orc.enc16(_f32([np.nan]))[0] & 0x7FFF > 0x7C00


def pin_quantize_page_rmse(orc):
    g = _golden("quantization_rmse.json")
    M, N = 256, 4096
    W = _f32(synth.uniform(21, 1, 0, M * N, -1.0, 1.0).reshape(M, N))
    _, _, e8 = orc.quantize("q8row", W, M, N)
    _, _, e4 = orc.quantize("q4", W, M, N)
    r8, r4 = (e8 / W.size) ** 0.5, (e4 / W.size) ** 0.5
    assert float(f"{r8:.1e}") == g["q8_per_row_rmse"], r8
    assert float(f"{r4:.1e}") == g["q4_group128_rmse"], r4


def pin_quantize_closed_forms(orc):
    # a group on the code grid: w = k * 0.25 with max 7 * 0.25 -> s = 0.25, codes k, no error
    k = np.arange(-7, 8)
    row = np.concatenate([k, np.zeros(128 - k.size)]) * 0.25
    A, S, e = orc.quantize("q4", _f32([row]), 1, 128)
    assert S[0, 0] == 0x3400 and e == 0.0  # binary16 0.25
    W = orc.dequant("q4", A, S, 1, 128)
    assert np.array_equal(W[0], row)
    # ties go to the even code: s = 0.5 (max 3.5 = 7 s); 0.25 -> 0, 0.75 -> 2,
    # 1.25 -> 2, -0.75 -> -2, -1.75 -> -4
    row = np.zeros(128)
    row[:6] = [3.5, 0.25, 0.75, 1.25, -0.75, -1.75]
    A, S, _ = orc.quantize("q4", _f32([row]), 1, 128)
    assert S[0, 0] == 0x3800
    assert list(orc.dequant("q4", A, S, 1, 128)[0, :6] / 0.5) == [7, 0, 2, 2, -2, -4]
    # an all-zero group: scale 0, codes 0; INT8 per row: the largest magnitude maps to +-127
    W = _f32(synth.uniform(22, 1, 0, 3 * 300, -2.0, 2.0).reshape(3, 300))
    W[1, 128:256] = 0.0
    A, S, _ = orc.quantize("q8", W, 3, 300)
    assert S[1, 1] == 0 and not np.any(A[1, 128:256])
    A, S, _ = orc.quantize("q8row", W, 3, 300)
    for i in range(3):
        assert abs(int(A[i, np.argmax(np.abs(W[i]))])) == 127


def pin_quantize_invariants(orc):
    M, N = 5, 1000
    W = _f32(synth.normal(23, 1, 0, M * N, 0.05).reshape(M, N))
    for dt, qmax in (("q8", 127), ("q8row", 127), ("q4", 7)):
        A, S, e = orc.quantize(dt, W, M, N)
        width = N if dt == "q8row" else 128
        # scales: binary16 of (FP32 max|w| / qmax), by numpy's own arithmetic
        amax = np.array([[np.abs(W[i, g * width:(g + 1) * width]).max() for g in range(S.shape[1])]
                         for i in range(M)], dtype=np.float32)
        assert np.array_equal(S, (amax / np.float32(qmax)).astype(np.float16).view(np.uint16)), dt
        # every weight within half a step of its reconstruction, codes in range
        s = S.view(np.float16).astype(np.float64)
        sc = s[:, np.arange(N) // width]
        if dt == "q4":
            Wq = orc.dequant("q4", A, S, M, N)
        else:
            Wq = A.astype(np.float64) * sc
        assert np.all(np.abs(W - Wq) <= sc / 2 * (1 + 2.0 ** -10)), dt
        codes = np.rint(Wq / np.where(sc == 0, 1, sc))
        assert np.abs(codes).max() == qmax, dt
        assert abs(e - ((W.astype(np.float64) - Wq) ** 2).sum()) <= 1e-12 * e, dt
        # scaling a row by 2^3 scales its scales by 2^3 and keeps the codes
        W2 = W.copy()
        W2[2] *= 8.0
        A2, S2, _ = orc.quantize(dt, W2, M, N)
        assert np.array_equal(A2, A), dt
        assert np.array_equal(S2[2].view(np.float16).astype(np.float64),
                              S[2].view(np.float16).astype(np.float64) * 8.0), dt
        # binary16 weights give the same result as their exact FP32 values
        Wh = W.astype(np.float16)
        Ah, Sh, eh = orc.quantize(dt, Wh.view(np.uint16), M, N)
        Af, Sf, ef = orc.quantize(dt, Wh.astype(np.float32), M, N)
        assert np.array_equal(Ah, Af) and np.array_equal(Sh, Sf) and eh == ef, dt


PINS = [pin_dec16_all_patterns, pin_rowmajor_worked_example, pin_identity, pin_unit_vectors,
        pin_format_options_unit_vectors, pin_int4_byte_table, pin_all_ones, pin_bruteforce_exact, pin_counts,
        pin_softmax_closed_forms, pin_softmax_sums_and_brute_force,
        pin_enc16_against_numpy, pin_quantize_page_rmse, pin_quantize_closed_forms,
        pin_quantize_invariants]


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


def test_threads_do_not_change_results(orc):
    w = synth.random_case("f16", 257, 1000, 77)
    inp = synth.make(w)
    y1, d1 = orc.gemv("f16", inp["A"], inp["x"], w.M, w.N, threads=1)
    y4, d4 = orc.gemv("f16", inp["A"], inp["x"], w.M, w.N, threads=4)
    assert y1.tobytes() == y4.tobytes() and d1.tobytes() == d4.tobytes()


def test_row_subset_matches_full(orc):
    w = synth.random_case("q4", 50, 260, 78)
    inp = synth.make(w)
    y, d = orc.gemv("q4", inp["A"], inp["x"], w.M, w.N, scales=inp["scales"])
    rows = [49, 0, 17, 17, 3]
    ys, ds = orc.gemv("q4", inp["A"], inp["x"], w.M, w.N, scales=inp["scales"], rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(ds, d[rows])


def test_zero_rows_and_empty(orc):
    A = np.zeros((2, 5), dtype=np.float32)
    A[1, 2] = 3.0
    y, d = orc.gemv("f32", A, np.ones(5, dtype=np.float32), 2, 5)
    assert y[0] == 0.0 and d[0] == 0.0 and y[1] == 3.0
    y, d = orc.gemv("f32", np.zeros((3, 0), np.float32), np.zeros(0, np.float32), 3, 0)
    assert np.array_equal(y, np.zeros(3)) and np.array_equal(d, np.zeros(3))
    y, d = orc.gemv("f16", np.zeros((0, 4), np.uint16), np.zeros(4, np.uint16), 0, 4)
    assert y.size == 0


def test_rejects_bad_arguments(orc):
    with pytest.raises(ValueError):
        orc.gemv("q4", np.zeros((1, 2), np.uint8), np.zeros(3, np.uint16), 1, 3,
                 scales=np.zeros((1, 1), np.uint16))
    with pytest.raises(ValueError):
        orc.gemv("f32", np.zeros((2, 2), np.float32), np.zeros(2, np.float32), 2, 2, rows=[2])


def test_error_metric():
    y_ref = np.array([1.0, 0.0, -2.0])
    den = np.array([2.0, 0.0, 4.0])
    assert oracle.max_normalised_error([1.0, 0.0, -2.0], y_ref, den) == 0.0
    assert oracle.max_normalised_error([1.5, 0.0, -2.0], y_ref, den) == 0.25
    assert oracle.max_normalised_error([1.0, 1e-30, -2.0], y_ref, den) == np.inf
    assert oracle.max_normalised_error([np.nan, 0.0, -2.0], y_ref, den) == np.inf


MUTANTS = {1: "int4 nibble order swapped", 2: "int4 read as offset-8",
           3: "scale group width 64", 4: "A read column-major",
           5: "binary16 subnormals decoded as normals", 6: "last column dropped",
           7: "scale row pitch floor(N/128)", 8: "softmax without the maximum subtracted",
           9: "softmax sum missing its last term", 10: "softmax normalised by N",
           11: "per-row scale taken from row 0", 12: "FP32 x of f16 weights read as binary16",
           13: "INT4 scale max/8", 14: "codes truncated, not rounded",
           15: "quantisation groups of 64 columns", 16: "binary16 encoder truncates"}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[MUTANTS[k] for k in sorted(MUTANTS)])
def test_mutants_are_caught(tmp_path, mutant):
    bad = oracle.Oracle(oracle.build(mutant, build_dir=str(tmp_path)))
    assert bad.mutant == mutant
    failed = []
    for pin in PINS:
        try:
            pin(bad)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {mutant} ({MUTANTS[mutant]})"
