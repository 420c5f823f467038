"""GPU parity: every kernel variant against the CPU oracle, through the C ABI.

Inputs are the seeded synthetic workloads; the bar is the maximum over rows
of |y_gpu - y_ref| / sum_j |w_ij||x_j|: 1e-5 for FP32, 2e-3 for FP16 and the
quantised types (rows whose normaliser is 0 must come out exactly 0).
"""

import numpy as np
import pytest

import memory_bound_gemv_gb300 as mbg
import oracle
import synth
from gpu_util import TOL, assert_close, reference, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

DTYPES = ("f32", "f16", "q8", "q4", "f16x32", "q8row")

# (M, N): several tiles, ragged tails, short rows for the multi-row variants,
# and row pitches that are / are not multiples of 16 bytes.
SHAPES = [(1, 1), (1, 8), (2, 3), (3, 7), (5, 32), (7, 33), (9, 64), (31, 65), (32, 126),
          (33, 128), (63, 130), (64, 254), (65, 256), (127, 258), (129, 512), (130, 1000),
          (257, 1024), (64, 2056), (33, 4096), (300, 4160), (17, 8200), (37, 14336)]


def _shapes(dtype):
    return [(M, N) for (M, N) in SHAPES if not (dtype == "q4" and N % 2)]


@pytest.mark.parametrize("dtype", DTYPES)
def test_every_variant_small_shapes(dtype):
    nvar = len(mbg.variants(dtype))
    checked = 0
    for (M, N) in _shapes(dtype):
        w = synth.random_case(dtype, M, N, seed=M * 1000 + N)
        inp = synth.make(w)
        y_ref, den = reference(dtype, inp, M, N)
        t = upload(dtype, inp)
        y = mbg.gemv(dtype, t["A"], t["x"], t.get("scales"))
        torch.cuda.synchronize()
        assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} auto {M}x{N}")
        for v in range(nvar):
            try:
                y = mbg.gemv_run_variant(dtype, v, t["A"], t["x"], t.get("scales"))
            except mbg.GemvError as e:
                assert e.status == mbg.ERR_UNSUPPORTED
                continue
            torch.cuda.synchronize()
            assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} variant {v} {M}x{N}")
            checked += 1
    assert mbg.gemv_get_device_error() == mbg.OK
    assert checked > 0


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_workloads_full_size(name):
    """The named workloads at full size, every row against the oracle, for the
    automatic choice and every row-tile, bulk-pipeline, row-band and
    warp-per-row variant that fits the workload."""
    w = synth.WORKLOADS[name]
    inp = synth.make(w)
    t = upload(w.dtype, inp)
    y_ref, den = reference(w.dtype, inp, w.M, w.N, threads=16)
    y = mbg.gemv(w.dtype, t["A"], t["x"], t.get("scales"))
    torch.cuda.synchronize()
    y_np = y.cpu().numpy()
    assert y_np.shape == (w.M,)
    assert_close(w.dtype, y_np, y_ref, den, f"{name} auto")
    checked = 0
    for v in mbg.variants(w.dtype):
        if v["kind"] == "elem" or (v["kind"] == "vec" and v["threads_per_row"] != 32):
            continue
        try:
            y2 = mbg.gemv_run_variant(w.dtype, v["id"], t["A"], t["x"], t.get("scales"))
        except mbg.GemvError as e:
            assert e.status == mbg.ERR_UNSUPPORTED
            continue
        torch.cuda.synchronize()
        assert_close(w.dtype, y2.cpu().numpy(), y_ref, den, f"{name} {v['name']}")
        checked += 1
    assert checked > 0
    # outputs are finite everywhere
    assert np.all(np.isfinite(y_np))
    assert mbg.gemv_get_device_error() == mbg.OK


@pytest.mark.parametrize("N", (4096, 14336))
def test_int8_code_minus_128(N):
    """INT8 codes span the whole byte, -128 included (the header admits it;
    the workload recipe draws only -127..127)."""
    M = 64
    A = synth.integers(77, 1, 0, M * N, -128, 127).astype(np.int8).reshape(M, N)
    A[::7, ::5] = -128
    scales = synth.to_f16_bits(synth.uniform(77, 3, 0, M * synth.n_groups(N), 0.001, 0.01)).reshape(M, -1)
    x = synth.to_f16_bits(synth.normal(77, 2, 0, N, 1.0))
    inp = {"A": A, "x": x, "scales": scales}
    y_ref, den = reference("q8", inp, M, N)
    t = upload("q8", inp)
    checked = 0
    for v in mbg.variants("q8"):
        try:
            y = mbg.gemv_run_variant("q8", v["id"], t["A"], t["x"], t["scales"])
        except mbg.GemvError as e:
            assert e.status == mbg.ERR_UNSUPPORTED
            continue
        torch.cuda.synchronize()
        assert_close("q8", y.cpu().numpy(), y_ref, den, f"q8 -128 {v['name']}")
        checked += 1
    assert checked > 5
    # -128 on the diagonal with unit scales: y = -128 x exactly (exact in FP32)
    n = N
    eye = np.zeros((n // 8, n), dtype=np.int8)
    eye[np.arange(n // 8), np.arange(n // 8) * 8] = -128
    ones = np.full((n // 8, synth.n_groups(n)), 0x3C00, dtype=np.uint16)
    t2 = upload("q8", {"A": eye, "x": x, "scales": ones})
    expect = -128.0 * x.view(np.float16).astype(np.float64)[::8][: n // 8]
    for v in mbg.variants("q8"):
        try:
            y = mbg.gemv_run_variant("q8", v["id"], t2["A"], t2["x"], t2["scales"])
        except mbg.GemvError:
            continue
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().astype(np.float64), expect), v["name"]
    # dequantisation keeps -128 exact
    W = mbg.gemv_dequant_q8(t["A"], t["scales"])
    torch.cuda.synchronize()
    assert np.array_equal(W.cpu().numpy().astype(np.float64), oracle.load().dequant("q8", A, scales, M, N))


@pytest.mark.parametrize("dtype", DTYPES)
def test_edge_sizes(dtype):
    t = upload(dtype, synth.make(synth.random_case(dtype, 4, 64, 9)))
    # M == 0: no-op
    y = torch.full((3,), 7.0, device="cuda")
    A0 = t["A"][:0]
    mbg.gemv(dtype, A0, t["x"], t.get("scales")[:0] if "scales" in t else None, y=y[:0])
    # N == 0: y = 0
    L = mbg.lib()
    if dtype == "q8row":
        st = L.gemv_q8_rowscale_run_variant(0, 0, 0, y.data_ptr(), 3, 0, None, None)
    else:
        st = L.gemv_run_variant(mbg.DTYPES[dtype], 0, 0, 0, y.data_ptr(), 3, 0, None, None)
    assert st == mbg.OK
    torch.cuda.synchronize()
    assert y.tolist() == [0.0, 0.0, 0.0]


@pytest.mark.parametrize("dtype", DTYPES)
def test_canary_and_determinism(dtype):
    M, N = 77, 4096
    inp = synth.make(synth.random_case(dtype, M, N, 21))
    t = upload(dtype, inp)
    guard = torch.full((M + 64,), 1234.5, device="cuda")
    y = guard[:M]
    mbg.gemv(dtype, t["A"], t["x"], t.get("scales"), y=y)
    torch.cuda.synchronize()
    first = y.clone()
    assert torch.all(guard[M:] == 1234.5)
    mbg.gemv(dtype, t["A"], t["x"], t.get("scales"), y=y)
    torch.cuda.synchronize()
    assert torch.equal(first, y)
    y_ref, den = reference(dtype, inp, M, N)
    assert_close(dtype, first.cpu().numpy(), y_ref, den, f"{dtype} canary")


@pytest.mark.parametrize("dtype", DTYPES)
def test_unaligned_layouts_take_the_element_path(dtype):
    """Offset base pointers and row pitches that are not 16-byte multiples."""
    M, N = 45, 1026 if dtype != "q4" else 1026
    inp = synth.make(synth.random_case(dtype, M, N, 31))
    y_ref, den = reference(dtype, inp, M, N)
    t = upload(dtype, inp)
    y = mbg.gemv(dtype, t["A"], t["x"], t.get("scales"))
    torch.cuda.synchronize()
    assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} pitch {N}")
    # A shifted by one element inside a larger buffer (pointer not 16-byte aligned)
    width = t["A"].shape[1]
    big = torch.empty(M * width + 1, dtype=t["A"].dtype, device="cuda")
    big[1:].copy_(t["A"].reshape(-1))
    A_off = big[1:].view(M, width)
    sel = mbg.select_variant(dtype, A_off, t["x"])
    assert mbg.variants(dtype)[sel]["xmode"] == "elem"
    y = mbg.gemv(dtype, A_off, t["x"], t.get("scales"))
    torch.cuda.synchronize()
    assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} offset A")


def _eye_inputs(dtype, n):
    eye = np.eye(n)
    x = synth.normal(3, 2, 0, n, 1.0)
    if dtype == "f32":
        return {"A": eye.astype(np.float32), "x": x.astype(np.float32)}, x.astype(np.float32).astype(np.float64)
    if dtype == "f16x32":
        return {"A": synth.to_f16_bits(eye), "x": x.astype(np.float32)}, x.astype(np.float32).astype(np.float64)
    xb = synth.to_f16_bits(x)
    xv = xb.view(np.float16).astype(np.float64)
    ones = np.full((n, synth.n_groups(n)), 0x3C00, dtype=np.uint16)
    if dtype == "f16":
        return {"A": synth.to_f16_bits(eye), "x": xb}, xv
    if dtype == "q8":
        return {"A": eye.astype(np.int8), "x": xb, "scales": ones}, xv
    if dtype == "q8row":
        return {"A": eye.astype(np.int8), "x": xb, "scales": ones[:, :1]}, xv
    return {"A": synth.pack_int4(eye.astype(np.int64)), "x": xb, "scales": ones}, xv


@pytest.mark.parametrize("dtype", DTYPES)
def test_identity_is_exact(dtype):
    n = 1024
    inp, expect = _eye_inputs(dtype, n)
    t = upload(dtype, inp)
    for v in mbg.variants(dtype):
        try:
            y = mbg.gemv_run_variant(dtype, v["id"], t["A"], t["x"], t.get("scales"))
        except mbg.GemvError:
            continue
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().astype(np.float64), expect), v["name"]


@pytest.mark.parametrize("dtype", ("q8", "q4"))
def test_exact_cases_every_variant(dtype):
    """Cases with exact answers, at a row length every quantised kernel family
    serves (4096 columns, 37 rows: an odd last tile), for every variant:
    - an identity (code 1 on the diagonal) with power-of-two scales that
      differ per (row, group) times an x of binary16 subnormals and normals:
      y_i = s_i x_i exactly (the MMA path multiplies binary16 operands, so a
      flushed subnormal or a wrong group scale would show);
    - rows of zero codes (with nonzero scales and x) come out exactly 0."""
    M, N = 37, 4096
    g = synth.n_groups(N)
    # x: every fourth value a binary16 subnormal (2^-24 .. 2^-15), the rest normal
    xv = synth.normal(404, 2, 0, N, 1.0)
    sub = (synth.integers(404, 3, 0, N, 1, 1023) * 2.0 ** -24)
    xv[::4] = sub[::4] * np.where(np.arange(N)[::4] % 8 == 0, 1.0, -1.0)
    xb = synth.to_f16_bits(xv)
    xd = xb.view(np.float16).astype(np.float64)
    assert np.count_nonzero(np.abs(xd) < 2.0 ** -14) >= N // 4 - 8  # subnormals present
    codes = np.zeros((M, N), dtype=np.int64)
    cols = (np.arange(M) * 97 + 5) % N           # one code per row, spread over the groups
    zero_rows = [3, 17, 36]
    for i in range(M):
        if i not in zero_rows:
            codes[i, cols[i]] = 1 if i % 2 else -1
    exps = synth.integers(404, 5, 0, M * g, -4, 4).reshape(M, g)
    scales = synth.to_f16_bits(np.ldexp(1.0, exps))
    A = codes.astype(np.int8) if dtype == "q8" else synth.pack_int4(codes)
    t = upload(dtype, {"A": A, "x": xb, "scales": scales})
    expect = np.zeros(M)
    for i in range(M):
        if i not in zero_rows:
            expect[i] = codes[i, cols[i]] * np.ldexp(1.0, exps[i, cols[i] // 128]) * xd[cols[i]]
    ran = set()
    for v in mbg.variants(dtype):
        try:
            y = mbg.gemv_run_variant(dtype, v["id"], t["A"], t["x"], t["scales"])
        except mbg.GemvError as e:
            assert e.status == mbg.ERR_UNSUPPORTED
            continue
        torch.cuda.synchronize()
        got = y.cpu().numpy().astype(np.float64)
        assert np.array_equal(got, expect), (v["name"], np.nonzero(got != expect)[0][:5])
        ran.add(v["kind"])
    assert {"mma", "smma", "bulk", "band"} <= ran or {"mma", "smma", "bulk"} <= ran, ran


@pytest.mark.parametrize("dtype", ("q8", "q4", "f16", "f16x32"))
def test_one_to_three_rows_every_variant(dtype):
    """1, 2 and 3 rows at the decode row lengths: grids with more blocks than
    tiles, a single tile whose second row does not exist, every variant
    against the oracle."""
    for N in (4096, 14336):
        for M in (1, 2, 3):
            inp = synth.make(synth.random_case(dtype, M, N, 700 + 10 * M + N))
            y_ref, den = reference(dtype, inp, M, N)
            t = upload(dtype, inp)
            for v in mbg.variants(dtype):
                try:
                    y = mbg.gemv_run_variant(dtype, v["id"], t["A"], t["x"], t.get("scales"))
                except mbg.GemvError as e:
                    assert e.status == mbg.ERR_UNSUPPORTED
                    continue
                torch.cuda.synchronize()
                assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} {M}x{N} {v['name']}")
    assert mbg.gemv_get_device_error() == mbg.OK


@pytest.mark.parametrize("dtype,N", [("q8", 4096), ("q4", 4096), ("q4", 14336)])
def test_scales_two_byte_aligned(dtype, N):
    """Scales that start 2 bytes past an aligned address (legal for binary16):
    every variant either computes the right result or refuses the call with
    GEMV_ERR_UNSUPPORTED before launching (the first INT4 MMA band layout reads
    two neighbouring scales as one 4-byte word, the staged kernels copy whole
    rows of scales in bulk; the row-contiguous layout takes them); the
    automatic choice still works."""
    M = 64
    inp = synth.make(synth.random_case(dtype, M, N, 606 + N))
    y_ref, den = reference(dtype, inp, M, N)
    t = upload(dtype, inp)
    sc = t["scales"].reshape(-1)
    buf = torch.empty(sc.numel() + 8, dtype=sc.dtype, device="cuda")
    buf[1:1 + sc.numel()].copy_(sc)
    s_off = buf[1:1 + sc.numel()].view(t["scales"].shape)
    assert s_off.data_ptr() % 4 == 2
    y = mbg.gemv(dtype, t["A"], t["x"], s_off)
    torch.cuda.synchronize()
    assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} offset scales auto")
    refused, ran = set(), set()
    for v in mbg.variants(dtype):
        try:
            y = mbg.gemv_run_variant(dtype, v["id"], t["A"], t["x"], s_off)
        except mbg.GemvError as e:
            assert e.status == mbg.ERR_UNSUPPORTED
            refused.add(v["kind"])
            continue
        torch.cuda.synchronize()
        assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} offset scales {v['name']}")
        ran.add(v["name"])
    assert "smma" in refused
    if dtype == "q4":
        assert "mma" in refused
        # the row-contiguous layout loads one scale at a time
        assert any(n.startswith("mma_") and n.endswith("_rc") for n in ran), sorted(ran)
    assert mbg.gemv_get_device_error() == mbg.OK


@pytest.mark.parametrize("dtype", ("q8", "q4"))
def test_dequant_bit_exact(dtype):
    orc = oracle.load()
    for (M, N) in ((5, 256), (33, 4096), (7, 130), (3, 1026)):
        w = synth.random_case(dtype, M, N, 5 + N)
        inp = synth.make(w)
        ref = orc.dequant(dtype, inp["A"], inp["scales"], M, N)
        assert np.array_equal(ref.astype(np.float32).astype(np.float64), ref)  # exact in FP32
        t = upload(dtype, inp)
        fn = mbg.gemv_dequant_q8 if dtype == "q8" else mbg.gemv_dequant_q4
        W = fn(t["A"], t["scales"])
        torch.cuda.synchronize()
        assert np.array_equal(W.cpu().numpy().astype(np.float64), ref), (M, N)


def test_probe_reads_every_word_once():
    rng = np.random.default_rng(5)
    words = rng.integers(0, 2 ** 32, size=(8 << 20) // 4 + 4 * 37, dtype=np.uint64).astype(np.uint32)
    expect = int(np.bitwise_xor.reduce(words))
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    for v, name in enumerate(mbg.probe_variants()):
        sink = torch.zeros(1, dtype=torch.int64, device="cuda")
        mbg.gemv_probe_read(buf, sink, v)
        torch.cuda.synchronize()
        assert int(sink.item()) & 0xFFFFFFFF == expect, name
        assert int(sink.item()) >> 32 == 0, name


def test_bounded_wait_reports_timeout_and_context_survives():
    dtype = "f16"
    M, N = 64, 1024
    inp = synth.make(synth.random_case(dtype, M, N, 44))
    t = upload(dtype, inp)
    bulk = [v["id"] for v in mbg.variants(dtype) if v["xmode"] == "bulk" and v["kind"] == "vec"][0]
    tile = [v["id"] for v in mbg.variants(dtype) if v["xmode"] == "bulk" and v["kind"] == "tile"
            and v["threads_per_row"] == 128][0]
    pipe = [v["id"] for v in mbg.variants(dtype) if v["kind"] == "bulk"][0]
    assert mbg.gemv_get_device_error() == mbg.OK
    y_ref, den = reference(dtype, inp, M, N)
    for vid in (bulk, tile, pipe):
        try:
            mbg.debug_set_wait_limit_ns(2_000_000)  # 2 ms
            mbg.debug_skip_x_copy(True)             # nothing is copied: the wait must run out
            mbg.gemv_run_variant(dtype, vid, t["A"], t["x"])
            assert mbg.gemv_get_device_error() == mbg.ERR_TIMEOUT
        finally:
            mbg.debug_skip_x_copy(False)
            mbg.debug_set_wait_limit_ns(0)
        y = mbg.gemv_run_variant(dtype, vid, t["A"], t["x"])
        assert mbg.gemv_get_device_error() == mbg.OK
        assert_close(dtype, y.cpu().numpy(), y_ref, den, "after timeout")


def _timeout_then_recovery(run, check, mask):
    """run() with the given skip hook and a 2 ms wait limit must report a
    timeout (and no undrained copy); without the hook it must be correct."""
    assert mbg.gemv_get_device_error() == mbg.OK
    try:
        mbg.debug_set_wait_limit_ns(2_000_000)
        mbg.debug_skip_copies(mask)
        run()
        status = mbg.gemv_get_device_error()
    finally:
        mbg.debug_skip_copies(0)
        mbg.debug_set_wait_limit_ns(0)
    assert status == mbg.ERR_TIMEOUT, mbg.STATUS.get(status, status)
    check(run())
    assert mbg.gemv_get_device_error() == mbg.OK


@pytest.mark.parametrize("dtype,M,N", [("q4", 300, 4096), ("q8", 300, 4096), ("q4", 37, 14336),
                                       ("f16", 300, 4096)])
def test_bulk_pipeline_stage_wait_runs_out(dtype, M, N):
    """Every bulk-pipeline, staged row-band and staged MMA row-band variant:
    the first weight stage of every block is armed but never copied.  Bulk
    pipeline: the consumers give up, the producer gives up on the
    reduced-stage barrier, drains its other stages and the block exits.
    Staged row bands (CUDA-core or MMA products): every thread gives up on the
    stage, the block agrees at the window barrier, thread 0 drains the other
    stages and the block exits."""
    inp = synth.make(synth.random_case(dtype, M, N, 515 + M))
    t = upload(dtype, inp)
    y_ref, den = reference(dtype, inp, M, N)
    ran = 0
    for v in mbg.variants(dtype):
        if v["kind"] not in ("bulk", "sband", "smma"):
            continue
        try:
            mbg.gemv_run_variant(dtype, v["id"], t["A"], t["x"], t.get("scales"))
        except mbg.GemvError as e:
            assert e.status == mbg.ERR_UNSUPPORTED
            continue
        torch.cuda.synchronize()

        def run(vid=v["id"]):
            return mbg.gemv_run_variant(dtype, vid, t["A"], t["x"], t.get("scales"))

        def check(y, name=v["name"]):
            torch.cuda.synchronize()
            assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{name} after timeout")

        _timeout_then_recovery(run, check, mbg.SKIP_STAGE)
        ran += 1
    assert ran > 0


def test_softmax_segment_wait_runs_out():
    """Softmax kernels that stage rows by bulk copies, single blocks and
    clusters of 2 to 8: the first segment copy of every block is skipped; the
    blocks give up, keep meeting the cluster barriers, write nothing and exit."""
    names = mbg.softmax_variants()
    orc = oracle.load()
    ran = set()
    for vid, name in enumerate(names):
        if not name.startswith("smb_"):
            continue
        T = int(name.split("_t")[1].split("_")[0])
        E = int(name.split("_e")[1].split("_")[0])
        C = int(name.split("_c")[1].split("_")[0])
        N = T * E * C
        M = 12
        bits = synth.to_f16_bits(synth.normal(600 + vid, 1, 0, M * N, 2.0)).reshape(M, N)
        x = torch.from_numpy(bits.view(np.float16)).cuda()
        ref = orc.softmax(bits, M, N)

        def run(v=vid, x=x):
            return mbg.gemv_softmax_f16(x, variant=v)

        def check(y, ref=ref, name=name):
            torch.cuda.synchronize()
            got = y.cpu().numpy().astype(np.float64)
            err = float(np.max(np.abs(got - ref) / np.maximum(ref, 1e-4)))
            assert err <= 1e-3, (name, err)

        _timeout_then_recovery(run, check, mbg.SKIP_SEGMENT)
        ran.add(C)
    assert {1, 2, 8} <= ran


def test_bulk_probe_wait_runs_out():
    """Bulk-copy probe patterns: the first chunk of every block is skipped; the
    probe sets bit 63 of the sink (not bit 62: nothing was left in flight)."""
    rng = np.random.default_rng(8)
    words = rng.integers(0, 2 ** 32, size=(4 << 20) // 4, dtype=np.uint64).astype(np.uint32)
    expect = int(np.bitwise_xor.reduce(words))
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    ran = 0
    for v, name in enumerate(mbg.probe_variants()):
        if not name.startswith("bulk"):
            continue
        sink = torch.zeros(1, dtype=torch.int64, device="cuda")
        try:
            mbg.debug_set_wait_limit_ns(2_000_000)
            mbg.debug_skip_copies(mbg.SKIP_PROBE)
            mbg.gemv_probe_read(buf, sink, v)
            torch.cuda.synchronize()
        finally:
            mbg.debug_skip_copies(0)
            mbg.debug_set_wait_limit_ns(0)
        word = int(sink.item()) & 0xFFFFFFFFFFFFFFFF
        assert (word >> 63) & 1 == 1 and (word >> 62) & 1 == 0, (name, hex(word))
        sink.zero_()
        mbg.gemv_probe_read(buf, sink, v)
        torch.cuda.synchronize()
        assert int(sink.item()) == expect, name
        ran += 1
    assert ran > 0


def test_host_call_waits_for_a_kernel_that_writes_the_weights():
    """gemv_ex_host without the overlap flag: the kernel before the call
    lets its successor start at once but writes A only later; the GEMV must
    see the written A (the copy of x waits for that kernel before it lets the
    GEMV start)."""
    L = mbg.lib()
    for dtype, M, N in (("f16", 2048, 4096), ("q4", 1024, 4096)):
        w = synth.random_case(dtype, M, N, 707)
        inp = synth.make(w)
        if dtype == "f16":
            A_final = np.full((M, N), 0x3C00, dtype=np.uint16)   # all ones
            word = 0x3C003C00
        else:
            A_final = np.full((M, N // 2), 0x11, dtype=np.uint8)  # every code 1
            word = 0x11111111
        inp_final = dict(inp, A=A_final)
        y_ref, den = reference(dtype, inp_final, M, N)
        t = upload(dtype, inp)
        A_dev = torch.zeros_like(t["A"])  # zero until the late kernel writes it
        x_np = inp["x"]
        x_host = torch.from_numpy(np.ascontiguousarray(x_np).view(np.float16)).pin_memory()
        x_dev = torch.empty_like(t["x"])
        y_host = torch.full((M,), np.nan, dtype=torch.float32).pin_memory()
        s_ptr = t["scales"].data_ptr() if "scales" in t else None
        s = torch.cuda.current_stream()
        for _ in range(3):
            A_dev.zero_()
            mbg.debug_late_fill(A_dev, word, 200_000, stream=s)
            st = L.gemv_ex_host(mbg.DTYPES[dtype], A_dev.data_ptr(), x_host.data_ptr(), x_dev.data_ptr(),
                                y_host.data_ptr(), M, N, s_ptr, 0, s.cuda_stream)
            assert st == mbg.OK, mbg.status_string(st)
            s.synchronize()
            assert_close(dtype, y_host.numpy().copy(), y_ref, den, f"{dtype} after a late write")
    assert mbg.gemv_get_device_error() == mbg.OK


def test_runs_on_a_side_stream():
    dtype = "q4"
    M, N = 300, 4096
    inp = synth.make(synth.random_case(dtype, M, N, 12))
    t = upload(dtype, inp)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = mbg.gemv_q4(t["A"], t["x"], t["scales"])
    s.synchronize()
    y_ref, den = reference(dtype, inp, M, N)
    assert_close(dtype, y.cpu().numpy(), y_ref, den, "side stream")


def test_tolerances_are_the_stated_ones():
    # FP32 arithmetic 1e-5, FP16 / quantised 2e-3; FP16 weights with an FP32 x
    # are multiplied and summed in FP32, so they take the FP32 bound
    assert TOL == {"f32": 1e-5, "f16": 2e-3, "q8": 2e-3, "q4": 2e-3, "f16x32": 1e-5, "q8row": 2e-3}


@pytest.mark.parametrize("dtype", DTYPES)
def test_overlap_flag_parity(dtype):
    for (M, N) in ((300, 4096), (64, 14336), (1000, 1024)):
        inp = synth.make(synth.random_case(dtype, M, N, 60 + M))
        y_ref, den = reference(dtype, inp, M, N)
        t = upload(dtype, inp)
        y = mbg.gemv(dtype, t["A"], t["x"], t.get("scales"), overlap=True)
        torch.cuda.synchronize()
        assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} overlap {M}x{N}")


def _chain_inputs():
    w1 = synth.random_case("f32", 4096, 1024, 71)
    w2 = synth.random_case("f32", 512, 4096, 72)
    i1, i2 = synth.make(w1), synth.make(w2)
    t1, t2 = upload("f32", i1), upload("f32", i2)
    return i1, i2, t1, t2


def test_overlapped_chain_sees_the_previous_result():
    """y1 = A1 x, then y2 = A2 y1 launched to overlap its predecessor: y2 must
    use the finished y1 (y1 is cleared before every round)."""
    i1, i2, t1, t2 = _chain_inputs()
    y1 = torch.empty(4096, device="cuda")
    y2 = torch.empty(512, device="cuda")
    mbg.gemv("f32", t1["A"], t1["x"], y=y1)
    torch.cuda.synchronize()
    y1_ref = y1.cpu().numpy().copy()
    y2_ref, den = oracle.load().gemv("f32", i2["A"], y1_ref, 512, 4096)
    for _ in range(20):
        y1.zero_()
        mbg.gemv("f32", t1["A"], t1["x"], y=y1, overlap=True)
        mbg.gemv("f32", t2["A"], y1, y=y2, overlap=True)
    torch.cuda.synchronize()
    assert np.array_equal(y1.cpu().numpy(), y1_ref)
    assert_close("f32", y2.cpu().numpy(), y2_ref, den, "overlapped chain")


def test_overlapped_chain_in_a_cuda_graph():
    i1, i2, t1, t2 = _chain_inputs()
    y1 = torch.empty(4096, device="cuda")
    y2 = torch.empty(512, device="cuda")
    mbg.gemv("f32", t1["A"], t1["x"], y=y1)
    torch.cuda.synchronize()
    y2_ref, den = oracle.load().gemv("f32", i2["A"], y1.cpu().numpy(), 512, 4096)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(2):
            mbg.gemv("f32", t1["A"], t1["x"], y=y1, overlap=True)
            mbg.gemv("f32", t2["A"], y1, y=y2, overlap=True)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(8):
            y1.zero_()
            mbg.gemv("f32", t1["A"], t1["x"], y=y1, overlap=True)
            mbg.gemv("f32", t2["A"], y1, y=y2, overlap=True)
    y2.fill_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    assert_close("f32", y2.cpu().numpy(), y2_ref, den, "overlapped chain in a graph")
    assert mbg.gemv_get_device_error() == mbg.OK


def test_row_scales_equal_broadcast_group_scales():
    """One scale per row gives the same bits as equal group scales, per variant."""
    M, N = 300, 4160
    w = synth.random_case("q8row", M, N, 71)
    inp = synth.make(w)
    y_ref, den = reference("q8row", inp, M, N)
    t = upload("q8row", inp)
    groups = t["scales"].reshape(M, 1).expand(M, synth.n_groups(N)).contiguous()
    compared = bulk = 0
    for v in mbg.variants("q8"):
        try:
            y_row = mbg.gemv_run_variant("q8row", v["id"], t["A"], t["x"], t["scales"])
        except mbg.GemvError as e:
            # a variant refuses row scales only where it refuses the shape
            assert e.status == mbg.ERR_UNSUPPORTED, v["name"]
            with pytest.raises(mbg.GemvError):
                mbg.gemv_run_variant("q8", v["id"], t["A"], t["x"], groups)
            continue
        torch.cuda.synchronize()
        assert_close("q8row", y_row.cpu().numpy(), y_ref, den, v["name"])
        bulk += v["kind"] == "bulk"
        try:
            y_grp = mbg.gemv_run_variant("q8", v["id"], t["A"], t["x"], groups)
        except mbg.GemvError as e:
            # 33 group scales per row (66 bytes) cannot be bulk-copied
            assert e.status == mbg.ERR_UNSUPPORTED and v["kind"] == "bulk", v["name"]
            continue
        torch.cuda.synchronize()
        assert torch.equal(y_row, y_grp), v["name"]
        compared += 1
    assert compared >= 5 and bulk >= 1


def test_concurrent_calls_from_threads_and_streams():
    """Entry points called from several host threads, each on its own stream,
    at the same time (the per-device state and the variant caches are shared)."""
    import threading
    cases = [("f16", 300, 4160), ("q4", 129, 4160), ("q8", 257, 4096), ("f32", 64, 1000)]
    prepared = []
    for dtype, M, N in cases:
        inp = synth.make(synth.random_case(dtype, M, N, 880 + M))
        y_ref, den = reference(dtype, inp, M, N)
        prepared.append((dtype, upload(dtype, inp), y_ref, den))
    results = [None] * len(prepared)
    errors = []

    def work(k):
        try:
            dtype, t, _, _ = prepared[k]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                ys = [mbg.gemv(dtype, t["A"], t["x"], t.get("scales")) for _ in range(20)]
            s.synchronize()
            results[k] = [y.cpu().numpy() for y in ys]
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(k,)) for k in range(len(prepared))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for (dtype, _, y_ref, den), ys in zip(prepared, results):
        for y in ys:
            assert_close(dtype, y, y_ref, den, f"{dtype} concurrent")
        assert all(np.array_equal(ys[0], y) for y in ys[1:])
    assert mbg.gemv_get_device_error() == mbg.OK


def test_fixed_chunk_bulk_variants_with_ragged_rows():
    """Bulk variants specialised for an exact chunk count per thread, on row
    counts that leave a partial last tile."""
    checked = set()
    for dtype, M, N in (("q4", 37, 14336), ("q4", 37, 4096), ("q8", 37, 4096), ("q8", 37, 14336),
                        ("q4", 3, 14336), ("q4", 2, 4096)):
        inp = synth.make(synth.random_case(dtype, M, N, 4000 + M))
        y_ref, den = reference(dtype, inp, M, N)
        t = upload(dtype, inp)
        for v in mbg.variants(dtype):
            if v["kind"] != "bulk" or v["unroll"] == 0:
                continue
            try:
                y = mbg.gemv_run_variant(dtype, v["id"], t["A"], t["x"], t.get("scales"))
            except mbg.GemvError as e:
                assert e.status == mbg.ERR_UNSUPPORTED
                continue
            torch.cuda.synchronize()
            assert_close(dtype, y.cpu().numpy(), y_ref, den, f"{dtype} {v['name']} {M}x{N}")
            checked.add((dtype, v["name"]))
    every = {(d, v["name"]) for d in ("q4", "q8") for v in mbg.variants(d)
             if v["kind"] == "bulk" and v["unroll"] > 0}
    assert checked == every, f"not exercised: {sorted(every - checked)}"
