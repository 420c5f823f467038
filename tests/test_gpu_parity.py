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
          (257, 1024), (64, 2056), (33, 4096), (300, 4160), (17, 8200)]


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


def _sample_rows(M, n=96, seed=0):
    rng = np.random.default_rng(seed)
    rows = set([0, 1, M // 2, M - 2, M - 1]) | set(rng.integers(0, M, n).tolist())
    return sorted(r for r in rows if 0 <= r < M)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_workloads_full_size(name):
    """The named workloads at full size: every row of the small one, sampled rows else."""
    w = synth.WORKLOADS[name]
    inp = synth.make(w)
    t = upload(w.dtype, inp)
    rows = None if w.M * w.N <= 1024 * 1024 else _sample_rows(w.M, seed=w.seed)
    y_ref, den = reference(w.dtype, inp, w.M, w.N, rows=rows)
    y = mbg.gemv(w.dtype, t["A"], t["x"], t.get("scales"))
    torch.cuda.synchronize()
    y_np = y.cpu().numpy()
    y_sel = y_np if rows is None else y_np[rows]
    assert_close(w.dtype, y_sel, y_ref, den, f"{name} auto")
    # every tile variant and the warp-per-row variants that fit this workload
    for v in mbg.variants(w.dtype):
        if v["kind"] == "elem" or (v["kind"] == "vec" and v["threads_per_row"] != 32):
            continue
        try:
            y2 = mbg.gemv_run_variant(w.dtype, v["id"], t["A"], t["x"], t.get("scales"))
        except mbg.GemvError as e:
            assert e.status == mbg.ERR_UNSUPPORTED
            continue
        torch.cuda.synchronize()
        y2 = y2.cpu().numpy()
        assert_close(w.dtype, y2 if rows is None else y2[rows], y_ref, den, f"{name} {v['name']}")
    # outputs are finite everywhere
    assert np.all(np.isfinite(y_np))


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
