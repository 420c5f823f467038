"""The seeded input generator: published SplitMix64 outputs, layouts, ranges."""

import numpy as np

import synth


def test_splitmix64_published_vector():
    # SplitMix64 started from state 0 yields 0xE220A8397B1DCDAF,
    # 0x6E789E6AA1B965F4, 0x06C45D188009454F first (Steele, Lea & Flood 2014
    # reference generator).
    z = synth._mix(np.array([1, 2, 3], dtype=np.uint64) * np.uint64(synth.GAMMA))
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert synth._mix_int(synth.GAMMA) == 0xE220A8397B1DCDAF


def test_counter_based_slices_agree():
    full = synth.raw_u64(5, 1, 0, 1000)
    part = synth.raw_u64(5, 1, 400, 100)
    assert np.array_equal(full[400:500], part)
    w = synth.WORKLOADS["q4_4096x14336"]
    rows = synth.weight_rows(w, 100, 3)
    assert np.array_equal(rows[1], synth.weight_rows(w, 101, 1)[0])


def test_distributions_in_range():
    u = synth.uniform(1, 1, 0, 100000, -1.0, 1.0)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    q = synth.integers(1, 1, 0, 100000, -127, 127)
    assert q.min() == -127 and q.max() == 127
    q4 = synth.integers(1, 1, 0, 100000, -8, 7)
    assert q4.min() == -8 and q4.max() == 7
    z = synth.normal(1, 2, 0, 200000, 0.02)
    assert abs(z.std() - 0.02) < 0.0005 and abs(z.mean()) < 0.0005


def test_pack_int4_layout():
    q = np.array([[1, 2, -1, -8, 7, 0]])
    packed = synth.pack_int4(q)
    assert packed.tolist() == [[0x21, 0x8F, 0x07]]


def test_workload_inputs_have_storage_shapes():
    for name, w in synth.WORKLOADS.items():
        if w.M * w.N > 4096 * 4096:
            continue
        rows = synth.weight_rows(w, 0, 2)
        width = w.N // 2 if w.dtype == "q4" else w.N
        assert rows.shape == (2, width), name
        x = synth.x_vector(w)
        assert x.shape == (w.N,)
        assert x.dtype == (np.float32 if w.dtype in ("f32", "f16x32") else np.uint16)
        if w.quantised:
            g = 1 if w.dtype == "q8row" else synth.n_groups(w.N)
            assert synth.scale_rows(w, 0, 2).shape == (2, g)
