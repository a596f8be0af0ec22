"""The seeded generator: determinism, addressability and rough distribution."""
import numpy as np

import synth


def test_subset_draw_equals_slice_of_full_draw():
    full = synth.normal(7, 1, 10000, 0.5, 0, "f64")
    part = synth.normal(7, 1, 999, 0.5, 4321, "f64")
    assert np.array_equal(full[4321:4321 + 999], part)
    rows = synth.normal_rows_bf16(7, 1, np.array([3, 0, 7]), 100, 0.5)
    fullb = synth.normal(7, 1, 800, 0.5, 0, "bf16").reshape(8, 100)
    assert np.array_equal(rows, fullb[[3, 0, 7]])


def test_streams_and_seeds_differ_and_moments_are_normal():
    a = synth.normal(1, 1, 200000)
    b = synth.normal(1, 2, 200000)
    c = synth.normal(2, 1, 200000)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    for x in (a, b, c):
        assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.01


def test_uniform_ints_and_permutation():
    u = synth.uniform_int(5, 5, 100000, 1, 32768)
    assert u.min() >= 1 and u.max() <= 32768 and abs(u.mean() - 16384.5) < 200
    p = synth.permutation(5, 6, 5000)
    assert np.array_equal(np.sort(p), np.arange(5000)) and not np.array_equal(p, np.arange(5000))


def test_workload_shapes():
    w = synth.ragged_paged()
    assert w.B == 128 and w.Q == 2 and w.lens.min() >= 1 and w.lens.max() <= 32768
    pt = w.page_table()
    used = np.concatenate([pt[b, :w.pages_per_seq[b]] for b in range(w.B)])
    assert np.array_equal(np.sort(used), np.arange(w.num_pages))
    t = synth.tiny_fp32()
    qn, qr = t.queries()
    assert qn.shape == (2, 1, 8, 64) and qr.shape == (2, 1, 8, 16) and qn.dtype == np.float32
