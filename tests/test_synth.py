"""The seeded input generator: its stream against the published SplitMix64 outputs, and
the value sets of each distribution."""
import numpy as np

import synth


def test_splitmix64_published_outputs():
    # First three outputs of SplitMix64 seeded with 0, as published with the algorithm's
    # reference implementations (Steele, Lea & Flood 2014; Vigna's splitmix64.c).
    out = synth.splitmix64(0, np.arange(3, dtype=np.uint64))
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_uniform_grid_and_range():
    a = synth.uniform(64, 129, 0)
    assert a.dtype == np.float32 and a.shape == (64, 129)
    assert a.min() >= -1.0 and a.max() < 1.0
    # every value sits on the 2**-23 grid of [-1, 1) (24-bit uniform, exact in fp32)
    scaled = (a.astype(np.float64) + 1.0) * 2.0 ** 23
    assert np.array_equal(scaled, np.round(scaled))
    assert abs(float(a.mean())) < 0.02


def test_row_subset_and_layout_independence():
    full = synth.normal(50, 37, 9, sigma=0.02)
    part = synth.normal(50, 37, 9, sigma=0.02, row0=13, nrows=7)
    assert np.array_equal(full[13:20], part)
    u = synth.uniform(33, 65, 4)
    assert np.array_equal(u[5:9], synth.uniform(33, 65, 4, row0=5, nrows=4))
    p = synth.padded(u, 70)
    assert p.shape == (33, 70) and np.isnan(p[:, 65:]).all() and np.array_equal(p[:, :65], u)


def test_normal_moments():
    z = synth.normal(256, 256, 1)
    assert abs(float(z.mean())) < 0.02 and abs(float(z.std()) - 1.0) < 0.02
    w = synth.normal(256, 256, 1, mu=0.0, sigma=0.02)
    assert abs(float(w.std()) - 0.02) < 0.001


def test_small_int_values():
    s = synth.small_int(100, 100, 3)
    assert set(np.unique(s).tolist()) == set(float(v) for v in range(-4, 5))


def test_streams_differ_by_seed():
    assert not np.array_equal(synth.uniform(8, 8, 0), synth.uniform(8, 8, 1))
    assert np.array_equal(synth.uniform(8, 8, 7), synth.uniform(8, 8, 7))
