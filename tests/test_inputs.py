"""The seeded input generators (no GPU)."""
import numpy as np

import cns_inputs as ci


def test_splitmix64_published_outputs():
    # first outputs of SplitMix64 seeded with 0, as published with the algorithm
    got = [int(x) for x in ci.splitmix64(0, 4)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F, 0xF88BB8A8724C81EC]


def test_offsets_regenerate_slices():
    a = ci.u32_uniform(5, 1000)
    b = ci.u32_uniform(5, 100, offset=900)
    np.testing.assert_array_equal(a[900:], b)


def test_float_field_range_and_exactness():
    f = ci.f32_uniform_pm1(3, 100000)
    assert f.dtype == np.float32 and f.min() >= -1.0 and f.max() < 1.0
    # every value is k * 2^-23 - 1 exactly
    k = (f.astype(np.float64) + 1.0) * 2.0 ** 23
    np.testing.assert_array_equal(k, np.round(k))


def test_notify_ops_shape_and_validity():
    o = ci.notify_ops(100000)
    assert o.shape == (100000, 4) and o.dtype == np.uint32
    rec = o[:, 0] == 0
    assert set(np.unique(o[rec, 1]).tolist()) == {0, 1, 2, 4}
    assert set(np.unique(o[~rec, 1]).tolist()) == {0, 1, 2, 3, 4}
    assert (o[rec, 3] == 0).all()
    frac_clear = o[~rec, 3].mean()
    assert 0.08 < frac_clear < 0.17
    assert 0.45 < rec.mean() < 0.55


def test_sample_indices_include_both_ends():
    s = ci.sample_indices(1, 1000, 20)
    assert s[0] == 0 and s[-1] == 999 and (np.diff(s) > 0).all()
