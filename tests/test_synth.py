"""The seeded input generators: reproducible, thread-count independent, right shapes
and distributions, and a d2t map that sends draft ids to distinct in-range targets."""
import numpy as np

from eagle_speculative_decode_gb300 import synth


def test_d2t_maps_to_distinct_sorted_in_range_targets():
    for geo in (synth.TINY, synth.FULL):
        d2t = synth.make_d2t(geo, seed=0)
        assert d2t.dtype == np.int64 and d2t.shape == (geo.draft_vocab,)
        tgt = np.arange(geo.draft_vocab) + d2t
        assert tgt.min() >= 0 and tgt.max() < geo.target_vocab
        assert np.all(np.diff(tgt) > 0)


def test_normal_bf16_reproducible_and_thread_independent():
    a = synth.normal_bf16((3, 1 << 21), seed=5, key=(9,), std=0.02, threads=1)
    b = synth.normal_bf16((3, 1 << 21), seed=5, key=(9,), std=0.02, threads=8)
    np.testing.assert_array_equal(a, b)
    c = synth.normal_bf16((3, 1 << 21), seed=6, key=(9,), std=0.02)
    assert not np.array_equal(a, c)
    x = (a.astype(np.uint32) << 16).view(np.float32)
    assert abs(float(x.mean())) < 1e-4 and abs(float(x.std()) - 0.02) < 2e-4


def test_f32_to_bf16_bits_rounds_to_nearest_even():
    x = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -2.5, 0.0], dtype=np.float32)
    np.testing.assert_array_equal(synth.f32_to_bf16_bits(x),
                                  np.array([0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000], dtype=np.uint16))


def test_make_weights_shapes_and_gain_modes():
    w = synth.make_weights(synth.TINY, seed=1)
    for name, shape in synth.weight_shapes(synth.TINY).items():
        assert w.bits[name].shape == shape and w.bits[name].dtype == np.uint16
    g = (w.bits["in_norm"].astype(np.uint32) << 16).view(np.float32)
    assert abs(float(g.mean()) - 1.0) < 0.01
    lit = synth.make_weights(synth.TINY, seed=1, gains="literal")
    g2 = (lit.bits["in_norm"].astype(np.uint32) << 16).view(np.float32)
    assert abs(float(g2.mean())) < 0.01
    np.testing.assert_array_equal(w.bits["q"], lit.bits["q"])


def test_accept_imposition():
    d = np.array([[5, 6, 7], [1, 2, 3]], dtype=np.int32)
    n = np.array([2, 0], dtype=np.int32)
    y = synth.impose_target_predictions(d, n, synth.TINY, seed=0)
    assert y.shape == (2, 4)
    assert list(y[0, :2]) == [5, 6] and y[0, 2] != 7
    assert y[1, 0] != 1
    lens = synth.imposed_accept_lengths(1000, 3, seed=1, p_accept=0.6)
    assert lens.min() >= 0 and lens.max() <= 3
    assert abs(lens.mean() - (0.6 + 0.36 + 0.216)) < 0.1
