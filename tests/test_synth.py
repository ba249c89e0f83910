"""The seeded input generator: published SplitMix64 outputs, moments, determinism."""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 seeded with 0 (the reference sequence of the
    # generator's published C implementation)
    assert synth.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert synth.splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert synth.splitmix64_at(0, 2) == 0x06C45D188009454F


def test_normal_moments_and_offsets():
    k = synth.key(0, 1, 2, 3)
    z = synth.normal64(k, 400_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.abs(z).max() <= 6.0
    # counter based: a slice drawn with an offset equals the same slice of a longer draw
    a = synth.normal(k, (1000,), 0.02)
    b = synth.normal(k, (300,), 0.02, first=700)
    assert np.array_equal(a[700:], b)
    # sigma * z rounded once to fp32
    assert np.array_equal(a, (0.02 * synth.normal64(k, 1000)).astype(np.float32))


def test_streams_differ_and_repeat():
    w1 = synth.expert_weights(synth.TINY, 3)[0]
    w2 = synth.expert_weights(synth.TINY, 3)[0]
    w3 = synth.expert_weights(synth.TINY, 4)[0]
    assert np.array_equal(w1, w2) and not np.array_equal(w1, w3)
    assert w1.shape == (2 * synth.TINY.I, synth.TINY.H)


def test_zipf_bias_is_a_log_distribution_over_a_permutation():
    b = synth.popularity_bias(synth.FULL, seed=0)
    p = np.exp(b.astype(np.float64))
    assert abs(p.sum() - 1.0) < 1e-5
    ranks = np.argsort(-p)
    ps = p[ranks]
    r = np.arange(1, 129, dtype=np.float64)
    assert np.allclose(ps / ps[0], r ** -1.1, rtol=1e-5)


def test_ar1_lag_one_correlation():
    x = synth.ar1(synth.key(0, 0, synth.T_AR1), 64, 2816, 0.9).astype(np.float64)
    c = np.mean(x[1:] * x[:-1]) / np.mean(x * x)
    assert abs(c - 0.9) < 0.02
