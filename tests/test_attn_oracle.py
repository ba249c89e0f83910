"""Pins of the oracle's attention block against facts fixed outside it.

The pages fix the pieces (4-bit affine projections, RoPE, attention over an FP16
key/value cache that is a bounded ring for sliding-window layers and a linear store
for full layers), not their formulas; the readings are the plain ones (rotate-half
RoPE, softmax attention with grouped key/value heads).  Each test pins one of them
to a closed form or an invariant that a plausible slip (a sign, a pairing, a slot
index, a window bound, a head mapping) would break:

* RoPE: hand-built exact weights make the cached key a known pair of inputs; the
  rotated values must match cos/sin of p * theta^(-2i/d) computed here.
* One attended position: the output is that position's value, so y = x + Wo v.
* Zero queries: every score is 0, so the output is the plain mean of the values of
  exactly the attended positions (window bounds, ring slots, full layers).
* Grouped queries equal ordinary multi-head attention with duplicated key/value heads.
* Scores depend only on position differences (shifting a whole sequence).
* A sliding layer ignores positions older than its window even while the ring
  still holds them.
* Pre-norm: the block equals the un-normed block on RMSNorm(x) plus x.
"""
import math

import numpy as np
import pytest

import oracle
import synth

H = 64


def _exact_rows(selectors, n_rows, K):
    """4-bit affine rows with scale 1, bias 0 and code 1 at the listed columns:
    selectors = {row: [columns]} -> (q, s, b) holding exactly those 0/1 weights."""
    q = np.zeros((n_rows, K // 8), np.uint32)
    s = np.zeros((n_rows, K // 64), np.uint16)
    b = np.zeros((n_rows, K // 64), np.uint16)
    one = np.float16(1.0).view(np.uint16)
    for r, cols in selectors.items():
        s[r, :] = one
        for j in cols:
            q[r, j // 8] |= np.uint32(1) << np.uint32(4 * (j % 8))
    return q, s, b


def _caches(nkv, kv_len, d, hist=None):
    if hist is None:
        k = np.zeros((nkv, kv_len, d), np.uint16)
        v = np.zeros((nkv, kv_len, d), np.uint16)
    else:
        k = np.ascontiguousarray(hist[0].astype(np.float16).view(np.uint16))
        v = np.ascontiguousarray(hist[1].astype(np.float16).view(np.uint16))
    return k, v


def _h(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _run(s, wqkv, wo, k, v, x, pos, **kw):
    return oracle.attn_step(s.H, s.nq, s.nkv, s.d, s.window, s.kv_len, s.theta, s.scale, wqkv, wo, k, v, x,
                            pos, **kw)


def test_rope_rotates_cached_keys_by_closed_form():
    nq, nkv, d, kv_len, theta = 1, 1, 64, 64, 10000.0
    rows = (nq + 2 * nkv) * d
    kb = nq * d  # first key row
    # key dims 0 and 1 read x0, their partners d/2 and d/2+1 read x1
    wqkv = _exact_rows({kb + 0: [0], kb + d // 2: [1], kb + 1: [0], kb + d // 2 + 1: [1]}, rows, H)
    wo = _exact_rows({}, H, nq * d)
    x = np.zeros((1, H), np.float32)
    x0, x1 = 0.75, -1.25
    x[0, 0], x[0, 1] = x0, x1
    for p in (0, 1, 5, 37):
        k, v = _caches(nkv, kv_len, d)
        oracle.attn_step(H, nq, nkv, d, 0, kv_len, theta, d ** -0.5, wqkv, wo, k, v, x, p)
        got = _h(k[0, p])
        for i in (0, 1):
            a = p * theta ** (-2.0 * i / d)
            lo = x0 * math.cos(a) - x1 * math.sin(a)
            hi = x1 * math.cos(a) + x0 * math.sin(a)
            for val, ref in ((got[i], lo), (got[i + d // 2], hi)):
                ulp = float(np.spacing(np.float16(abs(ref)))) if ref != 0 else 2.0 ** -24
                assert abs(val - ref) <= ulp, (p, i, val, ref)
        # the other key dimensions have all-zero rows
        assert np.all(got[2:d // 2] == 0) and np.all(got[d // 2 + 2:] == 0)


@pytest.mark.parametrize("window,kv_len,pos", [(0, 32, 0), (8, 11, 0)])
def test_single_position_output_is_its_value(window, kv_len, pos):
    s = synth.AttnShape("t", H, 2, 1, 64, window, kv_len, 10000.0)
    wqkv_f, wo_f = synth.attn_weights(s, seed=3)
    wqkv, wo = oracle.quantise(wqkv_f, 4), oracle.quantise(wo_f, 4)
    x = synth.normal(synth.key(11), (1, H), 1.0)
    k, v = _caches(s.nkv, s.kv_len, s.d)
    y, o = _run(s, wqkv, wo, k, v, x, pos)
    vrows = tuple(a[(s.nq + s.nkv) * s.d:] for a in wqkv)
    vref = oracle.qgemv(*vrows, H, 4, x)[0].astype(np.float16).astype(np.float64)
    # both query heads read the single key/value head
    np.testing.assert_array_equal(o[0], np.concatenate([vref, vref]))
    yref = x[0].astype(np.float64) + oracle.qgemv(*wo, s.nq * s.d, 4, o.astype(np.float32))[0]
    np.testing.assert_allclose(y[0], yref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("window,kv_len,pos,T", [(16, 23, 61, 1), (16, 23, 5, 1), (16, 20, 100, 3),
                                                 (0, 96, 0, 1), (0, 96, 70, 4)])
def test_zero_queries_average_exactly_the_attended_values(window, kv_len, pos, T):
    s = synth.AttnShape("t", 512, 4, 2, 64, window, kv_len, 10000.0)
    wqkv_f, wo_f = synth.attn_weights(s, seed=1)
    wqkv_f[:s.nq * s.d] = 0.0  # q = 0: every score is 0
    wqkv, wo = oracle.quantise(wqkv_f, 4), oracle.quantise(wo_f, 4)
    k, v = _caches(s.nkv, s.kv_len, s.d, synth.kv_history(s, seed=2))
    x = synth.tokens(synth.TINY, T, seed=0, stream=9)
    _, o = _run(s, wqkv, wo, k, v, x, pos)
    # after the call the cache holds every attended position (the chunk's own
    # tokens included; kv_len >= window + T - 1 keeps the oldest ones intact)
    vals = _h(v).reshape(s.nkv, s.kv_len, s.d)
    G = s.nq // s.nkv
    for t in range(T):
        p = pos + t
        first = max(0, p - window + 1) if window else 0
        slots = [(j % kv_len) if window else j for j in range(first, p + 1)]
        for h in range(s.nq):
            ref = vals[h // G, slots].mean(axis=0)
            np.testing.assert_allclose(o[t, h * s.d:(h + 1) * s.d], ref, rtol=0, atol=1e-12)


def test_grouped_queries_equal_duplicated_heads():
    s = synth.AttnShape("gqa", 512, 4, 2, 64, 16, 23, 10000.0)
    m = synth.AttnShape("mha", 512, 4, 4, 64, 16, 23, 10000.0)
    wqkv_f, wo_f = synth.attn_weights(s, seed=4)
    d, nq = s.d, s.nq
    qrows = wqkv_f[:nq * d]
    krows = wqkv_f[nq * d:(nq + 2) * d].reshape(2, d, -1)
    vrows = wqkv_f[(nq + 2) * d:].reshape(2, d, -1)
    dup = [0, 0, 1, 1]  # query head h reads key/value head h // 2
    wm = np.concatenate([qrows, krows[dup].reshape(4 * d, -1), vrows[dup].reshape(4 * d, -1)])
    hist = synth.kv_history(s, seed=5)
    kg, vg = _caches(2, 23, d, hist)
    km, vm = _caches(4, 23, d, hist[:, dup])
    wo = oracle.quantise(wo_f, 4)
    x = synth.tokens(synth.TINY, 3, seed=0, stream=10)
    yg, og = _run(s, oracle.quantise(wqkv_f, 4), wo, kg, vg, x, 30)
    ym, om = _run(m, oracle.quantise(wm, 4), wo, km, vm, x, 30)
    np.testing.assert_array_equal(og, om)
    np.testing.assert_array_equal(yg, ym)


def test_scores_depend_on_position_differences_only():
    # a sliding layer of window 8: from the eighth token on, each token attends to
    # the last eight tokens of the same sequence wherever the sequence starts
    s = synth.AttnShape("rel", 512, 4, 2, 64, 8, 1200, 10000.0)
    wqkv_f, wo_f = synth.attn_weights(s, seed=6)
    wqkv, wo = oracle.quantise(wqkv_f, 4), oracle.quantise(wo_f, 4)
    x = synth.tokens(synth.TINY, 14, seed=0, stream=11)
    outs = []
    for pos in (0, 1000):
        k, v = _caches(s.nkv, s.kv_len, s.d)
        outs.append(_run(s, wqkv, wo, k, v, x, pos)[1][s.window - 1:])
    # only the binary16 rounding of the rotated keys differs between the two
    np.testing.assert_allclose(outs[0], outs[1], rtol=0, atol=2e-3 * np.abs(outs[0]).max())
    assert np.abs(outs[0] - outs[1]).max() > 0  # the rotations did differ


def test_sliding_window_ignores_older_positions_still_in_the_ring():
    s = synth.AttnShape("win", 512, 4, 2, 64, 16, 23, 10000.0)
    wqkv_f, wo_f = synth.attn_weights(s, seed=7)
    wqkv, wo = oracle.quantise(wqkv_f, 4), oracle.quantise(wo_f, 4)
    hist = synth.kv_history(s, seed=8)
    x = synth.tokens(synth.TINY, 1, seed=0, stream=12)
    p = 50

    def run(edit_pos):
        k, v = _caches(s.nkv, s.kv_len, s.d, hist)
        if edit_pos is not None:
            sl = edit_pos % s.kv_len
            k[:, sl] = np.float16(3.0).view(np.uint16)
            v[:, sl] = np.float16(-5.0).view(np.uint16)
        return _run(s, wqkv, wo, k, v, x, p)[0]

    base = run(None)
    np.testing.assert_array_equal(run(p - s.window), base)       # just outside the window
    assert np.abs(run(p - s.window + 1) - base).max() > 1e-3    # oldest position inside it


def test_prenorm_is_the_block_on_the_normalised_input():
    s = synth.AttnShape("norm", 512, 4, 2, 64, 16, 23, 10000.0)
    wqkv_f, wo_f = synth.attn_weights(s, seed=9)
    wqkv, wo = oracle.quantise(wqkv_f, 4), oracle.quantise(wo_f, 4)
    g = synth.norm_weights(s.H, seed=9)
    x = 3.0 * synth.tokens(synth.TINY, 2, seed=0, stream=13)
    hist = synth.kv_history(s, seed=10)
    k1, v1 = _caches(s.nkv, s.kv_len, s.d, hist)
    y1, _ = _run(s, wqkv, wo, k1, v1, x, 40, norm_w=g, norm_eps=1e-6)
    xn = oracle.rmsnorm(x, g, 1e-6)
    k2, v2 = _caches(s.nkv, s.kv_len, s.d, hist)
    y2, _ = _run(s, wqkv, wo, k2, v2, xn.astype(np.float32), 40, residual=False)
    np.testing.assert_allclose(y1, x + y2, rtol=0, atol=1e-5)


def test_positions_outside_the_cache_are_refused():
    s = synth.AttnShape("cap", 512, 4, 2, 64, 0, 32, 10000.0)
    wqkv_f, wo_f = synth.attn_weights(s)
    wqkv, wo = oracle.quantise(wqkv_f, 4), oracle.quantise(wo_f, 4)
    k, v = _caches(s.nkv, s.kv_len, s.d)
    x = synth.tokens(synth.TINY, 2, seed=0, stream=14)
    _run(s, wqkv, wo, k, v, x, 30)  # positions 30, 31 fit
    with pytest.raises(ValueError):
        _run(s, wqkv, wo, k, v, x, 31)
    r = synth.AttnShape("ring", 512, 4, 2, 64, 16, 15, 10000.0)  # ring shorter than its window
    with pytest.raises(ValueError):
        _run(r, wqkv, wo, np.zeros((2, 15, 64), np.uint16), np.zeros((2, 15, 64), np.uint16), x, 0)
