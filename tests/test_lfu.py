"""The library's cache policy (moe_lfu_*, host code, no GPU) against the oracle's
policy and the hand-worked traces of tests/golden/lfu_traces.json.

Slot assignments, hit flags and the full policy state must agree bit for bit,
step by step, on hand-made and on seeded random request sequences (Zipf-like
popularity, correlated steps, ties).
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "lfu_traces.json")


@pytest.fixture(scope="module")
def moe():
    import bit_affine_quantised_affine4_b300 as m
    return m


def _cases():
    return {c["name"]: c for c in json.load(open(GOLDEN))["cases"]}


def test_hand_trace(moe):
    c = _cases()["fill_hit_evict_ties"]
    lfu = moe.LFU(c["slots"], c["E"])
    for st in c["steps"]:
        slot, hit = lfu.step(st["req"])
        assert list(slot) == st["slot"] and list(hit.astype(int)) == st["hit"], st
    eos, cnt, last, hits, misses = lfu.state()
    f = c["final"]
    assert list(eos) == f["expert_of_slot"] and list(cnt) == f["count"]
    assert list(last) == f["last"] and (hits, misses) == (f["hits"], f["misses"])


def test_cyclic_thrash(moe):
    c = _cases()["seventeen_cyclic_thrash"]
    lfu = moe.LFU(c["slots"], c["E"])
    for s in range(c["cyclic"]["steps"]):
        slot, hit = lfu.step([s % c["cyclic"]["period"]])
        assert not hit[0] and slot[0] == s % 16
    assert lfu.state()[3:] == (c["hits"], c["misses"])


def test_hot_set_stays(moe):
    c = _cases()["hot_eight_never_evicted"]
    lfu = moe.LFU(c["slots"], c["E"])
    for s in range(c["steps"]):
        req = c["hot"] + [c["cold_base"] + s % c["cold_count"]]
        slot, hit = lfu.step(req)
        assert list(slot[:8]) == c["hot_slots"]
        assert bool(hit[8]) is False
        assert all(hit[:8]) == (s > 0)
    assert lfu.state()[3:] == (c["hits"], c["misses"])


def test_rejects_bad_requests_without_change(moe):
    lfu = moe.LFU(4, 10)
    lfu.step([1, 2])
    before = lfu.state()
    for bad, status in (([3, 3], moe.MOE_EINVAL), ([10], moe.MOE_EINVAL), ([-1], moe.MOE_EINVAL),
                        ([0, 1, 2, 3, 4], moe.MOE_ECAPACITY)):
        with pytest.raises(moe.MoeError) as e:
            lfu.step(bad)
        assert e.value.status == status
    after = lfu.state()
    for a, b in zip(before, after):
        assert np.array_equal(a, b)


def _zipf_requests(rng, E, n_req, steps, s=1.1, corr=0.7):
    """Request lists of n_req distinct experts drawn by Zipf(s) popularity over a
    random permutation; each step keeps each previous expert with probability corr."""
    p = 1.0 / np.arange(1, E + 1) ** s
    p /= p.sum()
    perm = rng.permutation(E)
    prev = []
    for _ in range(steps):
        req = [e for e in prev if rng.random() < corr]
        while len(req) < n_req:
            e = int(perm[rng.choice(E, p=p)])
            if e not in req:
                req.append(e)
        rng.shuffle(req)
        prev = req
        yield req


@pytest.mark.parametrize("slots,E,n_req,seed", [(16, 128, 8, 0), (16, 128, 16, 1), (4, 12, 3, 2),
                                                (16, 32, 12, 3), (64, 256, 40, 4), (1, 3, 1, 5)])
def test_matches_oracle_on_random_sequences(moe, slots, E, n_req, seed):
    rng = np.random.default_rng(seed)
    ours, ref = moe.LFU(slots, E), oracle.LFU(slots, E)
    for req in _zipf_requests(rng, E, n_req, 300):
        s1, h1 = ours.step(req)
        s2, h2 = ref.step(req)
        assert np.array_equal(s1, s2) and np.array_equal(h1, h2), req
    for a, b in zip(ours.state(), ref.state()):
        assert np.array_equal(a, b)
