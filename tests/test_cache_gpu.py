"""Decode through the per-layer LFU expert cache, called through the C ABI.

Experts live in page-locked host memory (tile layout); the cache holds a few of
them on the device.  Every step is compared with the oracle (fp32 outputs within
2e-3 * (1 + |oracle|), expert indices bit-exact), and the cache's slot table and
hit/miss counts with the oracle's LFU policy run on the same request sequence
(bit-exact).  Workload: the tiny layer and the full-size layer with Zipf(1.1)
popularity, token sequences correlated across steps (AR(1), rho 0.9).
"""
import numpy as np
import pytest

import oracle
import synth
from layers import OracleLayer, gpu_layer, within_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _host_experts(gl):
    """The layer's tile-layout expert blobs, copied to page-locked host memory."""
    return gl.experts[0].cpu().pin_memory()


def _requests(idx):
    seen = []
    for e in idx.reshape(-1):
        if int(e) not in seen:
            seen.append(int(e))
    return seen


@pytest.mark.parametrize("policy", ["host", "device"])
@pytest.mark.parametrize("shape_name,slots,T,steps", [("tiny", 16, 1, 24), ("tiny", 10, 1, 30),
                                                      ("tiny", 16, 2, 12), ("full", 16, 1, 12)])
def test_cached_decode_matches_oracle_and_policy(shape_name, slots, T, steps, policy):
    """policy "device": the policy step runs on the GPU and the misses are fetched by
    a kernel from the mapped host blobs; same slot tables, counts and outputs."""
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.SHAPES[shape_name]
    bias = synth.popularity_bias(s, seed=0)
    gl = gpu_layer(s, seed=0, bias=bias)
    ol = OracleLayer(s, seed=0, bias=bias)
    cache = moe.Cache(s.H, s.E, s.I, _host_experts(gl), slots=slots)
    if policy == "device":
        cache.set_device_policy(True)
    policy = oracle.LFU(slots, s.E)
    layer = gl.view(experts=False)
    ws = moe.new_workspace(layer, T)
    xs = synth.token_sequence(s, steps * T, seed=0)
    idx = torch.empty((T, s.topk), dtype=torch.int32, device="cuda")
    for k in range(steps):
        x = xs[k * T:(k + 1) * T]
        y = moe.moe_layer_decode(layer, torch.from_numpy(x).cuda(), ws, idx=idx, cache=cache)
        torch.cuda.synchronize()
        gidx = idx.cpu().numpy()
        ry, ridx, _ = ol.layer(x)
        assert np.array_equal(gidx, ridx), k
        ok, worst = within_tol(y.cpu().numpy(), ry, TOL)
        assert ok, "step %d: worst err/bound %.3f" % (k, worst)
        policy.step(_requests(gidx))
        eos, cnt = cache.slots_state()
        reos, rcnt, _, rh, rm = policy.state()
        assert np.array_equal(eos, reos) and np.array_equal(cnt, rcnt), k
    hits, misses, h2d = cache.stats()
    assert (hits, misses) == policy.state()[3:]
    assert h2d == misses * moe.moe_tile_blob_bytes(s.H, s.I)
    assert misses > 0 and hits > 0
    cache.close()


def test_policy_switch_keeps_state():
    """Steps alternate between the host and the device policy; the slot table and the
    counts follow the oracle's policy throughout."""
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    bias = synth.popularity_bias(s, seed=0)
    gl, ol = gpu_layer(s, seed=0, bias=bias), OracleLayer(s, seed=0, bias=bias)
    cache = moe.Cache(s.H, s.E, s.I, _host_experts(gl), slots=12)
    policy = oracle.LFU(12, s.E)
    layer = gl.view(experts=False)
    ws = moe.new_workspace(layer, 1)
    xs = synth.token_sequence(s, 24, seed=1)
    idx = torch.empty((1, s.topk), dtype=torch.int32, device="cuda")
    for k in range(24):
        cache.set_device_policy(k % 6 >= 3)
        y = moe.moe_layer_decode(layer, torch.from_numpy(xs[k:k + 1]).cuda(), ws, idx=idx, cache=cache)
        torch.cuda.synchronize()
        ry, ridx, _ = ol.layer(xs[k:k + 1])
        assert np.array_equal(idx.cpu().numpy(), ridx), k
        assert within_tol(y.cpu().numpy(), ry, TOL)[0], k
        policy.step(_requests(idx.cpu().numpy()))
        eos, cnt = cache.slots_state()
        reos, rcnt, _, rh, rm = policy.state()
        assert np.array_equal(eos, reos) and np.array_equal(cnt, rcnt), k
        assert cache.stats()[:2] == (rh, rm), k
    assert cache.stats()[2] == cache.stats()[1] * moe.moe_tile_blob_bytes(s.H, s.I)
    cache.close()


def test_device_policy_capacity_error():
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    gl = gpu_layer(s, seed=0)
    cache = moe.Cache(s.H, s.E, s.I, _host_experts(gl), slots=12)
    cache.set_device_policy(True)
    layer = gl.view(experts=False)
    ws = moe.new_workspace(layer, 2)
    x = torch.from_numpy(synth.tokens(s, 2, seed=0, stream=3)).cuda()
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_decode(layer, x, ws, cache=cache)  # 2 tokens x top-8 > 12 slots
    assert e.value.status == moe.MOE_ECAPACITY
    assert cache.stats() == (0, 0, 0)
    cache.close()


def test_cache_capacity_error():
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    gl = gpu_layer(s, seed=0)
    cache = moe.Cache(s.H, s.E, s.I, _host_experts(gl), slots=4)
    layer = gl.view(experts=False)
    ws = moe.new_workspace(layer, 2)
    x = torch.from_numpy(synth.tokens(s, 2, seed=0, stream=3)).cuda()
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_decode(layer, x, ws, cache=cache)  # 2 tokens x top-8 > 4 slots
    assert e.value.status == moe.MOE_ECAPACITY
    assert cache.stats() == (0, 0, 0)
    cache.close()
