"""Failure paths, exercised without any GPU fault (called through the C ABI).

* A device-side wait that gives up: fault injection makes the decode kernel's
  routing wait expect one router row more than exist, with a 2 ms limit.  The
  wait runs out, the kernel drains without computing, moe_workspace_status
  reports MOE_ETIMEOUT once and re-initialises the workspace, and the next call
  matches the oracle again.
* A host -> device expert copy of a cached decode that fails: fault injection
  makes the call behave as if cudaMemcpyAsync had returned an error.  The call
  returns MOE_ECUDA, the cache's slot table, counts and statistics are those of
  before the call, and the next call (retrying the same step) matches the oracle
  and the oracle's LFU policy, which never saw the failed step.
* A prepared host call on a workspace whose error word is raised: the step
  completes, the status call reports and clears the error, the next step is right.
"""
import numpy as np
import pytest

import oracle
import synth
from layers import OracleLayer, gpu_layer, within_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _requests(idx):
    seen = []
    for e in idx.reshape(-1):
        if int(e) not in seen:
            seen.append(int(e))
    return seen


@pytest.mark.parametrize("T", [1, 4, 12])
def test_device_wait_times_out_and_recovers(T):
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    gl, ol = gpu_layer(s, seed=0), OracleLayer(s, seed=0)
    layer = gl.view()
    ws = moe.new_workspace(layer, T)
    x = synth.tokens(s, T, seed=0, stream=1400 + T)
    xd = torch.from_numpy(x).cuda()
    moe.moe_layer_decode(layer, xd, ws)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    moe.moe_debug_inject(moe.MOE_INJECT_WAIT)
    moe.moe_layer_decode(layer, xd, ws)
    assert moe.moe_workspace_status(ws) == moe.MOE_ETIMEOUT
    assert moe.moe_workspace_status(ws) == moe.MOE_OK  # re-initialised
    for _ in range(2):
        idx = torch.empty((T, s.topk), dtype=torch.int32, device="cuda")
        y = moe.moe_layer_decode(layer, xd, ws, idx=idx)
        assert moe.moe_workspace_status(ws) == moe.MOE_OK
        ry, ridx, _ = ol.layer(x)
        assert np.array_equal(idx.cpu().numpy(), ridx)
        ok, worst = within_tol(y.cpu().numpy(), ry, TOL)
        assert ok, worst


def test_prepared_host_call_after_a_wait_gave_up():
    # a prepared host call on a workspace whose error word another call raised: the
    # step still completes and signals (the kernel drains), moe_workspace_status
    # reports MOE_ETIMEOUT and re-initialises the workspace, and the handle's next
    # step equals its first bit for bit
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    gl = gpu_layer(s, seed=0)
    layer = gl.view()
    ws = moe.new_workspace(layer, 1)
    x = torch.from_numpy(synth.tokens(s, 1, seed=0, stream=1500)).pin_memory()
    hc = moe.HostCall(layer, ws, T=1)
    y0 = torch.empty_like(x)
    hc(x, y0)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    moe.moe_debug_inject(moe.MOE_INJECT_WAIT)
    moe.moe_layer_decode(layer, x.cuda(), ws)
    y1 = torch.empty_like(x)
    hc(x, y1)  # returns: the step ends without waiting on anything that will not come
    assert moe.moe_workspace_status(ws) == moe.MOE_ETIMEOUT
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    y2 = torch.empty_like(x)
    hc(x, y2)
    assert np.array_equal(y2.numpy(), y0.numpy())
    hc.close()


def test_inject_rejects_unknown_kind():
    import bit_affine_quantised_affine4_b300 as moe
    with pytest.raises(moe.MoeError) as e:
        moe.moe_debug_inject(9)
    assert e.value.status == moe.MOE_EINVAL
    moe.moe_debug_inject(moe.MOE_INJECT_NONE)


def test_failed_expert_copy_leaves_cache_unchanged():
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    bias = synth.popularity_bias(s, seed=0)
    gl, ol = gpu_layer(s, seed=0, bias=bias), OracleLayer(s, seed=0, bias=bias)
    slots = 10
    cache = moe.Cache(s.H, s.E, s.I, gl.experts[0].cpu().pin_memory(), slots=slots)
    policy = oracle.LFU(slots, s.E)
    layer = gl.view(experts=False)
    ws = moe.new_workspace(layer, 1)
    xs = synth.token_sequence(s, 16, seed=0)
    idx = torch.empty((1, s.topk), dtype=torch.int32, device="cuda")
    failed = 0
    for k in range(16):
        x = torch.from_numpy(xs[k:k + 1]).cuda()
        y = None
        if k in (0, 5, 11):
            before = (cache.slots_state(), cache.stats())
            moe.moe_debug_inject(moe.MOE_INJECT_COPY)
            try:
                y = moe.moe_layer_decode(layer, x, ws, idx=idx, cache=cache)
            except moe.MoeError as e:
                assert e.status == moe.MOE_ECUDA
                failed += 1
                after = (cache.slots_state(), cache.stats())
                assert np.array_equal(before[0][0], after[0][0]) and np.array_equal(before[0][1], after[0][1])
                assert before[1] == after[1]
                torch.cuda.synchronize()
                assert moe.moe_workspace_status(ws) == moe.MOE_OK
            moe.moe_debug_inject(moe.MOE_INJECT_NONE)  # a step without a miss consumed nothing
        if y is None:
            y = moe.moe_layer_decode(layer, x, ws, idx=idx, cache=cache)  # the step (or its retry)
        torch.cuda.synchronize()
        gidx = idx.cpu().numpy()
        ry, ridx, _ = ol.layer(xs[k:k + 1])
        assert np.array_equal(gidx, ridx), k
        assert within_tol(y.cpu().numpy(), ry, TOL)[0], k
        policy.step(_requests(gidx))
        eos, cnt = cache.slots_state()
        reos, rcnt, _, _, _ = policy.state()
        assert np.array_equal(eos, reos) and np.array_equal(cnt, rcnt), k
    assert failed >= 1  # step 0 starts from an empty cache: it has misses
    hits, misses, h2d = cache.stats()
    assert (hits, misses) == policy.state()[3:]
    cache.close()
