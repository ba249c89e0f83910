"""A stack of MoE layers decoded through per-layer LFU caches (the 30-layer stack
workload, scaled down in depth: the tiny layer, and 3 layers of the full-size
layer with 16 slots each), called through the C ABI.

Each layer has its own experts in page-locked host memory and its own device
cache; attention is the identity, so a step is h <- h + MoE_l(h) for l = 1..L.
Parity is teacher-forced per layer: the oracle layer runs on the GPU's input to
that layer, and each layer's LFU policy (oracle) runs on the GPU's request
sequence for that layer.  Checked every step: expert indices bit-exact, outputs
within 2e-3 * (1 + |oracle|), slot tables and hit/miss counts bit-exact.  A
free-running oracle stack (its own h) is also run, and the step at which its
routing first differs from the GPU's is reported (none is expected here).
"""
import numpy as np
import pytest

import oracle
import synth
from layers import OracleLayer, gpu_layer, norm_weights, within_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _requests(idx):
    seen = []
    for e in idx.reshape(-1):
        if int(e) not in seen:
            seen.append(int(e))
    return seen


@pytest.mark.parametrize("shape_name,layers,slots,steps,prenorm,policy", [("tiny", 3, 16, 10, False, "host"),
                                                                           ("tiny", 2, 10, 12, False, "device"),
                                                                           ("tiny", 3, 16, 8, True, "device"),
                                                                           ("full", 3, 16, 6, True, "host"),
                                                                           ("full", 3, 16, 6, True, "device")])
def test_stack_teacher_forced(shape_name, layers, slots, steps, prenorm, policy):
    """prenorm: each layer is the pre-norm block h <- h + MoE(RMSNorm(h)), which
    keeps the activations of a deep stack bounded (the plain residual stack grows
    layer over layer, GeGLU being quadratic)."""
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.SHAPES[shape_name]
    gls, ols, caches, views, policies, norms = [], [], [], [], [], []
    for l in range(layers):
        bias = synth.popularity_bias(s, seed=0, layer=l)
        norm = (norm_weights(s, 0, l), 1e-6) if prenorm else None
        norms.append(norm)
        gl = gpu_layer(s, seed=0, layer=l, bias=bias, norm=norm)
        gls.append(gl)
        ols.append(OracleLayer(s, seed=0, layer=l, bias=bias))
        caches.append(moe.Cache(s.H, s.E, s.I, gl.experts[0].cpu().pin_memory(), slots=slots))
        if policy == "device":
            caches[-1].set_device_policy(True)
        views.append(gl.view(experts=False))
        policies.append(oracle.LFU(slots, s.E))
    ws = moe.new_workspace(views[0], 1)
    idx = torch.empty((1, s.topk), dtype=torch.int32, device="cuda")
    xs = synth.token_sequence(s, steps, seed=0)
    h_free = None
    first_divergence = None
    for k in range(steps):
        h = torch.from_numpy(xs[k:k + 1]).cuda()
        h_free = xs[k:k + 1].astype(np.float64)
        for l in range(layers):
            h_in = h.cpu().numpy()
            flags = moe.MOE_RESIDUAL | (moe.MOE_PRENORM if prenorm else 0)
            y = moe.moe_layer_decode(views[l], h, ws, flags=flags, idx=idx, cache=caches[l])
            torch.cuda.synchronize()
            gidx = idx.cpu().numpy()
            if prenorm:
                ry, ridx, _ = ols[l].block(h_in, *norms[l])
            else:
                ry, ridx, _ = ols[l].layer(h_in, residual=True)
            assert np.array_equal(gidx, ridx), (k, l)
            ok, worst = within_tol(y.cpu().numpy(), ry, TOL)
            assert ok, "step %d layer %d: worst err/bound %.3f" % (k, l, worst)
            policies[l].step(_requests(gidx))
            eos, cnt = caches[l].slots_state()
            reos, rcnt, _, _, _ = policies[l].state()
            assert np.array_equal(eos, reos) and np.array_equal(cnt, rcnt), (k, l)
            # the free-running oracle stack, for the report only
            if prenorm:
                fy, fidx, _ = ols[l].block(h_free.astype(np.float32), *norms[l])
            else:
                fy, fidx, _ = ols[l].layer(h_free.astype(np.float32), residual=True)
            if first_divergence is None and not np.array_equal(fidx, gidx):
                first_divergence = (k, l)
            h_free = fy
            h = y
    for l in range(layers):
        hits, misses, h2d = caches[l].stats()
        assert (hits, misses) == policies[l].state()[3:]
        assert h2d == misses * moe.moe_tile_blob_bytes(s.H, s.I)
        caches[l].close()
    print("free-running routing: first divergence", first_divergence)
