"""Exact router ties and degenerate weight groups, CUDA path vs the oracle.

The tie rule (larger logit first, equal logits -> lower expert index) decides
only when two logits are exactly equal.  Duplicating a router row before
quantisation gives two quantised rows with identical bytes, hence bit-identical
fp32 logits in every kernel (each row is summed in an order that does not depend
on its index) and equal logits in the oracle.  Three ties are built from the
oracle's own ranking of one token:
  * inside the top-k: the 6th-ranked expert gets the 3rd-ranked expert's row;
  * across the k-th / (k+1)-th boundary: an expert outside the top-k gets the
    k-th expert's row, once with a lower index (it displaces the k-th expert)
    and once with a higher one (it stays out);
  * every row equal: experts 0..k-1 in that order, each with gate exactly 1/k.
Each router goes through the three routers of the library: moe_route (the
standalone router), moe_layer_decode (the decode kernel's own router) and
moe_layer_prefill_chunk.  Indices must match bit for bit; gates and outputs
within 2e-3 * (1 + |oracle|).

The degenerate groups (constant groups with scale 0, groups of codes 0 and 15
only, groups at the maximum but for one element, a zero row) are planted in every
expert, routed and shared, and run through decode and prefill.
"""
import numpy as np
import pytest

import synth
from layers import OracleLayer, distinct_margin, extreme_groups, gpu_layer, within_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _cuda(a):
    return torch.as_tensor(np.ascontiguousarray(a)).cuda()


def _tied_routers(shape, x):
    """-> {case: router fp32 [E, H]} built from the oracle's ranking of token x."""
    base = synth.router_weights(shape, 0)
    k = shape.topk
    ol = OracleLayer(shape, seed=0)
    logits, idx, _ = ol.route(x[:1])
    rank = list(np.argsort(-logits[0], kind="stable"))
    top, rest = rank[:k], rank[k:]
    out = {}
    r = base.copy()
    r[top[5]] = r[top[2]]
    out["inside"] = r
    a = top[k - 1]
    lower = [e for e in rest if e < a]
    higher = [e for e in rest if e > a]
    if lower:
        r = base.copy()
        r[lower[0]] = r[a]
        out["boundary_lower"] = r
    if higher:
        r = base.copy()
        r[higher[0]] = r[a]
        out["boundary_higher"] = r
    out["all_equal"] = np.repeat(base[:1], shape.E, axis=0)
    return out


def _check_route(moe, gl, ol, x, case):
    T = x.shape[0]
    layer = gl.view()
    ws = moe.new_workspace(layer, T)
    rlog, ridx, rgate = ol.route(x)
    # only exact ties may be close: any other pair of logits is far enough apart
    # that an fp32 sum cannot reorder it
    bound = 1e-5 * np.max(np.abs(rlog)) + 1e-6
    assert np.all(distinct_margin(rlog, gl.topk) > bound), (case, "near-tie between different logits")
    logits = torch.empty((T, gl.E), dtype=torch.float32, device="cuda")
    idx, gate = moe.moe_route(layer, _cuda(x), ws, logits=logits)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), ridx), case
    assert within_tol(gate.cpu().numpy(), rgate, TOL)[0], case
    return ridx, rgate


def _check_layer(moe, gl, ol, x, prefill, case):
    T = x.shape[0]
    layer = gl.view()
    ws = moe.new_workspace(layer, T)
    idx = torch.empty((T, gl.topk), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, gl.topk), dtype=torch.float32, device="cuda")
    fn = moe.moe_layer_prefill_chunk if prefill else moe.moe_layer_decode
    y = fn(layer, _cuda(x), ws, idx=idx, gate=gate)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    ry, ridx, rgate = ol.layer(x)
    assert np.array_equal(idx.cpu().numpy(), ridx), (case, prefill)
    assert within_tol(gate.cpu().numpy(), rgate, TOL)[0], (case, prefill)
    ok, worst = within_tol(y.cpu().numpy(), ry, TOL)
    assert ok, "%s prefill=%s: worst err/bound %.3f" % (case, prefill, worst)
    return idx.cpu().numpy(), gate.cpu().numpy()


def _set_router(gl, ol, rw):
    """Replaces the router of both copies of the layer (the experts stay)."""
    import oracle
    gl.set_router(torch.from_numpy(np.ascontiguousarray(rw, np.float32)))
    ol.router = oracle.quantise(np.ascontiguousarray(rw, np.float32), 8)
    torch.cuda.synchronize()


@pytest.mark.parametrize("shape", [synth.TINY, synth.FULL], ids=["tiny", "full"])
def test_exact_router_ties(shape):
    import bit_affine_quantised_affine4_b300 as moe
    k = shape.topk
    gl, ol = gpu_layer(shape, seed=0), OracleLayer(shape, seed=0)
    x1 = synth.tokens(shape, 1, seed=0, stream=1100)
    cases = _tied_routers(shape, x1)
    assert set(cases) >= {"inside", "all_equal"} and ("boundary_lower" in cases or "boundary_higher" in cases)
    for case, rw in cases.items():
        _set_router(gl, ol, rw)
        ridx, rgate = _check_route(moe, gl, ol, x1, case)
        tied = np.flatnonzero(np.all(rw == rw[ridx[0][-1]], axis=1))
        if case == "all_equal":
            assert list(ridx[0]) == list(range(k))
            assert np.all(rgate == 1.0 / k)
        elif case == "boundary_lower":
            assert tied.size == 2 and ridx[0][-1] == tied.min(), "the lower index must take the last place"
        elif case == "boundary_higher":
            assert tied.size == 2 and ridx[0][-1] == tied.min() and tied.max() not in ridx[0]
        else:
            pair = [i for i, e in enumerate(ridx[0]) if np.array_equal(rw[e], rw[ridx[0][2]])]
            assert len(pair) == 2 and pair[1] == pair[0] + 1, "the tied pair sits side by side"
            assert ridx[0][pair[0]] < ridx[0][pair[1]], "lower index first"
        for prefill in (False, True):
            idx, gate = _check_layer(moe, gl, ol, x1, prefill, case)
            if case == "all_equal":
                assert np.array_equal(idx[0], np.arange(k)) and np.all(gate == np.float32(1.0 / k))
    # every row equal, several tokens at once: each token picks experts 0..k-1
    _set_router(gl, ol, cases["all_equal"])
    for T, prefill in ((16, False), (5, False), (37, True)):
        x = synth.tokens(shape, T, seed=0, stream=1200 + T)
        idx, gate = _check_layer(moe, gl, ol, x, prefill, "all_equal_T%d" % T)
        assert np.array_equal(idx, np.tile(np.arange(k), (T, 1)))


@pytest.mark.parametrize("shape", [synth.TINY, synth.FULL], ids=["tiny", "full"])
def test_degenerate_groups(shape):
    import bit_affine_quantised_affine4_b300 as moe
    bias = synth.popularity_bias(shape, seed=0)
    gl = gpu_layer(shape, seed=0, bias=bias, edit=extreme_groups)
    ol = OracleLayer(shape, seed=0, bias=bias, edit=extreme_groups)
    # the planted groups really are degenerate once quantised, and the GPU's
    # packed bytes equal the oracle's
    import oracle
    gu, d = extreme_groups(*synth.shared_weights(shape, 0))
    q, sc, _ = oracle.quantise(gu, 4)
    assert sc[0, 0] == 0 and np.all(q[0, :8] == 0), "constant group: scale 0, codes 0"
    codes = np.array([(q[2, 16 + j // 8] >> (4 * (j % 8))) & 15 for j in range(64)])
    assert set(codes.tolist()) == {0, 15}, "two-valued group: codes 0 and 15 only"
    codes = np.array([(q[7, 24 + j // 8] >> (4 * (j % 8))) & 15 for j in range(64)])
    assert np.sum(codes == 15) == 63 and codes[17] == 0
    mlx = oracle.untile_expert(gl.shared_blob_host(), shape.H, shape.Is)
    assert np.array_equal(mlx, ol.shared)
    for T, prefill in ((1, False), (3, False), (16, False), (1, True), (40, True)):
        x = synth.tokens(shape, T, seed=0, stream=1300 + T)
        _check_layer(moe, gl, ol, x, prefill, "degenerate")
