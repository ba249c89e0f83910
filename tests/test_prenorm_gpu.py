"""The pre-norm MoE block, CUDA path vs the oracle, through the C ABI.

With MOE_PRENORM the router and the experts read RMSNorm(x) = x * w / rms(x)
and MOE_RESIDUAL adds the raw x: y = x + MoE(RMSNorm(x)).  The oracle computes
RMSNorm in fp64 and runs its layer on the result (rounded to fp32, the layer's
input type).  Checked: the standalone moe_rmsnorm; decode (tiny and full-size,
T up to 16); the prefill chunk; decode through the LFU cache.  Indices must match
bit for bit (with the usual near-tie guard); outputs within 2e-3 * (1 + |oracle|).
"""
import numpy as np
import pytest

import oracle
import synth
from layers import OracleLayer, gpu_layer, norm_weights, topk_margin, within_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3
EPS = 1e-6


def _cuda(a):
    return torch.as_tensor(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("T,H,eps", [(1, 512, 1e-6), (16, 2816, 1e-6), (5, 384, 0.5), (3, 4096, 0.0)])
def test_rmsnorm_matches_oracle(T, H, eps):
    import bit_affine_quantised_affine4_b300 as moe
    x = synth.normal(synth.key(3, T, H), (T, H), 1.5)
    x[0, :7] = 40.0  # a few large values
    w = synth.normal(synth.key(4, H), (H,), 1.0)
    y = moe.moe_rmsnorm(_cuda(x), _cuda(w), eps)
    ref = oracle.rmsnorm(x, w, eps)
    ok, worst = within_tol(y.cpu().numpy(), ref, 1e-5)
    assert ok, worst
    # in place
    xd = _cuda(x)
    moe.moe_rmsnorm(xd, _cuda(w), eps, y=xd)
    assert np.array_equal(xd.cpu().numpy(), y.cpu().numpy())


def _block_check(moe, s, gl, ol, x, norm, prefill=False, residual=True):
    T = x.shape[0]
    layer = gl.view()
    ws = moe.new_workspace(layer, T)
    idx = torch.empty((T, s.topk), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, s.topk), dtype=torch.float32, device="cuda")
    flags = moe.MOE_PRENORM | (moe.MOE_RESIDUAL if residual else 0)
    fn = moe.moe_layer_prefill_chunk if prefill else moe.moe_layer_decode
    y = fn(layer, _cuda(x), ws, flags=flags, idx=idx, gate=gate)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    rlog, _, _ = ol.route_normed(x, *norm)
    bound = 1e-5 * np.max(np.abs(rlog)) + 1e-6
    assert np.all(topk_margin(rlog, s.topk) > bound), "near-tie at the top-k boundary"
    ry, ridx, rgate = ol.block(x, *norm)
    if not residual:
        ry = ry - x.astype(np.float64)
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert within_tol(gate.cpu().numpy(), rgate, TOL)[0]
    ok, worst = within_tol(y.cpu().numpy(), ry, TOL)
    assert ok, "worst err/bound %.3f" % worst


@pytest.mark.parametrize("shape", [synth.TINY, synth.FULL], ids=["tiny", "full"])
def test_prenorm_decode_and_prefill(shape):
    import bit_affine_quantised_affine4_b300 as moe
    bias = synth.popularity_bias(shape, seed=0)
    norm = (norm_weights(shape, 0), EPS)
    gl = gpu_layer(shape, seed=0, bias=bias, norm=norm)
    ol = OracleLayer(shape, seed=0, bias=bias)
    for T in (1, 4, 16):
        # inputs of varied scale: the layer must see the normalised vector
        x = synth.tokens(shape, T, seed=0, stream=1500 + T) * np.float32(3.0 if T == 4 else 1.0)
        _block_check(moe, shape, gl, ol, x, norm)
    _block_check(moe, shape, gl, ol, synth.tokens(shape, 2, seed=0, stream=1520), norm, residual=False)
    _block_check(moe, shape, gl, ol, synth.tokens(shape, 37, seed=0, stream=1530), norm, prefill=True)
    if shape is synth.FULL:
        _block_check(moe, shape, gl, ol, synth.tokens(shape, 128, seed=0, stream=1540), norm, prefill=True)


def test_prenorm_cached_decode():
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    bias = synth.popularity_bias(s, seed=0)
    norm = (norm_weights(s, 0), EPS)
    gl = gpu_layer(s, seed=0, bias=bias, norm=norm)
    ol = OracleLayer(s, seed=0, bias=bias)
    cache = moe.Cache(s.H, s.E, s.I, gl.experts[0].cpu().pin_memory(), slots=10)
    layer = gl.view(experts=False)
    ws = moe.new_workspace(layer, 2)
    xs = synth.token_sequence(s, 16, seed=0)
    idx = torch.empty((2, s.topk), dtype=torch.int32, device="cuda")
    for k in range(8):
        x = xs[2 * k:2 * k + 2]
        y = moe.moe_layer_decode(layer, _cuda(x), ws, flags=moe.MOE_PRENORM | moe.MOE_RESIDUAL, idx=idx,
                                 cache=cache)
        torch.cuda.synchronize()
        ry, ridx, _ = ol.block(x, *norm)
        assert np.array_equal(idx.cpu().numpy(), ridx), k
        assert within_tol(y.cpu().numpy(), ry, TOL)[0], k
    cache.close()


def test_prenorm_requires_norm_weight():
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.TINY
    gl = gpu_layer(s, seed=0)
    layer = gl.view()
    ws = moe.new_workspace(layer, 1)
    x = torch.zeros((1, s.H), device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_decode(layer, x, ws, flags=moe.MOE_PRENORM)
    assert e.value.status == moe.MOE_EINVAL
