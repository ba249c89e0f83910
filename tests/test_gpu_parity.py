"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bars: quantiser bytes and expert indices bit-exact; fp32 outputs within
max|gpu - oracle| <= 2e-3 * (1 + |oracle|).  Inputs are the seeded synthetic
workloads (weights N(0, 0.02) quantised 4-bit g64 / router 8-bit g64, tokens
N(0, 1)); the tiny layer runs whole, the full-size layer is checked on every
output of the sampled tokens.
"""
import numpy as np
import pytest

import oracle
import synth
from layers import OracleLayer, gpu_layer, topk_margin, within_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def moe():
    import bit_affine_quantised_affine4_b300 as m
    return m


def _cuda(a, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


# ------------------------------------------------------------------ quantiser

@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("N,K", [(7, 64), (33, 2816), (1408, 704)])
def test_quantiser_bit_exact(moe, bits, N, K):
    w = synth.normal(synth.key(1, N, K, bits), (N, K), 0.02)
    w[0, :64] = 0.5  # constant group: scale 0
    w[-1, -64:] = np.linspace(-3, 3, 64, dtype=np.float32)
    q, s, b = moe.affine_quantise(_cuda(w), bits)
    oq, os_, ob = oracle.quantise(w, bits)
    assert np.array_equal(q.cpu().numpy().view(np.uint32), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint16), os_)
    assert np.array_equal(b.cpu().numpy().view(np.uint16), ob)


# ------------------------------------------------------------------ tile layout

@pytest.mark.parametrize("H,I", [(128, 64), (384, 192), (2816, 704), (2816, 2112)])
def test_expert_tile_bit_exact(moe, H, I):
    """moe_expert_tile on random bytes: the oracle's untile gives back the input."""
    n = oracle.expert_blob_bytes(H, I)
    rng = np.random.default_rng(H + I)
    mlx = rng.integers(0, 256, n, dtype=np.uint8)
    # padding between the MLX parts is not part of the expert: keep it zero
    off = oracle.expert_blob_offsets(H, I)
    sizes = [I * H, 2 * I * (H // 64) * 2, 2 * I * (H // 64) * 2, H * I // 2, H * (I // 64) * 2,
             H * (I // 64) * 2]
    keep = np.zeros(n, bool)
    for o, sz in zip(off, sizes):
        keep[o:o + sz] = True
    mlx[~keep] = 0
    tiles = torch.empty(moe.moe_tile_blob_bytes(H, I), dtype=torch.uint8, device="cuda")
    moe.moe_expert_tile(_cuda(mlx), H, I, tiles)
    back = oracle.untile_expert(tiles.cpu().numpy(), H, I)
    assert np.array_equal(back, mlx)


# ------------------------------------------------------------------ qgemv

@pytest.mark.parametrize("N,K", [(4, 64), (100, 320), (4224, 2816), (2816, 704), (2816, 2112), (16, 64),
                                 (48, 8192), (8192, 2816), (2816, 4096)])
def test_qgemv_affine4(moe, N, K):
    w = synth.normal(synth.key(2, N, K), (N, K), 0.02)
    x = synth.normal(synth.key(3, N, K), (K,), 1.0)
    q, s, b = oracle.quantise(w, 4)
    y = moe.qgemv_affine4(_cuda(q.view(np.int32)), _cuda(s.view(np.int16)), _cuda(b.view(np.int16)),
                          K, _cuda(x))
    ref = oracle.qgemv(q, s, b, K, 4, x)
    ok, worst = within_tol(y.cpu().numpy(), ref, TOL)
    assert ok, worst


# ------------------------------------------------------------------ layers

@pytest.fixture(scope="module")
def tiny(moe):
    s = synth.TINY
    return s, gpu_layer(s, seed=0), OracleLayer(s, seed=0)


@pytest.fixture(scope="module")
def full_zipf(moe):
    s = synth.FULL
    bias = synth.popularity_bias(s, seed=0)
    return s, gpu_layer(s, seed=0, bias=bias), OracleLayer(s, seed=0, bias=bias)


@pytest.fixture(scope="module")
def full_uniform(moe):
    s = synth.FULL
    return s, gpu_layer(s, seed=0), OracleLayer(s, seed=0)


def _blobs_match(gl, ol, experts):
    """The GPU's quantised weights (tile layout, read back through the oracle's
    untile) equal the oracle's own quantisation, bit for bit."""
    rq, rs, rb = gl.router_host()
    assert np.array_equal(rq, ol.router[0]) and np.array_equal(rs, ol.router[1])
    assert np.array_equal(rb, ol.router[2])
    assert np.array_equal(oracle.untile_expert(gl.shared_blob_host(), gl.H, gl.Is), ol.shared)
    for e in experts:
        assert np.array_equal(oracle.untile_expert(gl.expert_blob_host(int(e)), gl.H, gl.I),
                              ol.expert(int(e))), e


def _route_check(moe, shape, gl, ol, T, stream_id):
    x = synth.tokens(shape, T, seed=0, stream=stream_id)
    layer = gl.view()
    ws = moe.new_workspace(layer, T)
    logits = torch.empty((T, shape.E), dtype=torch.float32, device="cuda")
    idx, gate = moe.moe_route(layer, _cuda(x), ws, logits=logits)
    rlog, ridx, rgate = ol.route(x)
    # a near-tie within the fp32 error bound would make an index flip legitimate;
    # at these seeds there is none, and the test says so if one appears
    bound = 1e-5 * np.max(np.abs(rlog)) + 1e-6
    assert np.all(topk_margin(rlog, shape.topk) > bound), "near-tie at the top-k boundary"
    assert np.array_equal(idx.cpu().numpy(), ridx)
    assert within_tol(gate.cpu().numpy(), rgate, TOL)[0]
    assert within_tol(logits.cpu().numpy(), rlog, TOL)[0]
    return x


def test_route_tiny(moe, tiny):
    s, gl, ol = tiny
    _blobs_match(gl, ol, [])
    for T in (1, 5, 16, 128):
        _route_check(moe, s, gl, ol, T, 10 + T)


def test_route_full(moe, full_zipf):
    s, gl, ol = full_zipf
    _blobs_match(gl, ol, [])
    for T in (1, 16, 128):
        _route_check(moe, s, gl, ol, T, 20 + T)


def _layer_check(moe, shape, gl, ol, T, stream_id, prefill=False, residual=False, check_tokens=None):
    x = synth.tokens(shape, T, seed=0, stream=stream_id)
    layer = gl.view()
    ws = moe.new_workspace(layer, T)
    idx = torch.empty((T, shape.topk), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, shape.topk), dtype=torch.float32, device="cuda")
    fn = moe.moe_layer_prefill_chunk if prefill else moe.moe_layer_decode
    flags = moe.MOE_RESIDUAL if residual else 0
    y = fn(layer, _cuda(x), ws, flags=flags, idx=idx, gate=gate)
    torch.cuda.synchronize()
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    toks = list(range(T)) if check_tokens is None else check_tokens
    ry, ridx, rgate = ol.layer(x[toks], residual=residual)
    _blobs_match(gl, ol, np.unique(ridx))
    assert np.array_equal(idx.cpu().numpy()[toks], ridx)
    assert within_tol(gate.cpu().numpy()[toks], rgate, TOL)[0]
    ok, worst = within_tol(y.cpu().numpy()[toks], ry, TOL)
    assert ok, "worst err/bound %.3f" % worst
    return worst


@pytest.mark.parametrize("T", [1, 2, 3, 8, 16])
def test_decode_tiny(moe, tiny, T):
    s, gl, ol = tiny
    _layer_check(moe, s, gl, ol, T, 100 + T)


def test_decode_tiny_residual(moe, tiny):
    s, gl, ol = tiny
    _layer_check(moe, s, gl, ol, 4, 150, residual=True)


def test_decode_full_uniform_T1(moe, full_uniform):
    s, gl, ol = full_uniform
    for sid in range(3):
        _layer_check(moe, s, gl, ol, 1, 200 + sid)


@pytest.mark.parametrize("T", [1, 2, 4, 8, 16])
def test_decode_full_zipf_batch(moe, full_zipf, T):
    s, gl, ol = full_zipf
    _layer_check(moe, s, gl, ol, T, 300 + T)


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("T", [1, 5, 16])
def test_decode_host_buffers(moe, tiny, T, pinned):
    # moe_layer_decode_host: host x/y/idx/gate, copies and the stream wait inside the
    # call (pinned, mapped buffers: kernels read and write host memory directly;
    # pageable ones: DMA copies through the workspace); the result equals the
    # device-pointer call's and is within the oracle's tolerance
    s, gl, ol = tiny
    x = synth.tokens(s, T, seed=0, stream=700 + T)
    layer = gl.view()
    ws = moe.new_workspace(layer, T)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    xh = pin(torch.from_numpy(x))
    yh = pin(torch.full_like(xh, float("nan")))
    ih = pin(torch.full((T, s.topk), -1, dtype=torch.int32))
    gh = pin(torch.empty((T, s.topk), dtype=torch.float32))
    moe.moe_layer_decode_host(layer, xh, ws, y=yh, flags=moe.MOE_RESIDUAL, idx=ih, gate=gh)
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    yd = moe.moe_layer_decode(layer, _cuda(x), ws, flags=moe.MOE_RESIDUAL)
    torch.cuda.synchronize()
    assert np.array_equal(yh.numpy(), yd.cpu().numpy())
    ry, ridx, rgate = ol.layer(x, residual=True)
    assert np.array_equal(ih.numpy(), ridx)
    assert within_tol(gh.numpy(), rgate, TOL)[0]
    ok, worst = within_tol(yh.numpy(), ry, TOL)
    assert ok, "worst err/bound %.3f" % worst
    with pytest.raises(ValueError):
        moe.moe_layer_decode_host(layer, _cuda(x), ws)
    if T == 1:  # the reusable call object: the same call, arguments marshalled once
        call = moe.DecodeHostCall(layer, ws, flags=moe.MOE_RESIDUAL)
        y2 = pin(torch.full_like(xh, float("nan")))
        call(xh, y2)
        assert np.array_equal(y2.numpy(), yh.numpy())
        call(xh.data_ptr(), y2.data_ptr())  # plain addresses
        assert np.array_equal(y2.numpy(), yh.numpy())


@pytest.mark.parametrize("T", [1, 5])
def test_host_call(moe, tiny, T):
    # the prepared host call (a recorded graph per layer, workspace, T and flags):
    # consecutive steps on one handle equal the device-pointer call bit for bit,
    # from pinned and from pageable rows and from the handle's own staging rows
    s, gl, ol = tiny
    x = synth.tokens(s, 4 * T, seed=0, stream=720 + T)
    layer = gl.view()
    ws = moe.new_workspace(layer, 16)
    hc = moe.HostCall(layer, ws, T=T, flags=moe.MOE_RESIDUAL)
    for k in range(3):
        xk = torch.from_numpy(x[k * T:(k + 1) * T].copy())
        if k != 1:
            xk = xk.pin_memory()
        yk = torch.full_like(xk, float("nan"))
        hc(xk, yk)
        yd = moe.moe_layer_decode(layer, _cuda(xk.numpy()), ws, flags=moe.MOE_RESIDUAL)
        torch.cuda.synchronize()
        assert np.array_equal(yk.numpy(), yd.cpu().numpy())
    hc.x_row.copy_(torch.from_numpy(x[3 * T:]))
    hc(hc.x_row, hc.y_row)
    ry, _, _ = ol.layer(x[3 * T:], residual=True)
    ok, worst = within_tol(hc.y_row.numpy(), ry, TOL)
    assert ok, "worst err/bound %.3f" % worst
    assert moe.moe_workspace_status(ws) == moe.MOE_OK
    hc.close()
    for bad_T in (0, moe.MOE_MAX_DECODE_TOKENS + 1):
        with pytest.raises(moe.MoeError):
            moe.HostCall(layer, ws, T=bad_T)


@pytest.mark.parametrize("T", [1, 37, 128])
def test_prefill_tiny(moe, tiny, T):
    s, gl, ol = tiny
    _layer_check(moe, s, gl, ol, T, 400 + T, prefill=True)


def test_prefill_full_zipf_128(moe, full_zipf):
    # every one of the 128 tokens, outputs and routing
    s, gl, ol = full_zipf
    _layer_check(moe, s, gl, ol, 128, 500, prefill=True)


def test_odd_shapes(moe):
    """A small layer whose sizes are not powers of two: H 384, I 192, Is 320, E 13, top-5."""
    s = synth.Shape("odd", 384, 13, 5, 192, 320)
    gl, ol = gpu_layer(s, seed=3), OracleLayer(s, seed=3)
    for T in (1, 7):
        _layer_check(moe, s, gl, ol, T, 600 + T)
    _layer_check(moe, s, gl, ol, 29, 650, prefill=True)


def test_many_experts_topk1(moe):
    s = synth.Shape("wide", 256, 256, 1, 64, 64)
    gl, ol = gpu_layer(s, seed=4), OracleLayer(s, seed=4)
    _layer_check(moe, s, gl, ol, 16, 700)


def test_prefill_router_fallback(moe):
    # 256 experts with top-1: the chunk router's slice partials would not fit the
    # down GEMM's scratch (E * ceil(H/128) > topk * H), so the chunk takes the
    # decode path's router; three 16-token groups of it
    s = synth.Shape("wide", 256, 256, 1, 64, 64)
    gl, ol = gpu_layer(s, seed=4), OracleLayer(s, seed=4)
    _layer_check(moe, s, gl, ol, 40, 702, prefill=True)


def test_prefill_ragged_router_tiles(moe):
    # the chunk router's tiles with ragged edges: 100 experts (a partial second
    # 64-row block), 77 tokens (a partial third 32-token block), three K slices
    s = synth.Shape("ragged", 384, 100, 6, 128, 192)
    gl, ol = gpu_layer(s, seed=6), OracleLayer(s, seed=6)
    _layer_check(moe, s, gl, ol, 77, 703, prefill=True)


@pytest.mark.parametrize("shape", ["tiny", "full"])
def test_degenerate_routing(moe, shape):
    # every token picks the same top-k experts (a router bias of 10 on experts
    # 0..topk-1, far above the spread of the router's dot products): each routed
    # weight block is one item of all 128 tokens, the largest token tiles of the
    # chunk, and each down item reads h from a single expert's gate/up items
    s = synth.TINY if shape == "tiny" else synth.FULL
    bias = np.zeros(s.E, dtype=np.float32)
    bias[:s.topk] = 10.0
    gl, ol = gpu_layer(s, seed=7, bias=bias), OracleLayer(s, seed=7, bias=bias)
    _layer_check(moe, s, gl, ol, 128, 704, prefill=True)
    # and a 16-token decode step whose tokens all share their experts
    _layer_check(moe, s, gl, ol, 16, 705)


def test_rejects_bad_calls(moe, tiny):
    s, gl, ol = tiny
    layer = gl.view()
    ws = moe.new_workspace(layer, 4)
    x = torch.zeros((8, s.H), device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_prefill_chunk(layer, x, ws)  # 8 tokens > workspace T_max 4
    assert e.value.status == moe.MOE_EWORKSPACE
    small = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_decode(layer, x, small)  # far too small for 8 decode tokens
    assert e.value.status == moe.MOE_EWORKSPACE
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_decode(layer, torch.zeros((17, s.H), device="cuda"), moe.new_workspace(layer, 17))
    assert e.value.status == moe.MOE_EINVAL
    with pytest.raises(moe.MoeError) as e:
        moe.moe_layer_decode(layer, x[:2], ws, y=x[:2])  # y aliases x
    assert e.value.status == moe.MOE_EINVAL
