"""The attention block, CUDA path (moe_attn_step through the C ABI) vs the oracle.

Both sides start from the same quantised weights (the library's quantiser on the
GPU, the oracle's on the CPU; the two agree bit for bit) and the same binary16
cache contents, then run the same sequence of calls: a prefill chunk, decode steps
that wrap the ring of a sliding-window layer, chunks at the end of a full layer's
store.  After every call the outputs y and o (the attention output before Wo) and
the whole key/value cache are compared, elementwise, within
|gpu - oracle| <= 2e-3 (1 + |oracle|): the projections take fp16 activations on the
tensor cores and accumulate in fp32, the attention runs in fp32, the oracle in fp64
with the cache in binary16 on both sides.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL = 2e-3


def within(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref) - TOL * (1.0 + np.abs(ref))
    worst = np.unravel_index(np.argmax(err), err.shape) if err.size else None
    assert err.size == 0 or err.max() <= 0, "%s: worst %s gpu %r oracle %r" % (what, worst, got[worst], ref[worst])


def _bits_to_f(bits):
    return np.asarray(bits).view(np.float16).astype(np.float64)


class Pair:
    """One attention layer on both sides, fed the same calls."""

    def __init__(self, shape, seed=0, layer=0, history=True, norm=None, max_T=None):
        import torch
        import bit_affine_quantised_affine4_b300 as moe
        self.moe, self.torch, self.s = moe, torch, shape
        wqkv_f, wo_f = synth.attn_weights(shape, seed, layer)
        self.wqkv, self.wo = oracle.quantise(wqkv_f, 4), oracle.quantise(wo_f, 4)
        if history:
            hist = synth.kv_history(shape, seed, layer)
            self.k = np.ascontiguousarray(hist[0].astype(np.float16).view(np.uint16))
            self.v = np.ascontiguousarray(hist[1].astype(np.float16).view(np.uint16))
        else:
            self.k = np.zeros((shape.nkv, shape.kv_len, shape.d), np.uint16)
            self.v = np.zeros_like(self.k)
        self.g = moe.AttnLayer(shape.H, shape.nq, shape.nkv, shape.d, shape.window, shape.kv_len, shape.theta)
        self.g.set_weights(wqkv_f, wo_f)
        self.g.set_cache(self.k, self.v)
        self.norm = norm
        if norm is not None:
            self.g.set_norm(*norm)
        self.view = self.g.view()
        self.ws = moe.new_attn_workspace(self.view, max_T or moe.MOE_MAX_PREFILL_TOKENS)

    def quantised_weights_match(self):
        for dev, ref in zip(self.g.wqkv + self.g.wo, self.wqkv + self.wo):
            np.testing.assert_array_equal(dev.cpu().numpy().view(ref.dtype), ref)

    def step(self, x, pos, flags=None, check_cache=True):
        moe, torch, s = self.moe, self.torch, self.s
        if flags is None:
            flags = moe.MOE_RESIDUAL | (moe.MOE_PRENORM if self.norm is not None else 0)
        xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
        od = torch.empty((x.shape[0], s.nq * s.d), device="cuda")
        yd = moe.moe_attn_step(self.view, xd, self.ws, pos, flags=flags, attn_out=od)
        ry, ro = oracle.attn_step(s.H, s.nq, s.nkv, s.d, s.window, s.kv_len, s.theta, s.scale, self.wqkv, self.wo,
                                  self.k, self.v, x, pos, residual=bool(flags & moe.MOE_RESIDUAL),
                                  norm_w=None if not flags & moe.MOE_PRENORM else self.norm[0],
                                  norm_eps=0.0 if self.norm is None else self.norm[1])
        torch.cuda.synchronize()
        within(od.cpu().numpy(), ro, "attention output o at pos %d" % pos)
        within(yd.cpu().numpy(), ry, "y at pos %d" % pos)
        if check_cache:
            within(_bits_to_f(self.g.k_cache.cpu().numpy()), _bits_to_f(self.k), "key cache after pos %d" % pos)
            within(_bits_to_f(self.g.v_cache.cpu().numpy()), _bits_to_f(self.v), "value cache after pos %d" % pos)
        return yd


def _tokens(shape, T, stream):
    return synth.normal(synth.key(77, stream, shape.H), (T, shape.H), 1.0)


@pytest.mark.parametrize("shape", [synth.ATTN_TINY_SLIDING, synth.ATTN_TINY_FULL], ids=lambda s: s.name)
def test_tiny_sequence(shape):
    p = Pair(shape, history=False)
    p.quantised_weights_match()
    p.step(_tokens(shape, 7, 0), 0)  # prefill chunk from an empty cache
    pos = 7
    for i in range(40 if shape.window else 20):  # decode; wraps a sliding ring twice
        p.step(_tokens(shape, 1, 1 + i), pos)
        pos += 1
    if shape.window:
        # a chunk as long as the ring allows: kv_len >= window + T - 1
        T = shape.kv_len - shape.window + 1
        p.step(_tokens(shape, T, 100), pos)
    else:
        T = shape.kv_len - pos
        p.step(_tokens(shape, T, 100), pos)  # fills the store to its last entry


@pytest.mark.parametrize("nq,nkv,d", [(4, 4, 64), (8, 2, 128), (16, 1, 64), (2, 1, 512), (4, 2, 256)])
@pytest.mark.parametrize("window", [0, 40])
def test_head_layouts(nq, nkv, d, window):
    shape = synth.AttnShape("h", 512, nq, nkv, d, window, 300, 10000.0)
    p = Pair(shape, seed=1)
    p.step(_tokens(shape, 3, 0), 0)
    p.step(_tokens(shape, 13, 1), 3)      # several rows per tile, ragged tiles
    p.step(_tokens(shape, 1, 2), 250)     # long history, many slices
    p.step(_tokens(shape, 5, 3), 290)


def test_prenorm_and_flags():
    shape = synth.ATTN_TINY_SLIDING
    p = Pair(shape, seed=2, norm=(synth.norm_weights(shape.H, seed=2), 1e-6))
    moe = p.moe
    x = 4.0 * _tokens(shape, 2, 0)  # inputs of varied scale: the projections see RMSNorm(x)
    p.step(x, 30)
    p.step(_tokens(shape, 1, 1), 32, flags=moe.MOE_PRENORM)
    p.step(_tokens(shape, 1, 2), 33, flags=0)
    p.step(_tokens(shape, 1, 3), 34, flags=moe.MOE_RESIDUAL)


def test_full_length_chunks():
    # 128-token chunks: a full layer from position 0, a sliding layer with a ring of window + 127
    full = synth.AttnShape("f", 512, 4, 2, 64, 0, 384, 1000000.0)
    p = Pair(full, seed=3, history=False)
    p.step(_tokens(full, 128, 0), 0)
    p.step(_tokens(full, 128, 1), 128)
    p.step(_tokens(full, 128, 2), 256)
    slid = synth.AttnShape("s", 512, 4, 2, 64, 64, 64 + 127, 10000.0)
    q = Pair(slid, seed=4)
    for i in range(3):
        q.step(_tokens(slid, 128, 10 + i), 1000 + 128 * i)


def test_y_may_alias_x():
    import torch
    shape = synth.ATTN_TINY_FULL
    p = Pair(shape, seed=5)
    x = _tokens(shape, 4, 0)
    ref = p.step(x, 10).cpu().numpy()  # advances the cache; compare a second layer instead
    q = Pair(shape, seed=5)
    xd = torch.from_numpy(x).cuda()
    q.moe.moe_attn_step(q.view, xd, q.ws, 10, y=xd, flags=q.moe.MOE_RESIDUAL)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(xd.cpu().numpy(), ref)


@pytest.mark.parametrize("shape,pos,T", [(synth.ATTN_FULL_SLIDING, 5000, 1), (synth.ATTN_FULL_SLIDING, 777, 4),
                                         (synth.ATTN_FULL_GLOBAL, 4095, 1), (synth.ATTN_FULL_GLOBAL, 2000, 16)],
                         ids=["sliding-T1", "sliding-T4", "global-last", "global-T16"])
def test_full_size(shape, pos, T):
    """The full-size shapes of the decode stack: hidden 2816, 16 query heads and 8
    key/value heads of 256, a window of 1024 in a ring of 1151 or a linear store of
    4096, history filled with synthetic keys and values."""
    p = Pair(shape, seed=6, norm=(synth.norm_weights(shape.H, seed=6), 1e-6))
    p.quantised_weights_match()
    p.step(_tokens(shape, T, 0), pos)


def test_refusals():
    import ctypes as C
    import torch
    import bit_affine_quantised_affine4_b300 as moe
    shape = synth.ATTN_TINY_SLIDING
    p = Pair(shape, seed=7)
    p.step(_tokens(shape, 2, 0), 0)
    x = torch.zeros((2, shape.H), device="cuda")

    def rc(**kw):
        v = moe.moe_attn_t.from_buffer_copy(p.view)
        args = dict(T=2, pos=0, flags=0, ws=p.ws.data_ptr(), nbytes=p.ws.numel())
        for k, val in kw.items():
            if k in args:
                args[k] = val
            else:
                setattr(v, k, val)
        return moe.lib.moe_attn_step(C.byref(v), x.data_ptr(), args["T"], args["pos"], args["flags"],
                                     x.data_ptr(), None, args["ws"], args["nbytes"], None)

    assert rc(d=96) == moe.MOE_EINVAL
    assert rc(nkv=3) == moe.MOE_EINVAL
    assert rc(theta=0.0) == moe.MOE_EINVAL
    assert rc(T=0) == moe.MOE_EINVAL
    assert rc(T=129) == moe.MOE_EINVAL
    assert rc(pos=-1) == moe.MOE_EINVAL
    assert rc(flags=moe.MOE_PRENORM) == moe.MOE_EINVAL  # no norm weight
    assert rc(flags=8) == moe.MOE_EINVAL
    assert rc(k_cache=p.view.k_cache + 2) == moe.MOE_EINVAL  # misaligned cache
    assert rc(kv_len=shape.window) == moe.MOE_ECAPACITY      # ring too short for 2 tokens
    assert rc(window=0, pos=shape.kv_len - 1) == moe.MOE_ECAPACITY  # past the end of a full store
    assert rc(nbytes=1024) == moe.MOE_EWORKSPACE
    assert rc(ws=p.ws.data_ptr() + 8) == moe.MOE_EWORKSPACE
    # nothing ran for the refused calls: the next call still matches the oracle, cache included
    p.step(_tokens(shape, 1, 1), 2)


def test_attention_wait_times_out_and_recovers():
    """Fault injection (no GPU fault): the next call's attention CTAs expect 16
    bytes more than their copies bring, with a 2 ms limit.  The waits give up, the
    workspace status reports MOE_ETIMEOUT once, and the next call matches the oracle
    again (the timed-out call stored its keys and values, as the oracle's copy of the
    call does, and its slices still took their tickets)."""
    shape = synth.ATTN_TINY_SLIDING
    p = Pair(shape, seed=8)
    moe, torch = p.moe, p.torch
    p.step(_tokens(shape, 1, 0), 30)
    assert moe.moe_attn_workspace_status(p.ws) == moe.MOE_OK
    moe.moe_debug_inject(moe.MOE_INJECT_ATTN_WAIT)
    x = _tokens(shape, 2, 1)
    xd = torch.from_numpy(x).cuda()
    moe.moe_attn_step(p.view, xd, p.ws, 31, flags=moe.MOE_RESIDUAL)
    s = shape
    oracle.attn_step(s.H, s.nq, s.nkv, s.d, s.window, s.kv_len, s.theta, s.scale, p.wqkv, p.wo, p.k, p.v, x, 31)
    assert moe.moe_attn_workspace_status(p.ws) == moe.MOE_ETIMEOUT
    assert moe.moe_attn_workspace_status(p.ws) == moe.MOE_OK
    p.step(_tokens(shape, 1, 2), 33)
    p.step(_tokens(shape, 3, 3), 34)


def test_decode_step_stack_teacher_forced():
    """A decode step of a small stack as in the 30-layer workload: per layer the
    pre-norm attention block, then the pre-norm MoE block; layers 0 and 1 attend
    to a window (16 positions in a ring of 23, which wraps during the steps),
    layer 2 to the whole context (a store of 96).  Teacher-forced per block: each
    oracle block runs on the GPU's input to that block (the oracle keeps its own
    key/value caches, which track the GPU's to binary16 rounding).  Checked every
    step and block: outputs within 2e-3 (1 + |oracle|), expert indices bit-exact."""
    import bit_affine_quantised_affine4_b300 as moe
    from layers import OracleLayer, gpu_layer, norm_weights, within_tol
    s = synth.TINY
    eps = 1e-6
    attn, moes, omoes, mnorms = [], [], [], []
    for l in range(3):
        a = synth.ATTN_TINY_FULL if l == 2 else synth.ATTN_TINY_SLIDING
        attn.append(Pair(a, seed=20, layer=l, norm=(synth.norm_weights(a.H, seed=20, layer=l), eps)))
        bias = synth.popularity_bias(s, seed=0, layer=l)
        norm = (norm_weights(s, 0, l), eps)
        mnorms.append(norm)
        moes.append(gpu_layer(s, seed=0, layer=l, bias=bias, norm=norm))
        omoes.append(OracleLayer(s, seed=0, layer=l, bias=bias))
    mviews = [g.view() for g in moes]
    ws = moe.new_workspace(mviews[0], 1)
    import torch
    idx = torch.empty((1, s.topk), dtype=torch.int32, device="cuda")
    xs = synth.token_sequence(s, 8, seed=1)
    pos0 = 60
    for k in range(8):
        h = xs[k:k + 1].astype(np.float32)
        for l in range(3):
            ha = attn[l].step(h, pos0 + k).cpu().numpy()  # checks y, o and the caches against the oracle
            y = moe.moe_layer_decode(mviews[l], torch.from_numpy(ha).cuda(), ws,
                                     flags=moe.MOE_RESIDUAL | moe.MOE_PRENORM, idx=idx)
            torch.cuda.synchronize()
            ry, ridx, _ = omoes[l].block(ha, *mnorms[l])
            assert np.array_equal(idx.cpu().numpy(), ridx), (k, l)
            ok, worst = within_tol(y.cpu().numpy(), ry, 2e-3)
            assert ok, "step %d layer %d: worst err/bound %.3f" % (k, l, worst)
            h = y.cpu().numpy()
