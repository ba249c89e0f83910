"""Test-side builders: the same synthetic fp32 weights, quantised by the oracle (CPU)
and by the library's own quantiser (GPU).

Both builders take optional overrides so that a test can plant structure in the
weights (duplicated router rows for exact ties, constant or extreme-code groups):
``router_w`` replaces the router matrix, ``edit`` is applied to every expert's
(gate/up, down) fp32 pair -- routed and shared -- before quantisation.
"""
import numpy as np

import oracle
import synth


def _expert_w(shape, e, seed, layer, edit):
    gu, d = synth.expert_weights(shape, e, seed, layer)
    return edit(gu, d) if edit else (gu, d)


def _shared_w(shape, seed, layer, edit):
    gu, d = synth.shared_weights(shape, seed, layer)
    return edit(gu, d) if edit else (gu, d)


class OracleLayer:
    """Oracle-side copy of one layer; experts are generated and quantised on demand."""

    def __init__(self, shape, seed=0, layer=0, bias=None, router_w=None, edit=None):
        self.shape, self.seed, self.layer_id, self.edit = shape, seed, layer, edit
        rw = synth.router_weights(shape, seed, layer) if router_w is None else router_w
        self.router = oracle.quantise(np.ascontiguousarray(rw, np.float32), 8)
        gu, d = _shared_w(shape, seed, layer, edit)
        self.shared = oracle.pack_expert(shape.H, shape.Is, oracle.quantise(gu, 4), oracle.quantise(d, 4))
        self.bias = bias
        self._experts = {}

    def expert(self, e):
        if e not in self._experts:
            gu, d = _expert_w(self.shape, e, self.seed, self.layer_id, self.edit)
            self._experts[e] = oracle.pack_expert(self.shape.H, self.shape.I, oracle.quantise(gu, 4),
                                                  oracle.quantise(d, 4))
        return self._experts[e]

    def route(self, x):
        s = self.shape
        return oracle.route(*self.router, s.E, s.H, x, topk=s.topk, logit_bias=self.bias)

    def block(self, x, norm_w, norm_eps):
        """The pre-norm block y = x + MoE(RMSNorm(x)) -> (y, idx, gate)."""
        s = self.shape
        xn = oracle.rmsnorm(x, norm_w, norm_eps).astype(np.float32)
        _, idx, _ = self.route(xn)
        experts = [None] * s.E
        for e in np.unique(idx):
            experts[int(e)] = self.expert(int(e))
        return oracle.moe_block(s.H, s.E, s.topk, s.I, s.Is, self.router, experts, self.shared, x, norm_w,
                                norm_eps, logit_bias=self.bias)

    def route_normed(self, x, norm_w, norm_eps):
        return self.route(oracle.rmsnorm(x, norm_w, norm_eps).astype(np.float32))

    def layer(self, x, residual=False):
        s = self.shape
        _, idx, _ = self.route(x)
        experts = [None] * s.E
        for e in np.unique(idx):
            experts[int(e)] = self.expert(int(e))
        return oracle.moe_layer(s.H, s.E, s.topk, s.I, s.Is, self.router, experts, self.shared, x,
                                logit_bias=self.bias, residual=residual)


def gpu_layer(shape, seed=0, layer=0, bias=None, copies=1, router_w=None, edit=None, norm=None):
    """norm = (weight [H], eps) for the MOE_PRENORM calls, or None."""
    import bit_affine_quantised_affine4_b300 as moe
    rw = synth.router_weights(shape, seed, layer) if router_w is None else router_w
    L = moe.make_layer(shape.H, shape.E, shape.topk, shape.I, shape.Is,
                       np.ascontiguousarray(rw, np.float32),
                       lambda e: _expert_w(shape, e, seed, layer, edit),
                       _shared_w(shape, seed, layer, edit), bias=bias, copies=copies)
    if norm is not None:
        L.set_norm(norm[0], norm[1])
    return L


def norm_weights(shape, seed=0, layer=0):
    """A seeded RMSNorm weight: 1 + N(0, 0.1^2) per column."""
    return (1.0 + synth.normal(synth.key(seed, layer, 99), (shape.H,), 0.1)).astype(np.float32)


def within_tol(gpu, ref, rel=2e-3):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    bound = rel * (1.0 + np.abs(ref))
    return bool(np.all(err <= bound)), float(np.max(err / bound)) if err.size else 0.0


def topk_margin(logits, k):
    """Gap between the k-th and (k+1)-th largest fp64 logits per token."""
    s = np.sort(logits, axis=1)[:, ::-1]
    return s[:, k - 1] - s[:, k] if s.shape[1] > k else np.full(s.shape[0], np.inf)


def distinct_margin(logits, k):
    """Per token, the smallest gap between two different values among its k + 2
    largest logits.  Exact ties are decided by the index rule on both sides; only
    a near-tie between different values around the top-k could flip between an
    fp32 and an fp64 sum."""
    out = []
    for row in np.asarray(logits, np.float64):
        u = np.unique(np.sort(row)[::-1][:k + 2])
        out.append(np.min(np.diff(u)) if u.size > 1 else np.inf)
    return np.array(out)


def extreme_groups(gu, d):
    """Plants the quantiser's degenerate groups in one expert's weights (copies):
    constant groups (scale 0, every code 0), groups of two values (codes 0 and 15
    only), and groups at the maximum but for one element (codes 15 but one 0), in
    the gate rows, the up rows and the down rows."""
    gu, d = gu.copy(), d.copy()
    I = gu.shape[0] // 2
    H = gu.shape[1]
    alt = np.where(np.arange(64) % 2 == 0, 0.03, -0.03).astype(np.float32)
    top = np.full(64, 0.02, np.float32)
    top[17] = -0.02
    for r, g in ((0, 0), (3, H // 64 - 1)):            # gate rows
        gu[r, 64 * g:64 * g + 64] = 0.011
    gu[I + 1, 64:128] = -0.05                           # up row, constant negative
    gu[2, 128:192] = alt
    gu[I + 5, 0:64] = alt[::-1]
    gu[7, 192:256] = top
    gu[I + 7, 192:256] = -top
    d[0, 0:64] = 0.007
    d[1, 0:64] = alt
    d[-1, -64:] = top
    d[5, :] = 0.0                                       # a whole zero row
    return gu, d
