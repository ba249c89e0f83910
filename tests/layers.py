"""Test-side builders: the same synthetic fp32 weights, quantised by the oracle (CPU)
and by the library's own quantiser (GPU)."""
import numpy as np

import oracle
import synth


class OracleLayer:
    """Oracle-side copy of one layer; experts are generated and quantised on demand."""

    def __init__(self, shape, seed=0, layer=0, bias=None):
        self.shape, self.seed, self.layer_id = shape, seed, layer
        self.router = oracle.quantise(synth.router_weights(shape, seed, layer), 8)
        gu, d = synth.shared_weights(shape, seed, layer)
        self.shared = oracle.pack_expert(shape.H, shape.Is, oracle.quantise(gu, 4), oracle.quantise(d, 4))
        self.bias = bias
        self._experts = {}

    def expert(self, e):
        if e not in self._experts:
            gu, d = synth.expert_weights(self.shape, e, self.seed, self.layer_id)
            self._experts[e] = oracle.pack_expert(self.shape.H, self.shape.I, oracle.quantise(gu, 4),
                                                  oracle.quantise(d, 4))
        return self._experts[e]

    def route(self, x):
        s = self.shape
        return oracle.route(*self.router, s.E, s.H, x, topk=s.topk, logit_bias=self.bias)

    def layer(self, x, residual=False):
        s = self.shape
        _, idx, _ = self.route(x)
        experts = [None] * s.E
        for e in np.unique(idx):
            experts[int(e)] = self.expert(int(e))
        return oracle.moe_layer(s.H, s.E, s.topk, s.I, s.Is, self.router, experts, self.shared, x,
                                logit_bias=self.bias, residual=residual)


def gpu_layer(shape, seed=0, layer=0, bias=None, copies=1):
    import bit_affine_quantised_affine4_b300 as moe
    return moe.make_layer(shape.H, shape.E, shape.topk, shape.I, shape.Is,
                          synth.router_weights(shape, seed, layer),
                          lambda e: synth.expert_weights(shape, e, seed, layer),
                          synth.shared_weights(shape, seed, layer), bias=bias, copies=copies)


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
