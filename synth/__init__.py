"""Seeded synthetic inputs for the MoE layer workloads (no layer arithmetic).

Both the CPU oracle and the CUDA path are fed from here, so they see the same
bits.  The generator itself is ``synth.c`` (counter-based SplitMix64 and an
Irwin-Hall normal, exact in binary64); this module builds it, names the
workload shapes and hands out numpy arrays.

Workloads (weights N(0, 0.02) before quantisation, tokens N(0, 1)):

* ``tiny``   hidden 512, 32 experts, top-8, expert inter 256, shared inter 512
* ``full``   hidden 2816, 128 experts, top-8, expert inter 704, shared inter 2112
  (uniform router logits, or Zipf(1.1) popularity through a logit bias)

Attention blocks (``AttnShape``; weights N(0, 0.02), cached keys/values N(0, 1)):

* ``attn-tiny-sliding`` / ``attn-tiny-full``  hidden 512, 4 query heads, 2 key/value
  heads of 64, window 16 in a ring of 23 / linear store of 96
* ``attn-full-sliding`` / ``attn-full-global`` hidden 2816, 16 query heads, 8
  key/value heads of 256, window 1024 in a ring of 1151 / linear store of 4096
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

# sub-stream ids
(T_ROUTER, T_EXPERT_GU, T_EXPERT_D, T_SHARED_GU, T_SHARED_D, T_TOKENS, T_ZIPF, T_AR1, T_ATTN_QKV, T_ATTN_O,
 T_KV, T_NORM) = range(12)


@dataclass(frozen=True)
class Shape:
    name: str
    H: int
    E: int
    topk: int
    I: int
    Is: int


TINY = Shape("tiny", 512, 32, 8, 256, 512)
FULL = Shape("full", 2816, 128, 8, 704, 2112)
SHAPES = {"tiny": TINY, "full": FULL}

@dataclass(frozen=True)
class AttnShape:
    """One attention block: window > 0 is a sliding-window layer whose cache is a ring
    of kv_len entries; window == 0 is a full layer with a linear store of kv_len."""
    name: str
    H: int
    nq: int
    nkv: int
    d: int
    window: int
    kv_len: int
    theta: float

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    @property
    def n_qkv(self) -> int:
        return (self.nq + 2 * self.nkv) * self.d


ATTN_TINY_SLIDING = AttnShape("attn-tiny-sliding", 512, 4, 2, 64, 16, 23, 10000.0)
ATTN_TINY_FULL = AttnShape("attn-tiny-full", 512, 4, 2, 64, 0, 96, 1000000.0)
ATTN_FULL_SLIDING = AttnShape("attn-full-sliding", 2816, 16, 8, 256, 1024, 1151, 10000.0)
ATTN_FULL_GLOBAL = AttnShape("attn-full-global", 2816, 16, 8, 256, 0, 4096, 1000000.0)
ATTN_SHAPES = {a.name: a for a in (ATTN_TINY_SLIDING, ATTN_TINY_FULL, ATTN_FULL_SLIDING, ATTN_FULL_GLOBAL)}

WEIGHT_SIGMA = 0.02
ZIPF_S = 1.1
AR1_RHO = 0.9


def build(force: bool = False) -> str:
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                    _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        u64, i64 = C.c_uint64, C.c_int64
        L.synth_splitmix64_at.argtypes = [u64, u64]
        L.synth_splitmix64_at.restype = u64
        L.synth_key.argtypes = [u64, i64, i64, i64, i64]
        L.synth_key.restype = u64
        L.synth_normal_f32.argtypes = [u64, u64, i64, C.c_double, C.c_void_p]
        L.synth_normal_f64.argtypes = [u64, u64, i64, C.c_void_p]
        L.synth_permutation.argtypes = [u64, C.c_int, C.c_void_p]
        L.synth_zipf_bias.argtypes = [u64, C.c_int, C.c_double, C.c_void_p]
        L.synth_ar1.argtypes = [u64, C.c_int, C.c_int, C.c_double, C.c_void_p]
        _lib = L
    return _lib


def splitmix64_at(key: int, c: int) -> int:
    return int(lib().synth_splitmix64_at(key & (2**64 - 1), c))


def key(seed: int, a: int = 0, b: int = 0, c: int = 0, d: int = 0) -> int:
    return int(lib().synth_key(seed & (2**64 - 1), a, b, c, d))


def normal(k: int, shape, sigma: float = 1.0, first: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.float32)
    lib().synth_normal_f32(k, first, n, sigma, out.ctypes.data)
    return out.reshape(shape)


def normal64(k: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, np.float64)
    lib().synth_normal_f64(k, first, n, out.ctypes.data)
    return out


def permutation(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().synth_permutation(k, n, out.ctypes.data)
    return out


def zipf_bias(k: int, E: int, s: float = ZIPF_S) -> np.ndarray:
    out = np.empty(E, np.float32)
    lib().synth_zipf_bias(k, E, s, out.ctypes.data)
    return out


def ar1(k: int, steps: int, dim: int, rho: float = AR1_RHO) -> np.ndarray:
    out = np.empty((steps, dim), np.float32)
    lib().synth_ar1(k, steps, dim, rho, out.ctypes.data)
    return out


# ------------------------------------------------------------ workload pieces
# Every tensor has its own sub-stream keyed by (seed, layer, tensor id, expert).

def router_weights(shape: Shape, seed: int = 0, layer: int = 0) -> np.ndarray:
    return normal(key(seed, layer, T_ROUTER), (shape.E, shape.H), WEIGHT_SIGMA)


def expert_weights(shape: Shape, e: int, seed: int = 0, layer: int = 0):
    """-> (gate/up [2I, H] with gate rows first, down [H, I]) fp32."""
    gu = normal(key(seed, layer, T_EXPERT_GU, e), (2 * shape.I, shape.H), WEIGHT_SIGMA)
    d = normal(key(seed, layer, T_EXPERT_D, e), (shape.H, shape.I), WEIGHT_SIGMA)
    return gu, d


def shared_weights(shape: Shape, seed: int = 0, layer: int = 0):
    gu = normal(key(seed, layer, T_SHARED_GU), (2 * shape.Is, shape.H), WEIGHT_SIGMA)
    d = normal(key(seed, layer, T_SHARED_D), (shape.H, shape.Is), WEIGHT_SIGMA)
    return gu, d


def tokens(shape: Shape, T: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    return normal(key(seed, stream, T_TOKENS), (T, shape.H), 1.0)


def popularity_bias(shape: Shape, seed: int = 0, layer: int = 0, s: float = ZIPF_S) -> np.ndarray:
    return zipf_bias(key(seed, layer, T_ZIPF), shape.E, s)


def token_sequence(shape: Shape, steps: int, seed: int = 0, rho: float = AR1_RHO) -> np.ndarray:
    return ar1(key(seed, 0, T_AR1), steps, shape.H, rho)


def attn_weights(shape: AttnShape, seed: int = 0, layer: int = 0):
    """-> (Wqkv [(nq + 2 nkv) d, H]: query heads, key heads, value heads; Wo [H, nq d]) fp32."""
    wqkv = normal(key(seed, layer, T_ATTN_QKV), (shape.n_qkv, shape.H), WEIGHT_SIGMA)
    wo = normal(key(seed, layer, T_ATTN_O), (shape.H, shape.nq * shape.d), WEIGHT_SIGMA)
    return wqkv, wo


def kv_history(shape: AttnShape, seed: int = 0, layer: int = 0):
    """Stand-in for the keys and values of earlier tokens: fp32 N(0, 1), [2][nkv][kv_len][d]
    (keys, then values); the caller stores them at the cache's precision."""
    return normal(key(seed, layer, T_KV), (2, shape.nkv, shape.kv_len, shape.d), 1.0)


def norm_weights(H: int, seed: int = 0, layer: int = 0) -> np.ndarray:
    """RMSNorm gains around 1: 1 + 0.1 N(0, 1)."""
    return (1.0 + normal(key(seed, layer, T_NORM), (H,), 0.1)).astype(np.float32)
