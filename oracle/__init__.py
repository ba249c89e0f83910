"""CPU oracle for the routed MoE layer over affine group-quantised weights.

TEST INFRASTRUCTURE ONLY.  The oracle is the yardstick that the CUDA path is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
product package never does, and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 sums in index order);
this module only builds it and marshals numpy arrays through ctypes.  Each C
function's header comment cites the page passage it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

ORC_OK = 0
ORC_EINVAL = 1
ORC_ECAPACITY = 3


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmoe_oracle.so`` (plain gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O3", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


_p = C.c_void_p


def _declare(L):
    L.orc_half_to_double.argtypes = [C.c_uint16]
    L.orc_half_to_double.restype = C.c_double
    L.orc_float_to_half.argtypes = [C.c_float]
    L.orc_float_to_half.restype = C.c_uint16
    L.orc_gelu_tanh.argtypes = [C.c_double]
    L.orc_gelu_tanh.restype = C.c_double
    L.orc_dequant.argtypes = [_p, _p, _p, C.c_int, C.c_int, C.c_int, _p]
    L.orc_quantise.argtypes = [_p, C.c_int, C.c_int, C.c_int, _p, _p, _p]
    L.orc_qgemv.argtypes = [_p, _p, _p, C.c_int, C.c_int, C.c_int, _p, C.c_int, _p]
    L.orc_route.argtypes = [_p, _p, _p, C.c_int, C.c_int, _p, C.c_int, _p, C.c_int, _p, _p, _p]
    L.orc_expert_blob_bytes.argtypes = [C.c_int, C.c_int]
    L.orc_expert_blob_bytes.restype = C.c_size_t
    L.orc_expert_blob_offsets.argtypes = [C.c_int, C.c_int, _p]
    L.orc_tile_blob_bytes.argtypes = [C.c_int, C.c_int]
    L.orc_tile_blob_bytes.restype = C.c_size_t
    L.orc_untile_expert.argtypes = [_p, C.c_int, C.c_int, _p]
    L.orc_expert.argtypes = [_p, C.c_int, C.c_int, _p, _p, _p]
    L.orc_moe_layer.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, _p, _p, _p, _p, _p,
                                _p, C.c_int, _p, C.c_int, _p, _p, _p]
    L.orc_rmsnorm.argtypes = [_p, _p, C.c_double, C.c_int, C.c_int, _p]
    L.orc_sample.argtypes = [_p, C.c_int, C.c_double, C.c_int, C.c_double, C.c_double, _p, _p]
    L.orc_attn_step.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_double, C.c_double,
                                _p, _p, _p, _p, _p, _p, _p, C.c_double, C.c_int, _p, _p, _p, C.c_int, C.c_int,
                                _p, _p]
    L.orc_lfu_create.argtypes = [C.c_int, C.c_int]
    L.orc_lfu_create.restype = _p
    L.orc_lfu_destroy.argtypes = [_p]
    L.orc_lfu_step.argtypes = [_p, _p, C.c_int, _p, _p]
    L.orc_lfu_state.argtypes = [_p, _p, _p, _p, _p, _p]


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _check(rc, what):
    if rc != ORC_OK:
        raise ValueError("oracle %s failed with status %d" % (what, rc))


# ---------------------------------------------------------------- scalars

def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(int(h))


def float_to_half(f: float) -> int:
    return lib().orc_float_to_half(float(f))


def gelu_tanh(z: float) -> float:
    return lib().orc_gelu_tanh(float(z))


# ---------------------------------------------------------------- matrices

def words_per_row(K: int, bits: int) -> int:
    return K * bits // 32


def quantise(w: np.ndarray, bits: int):
    """Affine-quantise an fp32 [N, K] matrix -> (q uint32 [N, K*bits/32], s f16 bits, b f16 bits)."""
    w = _c(w, np.float32)
    N, K = w.shape
    q = np.zeros((N, words_per_row(K, bits)), np.uint32)
    s = np.zeros((N, K // 64), np.uint16)
    b = np.zeros((N, K // 64), np.uint16)
    _check(lib().orc_quantise(_ptr(w), N, K, bits, _ptr(q), _ptr(s), _ptr(b)), "quantise")
    return q, s, b


def dequant(q, s, b, K: int, bits: int) -> np.ndarray:
    q = _c(q, np.uint32); s = _c(s, np.uint16); b = _c(b, np.uint16)
    N = q.shape[0]
    out = np.empty((N, K), np.float64)
    _check(lib().orc_dequant(_ptr(q), _ptr(s), _ptr(b), N, K, bits, _ptr(out)), "dequant")
    return out


def qgemv(q, s, b, K: int, bits: int, x) -> np.ndarray:
    """y[t, n] = sum_j deq(W)[n, j] x[t, j] in fp64; x is [T, K] (or [K])."""
    q = _c(q, np.uint32); s = _c(s, np.uint16); b = _c(b, np.uint16)
    x2 = _c(np.atleast_2d(x), np.float32)
    N = q.shape[0]
    T = x2.shape[0]
    y = np.empty((T, N), np.float64)
    _check(lib().orc_qgemv(_ptr(q), _ptr(s), _ptr(b), N, K, bits, _ptr(x2), T, _ptr(y)), "qgemv")
    return y if np.ndim(x) == 2 else y[0]


def route(rq, rs, rb, E: int, H: int, x, topk: int = 8, logit_bias=None):
    """-> (logits fp64 [T, E], idx int32 [T, k], gate fp64 [T, k])."""
    rq = _c(rq, np.uint32); rs = _c(rs, np.uint16); rb = _c(rb, np.uint16)
    x2 = _c(np.atleast_2d(x), np.float32)
    T = x2.shape[0]
    bias = None if logit_bias is None else _c(logit_bias, np.float32)
    logits = np.empty((T, E), np.float64)
    idx = np.empty((T, topk), np.int32)
    gate = np.empty((T, topk), np.float64)
    _check(lib().orc_route(_ptr(rq), _ptr(rs), _ptr(rb), E, H, _ptr(x2), T, _ptr(bias), topk,
                           _ptr(logits), _ptr(idx), _ptr(gate)), "route")
    return logits, idx, gate


def expert_blob_bytes(H: int, I: int) -> int:
    return int(lib().orc_expert_blob_bytes(H, I))


def expert_blob_offsets(H: int, I: int):
    off = np.zeros(6, np.uint64)
    lib().orc_expert_blob_offsets(H, I, _ptr(off))
    return [int(v) for v in off]


def pack_expert(H: int, I: int, gu, d) -> np.ndarray:
    """Lay out one expert's quantised parts as a blob (uint8).

    gu = (q, s, b) of the [2I, H] gate/up matrix; d = (q, s, b) of the [H, I] down matrix.
    """
    blob = np.zeros(expert_blob_bytes(H, I), np.uint8)
    off = expert_blob_offsets(H, I)
    for o, a in zip(off, list(gu) + list(d)):
        a = np.ascontiguousarray(a)
        raw = a.view(np.uint8).reshape(-1)
        blob[o:o + raw.size] = raw
    return blob


def tile_blob_bytes(H: int, I: int) -> int:
    return int(lib().orc_tile_blob_bytes(H, I))


def untile_expert(tiled, H: int, I: int) -> np.ndarray:
    """The library's tile-layout blob of one expert -> the MLX-layout blob (uint8)."""
    tiled = _c(tiled, np.uint8)
    if tiled.size != tile_blob_bytes(H, I):
        raise ValueError("tile blob of %d bytes, expected %d" % (tiled.size, tile_blob_bytes(H, I)))
    blob = np.zeros(expert_blob_bytes(H, I), np.uint8)
    _check(lib().orc_untile_expert(_ptr(tiled), H, I, _ptr(blob)), "untile_expert")
    return blob


def expert(blob, H: int, I: int, x):
    """-> (out fp64 [H], h fp64 [I]) for one token x [H]."""
    blob = _c(blob, np.uint8)
    x = _c(x, np.float32)
    out = np.empty(H, np.float64)
    h = np.empty(I, np.float64)
    _check(lib().orc_expert(_ptr(blob), H, I, _ptr(x), _ptr(out), _ptr(h)), "expert")
    return out, h


def moe_layer(H, E, topk, I, Is, router, experts, shared, x, logit_bias=None, residual=False):
    """The layer on tokens x [T, H].

    router = (q, s, b); experts = list of E blobs (None allowed for experts that are
    never routed to); shared = blob.  -> (y fp64 [T, H], idx [T, k], gate fp64 [T, k]).
    """
    rq, rs, rb = (_c(router[0], np.uint32), _c(router[1], np.uint16), _c(router[2], np.uint16))
    x2 = _c(np.atleast_2d(x), np.float32)
    T = x2.shape[0]
    blobs = [None if e is None else _c(e, np.uint8) for e in experts]
    table = (C.c_void_p * E)(*[None if e is None else e.ctypes.data for e in blobs])
    shared = _c(shared, np.uint8)
    bias = None if logit_bias is None else _c(logit_bias, np.float32)
    y = np.empty((T, H), np.float64)
    idx = np.empty((T, topk), np.int32)
    gate = np.empty((T, topk), np.float64)
    rc = lib().orc_moe_layer(H, E, topk, I, Is, _ptr(rq), _ptr(rs), _ptr(rb),
                             C.cast(table, C.c_void_p), _ptr(shared), _ptr(x2), T, _ptr(bias),
                             1 if residual else 0, _ptr(y), _ptr(idx), _ptr(gate))
    _check(rc, "moe_layer")
    return y, idx, gate


def rmsnorm(x, g, eps: float) -> np.ndarray:
    """x [T, H] (or [H]) fp32, g [H] fp32 -> x * g / sqrt(mean(x^2) + eps), fp64."""
    x2 = _c(np.atleast_2d(x), np.float32)
    g = _c(g, np.float32)
    T, H = x2.shape
    out = np.empty((T, H), np.float64)
    _check(lib().orc_rmsnorm(_ptr(x2), _ptr(g), float(eps), T, H, _ptr(out)), "rmsnorm")
    return out if np.ndim(x) == 2 else out[0]


def sample(logits, temperature: float, top_k: int, top_p: float, u: float):
    """One token from a row of logits (temperature, top-K, top-P, uniform u).
    -> (token, margin): margin is the smallest gap between a decision's two sides,
    relative to the kept total (see orc_sample)."""
    lg = _c(logits, np.float32)
    tok = C.c_int32(0)
    m = C.c_double(0.0)
    _check(lib().orc_sample(_ptr(lg), lg.size, float(temperature), int(top_k), float(top_p), float(u),
                            C.byref(tok), C.byref(m)), "sample")
    return tok.value, m.value


def moe_block(H, E, topk, I, Is, router, experts, shared, x, norm_w, norm_eps, logit_bias=None):
    """The pre-norm MoE block y = x + MoE(RMSNorm(x)).  The layer's input is the
    normalised x rounded to fp32 (the layer's input type).  -> (y, idx, gate)."""
    xn = rmsnorm(x, norm_w, norm_eps).astype(np.float32)
    y, idx, gate = moe_layer(H, E, topk, I, Is, router, experts, shared, xn, logit_bias=logit_bias)
    return y + np.atleast_2d(x).astype(np.float64), idx, gate


def attn_step(H: int, nq: int, nkv: int, d: int, window: int, kv_len: int, theta: float, scale: float,
              wqkv, wo, k_cache, v_cache, x, pos: int, residual: bool = True, norm_w=None,
              norm_eps: float = 1e-6):
    """One attention block over the tokens x [T, H] at positions pos .. pos+T-1.

    wqkv / wo = (q, s, b) 4-bit affine of [(nq + 2 nkv) d, H] / [H, nq d].  k_cache,
    v_cache: uint16 (binary16 bits) [nkv, kv_len, d], updated in place.
    -> (y fp64 [T, H], o fp64 [T, nq d] the attention output before Wo)."""
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags.c_contiguous or c.shape != (nkv, kv_len, d):
            raise ValueError("caches must be C-contiguous uint16 [nkv, kv_len, d]")
    qq, qs, qb = (_c(a, t) for a, t in zip(wqkv, (np.uint32, np.uint16, np.uint16)))
    oq, os_, ob = (_c(a, t) for a, t in zip(wo, (np.uint32, np.uint16, np.uint16)))
    x2 = _c(np.atleast_2d(x), np.float32)
    T = x2.shape[0]
    nw = None if norm_w is None else _c(norm_w, np.float32)
    y = np.empty((T, H), np.float64)
    o = np.empty((T, nq * d), np.float64)
    rc = lib().orc_attn_step(H, nq, nkv, d, window, kv_len, theta, scale, _ptr(qq), _ptr(qs), _ptr(qb),
                             _ptr(oq), _ptr(os_), _ptr(ob), _ptr(nw), norm_eps, int(bool(residual)),
                             _ptr(k_cache), _ptr(v_cache), _ptr(x2), T, pos, _ptr(y), _ptr(o))
    if rc == ORC_ECAPACITY:
        raise ValueError("oracle attn_step: positions do not fit the cache")
    _check(rc, "attn_step")
    return y, o


def moe_prefill_chunk(*args, **kw):
    """A prefill chunk is, by definition, that many independent decodes."""
    return moe_layer(*args, **kw)


# ---------------------------------------------------------------- LFU

class LFU:
    """Per-layer expert cache policy (in-cache LFU), one step per call."""

    def __init__(self, slots: int = 16, E: int = 128):
        self.slots, self.E = slots, E
        self._c = lib().orc_lfu_create(slots, E)
        if not self._c:
            raise ValueError("bad LFU shape")

    def __del__(self):
        if getattr(self, "_c", None):
            lib().orc_lfu_destroy(self._c)
            self._c = None

    def step(self, request):
        """-> (slot per request int32, hit per request bool).  Raises on a bad request."""
        req = _c(request, np.int32)
        n = req.size
        slot = np.full(max(n, 1), -1, np.int32)
        hit = np.zeros(max(n, 1), np.uint8)
        rc = lib().orc_lfu_step(self._c, _ptr(req), n, _ptr(slot), _ptr(hit))
        if rc == ORC_ECAPACITY:
            raise OverflowError("more distinct experts requested than the cache has slots")
        _check(rc, "lfu_step")
        return slot[:n], hit[:n].astype(bool)

    def state(self):
        """-> (expert_of_slot, count, last, hits, misses)."""
        eos = np.empty(self.slots, np.int32)
        cnt = np.empty(self.slots, np.uint32)
        last = np.empty(self.slots, np.int64)
        h = C.c_uint64(0)
        m = C.c_uint64(0)
        lib().orc_lfu_state(self._c, _ptr(eos), _ptr(cnt), _ptr(last), C.byref(h), C.byref(m))
        return eos, cnt, last, h.value, m.value
