"""Thin Python binding of libmoe (include/moe.h).

Argument marshalling only: every step of the MoE layer runs in the CUDA kernels
of ``libmoe.so``.  Tensors are PyTorch CUDA tensors (used for device memory and
streams); each function has the name of the C entry point it calls and raises
``MoeError`` on a non-zero status.  There is no fallback: if the library cannot
be loaded, importing the binding raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

MOE_OK, MOE_EINVAL, MOE_ECUDA, MOE_ECAPACITY, MOE_ETIMEOUT, MOE_EWORKSPACE, MOE_ENOTREADY = range(7)
MOE_RESIDUAL = 1
MOE_PRENORM = 2
MOE_INJECT_NONE, MOE_INJECT_WAIT, MOE_INJECT_COPY, MOE_INJECT_ATTN_WAIT = range(4)
MOE_NOALLOC_SCRATCH_BYTES = 4 << 20
MOE_MAX_TOPK = 8
MOE_MAX_EXPERTS = 256
MOE_MAX_DECODE_TOKENS = 16
MOE_MAX_PREFILL_TOKENS = 128
MOE_MAX_CACHE_SLOTS = 64

# Every function the header declares (checked against include/moe.h by the tests).
ENTRY_POINTS = (
    "moe_status_string", "moe_expert_blob_bytes", "moe_expert_blob_offsets",
    "moe_tile_blob_bytes", "moe_expert_tile",
    "moe_workspace_bytes", "moe_workspace_init", "moe_workspace_status",
    "affine_quantise", "qgemv_affine4", "moe_route", "moe_layer_decode",
    "moe_layer_prefill_chunk", "moe_cache_create", "moe_cache_destroy",
    "moe_cache_slots", "moe_cache_stats", "moe_layer_decode_noalloc", "moe_layer_decode_host",
    "moe_lfu_create", "moe_lfu_destroy", "moe_lfu_step", "moe_lfu_state",
    "moe_decode_workspace_bytes", "moe_noalloc_status", "moe_debug_inject", "moe_rmsnorm", "moe_sample",
    "moe_cache_set_device_policy", "moe_attn_workspace_bytes", "moe_attn_step", "moe_attn_workspace_status",
    "moe_host_call_create", "moe_host_call_run", "moe_host_call_rows", "moe_host_call_destroy",
)
MOE_SAMPLE_MAX_K = 1024


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


class moe_layer_t(C.Structure):
    _fields_ = [
        ("H", C.c_int), ("E", C.c_int), ("topk", C.c_int), ("I", C.c_int), ("Is", C.c_int),
        ("r_q", C.c_void_p), ("r_s", C.c_void_p), ("r_b", C.c_void_p),
        ("experts", C.c_void_p), ("expert_stride", C.c_size_t),
        ("shared", C.c_void_p), ("logit_bias", C.c_void_p),
        ("norm_w", C.c_void_p), ("norm_eps", C.c_float),
    ]


class moe_attn_t(C.Structure):
    _fields_ = [
        ("H", C.c_int), ("nq", C.c_int), ("nkv", C.c_int), ("d", C.c_int),
        ("window", C.c_int), ("kv_len", C.c_int), ("theta", C.c_float), ("scale", C.c_float),
        ("wqkv_q", C.c_void_p), ("wqkv_s", C.c_void_p), ("wqkv_b", C.c_void_p),
        ("wo_q", C.c_void_p), ("wo_s", C.c_void_p), ("wo_b", C.c_void_p),
        ("norm_w", C.c_void_p), ("norm_eps", C.c_float),
        ("k_cache", C.c_void_p), ("v_cache", C.c_void_p),
    ]


def _load():
    path = _build.LIB
    if _build.stale():
        path = _build.build()
    if not os.path.exists(path):
        raise ImportError("libmoe.so is missing and could not be built")
    L = C.CDLL(path)
    p, i, sz = C.c_void_p, C.c_int, C.c_size_t
    L.moe_status_string.argtypes = [i]
    L.moe_status_string.restype = C.c_char_p
    L.moe_expert_blob_bytes.argtypes = [i, i]
    L.moe_expert_blob_bytes.restype = sz
    L.moe_expert_blob_offsets.argtypes = [i, i, p]
    L.moe_tile_blob_bytes.argtypes = [i, i]
    L.moe_tile_blob_bytes.restype = sz
    L.moe_expert_tile.argtypes = [p, i, i, p, p]
    L.moe_workspace_bytes.argtypes = [p, i]
    L.moe_workspace_bytes.restype = sz
    L.moe_workspace_init.argtypes = [p, sz, p]
    L.moe_workspace_status.argtypes = [p, sz, p]
    L.affine_quantise.argtypes = [p, i, i, i, p, p, p, p]
    L.qgemv_affine4.argtypes = [p, p, p, i, i, p, p, p]
    L.moe_route.argtypes = [p, p, i, p, p, p, p, sz, p]
    L.moe_layer_decode.argtypes = [p, p, i, i, p, p, p, p, p, sz, p]
    L.moe_layer_prefill_chunk.argtypes = [p, p, i, i, p, p, p, p, sz, p]
    L.moe_layer_decode_noalloc.argtypes = [p, p, i, i, p, p, p, p]
    L.moe_layer_decode_host.argtypes = [p, p, i, i, p, p, p, p, p, sz, p]
    L.moe_cache_create.argtypes = [p, i, i, i, p, sz, i]
    L.moe_cache_destroy.argtypes = [p]
    L.moe_cache_slots.argtypes = [p, p, p]
    L.moe_cache_stats.argtypes = [p, p, p, p]
    L.moe_cache_set_device_policy.argtypes = [p, i]
    L.moe_lfu_create.argtypes = [p, i, i]
    L.moe_lfu_destroy.argtypes = [p]
    L.moe_lfu_step.argtypes = [p, p, i, p, p]
    L.moe_lfu_state.argtypes = [p, p, p, p, p, p]
    L.moe_decode_workspace_bytes.argtypes = [p, i]
    L.moe_decode_workspace_bytes.restype = sz
    L.moe_noalloc_status.argtypes = [p]
    L.moe_debug_inject.argtypes = [i]
    L.moe_rmsnorm.argtypes = [p, p, C.c_float, i, i, p, p]
    L.moe_sample.argtypes = [p, i, i, C.c_float, i, C.c_float, p, p, p]
    L.moe_attn_workspace_bytes.argtypes = [p, i]
    L.moe_attn_workspace_bytes.restype = sz
    L.moe_attn_step.argtypes = [p, p, i, i, i, p, p, p, sz, p]
    L.moe_attn_workspace_status.argtypes = [p, sz, p]
    L.moe_host_call_create.argtypes = [p, p, i, i, p, sz, p]
    L.moe_host_call_run.argtypes = [p, p, p]
    L.moe_host_call_rows.argtypes = [p, p, p]
    L.moe_host_call_destroy.argtypes = [p]
    for name in ENTRY_POINTS:
        if name not in ("moe_status_string", "moe_expert_blob_bytes", "moe_workspace_bytes",
                        "moe_tile_blob_bytes", "moe_decode_workspace_bytes", "moe_attn_workspace_bytes"):
            getattr(L, name).restype = i
    return L


lib = _load()


def status_string(status: int) -> str:
    return lib.moe_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ layout

def moe_expert_blob_bytes(H: int, I: int) -> int:
    return int(lib.moe_expert_blob_bytes(H, I))


def moe_expert_blob_offsets(H: int, I: int):
    off = (C.c_size_t * 6)()
    _check(lib.moe_expert_blob_offsets(H, I, off), "moe_expert_blob_offsets")
    return list(off)


def moe_tile_blob_bytes(H: int, I: int) -> int:
    return int(lib.moe_tile_blob_bytes(H, I))


def moe_expert_tile(mlx_blob: torch.Tensor, H: int, I: int, tile_blob: torch.Tensor, stream=None):
    """MLX-layout expert blob -> tile-layout blob (both uint8 CUDA tensors)."""
    _check(lib.moe_expert_tile(_ptr(mlx_blob), H, I, _ptr(tile_blob), _stream(stream)), "moe_expert_tile")
    return tile_blob


# ------------------------------------------------------------------ kernels

def affine_quantise(w: torch.Tensor, bits: int, q=None, s=None, b=None, stream=None):
    """Quantise fp32 [N, K] on the GPU -> (q int32 [N, K*bits/32], s int16 [N, K/64], b int16)."""
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous()
    N, K = w.shape
    dev = w.device
    q = torch.empty((N, K * bits // 32), dtype=torch.int32, device=dev) if q is None else q
    s = torch.empty((N, K // 64), dtype=torch.int16, device=dev) if s is None else s
    b = torch.empty((N, K // 64), dtype=torch.int16, device=dev) if b is None else b
    _check(lib.affine_quantise(_ptr(w), N, K, bits, _ptr(q), _ptr(s), _ptr(b), _stream(stream)),
           "affine_quantise")
    return q, s, b


def qgemv_affine4(q, s, b, K: int, x, y=None, stream=None):
    N = q.shape[0]
    y = torch.empty(N, dtype=torch.float32, device=x.device) if y is None else y
    _check(lib.qgemv_affine4(_ptr(q), _ptr(s), _ptr(b), N, K, _ptr(x), _ptr(y), _stream(stream)),
           "qgemv_affine4")
    return y


def moe_rmsnorm(x, w, eps: float, y=None, stream=None):
    """RMSNorm of the rows of x (fp32 CUDA [T, H]) with weight w ([H])."""
    T, H = x.shape
    y = torch.empty_like(x) if y is None else y
    _check(lib.moe_rmsnorm(_ptr(x), _ptr(w), float(eps), T, H, _ptr(y), _stream(stream)), "moe_rmsnorm")
    return y


def moe_attn_workspace_bytes(attn: moe_attn_t, T_max: int) -> int:
    return int(lib.moe_attn_workspace_bytes(C.byref(attn), int(T_max)))


def new_attn_workspace(attn: moe_attn_t, T_max: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for moe_attn_step calls of up to T_max tokens."""
    n = moe_attn_workspace_bytes(attn, T_max)
    if n == 0:
        raise MoeError(MOE_EINVAL, "moe_attn_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def moe_attn_step(attn: moe_attn_t, x, ws, pos: int, y=None, flags: int = 0, attn_out=None, stream=None):
    """One attention block on the T tokens x [T, H] (device fp32) at positions pos .. pos+T-1;
    updates the layer's key/value cache and returns y [T, H]."""
    T = x.shape[0]
    y = torch.empty_like(x) if y is None else y
    _check(lib.moe_attn_step(C.byref(attn), _ptr(x), T, int(pos), flags, _ptr(y), _ptr(attn_out), _ptr(ws),
                             ws.numel(), _stream(stream)), "moe_attn_step")
    return y


def moe_attn_workspace_status(ws, stream=None) -> int:
    """MOE_ETIMEOUT if a bounded wait of an attention call on `ws` gave up since the last
    status call (and clears it), else MOE_OK; synchronises the stream."""
    return int(lib.moe_attn_workspace_status(_ptr(ws), ws.numel(), _stream(stream)))


def moe_sample(logits, temperature: float, top_k: int, top_p: float, u, tokens=None, stream=None):
    """One token per row of logits (fp32 CUDA [T, V]) with the caller's uniforms u ([T])."""
    T, V = logits.shape
    tokens = torch.empty(T, dtype=torch.int32, device=logits.device) if tokens is None else tokens
    _check(lib.moe_sample(_ptr(logits), T, V, float(temperature), int(top_k), float(top_p), _ptr(u),
                          _ptr(tokens), _stream(stream)), "moe_sample")
    return tokens


def moe_workspace_bytes(layer: moe_layer_t, T_max: int) -> int:
    return int(lib.moe_workspace_bytes(C.byref(layer), T_max))


def moe_decode_workspace_bytes(layer: moe_layer_t, T_max: int) -> int:
    return int(lib.moe_decode_workspace_bytes(C.byref(layer), T_max))


def moe_noalloc_status(stream=None) -> int:
    return int(lib.moe_noalloc_status(_stream(stream)))


def moe_debug_inject(what: int):
    _check(lib.moe_debug_inject(int(what)), "moe_debug_inject")


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib.moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def moe_workspace_status(ws: torch.Tensor, stream=None) -> int:
    return int(lib.moe_workspace_status(_ptr(ws), ws.numel(), _stream(stream)))


def new_workspace(layer: moe_layer_t, T_max: int, device="cuda", stream=None) -> torch.Tensor:
    n = moe_workspace_bytes(layer, T_max)
    if n == 0:
        raise MoeError(MOE_EINVAL, "moe_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_route(layer: moe_layer_t, x, ws, idx=None, gate=None, logits=None, stream=None):
    T = x.shape[0]
    dev = x.device
    idx = torch.empty((T, layer.topk), dtype=torch.int32, device=dev) if idx is None else idx
    gate = torch.empty((T, layer.topk), dtype=torch.float32, device=dev) if gate is None else gate
    _check(lib.moe_route(C.byref(layer), _ptr(x), T, _ptr(idx), _ptr(gate), _ptr(logits), _ptr(ws),
                         ws.numel(), _stream(stream)), "moe_route")
    return idx, gate


def moe_layer_decode(layer: moe_layer_t, x, ws, y=None, flags: int = 0, idx=None, gate=None,
                     cache=None, stream=None):
    T = x.shape[0]
    y = torch.empty_like(x) if y is None else y
    _check(lib.moe_layer_decode(C.byref(layer), _ptr(x), T, flags, _ptr(y), _ptr(idx), _ptr(gate),
                                None if cache is None else cache.handle, _ptr(ws), ws.numel(),
                                _stream(stream)), "moe_layer_decode")
    return y


def moe_layer_decode_host(layer: moe_layer_t, x, ws, y=None, flags: int = 0, idx=None, gate=None,
                          cache=None, stream=None):
    """moe_layer_decode on host (CPU) tensors: x, y, idx, gate live in host memory
    (pinned for asynchronous copies); returns once y is filled."""
    T = x.shape[0]
    y = torch.empty_like(x) if y is None else y
    for t in (x, y, idx, gate):
        if t is not None and t.is_cuda:
            raise ValueError("moe_layer_decode_host takes host tensors")
    _check(lib.moe_layer_decode_host(C.byref(layer), _ptr(x), T, flags, _ptr(y), _ptr(idx), _ptr(gate),
                                     None if cache is None else cache.handle, _ptr(ws), ws.numel(),
                                     _stream(stream)), "moe_layer_decode_host")
    return y


class DecodeHostCall:
    """moe_layer_decode_host for repeated one-token calls on the same layer,
    workspace and stream: the arguments are marshalled once, and each call passes
    only the host rows (tensors or plain addresses) -- the per-call Python work of
    a decode loop that feeds the library from host memory."""

    def __init__(self, layer: moe_layer_t, ws, flags: int = 0, stream=None):
        self._layer = layer  # kept alive for the pointer below
        self._lref = C.byref(layer)
        self._ws, self._nbytes = C.c_void_p(ws.data_ptr()), C.c_size_t(ws.numel())
        self._keep = ws
        self._flags = int(flags)
        self._stream = _stream(stream)
        self._fn = lib.moe_layer_decode_host

    def __call__(self, x, y):
        xp = x if isinstance(x, int) else x.data_ptr()
        yp = y if isinstance(y, int) else y.data_ptr()
        rc = self._fn(self._lref, xp, 1, self._flags, yp, None, None, None, self._ws, self._nbytes, self._stream)
        if rc != MOE_OK:
            raise MoeError(rc, "moe_layer_decode_host")


class HostCall:
    """moe_host_call: the decode step on host rows, prepared once for one layer,
    workspace, token count T, flags and stream (the step is a recorded CUDA graph;
    each call copies x in, launches it, waits for its completion word in host memory
    and copies y out).  `x_row` / `y_row` are the handle's page-locked staging rows
    (T x H fp32 tensors); passing them to the call skips the copies."""

    def __init__(self, layer: moe_layer_t, ws, T: int = 1, flags: int = 0, stream=None):
        self._layer, self._ws = layer, ws  # kept alive for the handle's pointers
        self.T, self.H = int(T), int(layer.H)
        h = C.c_void_p()
        _check(lib.moe_host_call_create(C.byref(h), C.byref(layer), self.T, int(flags), _ptr(ws), ws.numel(),
                                        _stream(stream)), "moe_host_call_create")
        self._h = h
        xr, yr = C.POINTER(C.c_float)(), C.POINTER(C.c_float)()
        _check(lib.moe_host_call_rows(h, C.byref(xr), C.byref(yr)), "moe_host_call_rows")
        n = self.T * self.H
        self.x_row = torch.frombuffer((C.c_float * n).from_address(C.addressof(xr.contents)),
                                      dtype=torch.float32).view(self.T, self.H)
        self.y_row = torch.frombuffer((C.c_float * n).from_address(C.addressof(yr.contents)),
                                      dtype=torch.float32).view(self.T, self.H)
        self._run = lib.moe_host_call_run

    def __call__(self, x, y):
        """x, y: host tensors (T x H fp32, contiguous) or plain addresses."""
        xp = x if isinstance(x, int) else x.data_ptr()
        yp = y if isinstance(y, int) else y.data_ptr()
        rc = self._run(self._h, xp, yp)
        if rc != MOE_OK:
            raise MoeError(rc, "moe_host_call_run")

    def close(self):
        if self._h:
            lib.moe_host_call_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_layer_decode_noalloc(layer: moe_layer_t, x, y=None, flags: int = 0, idx=None, gate=None,
                             stream=None):
    """moe_layer_decode with the library's own static scratch (no workspace argument)."""
    T = x.shape[0]
    y = torch.empty_like(x) if y is None else y
    _check(lib.moe_layer_decode_noalloc(C.byref(layer), _ptr(x), T, flags, _ptr(y), _ptr(idx),
                                        _ptr(gate), _stream(stream)), "moe_layer_decode_noalloc")
    return y


def moe_layer_prefill_chunk(layer: moe_layer_t, x, ws, y=None, flags: int = 0, idx=None, gate=None,
                            stream=None):
    T = x.shape[0]
    y = torch.empty_like(x) if y is None else y
    _check(lib.moe_layer_prefill_chunk(C.byref(layer), _ptr(x), T, flags, _ptr(y), _ptr(idx),
                                       _ptr(gate), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_layer_prefill_chunk")
    return y


# ------------------------------------------------------------------ LFU policy and cache

class LFU:
    """The cache policy on the host (moe_lfu_*), for inspection and tests."""

    def __init__(self, slots: int = 16, E: int = 128):
        self.slots, self.E = slots, E
        h = C.c_void_p()
        _check(lib.moe_lfu_create(C.byref(h), slots, E), "moe_lfu_create")
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None):
            lib.moe_lfu_destroy(self.handle)
            self.handle = None

    def step(self, request):
        import numpy as np
        req = np.ascontiguousarray(request, dtype=np.int32)
        n = req.size
        slot = np.full(max(n, 1), -1, np.int32)
        hit = np.zeros(max(n, 1), np.uint8)
        _check(lib.moe_lfu_step(self.handle, req.ctypes.data if n else None, n, slot.ctypes.data,
                                hit.ctypes.data), "moe_lfu_step")
        return slot[:n], hit[:n].astype(bool)

    def state(self):
        import numpy as np
        eos = np.empty(self.slots, np.int32)
        cnt = np.empty(self.slots, np.uint32)
        last = np.empty(self.slots, np.int64)
        h, m = C.c_uint64(0), C.c_uint64(0)
        _check(lib.moe_lfu_state(self.handle, eos.ctypes.data, cnt.ctypes.data, last.ctypes.data,
                                 C.byref(h), C.byref(m)), "moe_lfu_state")
        return eos, cnt, last, h.value, m.value


class Cache:
    """A per-layer expert cache (moe_cache_*) over tile-layout expert blobs held in
    host memory: `host_experts` is a uint8 CPU tensor [E, stride] (pin it for the
    copies to overlap compute); it must outlive the cache."""

    def __init__(self, H: int, E: int, I: int, host_experts: torch.Tensor, slots: int = 16):
        assert host_experts.device.type == "cpu" and host_experts.dtype == torch.uint8
        assert host_experts.dim() == 2 and host_experts.shape[0] == E and host_experts.is_contiguous()
        self.H, self.E, self.I, self.slots = H, E, I, slots
        self.host_experts = host_experts
        h = C.c_void_p()
        _check(lib.moe_cache_create(C.byref(h), H, E, I, C.c_void_p(host_experts.data_ptr()),
                                    host_experts.stride(0), slots), "moe_cache_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            _check(lib.moe_cache_destroy(self.handle), "moe_cache_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_device_policy(self, enable: bool = True):
        """Run the policy on the device: a cached decode then needs no host round trip."""
        _check(lib.moe_cache_set_device_policy(self.handle, 1 if enable else 0), "moe_cache_set_device_policy")

    def slots_state(self):
        import numpy as np
        eos = np.empty(self.slots, np.int32)
        cnt = np.empty(self.slots, np.uint32)
        _check(lib.moe_cache_slots(self.handle, eos.ctypes.data, cnt.ctypes.data), "moe_cache_slots")
        return eos, cnt

    def stats(self):
        h, m, b = C.c_uint64(0), C.c_uint64(0), C.c_uint64(0)
        _check(lib.moe_cache_stats(self.handle, C.byref(h), C.byref(m), C.byref(b)), "moe_cache_stats")
        return h.value, m.value, b.value


from .weights import AttnLayer, Layer, make_layer, pack_expert_blob, pack_expert_tiles  # noqa: E402
