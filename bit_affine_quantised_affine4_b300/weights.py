"""Device-side layer weights in the tile layout of include/moe.h.

Packing fp32 weights runs the library's own kernels on the GPU: the quantiser
(affine_quantise) writes an MLX-layout blob, which moe_expert_tile reorders into
the tile layout the layer kernels read.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import (affine_quantise, moe_attn_t, moe_expert_blob_bytes, moe_expert_blob_offsets, moe_expert_tile,
               moe_layer_t, moe_tile_blob_bytes)


def _part(blob: torch.Tensor, off: int, nbytes: int, dtype) -> torch.Tensor:
    return blob[off:off + nbytes].view(dtype)


def pack_expert_blob(gu_w: torch.Tensor, d_w: torch.Tensor, blob: torch.Tensor, stream=None):
    """Quantise one expert (gate/up [2I, H] gate rows first, down [H, I]; fp32 on the GPU)
    into `blob` in the MLX layout (uint8 CUDA tensor of at least moe_expert_blob_bytes(H, I) bytes)."""
    I2, H = gu_w.shape
    I = I2 // 2
    assert d_w.shape == (H, I)
    off = moe_expert_blob_offsets(H, I)
    gq = _part(blob, off[0], I2 * H // 2, torch.int32).view(I2, H // 8)
    gs = _part(blob, off[1], I2 * (H // 64) * 2, torch.int16).view(I2, H // 64)
    gb = _part(blob, off[2], I2 * (H // 64) * 2, torch.int16).view(I2, H // 64)
    dq = _part(blob, off[3], H * I // 2, torch.int32).view(H, I // 8)
    ds = _part(blob, off[4], H * (I // 64) * 2, torch.int16).view(H, I // 64)
    db = _part(blob, off[5], H * (I // 64) * 2, torch.int16).view(H, I // 64)
    affine_quantise(gu_w.contiguous(), 4, gq, gs, gb, stream)
    affine_quantise(d_w.contiguous(), 4, dq, ds, db, stream)
    return blob


def pack_expert_tiles(gu_w: torch.Tensor, d_w: torch.Tensor, tiles: torch.Tensor, stream=None):
    """Quantise one expert into `tiles` (uint8 CUDA tensor of at least
    moe_tile_blob_bytes(H, I) bytes) in the tile layout."""
    I2, H = gu_w.shape
    mlx = torch.empty(moe_expert_blob_bytes(H, I2 // 2), dtype=torch.uint8, device=tiles.device)
    pack_expert_blob(gu_w, d_w, mlx, stream)
    moe_expert_tile(mlx, H, I2 // 2, tiles, stream)
    return tiles


class Layer:
    """One MoE layer resident on the GPU: router (8-bit), E expert blobs, shared blob.

    `copies` > 1 allocates that many independent copies of the expert/shared/router
    memory (same values, different addresses) so that a benchmark can rotate through
    more bytes than the L2 cache holds; `view(c)` returns the C struct of copy c.
    """

    def __init__(self, H, E, topk, I, Is, device="cuda", copies=1):
        self.H, self.E, self.topk, self.I, self.Is = H, E, topk, I, Is
        self.device = torch.device(device)
        self.stride = moe_tile_blob_bytes(H, I)
        self.sstride = moe_tile_blob_bytes(H, Is)
        self.copies = copies
        self.r_q = torch.empty((copies, E, H // 4), dtype=torch.int32, device=self.device)
        self.r_s = torch.empty((copies, E, H // 64), dtype=torch.int16, device=self.device)
        self.r_b = torch.empty((copies, E, H // 64), dtype=torch.int16, device=self.device)
        self.experts = torch.empty((copies, E, self.stride), dtype=torch.uint8, device=self.device)
        self.shared = torch.empty((copies, self.sstride), dtype=torch.uint8, device=self.device)
        self.bias = None
        self.norm_w, self.norm_eps = None, 0.0

    # ---- filling
    def set_router(self, w: torch.Tensor):
        affine_quantise(w.to(self.device, torch.float32).contiguous(), 8, self.r_q[0], self.r_s[0],
                        self.r_b[0])

    def set_expert(self, e: int, gu_w: torch.Tensor, d_w: torch.Tensor):
        pack_expert_tiles(gu_w.to(self.device, torch.float32), d_w.to(self.device, torch.float32),
                          self.experts[0, e])

    def set_shared(self, gu_w: torch.Tensor, d_w: torch.Tensor):
        pack_expert_tiles(gu_w.to(self.device, torch.float32), d_w.to(self.device, torch.float32),
                          self.shared[0])

    def set_bias(self, bias):
        self.bias = None if bias is None else torch.as_tensor(bias, dtype=torch.float32).to(self.device)

    def set_norm(self, w, eps: float = 1e-6):
        """RMSNorm weight [H] and epsilon, read by the layer calls with MOE_PRENORM."""
        self.norm_w = None if w is None else torch.as_tensor(w, dtype=torch.float32).to(self.device).contiguous()
        self.norm_eps = float(eps)

    def replicate(self):
        for c in range(1, self.copies):
            self.r_q[c].copy_(self.r_q[0]); self.r_s[c].copy_(self.r_s[0]); self.r_b[c].copy_(self.r_b[0])
            self.experts[c].copy_(self.experts[0]); self.shared[c].copy_(self.shared[0])

    # ---- C view
    def view(self, c: int = 0, experts: bool = True) -> moe_layer_t:
        return moe_layer_t(
            H=self.H, E=self.E, topk=self.topk, I=self.I, Is=self.Is,
            r_q=self.r_q[c].data_ptr(), r_s=self.r_s[c].data_ptr(), r_b=self.r_b[c].data_ptr(),
            experts=self.experts[c].data_ptr() if experts else None,
            expert_stride=self.stride,
            shared=self.shared[c].data_ptr(),
            logit_bias=None if self.bias is None else self.bias.data_ptr(),
            norm_w=None if self.norm_w is None else self.norm_w.data_ptr(),
            norm_eps=self.norm_eps,
        )

    # ---- host copies of the tile-layout blobs
    def expert_blob_host(self, e: int, c: int = 0):
        return self.experts[c, e].cpu().numpy()

    def shared_blob_host(self, c: int = 0):
        return self.shared[c].cpu().numpy()

    def router_host(self, c: int = 0):
        return (self.r_q[c].cpu().numpy().view("uint32"), self.r_s[c].cpu().numpy().view("uint16"),
                self.r_b[c].cpu().numpy().view("uint16"))


def make_layer(H, E, topk, I, Is, router_w, expert_w, shared_w, bias=None, device="cuda", copies=1):
    """Build a Layer from fp32 weights: router_w [E, H]; expert_w(e) -> (gu [2I, H], d [H, I])
    (a callable, so that the host never holds every expert at once); shared_w = (gu, d)."""
    L = Layer(H, E, topk, I, Is, device=device, copies=copies)
    L.set_router(torch.as_tensor(router_w))
    for e in range(E):
        gu, d = expert_w(e)
        L.set_expert(e, torch.as_tensor(gu), torch.as_tensor(d))
    L.set_shared(*(torch.as_tensor(a) for a in shared_w))
    L.set_bias(bias)
    L.replicate()
    torch.cuda.synchronize(L.device)
    return L


class AttnLayer:
    """One attention block resident on the GPU: the 4-bit [q; k; v] and output
    projections (MLX layout) and the binary16 key/value cache [nkv, kv_len, d]."""

    def __init__(self, H, nq, nkv, d, window, kv_len, theta, scale=None, device="cuda"):
        self.H, self.nq, self.nkv, self.d = H, nq, nkv, d
        self.window, self.kv_len, self.theta = window, kv_len, float(theta)
        self.scale = d ** -0.5 if scale is None else float(scale)
        self.device = torch.device(device)
        nqkv = (nq + 2 * nkv) * d
        self.wqkv = (torch.zeros((nqkv, H // 8), dtype=torch.int32, device=self.device),
                     torch.zeros((nqkv, H // 64), dtype=torch.int16, device=self.device),
                     torch.zeros((nqkv, H // 64), dtype=torch.int16, device=self.device))
        K = nq * d
        self.wo = (torch.zeros((H, K // 8), dtype=torch.int32, device=self.device),
                   torch.zeros((H, K // 64), dtype=torch.int16, device=self.device),
                   torch.zeros((H, K // 64), dtype=torch.int16, device=self.device))
        self.k_cache = torch.zeros((nkv, kv_len, d), dtype=torch.int16, device=self.device)
        self.v_cache = torch.zeros((nkv, kv_len, d), dtype=torch.int16, device=self.device)
        self.norm_w, self.norm_eps = None, 0.0

    def set_weights(self, wqkv, wo):
        """Quantise fp32 Wqkv [(nq + 2 nkv) d, H] and Wo [H, nq d] with the library's quantiser."""
        affine_quantise(torch.as_tensor(wqkv).to(self.device, torch.float32).contiguous(), 4, *self.wqkv)
        affine_quantise(torch.as_tensor(wo).to(self.device, torch.float32).contiguous(), 4, *self.wo)

    def set_cache(self, k_bits, v_bits):
        """Cache contents as binary16 bits: uint16 numpy arrays or int16 tensors [nkv, kv_len, d]."""
        for dst, src in ((self.k_cache, k_bits), (self.v_cache, v_bits)):
            if not torch.is_tensor(src):
                src = torch.from_numpy(np.ascontiguousarray(src).view(np.int16))
            dst.copy_(src.view(torch.int16))

    def set_norm(self, w, eps: float = 1e-6):
        self.norm_w = None if w is None else torch.as_tensor(w, dtype=torch.float32).to(self.device).contiguous()
        self.norm_eps = float(eps)

    def view(self) -> moe_attn_t:
        return moe_attn_t(
            H=self.H, nq=self.nq, nkv=self.nkv, d=self.d, window=self.window, kv_len=self.kv_len,
            theta=self.theta, scale=self.scale,
            wqkv_q=self.wqkv[0].data_ptr(), wqkv_s=self.wqkv[1].data_ptr(), wqkv_b=self.wqkv[2].data_ptr(),
            wo_q=self.wo[0].data_ptr(), wo_s=self.wo[1].data_ptr(), wo_b=self.wo[2].data_ptr(),
            norm_w=None if self.norm_w is None else self.norm_w.data_ptr(), norm_eps=self.norm_eps,
            k_cache=self.k_cache.data_ptr(), v_cache=self.v_cache.data_ptr(),
        )
