"""The allocation-free decode entry point, called through the C ABI.

moe_layer_decode_noalloc serves callers that may not allocate device memory:
it runs the same decode as moe_layer_decode but keeps its scratch in a static
device array inside the library.  Each case below makes two calls in a row
(so the second one runs on the scratch the first one left behind) and checks
both against moe_layer_decode on the same inputs, within the tests' fp32
tolerance, with identical expert indices.  This file is collected last and
builds everything it needs itself, so it also passes alone in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest

import synth
from layers import gpu_layer, within_tol

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3


def _noalloc_call(moe, layer, x, T):
    """One call straight through the C entry point; returns (y, idx, gate)."""
    y = torch.empty((T, layer.H), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, layer.topk), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, layer.topk), dtype=torch.float32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = moe.lib.moe_layer_decode_noalloc(C.byref(layer), x.data_ptr(), T, 0, y.data_ptr(),
                                          idx.data_ptr(), gate.data_ptr(), stream)
    assert rc == moe.MOE_OK, moe.status_string(rc)
    return y, idx, gate


def _with_workspace(moe, layer, x, T):
    ws = moe.new_workspace(layer, T)
    idx = torch.empty((T, layer.topk), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, layer.topk), dtype=torch.float32, device="cuda")
    y = moe.moe_layer_decode(layer, x, ws, idx=idx, gate=gate)
    return y, idx, gate


@pytest.mark.parametrize("shape,T", [(synth.TINY, 1), (synth.TINY, 7), (synth.FULL, 1), (synth.FULL, 16)],
                         ids=["tiny-T1", "tiny-T7", "full-T1", "full-T16"])
def test_noalloc_matches_workspace_decode_twice(shape, T):
    import bit_affine_quantised_affine4_b300 as moe
    gl = gpu_layer(shape, seed=0, bias=synth.popularity_bias(shape, seed=0) if T > 1 else None)
    layer = gl.view()
    for call in range(2):
        x = torch.from_numpy(synth.tokens(shape, T, seed=0, stream=900 + 10 * T + call)).cuda()
        y_na, idx_na, gate_na = _noalloc_call(moe, layer, x, T)
        y_ws, idx_ws, gate_ws = _with_workspace(moe, layer, x, T)
        torch.cuda.synchronize()
        assert np.array_equal(idx_na.cpu().numpy(), idx_ws.cpu().numpy())
        assert within_tol(gate_na.cpu().numpy(), gate_ws.cpu().numpy(), TOL)[0]
        ok, worst = within_tol(y_na.cpu().numpy(), y_ws.cpu().numpy(), TOL)
        assert ok, "call %d: worst err/bound %.3f" % (call, worst)


def test_noalloc_scratch_fits_full_layer():
    # the full-size layer (hidden 2816, 128 experts, top-8, inter 704, shared
    # inter 2112) at the largest decode batch needs 2,602,240 bytes of scratch,
    # under the static array's 4 MiB
    import bit_affine_quantised_affine4_b300 as moe
    s = synth.FULL
    layer = moe.moe_layer_t(H=s.H, E=s.E, topk=s.topk, I=s.I, Is=s.Is, r_q=256, r_s=256, r_b=256,
                            experts=256, expert_stride=moe.moe_tile_blob_bytes(s.H, s.I), shared=256)
    need = moe.moe_decode_workspace_bytes(layer, moe.MOE_MAX_DECODE_TOKENS)
    assert need == 2_602_240
    assert need <= moe.MOE_NOALLOC_SCRATCH_BYTES


def test_noalloc_status_reports_a_wait_that_gave_up():
    """A routing wait made unreachable (fault injection, 2 ms limit) gives up: the
    kernel drains, moe_noalloc_status reports MOE_ETIMEOUT once and clears the
    array, and the next call is correct again."""
    import bit_affine_quantised_affine4_b300 as moe
    shape = synth.TINY
    gl = gpu_layer(shape, seed=0)
    layer = gl.view()
    x = torch.from_numpy(synth.tokens(shape, 1, seed=0, stream=990)).cuda()
    _noalloc_call(moe, layer, x, 1)
    assert moe.moe_noalloc_status() == moe.MOE_OK
    moe.moe_debug_inject(moe.MOE_INJECT_WAIT)
    _noalloc_call(moe, layer, x, 1)
    assert moe.moe_noalloc_status() == moe.MOE_ETIMEOUT
    assert moe.moe_noalloc_status() == moe.MOE_OK
    y_na, idx_na, _ = _noalloc_call(moe, layer, x, 1)
    y_ws, idx_ws, _ = _with_workspace(moe, layer, x, 1)
    torch.cuda.synchronize()
    assert moe.moe_noalloc_status() == moe.MOE_OK
    assert np.array_equal(idx_na.cpu().numpy(), idx_ws.cpu().numpy())
    assert within_tol(y_na.cpu().numpy(), y_ws.cpu().numpy(), TOL)[0]


def test_noalloc_rejects_oversized_layer():
    import bit_affine_quantised_affine4_b300 as moe
    # 256 experts of a wide layer at T = 16 need more scratch than the static array
    big = moe.moe_layer_t(H=8192, E=256, topk=8, I=1024, Is=4096, r_q=256, r_s=256, r_b=256,
                          experts=256, expert_stride=moe.moe_expert_blob_bytes(8192, 1024),
                          shared=256)
    x = torch.zeros((16, 8192), device="cuda")
    y = torch.empty_like(x)
    rc = moe.lib.moe_layer_decode_noalloc(C.byref(big), x.data_ptr(), 16, 0, y.data_ptr(), None,
                                          None, None)
    assert rc == moe.MOE_EWORKSPACE
