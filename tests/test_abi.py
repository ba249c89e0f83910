"""The C ABI without a GPU: the library loads, exports what the header declares,
and its host-side layout and argument checks behave."""
import ctypes as C
import os
import re

import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"#define MOE_API.*", "", src)
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    import bit_affine_quantised_affine4_b300 as moe
    names = header_functions()
    assert len(names) >= 15
    assert set(names) == set(moe.ENTRY_POINTS)
    for n in names:
        assert hasattr(moe.lib, n), n


def test_blob_sizes_match_oracle_and_known_figures():
    import bit_affine_quantised_affine4_b300 as moe
    for s in (synth.TINY, synth.FULL):
        for I in (s.I, s.Is):
            assert moe.moe_expert_blob_bytes(s.H, I) == oracle.expert_blob_bytes(s.H, I)
            assert moe.moe_expert_blob_offsets(s.H, I) == oracle.expert_blob_offsets(s.H, I)
    # 4.5 bits per weight: 3 I H weights at (32 + 2 + 2) / 64 bytes each
    assert moe.moe_expert_blob_bytes(2816, 704) == 3_345_408
    assert moe.moe_expert_blob_bytes(2816, 2112) == 10_036_224
    assert moe.moe_expert_blob_bytes(512, 256) == 221_184
    assert moe.moe_expert_blob_bytes(100, 64) == 0


def test_host_side_argument_checks():
    import bit_affine_quantised_affine4_b300 as moe
    L = moe.lib
    assert L.qgemv_affine4(None, None, None, 0, 64, None, None, None) == moe.MOE_EINVAL
    assert L.affine_quantise(None, 4, 64, 3, None, None, None, None) == moe.MOE_EINVAL
    bad = moe.moe_layer_t(H=100, E=8, topk=2, I=64, Is=64)
    assert L.moe_workspace_bytes(C.byref(bad), 1) == 0
    assert L.moe_route(C.byref(bad), None, 1, None, None, None, None, 0, None) == moe.MOE_EINVAL
    assert moe.status_string(moe.MOE_ECAPACITY).startswith("more distinct experts")
    good = moe.moe_layer_t(H=512, E=32, topk=8, I=256, Is=512, r_q=256, r_s=256, r_b=256,
                           experts=256, expert_stride=221184, shared=256)
    assert L.moe_workspace_bytes(C.byref(good), 1) > 0
    assert L.moe_workspace_bytes(C.byref(good), 129) == 0
    # a workspace too small is refused before any launch
    assert L.moe_layer_decode(C.byref(good), 256, 1, 0, 512, None, None, None, 256, 16, None) \
        == moe.MOE_EWORKSPACE
    assert L.moe_layer_decode(C.byref(good), 256, 17, 0, 512, None, None, None, 256, 1 << 30, None) \
        == moe.MOE_EINVAL
    # the prepared host call: refused before any allocation, capture or launch
    h = C.c_void_p(0)
    assert L.moe_host_call_create(None, C.byref(good), 1, 0, 256, 1 << 30, None) == moe.MOE_EINVAL
    assert L.moe_host_call_create(C.byref(h), C.byref(bad), 1, 0, 256, 1 << 30, None) == moe.MOE_EINVAL
    assert L.moe_host_call_create(C.byref(h), C.byref(good), 0, 0, 256, 1 << 30, None) == moe.MOE_EINVAL
    assert L.moe_host_call_create(C.byref(h), C.byref(good), 17, 0, 256, 1 << 30, None) == moe.MOE_EINVAL
    assert L.moe_host_call_create(C.byref(h), C.byref(good), 1, 0x100, 256, 1 << 30, None) == moe.MOE_EINVAL
    assert L.moe_host_call_create(C.byref(h), C.byref(good), 1, 0, 256, 16, None) == moe.MOE_EWORKSPACE
    assert h.value is None  # no handle on a refusal
    assert L.moe_host_call_run(None, 256, 256) == moe.MOE_EINVAL
    assert L.moe_host_call_rows(None, None, None) == moe.MOE_EINVAL
    assert L.moe_host_call_destroy(None) == moe.MOE_OK
