"""C-ABI checks that need no GPU: the library loads, exports every function
include/mf.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import packed_resolution_diffusion_plan_b300 as mf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mf.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mf_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mf.library_path):
        from packed_resolution_diffusion_plan_b300 import build
        build.build()
    return mf.lib()


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert set(declared) == set(mf.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(7):
        assert L.mf_status_string(code)
    assert L.mf_last_cuda_error() is not None


def _ws_size(L, samples, budget=0, head_dim=128, rope_axes=2):
    arr = mf._samples_array(samples)
    n = ctypes.c_size_t(0)
    st = L.mf_pack_plan_workspace_size(arr, len(samples), budget, head_dim, rope_axes, ctypes.byref(n))
    return st, n.value


def test_plan_validation_without_gpu(L):
    assert _ws_size(L, [(17, 128, 128), (9, 64, 256)])[0] == 0
    assert _ws_size(L, [])[0] == 0
    for bad in [(-1, 16, 16), (0, 0, 16), (0, 16, 24), (3, 17, 16), (0, -16, 16), (0, 0, 0)]:
        assert _ws_size(L, [bad])[0] == 1, bad
    assert _ws_size(L, [(7, 0, 0), (0, 16, 16)])[0] == 0   # text-only sample
    assert _ws_size(L, [(0, 16, 16)], head_dim=96)[0] == 2
    assert _ws_size(L, [(0, 16 * 1025, 16)])[0] == 2
    assert _ws_size(L, [(100, 64, 64)], budget=50)[0] == 3
    st, n_small = _ws_size(L, [(10, 64, 64)] * 3, budget=60)
    st2, n_all = _ws_size(L, [(10, 64, 64)] * 3)
    assert st == 0 and st2 == 0 and n_small < n_all
    # frames: an edit sample (frames 2) needs the 3-axis rotation; frames > 2 and
    # rope_axes other than 2 or 3 are rejected; 0 frames count as one
    assert _ws_size(L, [(4, 32, 32, 2)], rope_axes=3)[0] == 0
    assert _ws_size(L, [(4, 32, 32, 2)], rope_axes=2)[0] == 1
    assert _ws_size(L, [(4, 32, 32, 3)], rope_axes=3)[0] == 1
    assert _ws_size(L, [(4, 32, 32, 0)])[0] == 0
    assert _ws_size(L, [(4, 32, 32)], rope_axes=4)[0] == 1
    assert _ws_size(L, [(4, 512, 512, 2)], rope_axes=3)[1] > _ws_size(L, [(4, 512, 512)], rope_axes=3)[1]
    # null size pointer / null samples with n > 0
    assert L.mf_pack_plan_workspace_size(None, 1, 0, 128, 2, None) == 1
    n = ctypes.c_size_t(0)
    assert L.mf_pack_plan_workspace_size(None, 2, 0, 128, 2, ctypes.byref(n)) == 1
    assert L.mf_pack_plan_workspace_size(None, 5000, 0, 128, 2, ctypes.byref(n)) == 1
    arr = mf._samples_array([(0, 16, 16)] * 1)
    big = (mf.MfSample * 4097)()
    for i in range(4097):
        big[i] = mf.MfSample(1, 16, 16, 1)
    assert L.mf_pack_plan_workspace_size(big, 4097, 0, 128, 2, ctypes.byref(n)) == 2
    # pack call: null / misaligned workspace and bad theta fail before any CUDA call
    plan = mf.MfPlan()
    assert L.mf_pack_plan(arr, 1, 0, 128, 2, 10000.0, None, 0, ctypes.byref(plan), None) == 1
    assert L.mf_pack_plan(arr, 1, 0, 128, 2, 10000.0, ctypes.c_void_p(256 + 8), 1 << 20,
                          ctypes.byref(plan), None) == 1
    assert L.mf_pack_plan(arr, 1, 0, 128, 2, -1.0, ctypes.c_void_p(256), 1 << 20,
                          ctypes.byref(plan), None) == 1
    assert L.mf_pack_plan(arr, 1, 0, 128, 2, 10000.0, ctypes.c_void_p(256), 16,
                          ctypes.byref(plan), None) == 1
    assert L.mf_pack_plan(arr, 1, 0, 128, 5, 10000.0, ctypes.c_void_p(256), 1 << 20,
                          ctypes.byref(plan), None) == 1


def test_attn_validation_without_gpu(L):
    plan = mf.MfPlan()
    plan.total_tokens, plan.n_samples, plan.head_dim, plan.n_tiles, plan.rope_axes = 10, 1, 128, 1, 2
    for p in ("cu_seqlens", "pos", "frame", "rope_cs", "order", "status"):
        setattr(plan, p, 4096)
    vp = ctypes.c_void_p
    ok = vp(1 << 20)
    # null plan, bad heads, unsupported / mismatched head_dim, null or misaligned
    # tensors, null / short / misaligned workspace
    big = 1 << 30
    assert L.mf_attn_fwd(ok, ok, ok, None, 2, 128, 0.0, ok, big, ok, ok, None) == 1
    assert L.mf_attn_fwd(ok, ok, ok, ctypes.byref(plan), 0, 128, 0.0, ok, big, ok, ok, None) == 1
    assert L.mf_attn_fwd(ok, ok, ok, ctypes.byref(plan), 2, 96, 0.0, ok, big, ok, ok, None) == 2
    assert L.mf_attn_fwd(ok, ok, ok, ctypes.byref(plan), 2, 64, 0.0, ok, big, ok, ok, None) == 1
    assert L.mf_attn_fwd(None, ok, ok, ctypes.byref(plan), 2, 128, 0.0, ok, big, ok, ok, None) == 1
    assert L.mf_attn_fwd(vp((1 << 20) + 2), ok, ok, ctypes.byref(plan), 2, 128, 0.0, ok, big, ok, ok, None) == 1
    assert L.mf_attn_fwd(ok, ok, ok, ctypes.byref(plan), 2, 128, 0.0, None, big, ok, ok, None) == 1
    assert L.mf_attn_fwd(ok, ok, ok, ctypes.byref(plan), 2, 128, 0.0, ok, 16, ok, ok, None) == 1
    assert L.mf_attn_fwd(ok, ok, ok, ctypes.byref(plan), 2, 128, 0.0, vp((1 << 20) + 16), big, ok, ok, None) == 1
    n = ctypes.c_size_t(0)
    assert L.mf_attn_fwd_workspace_size(10, 2, 128, ctypes.byref(n)) == 0
    assert n.value >= 10 * 2 * 128 * 2 + 4
    assert L.mf_attn_fwd_workspace_size(10, 2, 96, ctypes.byref(n)) == 2
    assert L.mf_attn_bwd(ok, ok, ok, ok, ok, ok, ctypes.byref(plan), 2, 128, 0.0, ok, 16,
                         ok, ok, ok, None) == 1
    assert L.mf_attn_bwd(ok, ok, ok, ok, ok, None, ctypes.byref(plan), 2, 128, 0.0, ok, 1 << 30,
                         ok, ok, ok, None) == 1
    n = ctypes.c_size_t(0)
    assert L.mf_attn_bwd_workspace_size(10, 2, 128, ctypes.byref(n)) == 0
    assert n.value >= 10 * 2 * 4 + 10 * 2 * 128 * 4
    assert L.mf_attn_bwd_workspace_size(10, 2, 80, ctypes.byref(n)) == 2
    # an empty pack is a no-op that needs no tensors
    empty = mf.MfPlan()
    empty.head_dim, empty.rope_axes = 128, 2
    assert L.mf_attn_fwd(None, None, None, ctypes.byref(empty), 2, 128, 0.0, None, 0, None, None, None) == 0
    assert L.mf_attn_bwd(None, None, None, None, None, None, ctypes.byref(empty), 2, 128, 0.0, None, 0,
                         None, None, None, None) == 0
    assert L.mf_check(None, None) == 1
    # the chain calls: unsupported hidden sizes, null pointers, bad eps
    assert L.mf_norm_modulate(ok, ctypes.byref(plan), 1000, ok, ok, 1e-6, ok, None) == 2
    assert L.mf_norm_modulate(ok, ctypes.byref(plan), 3072, None, ok, 1e-6, ok, None) == 1
    assert L.mf_norm_modulate(ok, ctypes.byref(plan), 3072, ok, ok, -1.0, ok, None) == 1
    assert L.mf_norm_modulate(ok, None, 3072, ok, ok, 1e-6, ok, None) == 1
    assert L.mf_gate_residual(ok, ok, ctypes.byref(plan), 12, ok, ok, None) == 2
    assert L.mf_gate_residual(ok, None, ctypes.byref(plan), 16, ok, ok, None) == 1
    assert L.mf_attn_fwd_qkv(None, ctypes.byref(plan), 2, 128, 0.0, ok, big, ok, ok, None) == 1
    assert L.mf_attn_fwd_qkv(ok, ctypes.byref(plan), 2, 96, 0.0, ok, big, ok, ok, None) == 2
    assert L.mf_cfg_combine(ok, ctypes.byref(plan), 2, 128, 1.0, ok, None) == 1   # odd sample count
    # the timeout-path test aid takes only the documented bits
    assert L.mf_debug_inject(4) == 1 and L.mf_debug_inject(-1) == 1
    assert L.mf_debug_inject(3) == 0 and L.mf_debug_inject(0) == 0
