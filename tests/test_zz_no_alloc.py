"""The allocation-free backward, mf_attn_bwd_noalloc, called through the C ABI.

It exists for callers that cannot allocate device memory where they run the
backward (an engine plugin whose execute step may not allocate, a runtime
whose pool owns all device memory, a latency-critical loop that avoids
cudaMalloc because it can synchronize the device).  It must give the same
gradients as mf_attn_bwd with a caller workspace, call after call, although
every call reuses the same fixed scratch array.  This file is collected last
so that a run stopping at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import packed_resolution_diffusion_plan_b300 as mf
import synth
from _parity import assert_close, to64

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    fn = mf.lib().mf_attn_bwd_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.POINTER(mf.MfPlan), ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_float, vp, vp, vp, vp]
    fn.restype = ctypes.c_int32
    return fn


def _case(samples, heads, head_dim, seed):
    wl = synth.Workload("t", samples, heads, head_dim, "fwd+bwd", seed=seed)
    t = synth.draw_tensors(wl, with_grad=True)
    plan = mf.pack_plan(samples, head_dim=head_dim)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = mf.attn_fwd(q, k, v, plan)
    return plan, q, k, v, do, o, lse


def _call_noalloc(fn, plan, q, k, v, do, o, lse):
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = fn(p(q), p(k), p(v), p(o), p(lse), p(do), ctypes.byref(plan.raw), q.shape[1], q.shape[2], 0.0,
            p(dq), p(dk), p(dv), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, mf.STATUS.get(st, st)
    mf.check(plan)
    return dq, dk, dv


def test_noalloc_matches_workspace_backward_two_calls_in_a_row():
    """The larger pack first, then the smaller one, each called twice in a
    row: a call that read D or dQ partials left in the shared array by the
    call before it would differ from the caller-workspace backward."""
    fn = _noalloc_fn()
    cases = [
        (synth.single_1024().samples, 24, 128, 2),  # 4224 tokens: 104 MB of scratch
        ([(0, 16, 16), (7, 64, 32), (0, 128, 128), (200, 160, 48), (55, 96, 208)], 3, 128, 1),
    ]
    for samples, heads, head_dim, seed in cases:
        plan, q, k, v, do, o, lse = _case(samples, heads, head_dim, seed)
        want = mf.attn_bwd(q, k, v, o, lse, do, plan)
        mf.check(plan)
        for call in range(2):
            got = _call_noalloc(fn, plan, q, k, v, do, o, lse)
            for name, g, w in zip(("dQ", "dK", "dV"), got, want):
                assert_close(f"noalloc {name} (call {call + 1})", to64(g), to64(w), "grad")


def test_noalloc_rejects_packs_beyond_the_scratch():
    fn = _noalloc_fn()
    plan = mf.pack_plan(synth.native_res(0).samples, token_budget=32768)   # ~800 MB of scratch
    z = ctypes.c_void_p(1 << 20)
    st = fn(z, z, z, z, z, z, ctypes.byref(plan.raw), 24, 128, 0.0, z, z, z, None)
    assert mf.STATUS[st] == "MF_ERR_UNSUPPORTED"
