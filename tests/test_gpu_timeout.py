"""The timeout path of the attention kernels, on the GPU, without a fault.

mf_debug_inject makes the main kernel's TMA producer drop its streamed-tile
loads, so the consumers' bounded mbarrier waits run out (about 4 s).  The
kernel must then leave every loop, free its TMEM and exit with the timeout
status, which mf_check reports as MF_ERR_TIMEOUT and clears; the next normal
call on the same context must produce correct results.
"""
import re
import time

import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
import synth
from _parity import assert_close, to64

pytestmark = pytest.mark.gpu


def _inputs():
    wl = synth.tiny(0)
    t = synth.draw_tensors(wl, with_grad=True)
    plan = mf.pack_plan(wl.samples, head_dim=wl.head_dim)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    return wl, plan, q, k, v, do


def _expect_timeout(plan, kernel, n_ctas):
    """MF_ERR_TIMEOUT, with the record naming the kernel, a barrier of its
    barrier block and between one and n_ctas CTAs: every CTA of the
    persistent kernel that took a work item gives up, and with the loads
    dropped a CTA may take a second item before its first wait runs out,
    leaving others none."""
    t0 = time.time()
    with pytest.raises(mf.MfError) as ei:
        mf.check(plan)
    assert ei.value.code == "MF_ERR_TIMEOUT"
    assert time.time() - t0 < 60.0
    m = re.search(r"timed out in (\w+): first at barrier (\d+), (\d+) CTA", str(ei.value))
    assert m, str(ei.value)
    assert m.group(1) == kernel
    assert int(m.group(2)) < 40
    assert 1 <= int(m.group(3)) <= n_ctas
    mf.check(plan)  # the status word and the record were cleared


def test_fwd_dropped_loads_time_out_then_recover():
    wl, plan, q, k, v, _ = _inputs()
    mf.debug_inject(mf.DEBUG_DROP_FWD_KV)
    try:
        mf.attn_fwd(q, k, v, plan)
    finally:
        mf.debug_inject(0)
    _expect_timeout(plan, "attn_fwd_kernel", min(plan.n_pairs * q.shape[1], torch.cuda.get_device_properties(0).multi_processor_count))
    o, lse = mf.attn_fwd(q, k, v, plan)
    mf.check(plan)
    ref = oracle.pack_plan(wl.samples)
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), ref["cu_seqlens"], ref["pos"])
    assert_close("O", to64(o), O, "o")
    assert_close("LSE", to64(lse), L, "lse")


def test_bwd_dropped_loads_time_out_then_recover():
    wl, plan, q, k, v, do = _inputs()
    o, lse = mf.attn_fwd(q, k, v, plan)
    mf.check(plan)
    mf.debug_inject(mf.DEBUG_DROP_BWD_QDO)
    try:
        mf.attn_bwd(q, k, v, o, lse, do, plan)
    finally:
        mf.debug_inject(0)
    _expect_timeout(plan, "bwd_main_kernel", min(plan.n_tiles * q.shape[1], torch.cuda.get_device_properties(0).multi_processor_count))
    dq, dk, dv = mf.attn_bwd(q, k, v, o, lse, do, plan)
    mf.check(plan)
    ref = oracle.pack_plan(wl.samples)
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), ref["cu_seqlens"], ref["pos"])
    dQ, dK, dV = oracle.attn_bwd(to64(q), to64(k), to64(v), O, L, to64(do), ref["cu_seqlens"], ref["pos"])
    assert_close("dQ", to64(dq), dQ, "grad")
    assert_close("dK", to64(dk), dK, "grad")
    assert_close("dV", to64(dv), dV, "grad")


def test_debug_inject_rejects_unknown_bits():
    with pytest.raises(mf.MfError) as ei:
        mf.debug_inject(4)
    assert ei.value.code == "MF_ERR_INVALID_ARG"
