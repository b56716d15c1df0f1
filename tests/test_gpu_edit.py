"""Edit packs on the GPU: (frame, row, col) RoPE (rope_axes 3), forward and
backward vs the float64 oracle on the same bf16 inputs.

An edit sample (text, H, W, 2) carries its source and target latents as
frames 0 and 1 (review, editing-model section); the attention kernels are the
same as for 2D packs, only the once-per-token rotation passes, the plan and
the dK / dQ inverse rotations read the third axis.
"""
import numpy as np
import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
import synth
from _parity import assert_close, to64

pytestmark = pytest.mark.gpu


def _run(samples, heads, head_dim, seed, bwd=True):
    wl = synth.Workload("e", samples, heads, head_dim, "fwd+bwd", seed=seed, rope_axes=3)
    t = synth.draw_tensors(wl, with_grad=bwd)
    plan = mf.pack_plan(samples, head_dim=head_dim, rope_axes=3)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    wsf = torch.empty(max(256, mf.fwd_workspace_bytes(plan.total_tokens, heads, head_dim)), dtype=torch.uint8,
                      device="cuda")
    o, lse = mf.attn_fwd(q, k, v, plan, workspace=wsf)
    mf.check(plan)
    ref = oracle.pack_plan(samples)
    rope = dict(frame=ref["frame"], rope_axes=3)
    qn, kn, vn = to64(q), to64(k), to64(v)
    O, L = oracle.attn_fwd(qn, kn, vn, ref["cu_seqlens"], ref["pos"], **rope)
    assert_close("O", to64(o), O, "o")
    assert_close("LSE", to64(lse), L, "lse")
    if not bwd:
        return
    do = t["do"].cuda()
    rq, rk, rv = oracle.attn_bwd(qn, kn, vn, O, L, to64(do), ref["cu_seqlens"], ref["pos"], **rope)
    dq, dk, dv = mf.attn_bwd(q, k, v, o, lse, do, plan)
    mf.check(plan)
    assert_close("dV", to64(dv), rv, "grad")
    assert_close("dK", to64(dk), rk, "grad")
    assert_close("dQ", to64(dq), rq, "grad")


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("seed", range(3))
def test_edit_random_packs(head_dim, seed):
    _run(synth.random_pack(300 + seed, 6, 60, 14, edit=True), 2, head_dim, seed)


def test_edit_tile_edges_and_generation_only():
    # two-frame samples whose frames straddle 128-row tiles, a 1-token frame,
    # and a pack of one-frame samples planned with 3 axes
    _run([(5, 16 * 10, 16 * 13, 2), (0, 16, 16, 2), (127, 32, 64, 2), (3, 48, 48)], 2, 128, 7)
    _run(synth.random_pack(400, 5, 30, 10), 2, 128, 8)


def test_edit_frames_change_the_result():
    """The frame axis matters: the same pack planned as one long two-frame
    sample with 3 axes differs from the 2-axis rotation of the same tokens
    (frames are not rows)."""
    samples = [(8, 64, 64, 2)]
    wl = synth.Workload("e", samples, 2, 128, "fwd", seed=3, rope_axes=3)
    t = synth.draw_tensors(wl, with_grad=False)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o3, _ = mf.attn_fwd(q, k, v, mf.pack_plan(samples, head_dim=128, rope_axes=3))
    ref = oracle.pack_plan(samples)
    O2, _ = oracle.attn_fwd(to64(q), to64(k), to64(v), ref["cu_seqlens"], ref["pos"])
    assert np.abs(to64(o3) - O2).max() > 1e-2


def test_edit_full_size_sampled():
    """The edit training pack (about 27K tokens, 24 heads) in the bench's
    launch configuration: sampled forward rows on three heads, and the
    backward of its smallest edit sample on two heads."""
    wl = synth.edit_pack(0)
    t = synth.draw_tensors(wl, with_grad=True)
    plan = mf.pack_plan(wl.samples, head_dim=wl.head_dim, rope_axes=3)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = mf.attn_fwd(q, k, v, plan)
    dq, dk, dv = mf.attn_bwd(q, k, v, o, lse, do, plan)
    mf.check(plan)
    ref = oracle.pack_plan(wl.samples)
    cu = ref["cu_seqlens"]
    rng = np.random.default_rng(0)
    rows = []
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        t0 = wl.samples[i][0]
        rows += [a, a + t0, b - 1] + list(rng.integers(a, b, size=3))
    rows = sorted(set(int(r) for r in rows))
    qn, kn, vn = (x.float().numpy() for x in (t["q"], t["k"], t["v"]))
    o_c, lse_c = to64(o), to64(lse)
    for h in (0, 11, 23):
        O, L = oracle.attn_rows(qn, kn, vn, cu, ref["pos"], rows, h, frame=ref["frame"], rope_axes=3)
        assert_close(f"O[h{h}]", o_c[rows, h], O, "o")
        assert_close(f"LSE[h{h}]", lse_c[h, rows], L, "lse")
    si = 2  # the smallest edit sample
    a, b = int(cu[si]), int(cu[si + 1])
    sub = oracle.pack_plan([wl.samples[si]])
    rope = dict(frame=sub["frame"], rope_axes=3)
    for h in (0, 23):
        hs = slice(h, h + 1)
        qs, ks, vs, gs = (to64(x[a:b, hs]) for x in (q, k, v, do))
        O, L = oracle.attn_fwd(qs, ks, vs, sub["cu_seqlens"], sub["pos"], **rope)
        rq, rk, rv = oracle.attn_bwd(qs, ks, vs, O, L, gs, sub["cu_seqlens"], sub["pos"], **rope)
        assert_close(f"dV[h{h}]", to64(dv[a:b, hs]), rv, "grad")
        assert_close(f"dK[h{h}]", to64(dk[a:b, hs]), rk, "grad")
        assert_close(f"dQ[h{h}]", to64(dq[a:b, hs]), rq, "grad")
