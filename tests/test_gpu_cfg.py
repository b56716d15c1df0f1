"""mf_cfg_combine on the GPU vs the oracle: guided = u + g (c - u) on the
conditional image rows of each (cond, uncond) sample pair of a pack."""
import numpy as np
import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
import synth
from _parity import to64

pytestmark = pytest.mark.gpu


def _check(samples, guidance, heads=3, head_dim=128, seed=0, in_place=False):
    plan = mf.pack_plan(samples, head_dim=head_dim)
    g = torch.Generator("cpu").manual_seed(seed)
    o = torch.randn((plan.total_tokens, heads, head_dim), generator=g).to(torch.bfloat16).cuda()
    ref = oracle.pack_plan(samples)
    want = oracle.cfg_combine(to64(o), ref["cu_seqlens"], ref["pos"], guidance)
    out = mf.cfg_combine(o, plan, guidance, out=o if in_place else None)
    mf.check(plan)
    got = to64(out)
    # fp32 arithmetic rounded once to bf16: within half a bf16 ulp of the value
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30)


@pytest.mark.parametrize("guidance", [0.0, 1.0, 4.5, -2.0])
def test_cfg_small_pairs(guidance):
    # pairs with different text lengths, one image-only member, 1-token images
    _check([(5, 32, 48), (2, 32, 48), (0, 16, 16), (9, 16, 16), (17, 64, 32), (8, 64, 32)], guidance)


def test_cfg_head_dim_64_and_in_place():
    _check([(3, 48, 48), (1, 48, 48)], 3.0, head_dim=64, in_place=True)


def test_cfg_mismatched_pair_is_reported():
    plan = mf.pack_plan([(1, 16, 16), (1, 32, 16)])
    o = torch.zeros((plan.total_tokens, 1, 128), dtype=torch.bfloat16, device="cuda")
    mf.cfg_combine(o, plan, 2.0)
    with pytest.raises(mf.MfError) as ei:
        mf.check(plan)
    assert ei.value.code == "MF_ERR_INVALID_ARG"
    with pytest.raises(mf.MfError):
        mf.cfg_combine(o[:1], mf.pack_plan([(0, 16, 16)]), 2.0)  # odd sample count


def test_cfg_full_pack():
    """The CFG pair pack (4 prompts at 1024^2, 33,824 tokens, 24 heads): the
    GPU forward of the packed branches, then the guidance on its output."""
    wl = synth.cfg_pair(0)
    t = synth.draw_tensors(wl, with_grad=False)
    plan = mf.pack_plan(wl.samples, head_dim=wl.head_dim)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o, _ = mf.attn_fwd(q, k, v, plan)
    out = mf.cfg_combine(o, plan, 4.0)
    mf.check(plan)
    ref = oracle.pack_plan(wl.samples)
    want = oracle.cfg_combine(to64(o), ref["cu_seqlens"], ref["pos"], 4.0)
    got = to64(out)
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30)
