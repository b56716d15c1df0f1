"""mf_attn_fwd on the GPU vs the float64 oracle on the same bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
import synth
from _parity import assert_close, lse_tol_factor, to64

pytestmark = pytest.mark.gpu


def _run_full(samples, heads, head_dim, seed, scale=0.0, budget=0):
    wl = synth.Workload("t", samples, heads, head_dim, "fwd", token_budget=budget, seed=seed)
    t = synth.draw_tensors(wl, with_grad=False)
    plan = mf.pack_plan(samples, token_budget=budget, head_dim=head_dim)
    T = plan.total_tokens
    q, k, v = (t[n][:T].cuda() for n in ("q", "k", "v"))
    o, lse = mf.attn_fwd(q, k, v, plan, softmax_scale=scale)
    mf.check(plan)
    ref = oracle.pack_plan(samples, budget)
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), ref["cu_seqlens"], ref["pos"], softmax_scale=scale)
    assert_close("O", to64(o), O, "o")
    assert_close("LSE", to64(lse), L, "lse", factor=lse_tol_factor(scale, head_dim))
    return o, lse


@pytest.mark.parametrize("seed", range(3))
def test_fwd_tiny(seed):
    wl = synth.tiny(seed)
    _run_full(wl.samples, wl.heads, wl.head_dim, seed)


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("seed", range(3))
def test_fwd_ragged_multi_tile(head_dim, seed):
    # lengths span several 128-row tiles with ragged tails, image-only and
    # single-token samples
    samples = [(0, 16, 16), (7, 64, 32), (0, 128, 128), (200, 160, 48), (1, 16, 16), (55, 96, 208)]
    rng = np.random.default_rng(seed)
    rng.shuffle(samples)
    _run_full(samples, heads=3, head_dim=head_dim, seed=seed)


@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 255, 256, 257])
def test_fwd_tile_boundaries(L):
    # one image-only sample of exactly L tokens (1 x L grid)
    _run_full([(0, 16, 16 * L)], heads=2, head_dim=128, seed=L)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_fwd_text_only_and_image_only_samples(head_dim):
    # text-only samples (no image: unrotated), image-only samples, a 1-token
    # text-only sample, lengths around the tile edges
    _run_full([(40, 0, 0), (0, 48, 48), (1, 0, 0), (129, 0, 0), (3, 32, 32), (0, 16, 16 * 127)],
              heads=2, head_dim=head_dim, seed=head_dim)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_fwd_runs_of_short_ragged_samples(head_dim):
    # 200 samples of at most 124 tokens, 8 heads: every work item is one
    # ragged K/V tile, about 11 in a row per CTA, so the two sets of
    # ragged-tail barriers take turns many times within one launch
    samples = synth.random_pack(900 + head_dim, 200, 60, 8)
    assert max(t + (h // 16) * (w // 16) for t, h, w in samples) < 128
    _run_full(samples, heads=8, head_dim=head_dim, seed=head_dim)


def test_fwd_custom_scale_and_budget():
    samples = [(30, 96, 96), (12, 64, 48), (0, 48, 160)]
    _run_full(samples, heads=2, head_dim=64, seed=4, scale=0.3)
    _run_full(samples, heads=2, head_dim=128, seed=5, budget=80)


def test_fwd_empty_pack():
    plan = mf.pack_plan([], 0)
    z = torch.empty((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = mf.attn_fwd(z, z, z, plan)
    mf.check(plan)
    assert o.shape == (0, 4, 128) and lse.shape == (4, 0)


def _sample_rows(cu, per_sample, rng):
    rows = []
    for i in range(len(cu) - 1):
        a, b = int(cu[i]), int(cu[i + 1])
        cand = {a, b - 1, min(a + 127, b - 1), min(a + 128, b - 1), b - 1 - (b - a) % 128}
        cand |= set(int(x) for x in rng.integers(a, b, size=per_sample))
        rows += sorted(cand)
    return rows


@pytest.mark.parametrize("name", ["single_1024", "native_res_32k", "cfg_pair", "extreme_aspect", "native_res_50k"])
def test_fwd_full_size_sampled(name):
    """Full-size workloads in the launch configuration the bench times;
    sampled rows (sample edges, tile edges, random) of every head vs the
    oracle row by row."""
    wl = synth.WORKLOADS[name]()
    t = synth.draw_tensors(wl, with_grad=False)
    plan = mf.pack_plan(wl.samples, token_budget=wl.token_budget, head_dim=wl.head_dim)
    q, k, v = (t[n].cuda() for n in ("q", "k", "v"))
    o, lse = mf.attn_fwd(q, k, v, plan)
    mf.check(plan)
    ref = oracle.pack_plan(wl.samples, wl.token_budget)
    rng = np.random.default_rng(0)
    rows = _sample_rows(ref["cu_seqlens"], 4, rng)
    qn, kn, vn = t["q"].float().numpy(), t["k"].float().numpy(), t["v"].float().numpy()
    o_cpu, lse_cpu = to64(o), to64(lse)
    for h in range(wl.heads):
        O, L = oracle.attn_rows(qn, kn, vn, ref["cu_seqlens"], ref["pos"], rows, h)
        assert_close(f"O[{name},h{h}]", o_cpu[rows, h], O, "o")
        assert_close(f"LSE[{name},h{h}]", lse_cpu[h, rows], L, "lse")
    assert np.all(np.isfinite(o_cpu))
    if wl.cfg_pairs:
        # cond and uncond share image K/V but not text, so outputs differ;
        # each pair member is still its own sample: check the first pair fully
        a, b = int(ref["cu_seqlens"][0]), int(ref["cu_seqlens"][2])
        sub = oracle.pack_plan(wl.samples[:2])
        O, L = oracle.attn_fwd(qn[a:b, :2], kn[a:b, :2], vn[a:b, :2], sub["cu_seqlens"], sub["pos"])
        assert_close("O[cfg pair 0]", o_cpu[a:b, :2], O, "o")
        assert_close("LSE[cfg pair 0]", lse_cpu[:2, a:b], L, "lse")


def test_fwd_range_report_and_clear():
    """A rotated K row beyond the fp16 range of the logit product is reported
    by mf_check as MF_ERR_RANGE; the status word is then cleared."""
    samples = [(4, 32, 32)]
    plan = mf.pack_plan(samples, head_dim=128)
    T = plan.total_tokens
    q = torch.randn(T, 2, 128, device="cuda").to(torch.bfloat16)
    k = q.clone()
    v = q.clone()
    k[3, 1, 5] = 1.0e6
    mf.attn_fwd(q, k, v, plan)
    with pytest.raises(mf.MfError) as ei:
        mf.check(plan)
    assert ei.value.code == "MF_ERR_RANGE"
    k[3, 1, 5] = 1.0
    mf.attn_fwd(q, k, v, plan)
    mf.check(plan)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_fwd_non_finite_values_stay_in_their_sample(head_dim):
    """NaN and Inf in one sample's V (and NaN in its Q and K) leave every
    other sample's O and LSE exactly as without them: tiles that run past a
    sample's end read the next sample's rows, and a masked logit (P = 0)
    times a non-finite V value would otherwise be NaN.  The neighbours'
    lengths are ragged, so their last tiles reach into the poisoned sample."""
    samples = [(5, 256, 208), (3, 160, 160), (0, 16, 16 * 77), (9, 64, 16 * 30)]
    heads = 2
    wl = synth.Workload("t", samples, heads, head_dim, "fwd", seed=41)
    t = synth.draw_tensors(wl, with_grad=False)
    ref = oracle.pack_plan(samples)
    cu = ref["cu_seqlens"]
    a, b = int(cu[1]), int(cu[2])
    q, k, v = (t[n].clone() for n in ("q", "k", "v"))
    v[a:b, 0] = float("nan")
    v[a:b, 1] = float("inf")
    v[a + 3, 1, 7] = float("-inf")
    q[a + 1:b, :, :5] = float("nan")
    k[a:b - 2, :, 3:9] = float("nan")
    plan = mf.pack_plan(samples, head_dim=head_dim)
    o, lse = mf.attn_fwd(q.cuda(), k.cuda(), v.cuda(), plan)
    mf.check(plan)
    O, L = oracle.attn_fwd(to64(t["q"]), to64(t["k"]), to64(t["v"]), cu, ref["pos"])
    keep = np.r_[0:a, b:int(cu[-1])]
    assert_close("O outside the poisoned sample", to64(o)[keep], O[keep], "o")
    assert_close("LSE outside the poisoned sample", to64(lse)[:, keep], L[:, keep], "lse")
