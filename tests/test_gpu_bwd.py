"""mf_attn_bwd on the GPU vs the float64 oracle.  The GPU backward consumes
the GPU forward's O and LSE; the oracle computes its own from the same bf16
Q, K, V, dO, so the comparison covers forward + backward end to end."""
import numpy as np
import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
import synth
from _parity import assert_close, lse_tol_factor, to64

pytestmark = pytest.mark.gpu


def _gpu_fwd_bwd(samples, heads, head_dim, seed, budget=0, scale=0.0):
    wl = synth.Workload("t", samples, heads, head_dim, "fwd+bwd", token_budget=budget, seed=seed)
    t = synth.draw_tensors(wl, with_grad=True)
    plan = mf.pack_plan(samples, token_budget=budget, head_dim=head_dim)
    T = plan.total_tokens
    q, k, v, do = (t[n][:T].cuda() for n in ("q", "k", "v", "do"))
    wsf = torch.empty(max(256, mf.fwd_workspace_bytes(T, heads, head_dim)), dtype=torch.uint8, device="cuda")
    o, lse = mf.attn_fwd(q, k, v, plan, softmax_scale=scale, workspace=wsf)
    dq, dk, dv = mf.attn_bwd(q, k, v, o, lse, do, plan, softmax_scale=scale)
    mf.check(plan)
    return plan, (q, k, v, do), (dq, dk, dv)


def _run_full(samples, heads, head_dim, seed, budget=0, scale=0.0):
    plan, (q, k, v, do), (dq, dk, dv) = _gpu_fwd_bwd(samples, heads, head_dim, seed, budget, scale)
    ref = oracle.pack_plan(samples, budget)
    cu, pos = ref["cu_seqlens"], ref["pos"]
    qn, kn, vn, gn = to64(q), to64(k), to64(v), to64(do)
    O, L = oracle.attn_fwd(qn, kn, vn, cu, pos, softmax_scale=scale)
    rq, rk, rv = oracle.attn_bwd(qn, kn, vn, O, L, gn, cu, pos, softmax_scale=scale)
    f = lse_tol_factor(scale, head_dim)
    assert_close("dV", to64(dv), rv, "grad", f)
    assert_close("dK", to64(dk), rk, "grad", f)
    assert_close("dQ", to64(dq), rq, "grad", f)


@pytest.mark.parametrize("seed", range(3))
def test_bwd_tiny(seed):
    wl = synth.tiny(seed)
    _run_full(wl.samples, wl.heads, wl.head_dim, seed)


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("seed", range(2))
def test_bwd_ragged_multi_tile(head_dim, seed):
    samples = [(0, 16, 16), (7, 64, 32), (0, 128, 128), (200, 160, 48), (1, 16, 16), (55, 96, 208)]
    rng = np.random.default_rng(seed)
    rng.shuffle(samples)
    _run_full(samples, heads=3, head_dim=head_dim, seed=seed)


@pytest.mark.parametrize("L", [1, 127, 128, 129, 256, 300])
def test_bwd_tile_boundaries(L):
    _run_full([(0, 16, 16 * L)], heads=2, head_dim=128, seed=L)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_bwd_text_only_and_image_only_samples(head_dim):
    _run_full([(40, 0, 0), (0, 48, 48), (1, 0, 0), (129, 0, 0), (3, 32, 32), (0, 16, 16 * 127)],
              heads=2, head_dim=head_dim, seed=head_dim)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_bwd_runs_of_short_ragged_samples(head_dim):
    # 200 samples of at most 124 tokens, 8 heads: every work item is one
    # K/V tile whose only Q tile is ragged, about 11 in a row per CTA, so
    # the two sets of ragged-tail barriers take turns many times
    samples = synth.random_pack(950 + head_dim, 200, 60, 8)
    assert max(t + (h // 16) * (w // 16) for t, h, w in samples) < 128
    _run_full(samples, heads=8, head_dim=head_dim, seed=head_dim)


def test_bwd_single_token_closed_form():
    """One key: P = 1, dS = 0, so dQ = dK = 0 and dV = dO."""
    plan, (q, k, v, do), (dq, dk, dv) = _gpu_fwd_bwd([(0, 16, 16), (1, 16, 16)], 2, 128, 3)
    assert float(dq[0].abs().max()) < 1e-4 and float(dk[0].abs().max()) < 1e-4
    assert torch.equal(dv[0], do[0])


def test_bwd_budget_prefix():
    _run_full([(30, 96, 96), (12, 64, 48), (0, 48, 160)], heads=2, head_dim=64, seed=6, budget=80)


@pytest.mark.parametrize("scale", [0.05, 0.3])
def test_bwd_explicit_softmax_scale(scale):
    """A scale other than 1/sqrt(d), carried by one fp16 logit operand and
    multiplied back out of dK and dQ."""
    _run_full([(9, 64, 96), (0, 160, 32), (33, 0, 0)], heads=2, head_dim=128, seed=11, scale=scale)


def test_bwd_empty_pack():
    plan = mf.pack_plan([], 0)
    z = torch.empty((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 0), dtype=torch.float32, device="cuda")
    plan_d = mf.pack_plan([], 0, head_dim=64)
    dq, dk, dv = mf.attn_bwd(z, z, z, z, lse, z, plan_d)
    mf.check(plan_d)
    assert dq.shape == (0, 2, 64)


@pytest.mark.parametrize("name,samples_idx", [("native_res_32k", [2, 5]), ("extreme_aspect", [0])])
def test_bwd_full_size_per_sample(name, samples_idx):
    """Full-size pack in the bench's launch configuration; the oracle
    recomputes selected samples on a few heads (samples are independent, so a
    sample's gradients depend only on its own rows)."""
    wl = synth.WORKLOADS[name]()
    plan, (q, k, v, do), (dq, dk, dv) = _gpu_fwd_bwd(wl.samples, wl.heads, wl.head_dim, wl.seed,
                                                     wl.token_budget)
    ref = oracle.pack_plan(wl.samples, wl.token_budget)
    cu = ref["cu_seqlens"]
    dq_c, dk_c, dv_c = to64(dq), to64(dk), to64(dv)
    assert np.all(np.isfinite(dq_c)) and np.all(np.isfinite(dk_c)) and np.all(np.isfinite(dv_c))
    for si in samples_idx:
        a, b = int(cu[si]), int(cu[si + 1])
        sub = oracle.pack_plan([wl.samples[si]])
        for h in (0, wl.heads - 1):
            hs = slice(h, h + 1)
            qn, kn, vn, gn = (to64(x[a:b, hs]) for x in (q, k, v, do))
            O, L = oracle.attn_fwd(qn, kn, vn, sub["cu_seqlens"], sub["pos"])
            rq, rk, rv = oracle.attn_bwd(qn, kn, vn, O, L, gn, sub["cu_seqlens"], sub["pos"])
            assert_close(f"dV[{name},s{si},h{h}]", dv_c[a:b, hs], rv, "grad")
            assert_close(f"dK[{name},s{si},h{h}]", dk_c[a:b, hs], rk, "grad")
            assert_close(f"dQ[{name},s{si},h{h}]", dq_c[a:b, hs], rq, "grad")


def _edge_rows(a, b, rng, n_random):
    """Rows of sample [a, b): its first and last rows, both sides of every
    fourth 128-row tile edge, the last tile's first row and a few random rows."""
    rows = {a, a + 1, b - 2, b - 1, b - 1 - (b - a - 1) % 128}
    for e in range(a + 128, b, 512):
        rows |= {e - 1, e}
    rows |= set(int(x) for x in rng.integers(a, b, size=n_random))
    return sorted(r for r in rows if a <= r < b)


@pytest.mark.parametrize("name,samples_idx", [("native_res_32k", [0, 3]), ("extreme_aspect", [2])])
def test_bwd_full_size_long_samples_rows(name, samples_idx):
    """The long samples that dominate the benched fwd+bwd packs (10,749 and
    10,577 tokens of the training pack, 16,640 of the extreme-aspect pack: up
    to 130 K/V tiles whose dQ partials meet in one accumulator row), in the
    bench's launch configuration, on every head: sampled query rows (dQ) and
    key rows (dK, dV) against the row-wise oracle, which takes each sample's
    full-row statistics."""
    wl = synth.WORKLOADS[name]()
    t = synth.draw_tensors(wl, with_grad=True)
    plan = mf.pack_plan(wl.samples, token_budget=wl.token_budget, head_dim=wl.head_dim)
    T = plan.total_tokens
    q, k, v, do = (t[n][:T].cuda() for n in ("q", "k", "v", "do"))
    wsf = torch.empty(mf.fwd_workspace_bytes(T, wl.heads, wl.head_dim), dtype=torch.uint8, device="cuda")
    o, lse = mf.attn_fwd(q, k, v, plan, workspace=wsf)
    got = {"bwd": mf.attn_bwd(q, k, v, o, lse, do, plan)}
    mf.check(plan)
    got = {e: [to64(x) for x in g] for e, g in got.items()}
    for g in got.values():
        assert all(np.all(np.isfinite(x)) for x in g)
    ref = oracle.pack_plan(wl.samples, wl.token_budget)
    cu, pos = ref["cu_seqlens"], ref["pos"]
    rng = np.random.default_rng(1)
    q_rows, kv_rows = [], []
    for si in samples_idx:
        a, b = int(cu[si]), int(cu[si + 1])
        q_rows += _edge_rows(a, b, rng, 6)
        kv_rows += _edge_rows(a, b, rng, 6)
    qn, kn, vn, gn = (t[n].float().numpy() for n in ("q", "k", "v", "do"))
    for h in range(wl.heads):
        rq, rk, rv = oracle.attn_bwd_rows(qn, kn, vn, gn, cu, pos, h, q_rows=q_rows, kv_rows=kv_rows)
        for e, (dq, dk, dv) in got.items():
            assert_close(f"dQ[{name},{e},h{h}]", dq[q_rows, h], rq, "grad")
            assert_close(f"dK[{name},{e},h{h}]", dk[kv_rows, h], rk, "grad")
            assert_close(f"dV[{name},{e},h{h}]", dv[kv_rows, h], rv, "grad")


@pytest.mark.parametrize("head_dim", [64, 128])
def test_bwd_non_finite_values_stay_in_their_sample(head_dim):
    """NaN and Inf in one sample's V and dO (and NaN in its Q and K) leave
    every other sample's dQ, dK, dV as without them.  Tiles that run past a
    sample's end read the next sample's rows: a zero P or dS times a
    non-finite q~, dO or k~ value would otherwise be NaN, and dQ rows past a
    sample's end are reduced into the next sample's rows."""
    samples = [(5, 256, 208), (3, 160, 160), (0, 16, 16 * 77), (9, 64, 16 * 30)]
    heads = 2
    wl = synth.Workload("t", samples, heads, head_dim, "fwd+bwd", seed=43)
    t = synth.draw_tensors(wl, with_grad=True)
    ref = oracle.pack_plan(samples)
    cu = ref["cu_seqlens"]
    a, b = int(cu[1]), int(cu[2])
    q, k, v, do = (t[n].clone() for n in ("q", "k", "v", "do"))
    v[a:b, 0] = float("nan")
    v[a:b, 1] = float("inf")
    do[a:b, 0] = float("-inf")
    do[a + 2:b, 1, 9:] = float("nan")
    q[a + 1:b, :, :5] = float("nan")
    k[a:b - 2, :, 3:9] = float("nan")
    plan = mf.pack_plan(samples, head_dim=head_dim)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = mf.attn_fwd(qd, kd, vd, plan)
    dq, dk, dv = mf.attn_bwd(qd, kd, vd, o, lse, dod, plan)
    mf.check(plan)
    qn, kn, vn, gn = (to64(t[n]) for n in ("q", "k", "v", "do"))
    O, L = oracle.attn_fwd(qn, kn, vn, cu, ref["pos"])
    rq, rk, rv = oracle.attn_bwd(qn, kn, vn, O, L, gn, cu, ref["pos"])
    keep = np.r_[0:a, b:int(cu[-1])]
    assert_close("dV outside the poisoned sample", to64(dv)[keep], rv[keep], "grad")
    assert_close("dK outside the poisoned sample", to64(dk)[keep], rk[keep], "grad")
    assert_close("dQ outside the poisoned sample", to64(dq)[keep], rq[keep], "grad")
