"""The binding on a stream other than torch's current one.

Plan, forward and backward are enqueued on a side stream,
with their scratch workspaces allocated by the binding, while the current
stream keeps allocating and overwriting memory.  The scratch buffers are tied
to the side stream, so that memory cannot be handed out again under the
running kernels: the results must equal those of the same calls on the
current stream (the forward bit for bit; the backward within the rounding
of its unordered dQ reductions).
"""
import pytest
import torch

import packed_resolution_diffusion_plan_b300 as mf
import synth

pytestmark = pytest.mark.gpu


def _run(samples, q, k, v, do, stream):
    plan = mf.pack_plan(samples, head_dim=q.shape[2], stream=stream)
    wsf = mf._workspace(mf.fwd_workspace_bytes(q.shape[0], q.shape[1], q.shape[2]), q.device, stream)
    o, lse = mf.attn_fwd(q, k, v, plan, workspace=wsf, stream=stream)
    g = mf.attn_bwd(q, k, v, o, lse, do, plan, stream=stream)
    return plan, o, lse, g


def test_side_stream_matches_current_stream():
    samples = [(40, 256, 192), (7, 128, 384), (0, 96, 96), (120, 0, 0)]
    wl = synth.Workload("s", samples, 4, 128, "fwd+bwd", seed=5)
    t = synth.draw_tensors(wl, with_grad=True)
    q, k, v, do = (t[n].cuda() for n in ("q", "k", "v", "do"))
    plan0, o0, lse0, g0 = _run(samples, q, k, v, do, None)
    mf.check(plan0)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    plan1, o1, lse1, g1 = _run(samples, q, k, v, do, side)
    # meanwhile the current stream recycles and scribbles over free memory
    for _ in range(8):
        junk = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
        junk.fill_(0xff)
        del junk
    side.synchronize()
    mf.check(plan1, stream=side)
    torch.cuda.synchronize()

    assert torch.equal(o0, o1) and torch.equal(lse0, lse1)
    for a, b in zip(g0, g1):
        a, b = a.double(), b.double()
        assert torch.isfinite(b).all()
        assert float((a - b).norm() / a.norm()) < 1e-3
