"""A pack whose tensors pass 2^31 elements (~788K tokens at 24 heads x 128),
so that every offset into Q/K/V/O, the gradients, the rotated copies, the dQ
accumulator and LSE must be 64-bit.

The inputs come from a seeded CUDA generator (drawing 19 GB on the host
would take minutes); the oracle gets the slices it checks.  The last sample
lies wholly past element 2^31: its forward and both backward entries are
compared in full on two heads, and sampled rows of the big sample before it
(also past 2^31) check the forward over 52K keys.
"""
import numpy as np
import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
from _parity import assert_close, to64

pytestmark = pytest.mark.gpu

H, D = 24, 128
BIG = (100, 3664, 3664)     # 100 + 229 * 229 = 52,541 tokens
SMALL = (20, 256, 256)      # 276 tokens


def _draw(T, g):
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    for a in range(0, T, 65536):
        b = min(T, a + 65536)
        out[a:b] = torch.randn((b - a, H, D), generator=g, device="cuda").to(torch.bfloat16)
    return out


def test_pack_past_2_31_elements():
    samples = [BIG] * 15 + [SMALL]
    plan = mf.pack_plan(samples, head_dim=D)
    T = plan.total_tokens
    ref = oracle.pack_plan(samples)
    cu = ref["cu_seqlens"]
    assert T == int(cu[-1]) and T * H * D > 2 ** 31

    g = torch.Generator("cuda").manual_seed(31)
    q, k, v, do = (_draw(T, g) for _ in range(4))
    wsf = torch.empty(mf.fwd_workspace_bytes(T, H, D), dtype=torch.uint8, device="cuda")
    o, lse = mf.attn_fwd(q, k, v, plan, workspace=wsf)
    grads = {"bwd": mf.attn_bwd(q, k, v, o, lse, do, plan)}
    mf.check(plan)
    for t in (o, lse, *grads["bwd"]):
        assert torch.isfinite(t).all()

    # the last sample, wholly past element 2^31: everything on two heads
    a, b = int(cu[-2]), int(cu[-1])
    assert a * H * D > 2 ** 31
    sub = oracle.pack_plan([SMALL])
    for h in (0, H - 1):
        hs = slice(h, h + 1)
        qn, kn, vn, gn = (to64(x[a:b, hs]) for x in (q, k, v, do))
        O, L = oracle.attn_fwd(qn, kn, vn, sub["cu_seqlens"], sub["pos"])
        assert_close(f"O h{h}", to64(o[a:b, hs]), O, "o")
        assert_close(f"LSE h{h}", to64(lse[hs, a:b]), L, "lse")
        rq, rk, rv = oracle.attn_bwd(qn, kn, vn, O, L, gn, sub["cu_seqlens"], sub["pos"])
        for name, (dq, dk, dv) in grads.items():
            assert_close(f"dQ {name} h{h}", to64(dq[a:b, hs]), rq, "grad")
            assert_close(f"dK {name} h{h}", to64(dk[a:b, hs]), rk, "grad")
            assert_close(f"dV {name} h{h}", to64(dv[a:b, hs]), rv, "grad")

    # sampled rows of the big sample before it (text edge, first and last
    # image rows, a middle row), each attending over its 52,541 keys
    a2, b2 = int(cu[-3]), int(cu[-2])
    assert a2 * H * D > 2 ** 31
    big = oracle.pack_plan([BIG])
    rows = [0, 99, 100, 101, 26000, b2 - a2 - 1]
    for h in (0, H - 1):
        hs = slice(h, h + 1)
        qn, kn, vn = (to64(x[a2:b2, hs]) for x in (q, k, v))
        O, L = oracle.attn_rows(qn, kn, vn, big["cu_seqlens"], big["pos"], rows, 0)
        assert_close(f"O rows h{h}", to64(o[a2:b2][rows, h]), O, "o")
        assert_close(f"LSE rows h{h}", to64(lse[h, a2:b2][rows]), L, "lse")
    assert np.isfinite(to64(lse[:, a2:b2])).all()
