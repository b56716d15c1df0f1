"""The memory-bound chains around a joint-attention block on the GPU vs the
float64 oracle: LayerNorm + adaptive modulation, the attention forward fed
by a QKV projection's rows (RoPE fused into its first pass), and gate +
residual; then the whole block with the two projections as plain cuBLAS
products (synthetic weights)."""
import numpy as np
import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
import synth
from _parity import assert_close, rel_l2, to64

pytestmark = pytest.mark.gpu


def _bf16(g, *shape, scale=1.0, shift=0.0):
    return (torch.randn(shape, generator=g) * scale + shift).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("hidden", [1024, 3072, 4096])
def test_norm_modulate(hidden):
    samples = [(7, 64, 48), (0, 16, 16), (130, 96, 80)]
    plan = mf.pack_plan(samples, head_dim=128)
    g = torch.Generator("cpu").manual_seed(hidden)
    T = plan.total_tokens
    x = _bf16(g, T, hidden, scale=2.0, shift=0.5)
    shift = _bf16(g, len(samples), hidden, scale=0.3)
    scale = _bf16(g, len(samples), hidden, scale=0.3)
    y = mf.norm_modulate(x, plan, shift, scale)
    mf.check(plan)
    ref = oracle.norm_modulate(to64(x), plan.cu_seqlens().cpu().numpy(), to64(shift), to64(scale))
    got = to64(y)
    # fp32 statistics, one bf16 rounding of an O(1) result
    assert np.abs(got - ref).max() <= 2.0 ** -8 * np.abs(ref).max() + 1e-3
    assert rel_l2(got, ref) < 3e-3


def test_gate_residual_in_place():
    samples = [(3, 32, 32), (5, 48, 16)]
    plan = mf.pack_plan(samples, head_dim=128)
    g = torch.Generator("cpu").manual_seed(1)
    T, C = plan.total_tokens, 2048
    x, z = _bf16(g, T, C), _bf16(g, T, C, scale=4.0)
    gate = _bf16(g, 2, C, scale=0.5)
    ref = oracle.gate_residual(to64(x), to64(z), plan.cu_seqlens().cpu().numpy(), to64(gate))
    out = mf.gate_residual(x, z, plan, gate, out=x)
    mf.check(plan)
    got = to64(out)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)


@pytest.mark.parametrize("head_dim,heads", [(128, 8), (64, 16)])
def test_attn_fwd_qkv_equals_split_tensors(head_dim, heads):
    """Same kernels on the same values: the QKV-row entry must match the
    plain entry on contiguous copies bit for bit, and the oracle."""
    samples = synth.random_pack(500 + head_dim, 5, 90, 14)
    plan = mf.pack_plan(samples, head_dim=head_dim)
    g = torch.Generator("cpu").manual_seed(head_dim)
    T, C = plan.total_tokens, heads * head_dim
    qkv = _bf16(g, T, 3 * C)
    q, k, v = (qkv[:, i * C:(i + 1) * C].contiguous().view(T, heads, head_dim) for i in range(3))
    o1, l1 = mf.attn_fwd_qkv(qkv, plan, heads)
    o2, l2 = mf.attn_fwd(q, k, v, plan)
    mf.check(plan)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref = oracle.pack_plan(samples)
    O, L = oracle.attn_fwd(to64(q), to64(k), to64(v), ref["cu_seqlens"], ref["pos"])
    assert_close("O", to64(o1), O, "o")
    assert_close("LSE", to64(l1), L, "lse")


@pytest.mark.parametrize("rope_axes", [2, 3])
def test_bwd_after_qkv_forward(rope_axes):
    """The backward of the QKV-row forward (its O and LSE, the projection's
    thirds as Q, K, V), against the oracle's gradients."""
    heads, head_dim = 4, 128
    samples = synth.random_pack(700 + rope_axes, 4, 70, 12, edit=rope_axes == 3)
    plan = mf.pack_plan(samples, head_dim=head_dim, rope_axes=rope_axes)
    g = torch.Generator("cpu").manual_seed(rope_axes)
    T, C = plan.total_tokens, heads * head_dim
    qkv = _bf16(g, T, 3 * C)
    do = _bf16(g, T, heads, head_dim)
    wsf = torch.empty(max(256, mf.fwd_workspace_bytes(T, heads, head_dim)), dtype=torch.uint8, device="cuda")
    o, lse = mf.attn_fwd_qkv(qkv, plan, heads, workspace=wsf)
    q, k, v = (qkv[:, i * C:(i + 1) * C].contiguous().view(T, heads, head_dim) for i in range(3))
    dq, dk, dv = mf.attn_bwd(q, k, v, o, lse, do, plan)
    mf.check(plan)
    ref = oracle.pack_plan(samples)
    rope = dict(frame=ref["frame"], rope_axes=rope_axes)
    qn, kn, vn = to64(q), to64(k), to64(v)
    O, L = oracle.attn_fwd(qn, kn, vn, ref["cu_seqlens"], ref["pos"], **rope)
    rq, rk, rv = oracle.attn_bwd(qn, kn, vn, O, L, to64(do), ref["cu_seqlens"], ref["pos"], **rope)
    assert_close("dV", to64(dv), rv, "grad")
    assert_close("dK", to64(dk), rk, "grad")
    assert_close("dQ", to64(dq), rq, "grad")


@pytest.mark.parametrize("rope_axes", [2, 3])
def test_attention_block_end_to_end(rope_axes):
    """x -> norm_modulate -> @W_qkv -> attn_fwd_qkv -> @W_o -> gate_residual
    against the oracle's float64 block (bf16 intermediates on the GPU: the
    gated update out - x is compared)."""
    heads, D = 8, 128
    C = heads * D
    samples = [(20, 128, 96), (5, 64, 64, 2 if rope_axes == 3 else 1), (0, 48, 80)]
    plan = mf.pack_plan(samples, head_dim=D, rope_axes=rope_axes)
    g = torch.Generator("cpu").manual_seed(rope_axes)
    T = plan.total_tokens
    # small x and large gates keep the gated update well above out's bf16 rounding
    x = _bf16(g, T, C, scale=0.1)
    w_qkv = _bf16(g, C, 3 * C, scale=C ** -0.5)
    w_o = _bf16(g, C, C, scale=C ** -0.5)
    shift, scale = (_bf16(g, len(samples), C, scale=0.2) for _ in range(2))
    gate = _bf16(g, len(samples), C, scale=2.0)
    y = mf.norm_modulate(x, plan, shift, scale)
    qkv = y @ w_qkv
    o, _ = mf.attn_fwd_qkv(qkv, plan, heads)
    z = o.view(T, C) @ w_o
    out = mf.gate_residual(x, z, plan, gate)
    mf.check(plan)
    ref_p = oracle.pack_plan(samples)
    ref = oracle.attn_block_fwd(to64(x), ref_p["cu_seqlens"], ref_p["pos"], heads, to64(w_qkv), to64(w_o),
                                to64(shift), to64(scale), to64(gate), frame=ref_p["frame"], rope_axes=rope_axes)
    dx = to64(out) - to64(x)
    dref = ref - to64(x)
    assert rel_l2(dx, dref) < 3e-2
    assert np.abs(dx - dref).max() < 5e-2
