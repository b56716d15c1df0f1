"""mf_pack_plan on the GPU vs the oracle: bit-exact plans on every workload,
random ragged packs, budgets and edge cases."""
import math

import numpy as np
import pytest
import torch

import oracle
import packed_resolution_diffusion_plan_b300 as mf
import synth

pytestmark = pytest.mark.gpu


def _check_plan(samples, budget, head_dim=128, theta=10000.0, rope_axes=2):
    ref = oracle.pack_plan(samples, budget)
    p = mf.pack_plan(samples, token_budget=budget, head_dim=head_dim, rope_theta=theta, rope_axes=rope_axes)
    assert p.rope_axes == rope_axes
    mf.check(p)   # also fails if the device scan's scalars differ from the host's
    # the scan's own scalars (the workspace's first 32 bytes) are the plan's
    got = p.workspace[:32].view(torch.int32).cpu().tolist()
    assert got[:5] + got[6:7] == [p.n_samples, p.total_tokens, p.max_seqlen, p.max_grid, p.n_tiles, p.n_pairs]
    assert p.n_samples == ref["n_samples"]
    assert p.total_tokens == ref["total_tokens"]
    assert p.max_seqlen == ref["max_seqlen"]
    assert p.max_grid == ref["max_grid"]
    assert np.array_equal(p.cu_seqlens().cpu().numpy(), ref["cu_seqlens"])
    assert np.array_equal(p.pos().cpu().numpy(), ref["pos"])
    assert np.array_equal(p.frame().cpu().numpy(), ref["frame"])
    lens = np.diff(ref["cu_seqlens"])
    # work order: longest first, ties by sample index, tile starts = prefix of ceil(L/128)
    order = p.order().cpu().numpy()
    want = sorted(range(len(lens)), key=lambda i: (-lens[i], i))
    assert list(order[:, 0]) == want
    tiles = [math.ceil(lens[i] / 128) for i in want]
    pairs = [math.ceil(lens[i] / 256) for i in want]
    if want:
        assert list(order[:, 1]) == list(np.concatenate([[0], np.cumsum(tiles)[:-1]]).astype(int))
        assert list(order[:, 2]) == list(np.concatenate([[0], np.cumsum(pairs)[:-1]]).astype(int))
        assert list(order[:, 3]) == [0] * len(want)
    assert p.n_tiles == sum(tiles) and p.n_pairs == sum(pairs)
    # RoPE tables: cos/sin of p * theta^(-2i/a) rounded once to float32, a =
    # the row/col slice width (head_dim/2, or 7 head_dim/16 with 3 axes), and
    # with 3 axes the frame slice's (a = head_dim/8) for frames 0 and 1
    if p.max_grid:
        tab = p.rope_table().cpu().numpy().astype(np.float64)
        a = head_dim // 2 if rope_axes == 2 else 7 * head_dim // 16
        f = theta ** (-2.0 * np.arange(a // 2) / a)
        ang = np.arange(p.max_grid)[:, None] * f[None, :]
        assert np.abs(tab[..., 0] - np.cos(ang)).max() < 1e-7
        assert np.abs(tab[..., 1] - np.sin(ang)).max() < 1e-7
        if rope_axes == 3:
            tf = p.rope_table_frame().cpu().numpy().astype(np.float64)
            af = head_dim // 8
            ff = theta ** (-2.0 * np.arange(af // 2) / af)
            angf = np.arange(2)[:, None] * ff[None, :]
            assert np.abs(tf[..., 0] - np.cos(angf)).max() < 1e-7
            assert np.abs(tf[..., 1] - np.sin(angf)).max() < 1e-7
    return p


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_plan_workloads_bit_exact(name):
    wl = synth.WORKLOADS[name]()
    _check_plan(wl.samples, wl.token_budget, wl.head_dim, rope_axes=wl.rope_axes)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("head_dim", [64, 128])
def test_plan_edit_packs(seed, head_dim):
    """Random edit packs (frames 1 or 2 per sample) with the (frame, row, col)
    rotation, and a generation-only pack planned with 3 axes."""
    _check_plan(synth.random_pack(100 + seed, 9, 40, 12, edit=True), 0, head_dim, rope_axes=3)
    _check_plan(synth.random_pack(200 + seed, 5, 40, 12), 0, head_dim, rope_axes=3)


def test_plan_text_only_samples():
    _check_plan([(40, 0, 0), (3, 32, 32), (1, 0, 0), (0, 16, 16)], 0)
    _check_plan([(5, 0, 0), (2, 32, 16, 2)], 0, rope_axes=3)


def test_plan_edit_needs_three_axes():
    with pytest.raises(mf.MfError) as ei:
        mf.pack_plan([(4, 32, 32, 2)], rope_axes=2)
    assert ei.value.code == "MF_ERR_INVALID_ARG"


@pytest.mark.parametrize("seed", range(8))
def test_plan_native_res_seeds(seed):
    wl = synth.native_res(seed)
    _check_plan(wl.samples, wl.token_budget)


@pytest.mark.parametrize("seed", range(5))
def test_plan_random_ragged(seed):
    samples = synth.random_pack(100 + seed, n_samples=3 + 7 * seed, max_text=300, max_side_tokens=40)
    _check_plan(samples, 0, head_dim=64)
    ref = oracle.pack_plan(samples)
    first = int(ref["cu_seqlens"][1])
    _check_plan(samples, max(first, ref["total_tokens"] // 2 + 1), head_dim=128)


def test_plan_edge_cases():
    _check_plan([(0, 16, 16)], 0)                  # one token
    _check_plan([(0, 16, 16)] * 7, 0)              # many one-token samples, all tied
    _check_plan([(128, 16, 16), (0, 2048, 16)], 0)  # thin grids
    _check_plan([(5, 16 * 1024, 16 * 2)], 0)       # maximum grid side
    e = mf.pack_plan([], 0)
    assert e.total_tokens == 0 and e.n_samples == 0 and e.n_tiles == 0
    assert list(e.cu_seqlens().cpu().numpy()) == [0]
    big = [(1, 16, 16)] * 4096                     # maximum sample count
    _check_plan(big, 0)
    with pytest.raises(mf.MfError) as ei:
        mf.pack_plan([(100, 64, 64)], token_budget=50)
    assert ei.value.code == "MF_ERR_BUDGET"
