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


def _check_plan(samples, budget, head_dim=128, theta=10000.0):
    ref = oracle.pack_plan(samples, budget)
    p = mf.pack_plan(samples, token_budget=budget, head_dim=head_dim, rope_theta=theta)
    mf.check(p)
    assert p.n_samples == ref["n_samples"]
    assert p.total_tokens == ref["total_tokens"]
    assert p.max_seqlen == ref["max_seqlen"]
    assert p.max_grid == ref["max_grid"]
    assert np.array_equal(p.cu_seqlens().cpu().numpy(), ref["cu_seqlens"])
    assert np.array_equal(p.pos().cpu().numpy(), ref["pos"])
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
    # RoPE table: cos/sin of p * theta^(-2i/(D/2)) rounded once to float32
    if p.max_grid:
        tab = p.rope_table().cpu().numpy().astype(np.float64)
        half = head_dim // 2
        f = theta ** (-2.0 * np.arange(head_dim // 4) / half)
        ang = np.arange(p.max_grid)[:, None] * f[None, :]
        assert np.abs(tab[..., 0] - np.cos(ang)).max() < 1e-7
        assert np.abs(tab[..., 1] - np.sin(ang)).max() < 1e-7
    return p


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_plan_workloads_bit_exact(name):
    wl = synth.WORKLOADS[name]()
    _check_plan(wl.samples, wl.token_budget, wl.head_dim)


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
