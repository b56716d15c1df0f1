"""Pins for the float64 oracle: values derived by hand from the pages'
definitions, closed forms, invariants, library special cases and finite
differences.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_qkv(T, H, D, seed):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((T, H, D)) for _ in range(4)]


# --------------------------------------------------------------------------
# pack plan
# --------------------------------------------------------------------------

def _read_golden_plan():
    out = {"pos": []}
    with open(os.path.join(GOLDEN, "pack_plan_tiny.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "samples":
                out[key] = [tuple(int(x) for x in v.split(",")) for v in vals]
            elif key == "pos":
                out["pos"].append(tuple(int(x) for x in vals))
            elif key == "cu_seqlens":
                out[key] = [int(x) for x in vals]
            else:
                out[key] = int(vals[0])
    return out


def test_pack_plan_golden_tiny():
    g = _read_golden_plan()
    p = oracle.pack_plan(g["samples"], g["budget"])
    assert p["n_samples"] == g["n_samples"]
    assert list(p["cu_seqlens"]) == g["cu_seqlens"]
    assert p["total_tokens"] == g["total_tokens"]
    assert p["max_seqlen"] == g["max_seqlen"]
    assert p["max_grid"] == g["max_grid"]
    for tok, r, c in g["pos"]:
        assert tuple(p["pos"][tok]) == (r, c), tok


def test_workload_token_totals_golden():
    with open(os.path.join(GOLDEN, "workload_tokens.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for name, total, _ in rows:
        wl = synth.WORKLOADS[name]()
        assert oracle.pack_plan(wl.samples, wl.token_budget)["total_tokens"] == int(total)


def test_native_res_seed0_lengths():
    # Draw-and-skip recipe, seed 0: six samples filling 32,688 of 32,768.
    wl = synth.native_res(0)
    p = oracle.pack_plan(wl.samples, wl.token_budget)
    assert list(np.diff(p["cu_seqlens"])) == [10749, 3579, 1358, 10577, 3906, 2519]
    assert p["total_tokens"] == 32688


def _brute_positions(samples):
    """Independent construction of the per-token ids with numpy index grids."""
    rows = []
    for (t, h, w) in samples:
        gh, gw = h // 16, w // 16
        rr, cc = np.meshgrid(np.arange(gh), np.arange(gw), indexing="ij")
        rows.append(np.full((t, 2), -1))
        rows.append(np.stack([rr.ravel(), cc.ravel()], axis=1))
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, 2))


@pytest.mark.parametrize("seed", range(6))
def test_pack_plan_brute_force_and_invariants(seed):
    samples = synth.random_pack(seed, n_samples=1 + seed, max_text=20, max_side_tokens=9)
    p = oracle.pack_plan(samples, 0)
    assert np.array_equal(p["pos"], _brute_positions(samples))
    lens = [t + (h // 16) * (w // 16) for (t, h, w) in samples]
    assert p["cu_seqlens"][-1] == sum(lens) == p["total_tokens"]
    for i, (t, h, w) in enumerate(samples):
        a, b = p["cu_seqlens"][i], p["cu_seqlens"][i + 1]
        seg = p["pos"][a:b]
        img = seg[seg[:, 0] >= 0]
        assert len(img) == (h // 16) * (w // 16)
        assert img[:, 0].max() == h // 16 - 1 and img[:, 1].max() == w // 16 - 1
        assert np.all(seg[:t] == -1)


def test_pack_plan_budget_prefix():
    samples = [(10, 64, 64), (5, 32, 32), (7, 48, 16)]   # L = 26, 9, 10
    assert oracle.pack_plan(samples, 35)["n_samples"] == 2
    assert oracle.pack_plan(samples, 34)["n_samples"] == 1
    assert oracle.pack_plan(samples, 45)["n_samples"] == 3
    assert oracle.pack_plan(samples, 0)["n_samples"] == 3
    with pytest.raises(ValueError):
        oracle.pack_plan(samples, 25)
    for bad in [(-1, 16, 16), (0, 0, 16), (0, 16, 24), (3, 17, 16), (0, 0, 0)]:
        with pytest.raises(ValueError):
            oracle.pack_plan([bad], 0)
    # a text-only sample (no image): all of its rows are text, none rotated
    p = oracle.pack_plan([(4, 0, 0), (1, 16, 16)])
    assert list(p["cu_seqlens"]) == [0, 4, 6] and p["max_grid"] == 1
    assert [tuple(r) for r in p["pos"]] == [(-1, -1)] * 5 + [(0, 0)]
    empty = oracle.pack_plan([], 0)
    assert empty["total_tokens"] == 0 and list(empty["cu_seqlens"]) == [0]


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_golden_angles():
    rows = np.loadtxt(os.path.join(GOLDEN, "rope_angles_d8.txt"))
    for r, c, *ang in rows:
        pos = np.array([[int(r), int(c)]], dtype=np.int32)
        for m in range(4):
            x = np.zeros((1, 1, 8))
            x[0, 0, 2 * m] = 1.0              # unit vector of pair m
            y = oracle.rope(x, pos)[0, 0]
            got = math.atan2(y[2 * m + 1], y[2 * m])
            want = math.remainder(ang[m], 2 * math.pi)
            assert abs(got - want) < 1e-12, (r, c, m)
            others = np.delete(y, [2 * m, 2 * m + 1])
            assert np.all(others == 0)


def test_rope_norm_inverse_and_text():
    rng = np.random.default_rng(1)
    pos = np.array([[-1, -1], [0, 0], [5, 9], [127, 3], [40, 127]], dtype=np.int32)
    x = rng.standard_normal((5, 3, 128))
    y = oracle.rope(x, pos)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    assert np.allclose(oracle.rope(y, pos, inverse=True), x, atol=1e-12)
    assert np.array_equal(y[0], x[0]) and np.array_equal(y[1], x[1])


def test_rope_relative_position():
    rng = np.random.default_rng(2)
    D = 64
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    p, pp = np.array([[3, 11]]), np.array([[7, 2]])
    base = (oracle.rope(q, p) * oracle.rope(k, pp)).sum()
    for dr, dc in [(1, 0), (0, 5), (13, 21)]:
        d = np.array([[dr, dc]])
        moved = (oracle.rope(q, p + d) * oracle.rope(k, pp + d)).sum()
        assert abs(moved - base) < 1e-10


def test_rope_single_axis_is_1d_rope():
    """Column 0 everywhere: the second half is untouched and the first half is
    the textbook 1D RoPE of its 32 pairs, written here in complex form."""
    rng = np.random.default_rng(3)
    D, theta = 128, 10000.0
    x = rng.standard_normal((6, 2, D))
    pos = np.stack([np.arange(6) * 7, np.zeros(6, dtype=np.int64)], axis=1)
    y = oracle.rope(x, pos)
    assert np.array_equal(y[..., D // 2:], x[..., D // 2:])
    half = D // 2
    f = theta ** (-np.arange(half // 2) * 2.0 / half)
    z = x[..., 0:half:2] + 1j * x[..., 1:half:2]
    zr = z * np.exp(1j * pos[:, 0:1, None] * f[None, None, :])
    assert np.allclose(y[..., 0:half:2], zr.real, atol=1e-12)
    assert np.allclose(y[..., 1:half:2], zr.imag, atol=1e-12)


# --------------------------------------------------------------------------
# (h, w, f) RoPE of edit packs
# --------------------------------------------------------------------------

def test_pack_plan_edit_frames():
    """An edit sample (text, H, W, 2) carries its source and target latents as
    frames 0 and 1 after its text, each in row-major order (hand-derived)."""
    p = oracle.pack_plan([(5, 32, 48, 2), (2, 16, 16)])   # grids 2x3 (two frames), 1x1
    assert list(p["cu_seqlens"]) == [0, 17, 20]
    assert p["total_tokens"] == 20 and p["max_seqlen"] == 17 and p["max_grid"] == 3
    want_pos = [(-1, -1)] * 5 + [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 2)] * 2 + [(-1, -1)] * 2 + [(0, 0)]
    assert [tuple(r) for r in p["pos"]] == want_pos
    assert list(p["frame"]) == [-1] * 5 + [0] * 6 + [1] * 6 + [-1, -1, 0]
    with pytest.raises(ValueError):
        oracle.pack_plan([(1, 16, 16, 3)])


def test_rope3d_golden_angles():
    rows = np.loadtxt(os.path.join(GOLDEN, "rope3d_angles_d32.txt"))
    for r, c, f, *ang in rows:
        pos = np.array([[int(r), int(c)]], dtype=np.int32)
        frame = np.array([int(f)], dtype=np.int32)
        for m, a in zip((0, 1, 2, 3, 9, 10), ang):
            x = np.zeros((1, 1, 32))
            x[0, 0, 2 * m] = 1.0
            y = oracle.rope(x, pos, frame=frame, rope_axes=3)[0, 0]
            got = math.atan2(y[2 * m + 1], y[2 * m])
            assert abs(got - math.remainder(a, 2 * math.pi)) < 1e-12, (r, c, f, m)
            assert np.all(np.delete(y, [2 * m, 2 * m + 1]) == 0)


def test_rope3d_axes_dims():
    assert oracle.rope_axes_dims(128, 3) == [("frame", 16), ("row", 56), ("col", 56)]
    assert oracle.rope_axes_dims(64, 3) == [("frame", 8), ("row", 28), ("col", 28)]
    assert oracle.rope_axes_dims(128, 2) == [("row", 64), ("col", 64)]


def test_rope3d_norm_inverse_and_text():
    rng = np.random.default_rng(4)
    pos = np.array([[-1, -1], [0, 0], [5, 9], [127, 3], [40, 127]], dtype=np.int32)
    frame = np.array([-1, 1, 0, 1, 1], dtype=np.int32)
    x = rng.standard_normal((5, 3, 128))
    y = oracle.rope(x, pos, frame=frame, rope_axes=3)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
    assert np.allclose(oracle.rope(y, pos, inverse=True, frame=frame, rope_axes=3), x, atol=1e-12)
    assert np.array_equal(y[0], x[0])


def test_rope3d_relative_position_including_frame():
    rng = np.random.default_rng(5)
    D = 128
    q = rng.standard_normal((1, 1, D))
    k = rng.standard_normal((1, 1, D))
    p, pp = np.array([[3, 11]]), np.array([[7, 2]])
    f, ff = np.array([1]), np.array([0])
    base = (oracle.rope(q, p, frame=f, rope_axes=3) * oracle.rope(k, pp, frame=ff, rope_axes=3)).sum()
    for dr, dc, df in [(1, 0, 0), (0, 5, 0), (0, 0, 1), (13, 21, 3)]:
        d = np.array([[dr, dc]])
        moved = (oracle.rope(q, p + d, frame=f + df, rope_axes=3) *
                 oracle.rope(k, pp + d, frame=ff + df, rope_axes=3)).sum()
        assert abs(moved - base) < 1e-10
    # the frame does tell source from target: same (row, col), other frame
    other = (oracle.rope(q, p, frame=f, rope_axes=3) * oracle.rope(k, p, frame=ff, rope_axes=3)).sum()
    same = (oracle.rope(q, p, frame=ff, rope_axes=3) * oracle.rope(k, p, frame=ff, rope_axes=3)).sum()
    assert abs(other - same) > 1e-6


def test_rope3d_frame_slice_is_1d_rope():
    """Row = col = 0 everywhere: the row and column slices are untouched and
    the frame slice (head_dim/8 dims) is the textbook 1D RoPE of its pairs,
    written here in complex form."""
    rng = np.random.default_rng(6)
    D, theta = 128, 10000.0
    a = D // 8
    x = rng.standard_normal((4, 2, D))
    pos = np.zeros((4, 2), dtype=np.int32)
    frame = np.array([0, 1, 2, 5], dtype=np.int32)
    y = oracle.rope(x, pos, frame=frame, rope_axes=3)
    assert np.array_equal(y[..., a:], x[..., a:])
    f = theta ** (-np.arange(a // 2) * 2.0 / a)
    z = x[..., 0:a:2] + 1j * x[..., 1:a:2]
    zr = z * np.exp(1j * frame[:, None, None] * f[None, None, :])
    assert np.allclose(y[..., 0:a:2], zr.real, atol=1e-12)
    assert np.allclose(y[..., 1:a:2], zr.imag, atol=1e-12)


def test_bwd3d_central_finite_differences():
    """The exact gradient with the (h, w, f) rotation: directional central
    differences on a small edit pack (two frames) plus a one-frame sample."""
    samples = [(3, 32, 32, 2), (2, 16, 48)]
    p = oracle.pack_plan(samples)
    rng = np.random.default_rng(7)
    T = p["total_tokens"]
    q, k, v, g = (rng.standard_normal((T, 2, 64)) for _ in range(4))
    kw = dict(frame=p["frame"], rope_axes=3)
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"], **kw)
    dq, dk, dv = oracle.attn_bwd(q, k, v, O, L, g, p["cu_seqlens"], p["pos"], **kw)

    def loss(q_, k_, v_):
        return float((oracle.attn_fwd(q_, k_, v_, p["cu_seqlens"], p["pos"], **kw)[0] * g).sum())

    eps = 1e-6
    for x, dx in ((q, dq), (k, dk), (v, dv)):
        u = rng.standard_normal(x.shape)
        ap = [x + eps * u if y is x else y for y in (q, k, v)]
        am = [x - eps * u if y is x else y for y in (q, k, v)]
        fd = (loss(*ap) - loss(*am)) / (2 * eps)
        an = float((dx * u).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)


# --------------------------------------------------------------------------
# classifier-free guidance over (cond, uncond) pairs
# --------------------------------------------------------------------------

def test_cfg_combine_closed_forms():
    """guidance 1 keeps the conditional rows, 0 gives the unconditional ones,
    2 gives the extrapolation 2c - u; text rows and the unconditional sample
    are untouched; rows pair up from the end of each sample (text lengths
    differ, image rows match)."""
    samples = [(5, 32, 48), (2, 32, 48), (3, 16, 16), (0, 16, 16)]
    p = oracle.pack_plan(samples)
    rng = np.random.default_rng(8)
    o = rng.standard_normal((p["total_tokens"], 2, 8))
    cu = p["cu_seqlens"]
    c_img = slice(int(cu[0]) + 5, int(cu[1]))
    u_img = slice(int(cu[1]) + 2, int(cu[2]))
    for g, want in ((1.0, o[c_img]), (0.0, o[u_img]), (2.0, 2 * o[c_img] - o[u_img])):
        out = oracle.cfg_combine(o, cu, p["pos"], g)
        assert np.allclose(out[c_img], want, atol=1e-15)
        assert np.array_equal(out[int(cu[0]):int(cu[0]) + 5], o[int(cu[0]):int(cu[0]) + 5])
        assert np.array_equal(out[int(cu[1]):int(cu[2])], o[int(cu[1]):int(cu[2])])
    # second pair: one image row each, no text in the unconditional sample
    out = oracle.cfg_combine(o, cu, p["pos"], 3.0)
    assert np.allclose(out[int(cu[2]) + 3], o[int(cu[3])] + 3.0 * (o[int(cu[2]) + 3] - o[int(cu[3])]))
    with pytest.raises(ValueError):
        oracle.cfg_combine(o[:int(cu[3])], cu[:4], p["pos"], 1.0)        # odd sample count
    q = oracle.pack_plan([(1, 16, 16), (1, 32, 16)])
    with pytest.raises(ValueError):
        oracle.cfg_combine(np.zeros((q["total_tokens"], 1, 8)), q["cu_seqlens"], q["pos"], 1.0)


# --------------------------------------------------------------------------
# the memory-bound chains around a joint-attention block
# --------------------------------------------------------------------------

def test_norm_modulate_closed_form_and_library():
    """Hand-derived: x = (1, 3) has mean 2 and variance 1, so LN(x) =
    (-1, 1)/sqrt(1 + eps); modulation scales by 1 + scale and shifts.  The
    normalisation also matches torch's layer_norm in float64 (a library
    routine), and each token takes its own sample's vectors."""
    eps = 1e-6
    cu = np.array([0, 1, 3])
    x = np.array([[1.0, 3.0], [0.0, 4.0], [2.0, -2.0]])
    shift = np.array([[0.25, -0.5], [1.0, 2.0]])
    scale = np.array([[0.5, 0.0], [-1.0, 3.0]])
    y = oracle.norm_modulate(x, cu, shift, scale, eps)
    r = 1.0 / math.sqrt(1.0 + eps)
    assert np.allclose(y[0], [-r * 1.5 + 0.25, r * 1.0 - 0.5], atol=1e-15)
    r4 = 2.0 / math.sqrt(4.0 + eps)
    assert np.allclose(y[1], [-r4 * 0.0 + 1.0, r4 * 4.0 + 2.0], atol=1e-15)
    rng = np.random.default_rng(9)
    xr = rng.standard_normal((7, 64)) * 3 + 1
    zero = np.zeros((1, 64))
    ln = torch.nn.functional.layer_norm(torch.from_numpy(xr), (64,), eps=eps).numpy()
    assert np.allclose(oracle.norm_modulate(xr, np.array([0, 7]), zero, zero, eps), ln, atol=1e-12)


def test_gate_residual_closed_form():
    cu = np.array([0, 2, 3])
    x = np.arange(6.0).reshape(3, 2)
    z = np.ones((3, 2))
    gate = np.array([[2.0, -1.0], [0.5, 0.0]])
    out = oracle.gate_residual(x, z, cu, gate)
    assert np.array_equal(out, np.array([[2.0, 0.0], [4.0, 2.0], [4.5, 5.0]]))


def test_attn_block_closed_forms():
    """gate 0 leaves x unchanged; with zero Q/K weights every logit is 0, the
    attention of a sample is the mean of its v rows, and the block reduces to
    x + gate * mean_s(v) W_o in closed form."""
    rng = np.random.default_rng(10)
    heads, D = 2, 8
    C = heads * D
    samples = [(3, 32, 16), (2, 16, 16)]
    p = oracle.pack_plan(samples)
    T = p["total_tokens"]
    cu = p["cu_seqlens"]
    x = rng.standard_normal((T, C))
    w_qkv = rng.standard_normal((C, 3 * C)) / math.sqrt(C)
    w_o = rng.standard_normal((C, C)) / math.sqrt(C)
    shift, scale, gate = (rng.standard_normal((2, C)) * 0.1 for _ in range(3))
    out0 = oracle.attn_block_fwd(x, cu, p["pos"], heads, w_qkv, w_o, shift, scale, np.zeros((2, C)))
    assert np.array_equal(out0, x)
    w_v = w_qkv.copy()
    w_v[:, :2 * C] = 0.0
    out = oracle.attn_block_fwd(x, cu, p["pos"], heads, w_v, w_o, shift, scale, gate)
    y = oracle.norm_modulate(x, cu, shift, scale)
    v = y @ w_v[:, 2 * C:]
    want = x.copy()
    for i in range(2):
        a, b = int(cu[i]), int(cu[i + 1])
        want[a:b] += gate[i] * (v[a:b].mean(axis=0) @ w_o)
    assert np.allclose(out, want, atol=1e-12)


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------

def _tiny_inputs(seed=0):
    wl = synth.tiny(seed)
    p = oracle.pack_plan(wl.samples)
    t = synth.draw_tensors(wl)
    f64 = {k: v.to(torch.float64).numpy() for k, v in t.items()}
    return wl, p, f64


def test_fwd_equals_brute_force_masked():
    for seed in range(3):
        _, p, t = _tiny_inputs(seed)
        O, L = oracle.attn_fwd(t["q"], t["k"], t["v"], p["cu_seqlens"], p["pos"])
        Ob, Lb = oracle.brute_force_masked(t["q"], t["k"], t["v"], p["cu_seqlens"], p["pos"])
        assert np.abs(O - Ob).max() < 1e-12
        assert np.abs(L - Lb).max() < 1e-12
    samples = synth.random_pack(7, 5, 12, 5)
    p = oracle.pack_plan(samples)
    q, k, v, _ = _rand_qkv(p["total_tokens"], 3, 16, 7)
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    Ob, Lb = oracle.brute_force_masked(q, k, v, p["cu_seqlens"], p["pos"])
    assert np.abs(O - Ob).max() < 1e-12 and np.abs(L - Lb).max() < 1e-12


def test_fwd_samples_independent_and_permutation():
    samples = synth.random_pack(11, 4, 15, 6)
    p = oracle.pack_plan(samples)
    q, k, v, _ = _rand_qkv(p["total_tokens"], 2, 32, 11)
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    cu = p["cu_seqlens"]
    for i, s in enumerate(samples):
        a, b = cu[i], cu[i + 1]
        pi = oracle.pack_plan([s])
        Oi, Li = oracle.attn_fwd(q[a:b], k[a:b], v[a:b], pi["cu_seqlens"], pi["pos"])
        assert np.abs(Oi - O[a:b]).max() < 1e-12
        assert np.abs(Li - L[:, a:b]).max() < 1e-12
    perm = [2, 0, 3, 1]
    ps = oracle.pack_plan([samples[i] for i in perm])
    idx = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in perm])
    Op, Lp = oracle.attn_fwd(q[idx], k[idx], v[idx], ps["cu_seqlens"], ps["pos"])
    assert np.abs(Op - O[idx]).max() < 1e-12 and np.abs(Lp - L[:, idx]).max() < 1e-12


def test_fwd_cfg_pair_packed_equals_separate():
    """Cond and uncond branches packed in one pass give the two separate passes."""
    cond, unc = (12, 64, 48), (3, 64, 48)
    p = oracle.pack_plan([cond, unc])
    q, k, v, _ = _rand_qkv(p["total_tokens"], 2, 32, 5)
    a = p["cu_seqlens"][1]
    img = (64 // 16) * (48 // 16)            # 4x3 grid -> 12 image tokens
    for x in (q, k, v):                      # uncond image rows = cond image rows
        x[a + 3:a + 3 + img] = x[12:12 + img]
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    pc, pu = oracle.pack_plan([cond]), oracle.pack_plan([unc])
    Oc, Lc = oracle.attn_fwd(q[:a], k[:a], v[:a], pc["cu_seqlens"], pc["pos"])
    Ou, Lu = oracle.attn_fwd(q[a:], k[a:], v[a:], pu["cu_seqlens"], pu["pos"])
    assert np.abs(np.concatenate([Oc, Ou]) - O).max() < 1e-12
    assert np.abs(np.concatenate([Lc, Lu], axis=1) - L).max() < 1e-12


def test_fwd_closed_forms():
    rng = np.random.default_rng(4)
    # One-token sample: O = V, LSE = s * q.k (same rotation on both sides).
    p = oracle.pack_plan([(0, 16, 16), (1, 16, 16)])
    q, k, v = (rng.standard_normal((3, 2, 64)) for _ in range(3))
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    assert np.allclose(O[0], v[0], atol=1e-14)
    assert np.allclose(L[:, 0], (q[0] * k[0]).sum(-1) / 8.0, atol=1e-13)
    # Constant V inside a sample: O = that constant.
    p = oracle.pack_plan([(5, 48, 32)])
    T = p["total_tokens"]
    q, k = rng.standard_normal((T, 2, 64)), rng.standard_normal((T, 2, 64))
    v = np.broadcast_to(rng.standard_normal((1, 2, 64)), (T, 2, 64)).copy()
    O, _ = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    assert np.allclose(O, v, atol=1e-13)


def test_fwd_zero_rotation_equals_torch_sdpa():
    """Text-only positions (no rotation): per-sample attention is plain
    scaled-dot-product attention; cross-checked with torch's float64 SDPA."""
    samples = [(6, 32, 48), (4, 48, 16)]
    p = oracle.pack_plan(samples)
    T = p["total_tokens"]
    q, k, v, _ = _rand_qkv(T, 3, 32, 9)
    pos0 = np.full_like(p["pos"], -1)
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], pos0)
    cu = p["cu_seqlens"]
    for i in range(2):
        a, b = cu[i], cu[i + 1]
        tq = torch.from_numpy(q[a:b]).transpose(0, 1)
        tk = torch.from_numpy(k[a:b]).transpose(0, 1)
        tv = torch.from_numpy(v[a:b]).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)
        assert np.abs(ref.transpose(0, 1).numpy() - O[a:b]).max() < 1e-12
        S = torch.einsum("hqd,hkd->hqk", tq, tk) / math.sqrt(32)
        assert np.abs(torch.logsumexp(S, -1).numpy() - L[:, a:b]).max() < 1e-12


def test_attn_rows_matches_fwd():
    _, p, t = _tiny_inputs(1)
    O, L = oracle.attn_fwd(t["q"], t["k"], t["v"], p["cu_seqlens"], p["pos"])
    rows = [0, 16, 17, 80, 81, 100, 153]
    for h in range(2):
        Or, Lr = oracle.attn_rows(t["q"], t["k"], t["v"], p["cu_seqlens"], p["pos"], rows, h)
        assert np.abs(Or - O[rows, h]).max() < 1e-12
        assert np.abs(Lr - L[h, rows]).max() < 1e-12


def test_image_only_sample_shift_invariance():
    """Image-only sample: logits depend on position offsets only, so moving
    the grid origin leaves O and LSE unchanged."""
    p = oracle.pack_plan([(0, 80, 64)])
    q, k, v, _ = _rand_qkv(p["total_tokens"], 2, 64, 13)
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    moved = p["pos"] + np.array([[9, 31]], dtype=np.int32)
    Om, Lm = oracle.attn_fwd(q, k, v, p["cu_seqlens"], moved)
    assert np.abs(O - Om).max() < 1e-10 and np.abs(L - Lm).max() < 1e-10


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------

def _loss(q, k, v, g, p):
    O, _ = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    return float((O * g).sum())


def test_bwd_central_finite_differences():
    _, p, t = _tiny_inputs(2)
    q, k, v, g = t["q"], t["k"], t["v"], t["do"]
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    dq, dk, dv = oracle.attn_bwd(q, k, v, O, L, g, p["cu_seqlens"], p["pos"])
    eps = 1e-6
    rng = np.random.default_rng(0)
    # Directional derivatives cover every entry at once ...
    for x, dx in ((q, dq), (k, dk), (v, dv)):
        u = rng.standard_normal(x.shape)
        xp, xm = x + eps * u, x - eps * u
        args_p = [xp if y is x else y for y in (q, k, v)]
        args_m = [xm if y is x else y for y in (q, k, v)]
        fd = (_loss(*args_p, g, p) - _loss(*args_m, g, p)) / (2 * eps)
        an = float((dx * u).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)
    # ... and single entries pin individual indices (text and image rows,
    # both halves of the head, both heads).
    for (tok, h, d) in [(0, 0, 0), (20, 1, 5), (40, 0, 33), (80, 1, 63), (95, 0, 31), (150, 1, 40)]:
        for x, dx in ((q, dq), (k, dk), (v, dv)):
            e = np.zeros_like(x)
            e[tok, h, d] = 1.0
            args_p = [x + eps * e if y is x else y for y in (q, k, v)]
            args_m = [x - eps * e if y is x else y for y in (q, k, v)]
            fd = (_loss(*args_p, g, p) - _loss(*args_m, g, p)) / (2 * eps)
            assert abs(fd - dx[tok, h, d]) <= 1e-6 * max(1.0, abs(fd)), (tok, h, d)


def test_bwd_invariants():
    samples = synth.random_pack(3, 3, 10, 5)
    p = oracle.pack_plan(samples)
    q, k, v, g = _rand_qkv(p["total_tokens"], 2, 32, 3)
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], p["pos"])
    dq, dk, dv = oracle.attn_bwd(q, k, v, O, L, g, p["cu_seqlens"], p["pos"])
    cu = p["cu_seqlens"]
    for i in range(len(samples)):
        a, b = cu[i], cu[i + 1]
        for h in range(2):
            # O is linear in V:  <dV, V> = <dO, O>.
            assert abs((dv[a:b, h] * v[a:b, h]).sum() - (g[a:b, h] * O[a:b, h]).sum()) < 1e-10
            # Logits are bilinear in (q, k): scaling q or k by a is the same,
            # so <dQ, Q> = <dK, K>.
            assert abs((dq[a:b, h] * q[a:b, h]).sum() - (dk[a:b, h] * k[a:b, h]).sum()) < 1e-10
    # Identical rotated keys: softmax-Jacobian rows sum to zero, so dQ = 0.
    T = 12
    pos = np.zeros((T, 2), dtype=np.int32)
    cu1 = np.array([0, T], dtype=np.int32)
    k1 = np.broadcast_to(k[:1], (T,) + k.shape[1:]).copy()
    O, L = oracle.attn_fwd(q[:T], k1, v[:T], cu1, pos)
    dq, _, _ = oracle.attn_bwd(q[:T], k1, v[:T], O, L, g[:T], cu1, pos)
    assert np.abs(dq).max() < 1e-12


def test_bwd_zero_rotation_equals_torch_autograd():
    samples = [(7, 32, 32), (2, 16, 64)]
    p = oracle.pack_plan(samples)
    T = p["total_tokens"]
    q, k, v, g = _rand_qkv(T, 2, 16, 21)
    pos0 = np.full_like(p["pos"], -1)
    O, L = oracle.attn_fwd(q, k, v, p["cu_seqlens"], pos0)
    dq, dk, dv = oracle.attn_bwd(q, k, v, O, L, g, p["cu_seqlens"], pos0)
    cu = p["cu_seqlens"]
    for i in range(2):
        a, b = cu[i], cu[i + 1]
        tq, tk, tv = (torch.from_numpy(x[a:b]).transpose(0, 1).requires_grad_() for x in (q, k, v))
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv)
        out.backward(torch.from_numpy(g[a:b]).transpose(0, 1))
        for ref, mine in ((tq, dq), (tk, dk), (tv, dv)):
            assert np.abs(ref.grad.transpose(0, 1).numpy() - mine[a:b]).max() < 1e-12


def test_attn_bwd_rows_matches_bwd():
    """The row-wise backward gives attn_bwd's gradients row by row (tiny pack,
    a ragged pack with text-only and one-token samples, an edit pack with
    (h, w, f) RoPE and a non-default scale); a small block size exercises the
    statistics pass over several row blocks and a ragged last block."""
    cases = []
    _, p, t = _tiny_inputs(3)
    cases.append((p, t["q"], t["k"], t["v"], t["do"], {}, 0.0))
    samples = [(5, 32, 48), (9, 0, 0), (1, 16, 16), (0, 48, 16)]
    p = oracle.pack_plan(samples)
    q, k, v, g = _rand_qkv(p["total_tokens"], 2, 32, 17)
    cases.append((p, q, k, v, g, {}, 0.3))
    p = oracle.pack_plan([(4, 32, 32, 2), (3, 16, 48)])
    q, k, v, g = _rand_qkv(p["total_tokens"], 2, 32, 18)
    cases.append((p, q, k, v, g, {"frame": p["frame"], "rope_axes": 3}, 0.0))
    for p, q, k, v, g, ro, sc in cases:
        cu, pos = p["cu_seqlens"], p["pos"]
        O, L = oracle.attn_fwd(q, k, v, cu, pos, softmax_scale=sc, **ro)
        dq, dk, dv = oracle.attn_bwd(q, k, v, O, L, g, cu, pos, softmax_scale=sc, **ro)
        T = p["total_tokens"]
        rows = sorted({0, 1, T // 3, T // 2, T - 2, T - 1} | {int(c) for c in cu[1:-1]})
        for h in range(q.shape[1]):
            rq, rk, rv = oracle.attn_bwd_rows(q, k, v, g, cu, pos, h, q_rows=rows, kv_rows=rows[::-1],
                                              softmax_scale=sc, block=7, **ro)
            assert np.abs(rq - dq[rows, h]).max() < 1e-12
            assert np.abs(rk - dk[rows[::-1], h]).max() < 1e-12
            assert np.abs(rv - dv[rows[::-1], h]).max() < 1e-12


def test_attn_bwd_rows_finite_differences():
    """Single entries of the row-wise gradients against central finite
    differences of the forward (independently of attn_bwd)."""
    _, p, t = _tiny_inputs(4)
    q, k, v, g = t["q"], t["k"], t["v"], t["do"]
    cu, pos = p["cu_seqlens"], p["pos"]
    eps = 1e-6
    for tok, h, d in [(3, 0, 1), (30, 1, 40), (90, 0, 63), (120, 1, 17)]:
        rq, rk, rv = oracle.attn_bwd_rows(q, k, v, g, cu, pos, h, q_rows=[tok], kv_rows=[tok])
        for x, got in ((q, rq[0, d]), (k, rk[0, d]), (v, rv[0, d])):
            e = np.zeros_like(x)
            e[tok, h, d] = 1.0
            args_p = [x + eps * e if y is x else y for y in (q, k, v)]
            args_m = [x - eps * e if y is x else y for y in (q, k, v)]
            fd = (_loss(*args_p, g, p) - _loss(*args_m, g, p)) / (2 * eps)
            assert abs(fd - got) <= 1e-6 * max(1.0, abs(fd)), (tok, h, d, fd, got)
