"""Float64 CPU oracle for packed native-resolution joint attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run this module.  The CUDA
library never calls it and shares no code, table or helper with it.

What it computes, and where each step comes from:

* ``pack_plan`` -- Mage-Flow review (startedourmission.github.io),
  section "Native-Resolution MMDiT": images of different sizes are encoded to
  variable-length latent token rows and packed back to back into one batch
  under a fixed token budget; text is packed the same way, unpadded; attention
  is confined to each sample by per-sample cumulative offsets instead of a
  block-diagonal mask.  Section "Mage-VAE": the latent is 16x downsampled with
  patchification absorbed, so an H x W image gives (H/16)(W/16) tokens.
* ``rope`` -- per-sample 2D rotary embedding (Hugging Face paper page,
  Highlights, "System-level speed"; model card, section "Architecture").  The
  pages do not give the layout; this library fixes it: head_dim split in half,
  first half rotated by the token's latent row, second half by its column,
  pair (2i, 2i+1) of each half at frequency theta^(-2i/(head_dim/2)),
  theta = 10000, rotation x0' = x0 cos - x1 sin, x1' = x0 sin + x1 cos; text
  tokens are not rotated.
* ``rope`` with ``rope_axes=3`` -- the edit model's (h, w, f) positions
  (Mage-Flow review, section on the editing model: a frame dimension is added
  to the 2D RoPE so that source and target latents are told apart).  The
  pages give no layout; this library fixes it: head_dim split into three
  contiguous slices, frame | row | col, of head_dim/8, 7 head_dim/16 and
  7 head_dim/16 dimensions; pair i of an a-dimension slice turns at
  theta^(-2i/a) times the token's index on that axis.
* ``attn_fwd`` / ``attn_bwd`` -- joint text+image self-attention of each
  sample (review, "Native-Resolution MMDiT": text and image tokens are
  concatenated and processed by joint self-attention), i.e. plain
  softmax(s * q~ k~^T) v per sample and head, with s = 1/sqrt(head_dim) unless
  given; the backward is the exact gradient of that definition with respect
  to the un-rotated q, k and v.
* ``attn_rows`` / ``attn_bwd_rows`` -- the same forward and backward for
  selected rows of one head, row by row (O(L D) per row once a sample's row
  statistics are known), so that full-size packs can be checked.
* ``cfg_combine`` -- classifier-free guidance over a pack whose samples come
  in (conditional, unconditional) pairs (review, section on CFG: the two
  branches run in one packed forward).  The pages do not print the
  combination; the standard reading is taken: guided = u + g (c - u) for the
  image rows of each pair, written over the conditional sample's image rows.
* ``norm_modulate``, ``gate_residual``, ``attn_block_fwd`` -- the memory-bound
  chains around one joint-attention block (review, kernel-fusion section:
  normalisation, adaptive modulation, RoPE application, gating and the
  residual add are fused instead of run as separate kernels).  The pages do
  not give the operations' exact form; the plainest reading of adaptive
  modulation in a diffusion transformer is taken: y = LN(x) (1 + scale_s) +
  shift_s with a LayerNorm over the hidden size (no affine, eps 1e-6) and
  per-sample modulation vectors, and out = x + gate_s * z after the output
  projection.  The projections are plain matrix products (synthetic weights).
* ``brute_force_masked`` -- the thing the offsets replace: dense attention
  over the whole pack with an explicit block-diagonal mask.  Written
  separately from ``attn_fwd`` on purpose.

Every array is float64; bf16 inputs are widened exactly.  Nothing is blocked,
fused or reordered beyond the definitions above.
"""
from __future__ import annotations

import math

import numpy as np

PATCH = 16
TEXT_POS = -1


# --------------------------------------------------------------------------
# Pack plan
# --------------------------------------------------------------------------

def pack_plan(samples, token_budget: int = 0):
    """Plan a pack from per-sample (text_len, height_px, width_px[, frames]).

    A sample with height = width = 0 and text is text-only (no image rows).
    ``frames`` (default 1) is 1 for a generation sample and 2 for an edit
    sample, whose source and target latents (same size) follow its text as
    frames 0 and 1.  The samples are taken in order; the pack is the longest
    prefix whose total token count stays within ``token_budget`` (0 = no
    budget).  Tokens of one sample are [text; frame 0; frame 1 ...], each
    frame in row-major latent order (row = index along the height).  Returns
    a dict with ``n_samples`` (packed prefix), ``cu_seqlens`` int32 [n+1],
    ``pos`` int32 [T, 2] ((-1, -1) for text), ``frame`` int32 [T] (-1 for
    text), ``total_tokens``, ``max_seqlen`` and ``max_grid`` (largest grid
    side).  Raises ValueError for invalid shapes and when not even the first
    sample fits the budget.
    """
    lens, grids, frames = [], [], []
    for smp in samples:
        t, h, w = smp[:3]
        nf = smp[3] if len(smp) > 3 else 1
        text_only = h == 0 and w == 0 and t > 0       # a sample without an image
        if t < 0 or (not text_only and (h <= 0 or w <= 0)) or h % PATCH or w % PATCH or nf not in (1, 2):
            raise ValueError(f"invalid sample {tuple(smp)}")
        gh, gw = h // PATCH, w // PATCH
        lens.append(t + nf * gh * gw)
        grids.append((gh, gw))
        frames.append(nf)
    n = 0
    used = 0
    for L in lens:
        if token_budget > 0 and used + L > token_budget:
            break
        used += L
        n += 1
    if n == 0 and len(samples) > 0:
        raise ValueError("first sample exceeds the token budget")
    cu = np.zeros(n + 1, dtype=np.int32)
    for i in range(n):
        cu[i + 1] = cu[i] + lens[i]
    T = int(cu[n])
    pos = np.full((T, 2), TEXT_POS, dtype=np.int32)
    frame = np.full(T, TEXT_POS, dtype=np.int32)
    for i in range(n):
        t = samples[i][0]
        gh, gw = grids[i]
        for j in range(frames[i] * gh * gw):
            f, r = divmod(j, gh * gw)
            pos[cu[i] + t + j, 0] = r // gw
            pos[cu[i] + t + j, 1] = r % gw
            frame[cu[i] + t + j] = f
    return {
        "n_samples": n,
        "cu_seqlens": cu,
        "pos": pos,
        "frame": frame,
        "total_tokens": T,
        "max_seqlen": int(max(lens[:n])) if n else 0,
        "max_grid": int(max(max(g) for g in grids[:n])) if n else 0,
    }


# --------------------------------------------------------------------------
# 2D RoPE
# --------------------------------------------------------------------------

def rope_axes_dims(head_dim: int, rope_axes: int):
    """Sizes of the contiguous head_dim slices and the position axis each
    turns by: 2 axes -> [(row, d/2), (col, d/2)]; 3 axes -> [(frame, d/8),
    (row, 7d/16), (col, 7d/16)]."""
    if rope_axes == 2:
        return [("row", head_dim // 2), ("col", head_dim // 2)]
    if rope_axes == 3:
        a = 7 * head_dim // 16
        return [("frame", head_dim - 2 * a), ("row", a), ("col", a)]
    raise ValueError(f"rope_axes must be 2 or 3, got {rope_axes}")


def rope_angles(pos, head_dim: int, theta: float = 10000.0, frame=None, rope_axes: int = 2):
    """Angle of every rotation pair: [T, head_dim/2] float64.

    The head is cut into the slices of ``rope_axes_dims``; pair i of a slice
    of a dimensions turns by (the token's index on that slice's axis) *
    theta^(-2i/a).  With 2 axes that is: pair p < head_dim/4 in the first
    half turns by row * f_p, pair head_dim/4 + p by col * f_p, with
    f_p = theta^(-2p/(head_dim/2)).  Text rows get angle 0.
    """
    pos = np.asarray(pos)
    idx = {"row": pos[:, 0].astype(np.float64), "col": pos[:, 1].astype(np.float64)}
    if frame is not None:
        idx["frame"] = np.asarray(frame).astype(np.float64)
    parts = []
    for axis, a in rope_axes_dims(head_dim, rope_axes):
        f = np.array([theta ** (-2.0 * i / a) for i in range(a // 2)], dtype=np.float64)
        parts.append(idx[axis][:, None] * f[None, :])
    ang = np.concatenate(parts, axis=1)
    ang[pos[:, 0] < 0] = 0.0
    return ang


def rope(x, pos, theta: float = 10000.0, inverse: bool = False, frame=None, rope_axes: int = 2):
    """Rotate x [T, heads, head_dim] by each token's 2D (or (h, w, f)) position.

    Pair m covers dims (2m, 2m+1) over the whole head (m < head_dim/2), which
    puts the first head_dim/4 pairs in the first half and the rest in the
    second half (2 axes).  ``inverse`` rotates by the negated angles (R^T),
    which is the adjoint needed to pull gradients back to un-rotated inputs.
    """
    x = np.asarray(x, dtype=np.float64)
    T, H, D = x.shape
    ang = rope_angles(pos, D, theta, frame, rope_axes)
    if inverse:
        ang = -ang
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------

def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def _logsumexp_rows(S):
    m = S.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(S - m).sum(axis=1, keepdims=True)))[:, 0]


def attn_fwd(q, k, v, cu_seqlens, pos, softmax_scale: float = 0.0, theta: float = 10000.0,
             frame=None, rope_axes: int = 2):
    """Per-sample, per-head softmax attention on RoPE-rotated q and k.

    q, k, v: [T, H, D] (any float dtype, widened to float64).  ``frame`` and
    ``rope_axes`` select the (h, w, f) rotation (see ``rope``).
    Returns O [T, H, D] float64 and LSE [H, T] float64, where LSE is the
    natural log-sum-exp of the scaled logits of each query row.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, H, D = q.shape
    s = softmax_scale if softmax_scale > 0 else default_scale(D)
    qr = rope(q, pos, theta, frame=frame, rope_axes=rope_axes)
    kr = rope(k, pos, theta, frame=frame, rope_axes=rope_axes)
    O = np.zeros((T, H, D))
    LSE = np.zeros((H, T))
    for i in range(len(cu_seqlens) - 1):
        a, b = int(cu_seqlens[i]), int(cu_seqlens[i + 1])
        for h in range(H):
            S = s * (qr[a:b, h, :] @ kr[a:b, h, :].T)
            lse = _logsumexp_rows(S)
            P = np.exp(S - lse[:, None])
            O[a:b, h, :] = P @ v[a:b, h, :]
            LSE[h, a:b] = lse
    return O, LSE


def attn_bwd(q, k, v, o, lse, do, cu_seqlens, pos, softmax_scale: float = 0.0,
             theta: float = 10000.0, frame=None, rope_axes: int = 2):
    """Gradients dQ, dK, dV of sum(O * dO) w.r.t. the un-rotated q, k, v.

    With q~ = R q, k~ = R k, S = s q~ k~^T, P = exp(S - LSE):
      dV = P^T dO;  dP = dO V^T;  D = rowsum(dO * O);  dS = P * (dP - D);
      dq~ = s dS k~;  dk~ = s dS^T q~;  dq = R^T dq~;  dk = R^T dk~.
    ``o`` and ``lse`` are the forward's outputs (as the backward of the
    library receives them).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    T, H, D = q.shape
    s = softmax_scale if softmax_scale > 0 else default_scale(D)
    qr = rope(q, pos, theta, frame=frame, rope_axes=rope_axes)
    kr = rope(k, pos, theta, frame=frame, rope_axes=rope_axes)
    dqr = np.zeros((T, H, D))
    dkr = np.zeros((T, H, D))
    dv = np.zeros((T, H, D))
    for i in range(len(cu_seqlens) - 1):
        a, b = int(cu_seqlens[i]), int(cu_seqlens[i + 1])
        for h in range(H):
            S = s * (qr[a:b, h, :] @ kr[a:b, h, :].T)
            P = np.exp(S - lse[h, a:b][:, None])
            dv[a:b, h, :] = P.T @ do[a:b, h, :]
            dP = do[a:b, h, :] @ v[a:b, h, :].T
            Drow = (do[a:b, h, :] * o[a:b, h, :]).sum(axis=1)
            dS = P * (dP - Drow[:, None])
            dqr[a:b, h, :] = s * (dS @ kr[a:b, h, :])
            dkr[a:b, h, :] = s * (dS.T @ qr[a:b, h, :])
    dq = rope(dqr, pos, theta, inverse=True, frame=frame, rope_axes=rope_axes)
    dk = rope(dkr, pos, theta, inverse=True, frame=frame, rope_axes=rope_axes)
    return dq, dk, dv


def attn_rows(q, k, v, cu_seqlens, pos, rows, head: int, softmax_scale: float = 0.0,
              theta: float = 10000.0, frame=None, rope_axes: int = 2):
    """O and LSE of selected query rows of one head, one row at a time.

    For full-size packs: each row touches only its own sample's keys, so it
    costs O(L * D) (the sample's rotated keys are formed once for all of its
    requested rows).  Returns (O [len(rows), D], LSE [len(rows)]).
    """
    q = np.asarray(q[:, head, :], dtype=np.float64)[:, None, :]
    k = np.asarray(k[:, head, :], dtype=np.float64)[:, None, :]
    v = np.asarray(v[:, head, :], dtype=np.float64)
    D = q.shape[2]
    s = softmax_scale if softmax_scale > 0 else default_scale(D)
    cu = np.asarray(cu_seqlens)
    rows = [int(r) for r in rows]
    O = np.zeros((len(rows), D))
    LSE = np.zeros(len(rows))
    sample = [int(np.searchsorted(cu, r, side="right") - 1) for r in rows]
    for i in sorted(set(sample)):
        a, b = int(cu[i]), int(cu[i + 1])
        fk = None if frame is None else frame[a:b]
        kr = rope(k[a:b], pos[a:b], theta, frame=fk, rope_axes=rope_axes)[:, 0, :]
        for n, r in enumerate(rows):
            if sample[n] != i:
                continue
            fq = None if frame is None else frame[r:r + 1]
            qr = rope(q[r:r + 1], pos[r:r + 1], theta, frame=fq, rope_axes=rope_axes)[0, 0]
            srow = s * (kr @ qr)
            m = srow.max()
            lse = m + math.log(np.exp(srow - m).sum())
            O[n] = np.exp(srow - lse) @ v[a:b]
            LSE[n] = lse
    return O, LSE


def attn_bwd_rows(q, k, v, do, cu_seqlens, pos, head: int, q_rows=(), kv_rows=(), softmax_scale: float = 0.0,
                  theta: float = 10000.0, frame=None, rope_axes: int = 2, block: int = 1024):
    """dQ of selected query rows and dK, dV of selected key rows of one head.

    The same gradients as ``attn_bwd`` (the exact gradient of per-sample
    softmax(s q~ k~^T) v with respect to the un-rotated q, k, v), taken one
    row at a time so that full-size packs stay affordable:

      * the sample's row statistics first: for every query row r of a sample
        that holds a requested row, LSE_r = logsumexp_j S[r, j],
        O_r = sum_j exp(S[r, j] - LSE_r) v_j and D_r = dO_r . O_r
        (S = s q~ k~^T; the rows are visited ``block`` at a time only to bound
        memory, each row on its own);
      * query row r:  dS[r, :] = P[r, :] (dP[r, :] - D_r) with
        P[r, j] = exp(S[r, j] - LSE_r) and dP[r, j] = dO_r . v_j;
        dq_r = R^T (s sum_j dS[r, j] k~_j);
      * key row c:    dv_c = sum_r P[r, c] dO_r;
        dS[:, c] = P[:, c] (dP[:, c] - D);  dk_c = R^T (s sum_r dS[r, c] q~_r).

    Each requested row costs O(L D) once the statistics are known.  D_r here
    uses this oracle's own O (the library's backward receives the forward's
    O; the two agree within the forward's tolerance).  Returns (dq
    [len(q_rows), D], dk [len(kv_rows), D], dv [len(kv_rows), D]) in float64.
    """
    q = np.asarray(q[:, head, :], dtype=np.float64)
    k = np.asarray(k[:, head, :], dtype=np.float64)
    v = np.asarray(v[:, head, :], dtype=np.float64)
    do = np.asarray(do[:, head, :], dtype=np.float64)
    D = q.shape[1]
    s = softmax_scale if softmax_scale > 0 else default_scale(D)
    cu = np.asarray(cu_seqlens)
    pos = np.asarray(pos)
    q_rows = [int(r) for r in q_rows]
    kv_rows = [int(r) for r in kv_rows]
    dq = np.zeros((len(q_rows), D))
    dk = np.zeros((len(kv_rows), D))
    dv = np.zeros((len(kv_rows), D))

    def sample_of(r):
        return int(np.searchsorted(cu, r, side="right") - 1)

    def rot(x, a, b, inverse=False):
        fr = None if frame is None else np.asarray(frame)[a:b]
        return rope(x[:, None, :], pos[a:b], theta, inverse=inverse, frame=fr, rope_axes=rope_axes)[:, 0, :]

    for i in sorted({sample_of(r) for r in q_rows + kv_rows}):
        a, b = int(cu[i]), int(cu[i + 1])
        qr, kr = rot(q[a:b], a, b), rot(k[a:b], a, b)
        vs, dos = v[a:b], do[a:b]
        L = b - a
        lse = np.zeros(L)
        dsum = np.zeros(L)
        for r0 in range(0, L, block):
            S = s * (qr[r0:r0 + block] @ kr.T)
            m = S.max(axis=1, keepdims=True)
            E = np.exp(S - m)
            z = E.sum(axis=1, keepdims=True)
            lse[r0:r0 + block] = (m + np.log(z))[:, 0]
            O = (E / z) @ vs
            dsum[r0:r0 + block] = (dos[r0:r0 + block] * O).sum(axis=1)
        for n, r in enumerate(q_rows):
            if sample_of(r) != i:
                continue
            j = r - a
            P = np.exp(s * (kr @ qr[j]) - lse[j])
            dS = P * (vs @ dos[j] - dsum[j])
            dq[n] = rot((s * (dS @ kr))[None, :], r, r + 1, inverse=True)[0]
        for n, c in enumerate(kv_rows):
            if sample_of(c) != i:
                continue
            j = c - a
            P = np.exp(s * (qr @ kr[j]) - lse)
            dv[n] = P @ dos
            dS = P * (dos @ vs[j] - dsum)
            dk[n] = rot((s * (dS @ qr))[None, :], c, c + 1, inverse=True)[0]
    return dq, dk, dv


def cfg_combine(o, cu_seqlens, pos, guidance: float):
    """Guided outputs of a pack of (cond, uncond) sample pairs.

    ``o`` [T, H, D].  Samples 2p and 2p+1 are the conditional and the
    unconditional branch of prompt p; their image rows (the rows with
    pos >= 0, which end each sample) must have the same count.  Returns a
    float64 copy of ``o`` whose conditional image rows hold
    u + guidance * (c - u); every other row is unchanged.
    """
    o = np.asarray(o, dtype=np.float64)
    out = o.copy()
    cu = np.asarray(cu_seqlens)
    pos = np.asarray(pos)
    n = len(cu) - 1
    if n % 2:
        raise ValueError("a CFG pack holds (cond, uncond) pairs")
    for p in range(n // 2):
        ca, cb = int(cu[2 * p]), int(cu[2 * p + 1])
        ua, ub = int(cu[2 * p + 1]), int(cu[2 * p + 2])
        c_img = [r for r in range(ca, cb) if pos[r, 0] >= 0]
        u_img = [r for r in range(ua, ub) if pos[r, 0] >= 0]
        if len(c_img) != len(u_img):
            raise ValueError(f"pair {p}: image row counts differ")
        for rc, ru in zip(c_img, u_img):
            out[rc] = o[ru] + guidance * (o[rc] - o[ru])
    return out


def _sample_of_token(cu_seqlens):
    cu = np.asarray(cu_seqlens)
    return np.repeat(np.arange(len(cu) - 1), np.diff(cu))


def norm_modulate(x, cu_seqlens, shift, scale, eps: float = 1e-6):
    """y = LN(x) * (1 + scale_s) + shift_s for every token of sample s.

    x [T, C]; shift, scale [n_samples, C].  LN normalises each row over C to
    zero mean and unit variance (population variance, eps inside the square
    root), without a learned affine.
    """
    x = np.asarray(x, dtype=np.float64)
    s = _sample_of_token(cu_seqlens)
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    n = (x - mu) / np.sqrt(var + eps)
    return n * (1.0 + np.asarray(scale, dtype=np.float64)[s]) + np.asarray(shift, dtype=np.float64)[s]


def gate_residual(x, z, cu_seqlens, gate):
    """out = x + gate_s * z for every token of sample s (x, z [T, C])."""
    s = _sample_of_token(cu_seqlens)
    return np.asarray(x, dtype=np.float64) + np.asarray(gate, dtype=np.float64)[s] * np.asarray(z, dtype=np.float64)


def attn_block_fwd(x, cu_seqlens, pos, heads: int, w_qkv, w_o, shift, scale, gate, softmax_scale: float = 0.0,
                   eps: float = 1e-6, frame=None, rope_axes: int = 2):
    """One joint-attention block: x + gate * (Attn(R(q), R(k), v) W_o) with
    [q | k | v] = norm_modulate(x) W_qkv; x [T, C], W_qkv [C, 3C], W_o [C, C],
    C = heads * head_dim, the columns of each third ordered [head][dim]."""
    x = np.asarray(x, dtype=np.float64)
    T, C = x.shape
    D = C // heads
    y = norm_modulate(x, cu_seqlens, shift, scale, eps)
    qkv = y @ np.asarray(w_qkv, dtype=np.float64)
    q, k, v = (qkv[:, i * C:(i + 1) * C].reshape(T, heads, D) for i in range(3))
    O, _ = attn_fwd(q, k, v, cu_seqlens, pos, softmax_scale, frame=frame, rope_axes=rope_axes)
    z = O.reshape(T, C) @ np.asarray(w_o, dtype=np.float64)
    return gate_residual(x, z, cu_seqlens, gate)


def brute_force_masked(q, k, v, cu_seqlens, pos, softmax_scale: float = 0.0,
                       theta: float = 10000.0):
    """Dense attention over all T tokens with an explicit block-diagonal mask.

    Independent of ``attn_fwd``: the rotation is applied through complex
    multiplication of (x_{2m} + i x_{2m+1}) by exp(i * angle), the mask is a
    T x T boolean matrix built from a per-token sample id, and the softmax is
    taken over the full masked row.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, H, D = q.shape
    s = softmax_scale if softmax_scale > 0 else default_scale(D)
    ang = rope_angles(pos, D, theta)                     # [T, D/2]
    rot = np.exp(1j * ang)[:, None, :]
    qc = (q[..., 0::2] + 1j * q[..., 1::2]) * rot
    kc = (k[..., 0::2] + 1j * k[..., 1::2]) * rot
    sid = np.zeros(T, dtype=np.int64)
    for i in range(len(cu_seqlens) - 1):
        sid[int(cu_seqlens[i]):int(cu_seqlens[i + 1])] = i
    allowed = sid[:, None] == sid[None, :]
    O = np.zeros((T, H, D))
    LSE = np.zeros((H, T))
    for h in range(H):
        # Re(a * conj(b)) = a0 b0 + a1 b1 is the real dot product of the pairs.
        S = s * np.real(qc[:, h, :] @ np.conj(kc[:, h, :]).T)
        S = np.where(allowed, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        E = np.where(allowed, np.exp(S - m), 0.0)
        Z = E.sum(axis=1, keepdims=True)
        O[:, h, :] = (E / Z) @ v[:, h, :]
        LSE[h] = (m + np.log(Z))[:, 0]
    return O, LSE
