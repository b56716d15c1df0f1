"""Seeded synthetic workloads for packed native-resolution attention.

This module only *draws inputs*: per-sample shapes (text length, image height
and width in pixels) and the bf16 Q/K/V/dO values.  It holds none of the
attention arithmetic, so both the float64 oracle and the CUDA library can be
fed from it without sharing code with each other.

The workloads stand in for the training and inference packs the Mage-Flow
pages describe (images of 512..2048 px per side, aspect up to 4:1, packed
under a token budget with unpadded text; the 16x latent downsampling makes one
latent pixel one token).  No dataset is involved: every value is seeded.

Recipe (stated once, used everywhere):

* pack shapes come from ``numpy.random.default_rng(seed)`` (PCG64), drawing
  grid height, grid width and text length in that order per sample;
* Q, K, V and dO are drawn in that order from
  ``torch.Generator('cpu').manual_seed(seed)`` as ``randn`` float32 of shape
  ``[total_tokens, heads, head_dim]`` and rounded to bfloat16 (round to
  nearest even) -- the oracle and the GPU read the same bf16 values;
* in the CFG pack, each uncond sample's image rows are copies of its cond
  partner's image rows (Q, K, V and dO alike); text rows stay independent.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

PATCH = 16  # pixels per latent token side (16x downsampling tokenizer)


@dataclass
class Workload:
    name: str
    samples: list            # [(text_len, height_px, width_px)]
    heads: int
    head_dim: int
    passes: str              # "fwd" or "fwd+bwd"
    token_budget: int = 0    # 0 = unlimited
    cfg_pairs: bool = False  # uncond image rows copy the cond partner's
    notes: str = ""
    seed: int = 0
    extra: dict = field(default_factory=dict)
    rope_axes: int = 2       # 3: the (frame, row, col) rotation of edit packs

    def segments(self):
        """Per-sample (text rows, image rows) counts in pack order (an edit
        sample (t, h, w, 2) has two frames of image rows)."""
        return [(smp[0], (smp[3] if len(smp) > 3 else 1) * (smp[1] // PATCH) * (smp[2] // PATCH))
                for smp in self.samples]

    @property
    def total_tokens(self) -> int:
        return int(sum(a + b for a, b in self.segments()))


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    """Two samples: text 17 + 8x8 grid (128x128 px), text 9 + 4x16 grid
    (64x256 px); 2 heads, head_dim 64."""
    return Workload("tiny", [(17, 128, 128), (9, 64, 256)], heads=2, head_dim=64,
                    passes="fwd+bwd", seed=seed)


def single_1024(seed: int = 0) -> Workload:
    """One 1024x1024 image (64x64 = 4096 tokens) with 128 text tokens."""
    return Workload("single_1024", [(128, 1024, 1024)], heads=24, head_dim=128,
                    passes="fwd", seed=seed)


def native_res_shapes(seed: int, budget: int = 32768, max_draws: int = 1000):
    """Draw-and-skip fill of one token budget.

    Per draw: grid sides uniform over {32..128} latent tokens (512..2048 px in
    steps of 16 px), text length uniform over {32..256}.  A draw that does not
    fit the remaining budget is skipped; filling stops once the remainder is
    below the smallest possible sample (32 + 32*32 = 1056 tokens) or after
    ``max_draws`` draws.  The 4:1 aspect limit is checked but cannot bind for
    sides in [512, 2048].
    """
    rng = np.random.default_rng(seed)
    out, used = [], 0
    smallest = 32 + 32 * 32
    for _ in range(max_draws):
        gh = int(rng.integers(32, 129))
        gw = int(rng.integers(32, 129))
        t = int(rng.integers(32, 257))
        if max(gh, gw) > 4 * min(gh, gw):
            continue
        n = t + gh * gw
        if used + n <= budget:
            out.append((t, gh * PATCH, gw * PATCH))
            used += n
        if budget - used < smallest:
            break
    return out


def native_res(seed: int = 0, budget: int = 32768) -> Workload:
    return Workload("native_res_32k", native_res_shapes(seed, budget), heads=24,
                    head_dim=128, passes="fwd+bwd", token_budget=budget, seed=seed)


def cfg_pair(seed: int = 0) -> Workload:
    """4 prompts at 1024x1024: cond (256 text + 4096 image) then uncond
    (8 text + the same 4096 image rows), interleaved cond1, uncond1, ..."""
    s = []
    for _ in range(4):
        s.append((256, 1024, 1024))
        s.append((8, 1024, 1024))
    return Workload("cfg_pair", s, heads=24, head_dim=128, passes="fwd",
                    cfg_pairs=True, seed=seed,
                    notes="parts sum to 33,824 tokens (the stated 33,088 does not match its parts)")


def extreme_aspect(seed: int = 0) -> Workload:
    return Workload("extreme_aspect", [(200, 512, 2048), (64, 2048, 512), (256, 2048, 2048)],
                    heads=24, head_dim=128, passes="fwd+bwd", seed=seed,
                    notes="parts sum to 25,096 tokens (the stated 24,840 omits the 2048^2 text)")


def native_res_50k(seed: int = 0) -> Workload:
    """The training-pack recipe at the pages' 50,000 packed tokens per GPU
    (review, kernel-fusion section: 8 GPUs, global batch 8, ~50K tokens per
    GPU)."""
    return Workload("native_res_50k", native_res_shapes(seed, 50000), heads=24,
                    head_dim=128, passes="fwd+bwd", token_budget=50000, seed=seed)


def padded(wl: Workload) -> Workload:
    """The same samples as a padded batch: every sample grown to the longest
    one's token count with extra text rows (a dense kernel over a padded
    batch computes the masked positions too, so this is the padded batch's
    work; the padding rows are not masked).  No token budget."""
    segs = wl.segments()
    L = max(a + b for a, b in segs)
    out = []
    for smp, (a, b) in zip(wl.samples, segs):
        out.append((smp[0] + (L - a - b),) + tuple(smp[1:]))
    return Workload(wl.name + "_padded", out, wl.heads, wl.head_dim, wl.passes, token_budget=0,
                    seed=wl.seed, rope_axes=wl.rope_axes,
                    notes=f"{len(out)} samples padded to {L} tokens")


def edit_pack(seed: int = 0) -> Workload:
    """An edit training pack (not one of the five headline configs): three
    edit samples whose source and target latents (frames 0 and 1, same size)
    follow their instruction text, plus one generation sample, drawn like the
    training pack (sides 512-1536 px, text 32-256 tokens) until about 24K
    tokens; (frame, row, col) RoPE."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(4):
        gh, gw = (int(x) for x in rng.integers(32, 97, size=2))
        t = int(rng.integers(32, 257))
        out.append((t, gh * PATCH, gw * PATCH, 2 if i < 3 else 1))
    return Workload("edit_pack", out, heads=24, head_dim=128, passes="fwd+bwd", seed=seed, rope_axes=3)


WORKLOADS = {
    "tiny": tiny,
    "single_1024": single_1024,
    "native_res_32k": native_res,
    "cfg_pair": cfg_pair,
    "extreme_aspect": extreme_aspect,
    "edit_pack": edit_pack,
    "native_res_50k": native_res_50k,
    "native_res_32k_padded": lambda seed=0: padded(native_res(seed)),
    "native_res_50k_padded": lambda seed=0: padded(native_res_50k(seed)),
}


# --------------------------------------------------------------------------
# Tensors
# --------------------------------------------------------------------------

def draw_tensors(wl: Workload, with_grad: bool = True):
    """Seeded bf16 CPU tensors Q, K, V (and dO) of shape [T, heads, head_dim]."""
    g = torch.Generator("cpu").manual_seed(int(wl.seed))
    shape = (wl.total_tokens, wl.heads, wl.head_dim)
    names = ["q", "k", "v"] + (["do"] if with_grad else [])
    out = {}
    for nm in names:
        out[nm] = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    if wl.cfg_pairs:
        segs = wl.segments()
        starts = np.concatenate([[0], np.cumsum([a + b for a, b in segs])])
        for i in range(0, len(segs), 2):
            tc, ic = segs[i]
            tu, iu = segs[i + 1]
            assert ic == iu
            src = slice(int(starts[i]) + tc, int(starts[i]) + tc + ic)
            dst = slice(int(starts[i + 1]) + tu, int(starts[i + 1]) + tu + iu)
            for nm in names:
                out[nm][dst] = out[nm][src]
    return out


def random_pack(seed: int, n_samples: int, max_text: int, max_side_tokens: int, edit: bool = False):
    """Small random packs for edge-case parity tests: ragged lengths, image-only
    samples (text 0) and single-token samples (text 0, 16x16 px).  Every sample
    has at least one image token.  Returns [(text_len, height_px, width_px)],
    or with ``edit`` [(text_len, height_px, width_px, frames)] with frames
    drawn from {1, 2}.
    """
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n_samples):
        gh = int(rng.integers(1, max_side_tokens + 1))
        gw = int(rng.integers(1, max_side_tokens + 1))
        t = int(rng.integers(0, max_text + 1))
        if edit:
            out.append((t, gh * PATCH, gw * PATCH, int(rng.integers(1, 3))))
        else:
            out.append((t, gh * PATCH, gw * PATCH))
    return out
