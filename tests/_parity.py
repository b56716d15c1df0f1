"""Shared helpers for the GPU parity tests (tolerances and comparisons)."""
import numpy as np
import torch

# Tolerances of the library's contract: bf16 inputs, fp32 accumulation,
# compared with the float64 oracle on the same bf16 values.
TOL = {
    "o": {"max_abs": 2e-2, "rel_l2": 5e-3},
    "grad": {"max_abs": 2e-2, "rel_l2": 1e-2},
    "lse": {"max_abs": 1e-3},
}


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def lse_tol_factor(scale, head_dim):
    """The LSE and gradient bounds are stated for the default scale 1/sqrt(d).
    The logit rounding error is proportional to the logits' size,
    s * |q~||k~| ~ s*sqrt(d), and dQ, dK carry the factor s themselves, so a
    non-default scale widens the bounds by s * sqrt(d) (never tightens them)."""
    if not scale or scale <= 0:
        return 1.0
    return max(1.0, scale * np.sqrt(head_dim))


def assert_close(name, got, want, kind, factor=1.0):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    tol = {k: v * factor for k, v in TOL[kind].items()}
    mab = float(np.abs(got - want).max()) if got.size else 0.0
    assert mab <= tol["max_abs"], f"{name}: max-abs {mab:.3e} > {tol['max_abs']}"
    # relative L2 is undefined against an all-zero reference (e.g. dQ, dK of a
    # one-token sample, whose softmax is constant); max-abs still applies.
    if "rel_l2" in tol and got.size and np.linalg.norm(want) > 0:
        r = rel_l2(got, want)
        assert r <= tol["rel_l2"], f"{name}: rel-L2 {r:.3e} > {tol['rel_l2']}"
    return mab
