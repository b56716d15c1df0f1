"""Float64 CPU oracle (test infrastructure only; see ``oracle.ref``)."""
from .ref import (attn_block_fwd, attn_bwd, attn_bwd_rows, attn_fwd, attn_rows, brute_force_masked, cfg_combine,
                  default_scale, gate_residual, norm_modulate, pack_plan, rope, rope_angles, rope_axes_dims)

__all__ = ["pack_plan", "rope", "rope_angles", "rope_axes_dims", "attn_fwd", "attn_bwd", "attn_bwd_rows", "attn_rows", "cfg_combine", "norm_modulate", "gate_residual", "attn_block_fwd",
           "brute_force_masked", "default_scale"]
