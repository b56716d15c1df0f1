"""Packed native-resolution joint attention for B300 -- Python binding.

A thin ctypes layer over ``libmf.so`` (declared in ``include/mf.h``): it
marshals arguments and allocates caller-side buffers with PyTorch; every step
of the computation runs in the library's CUDA kernels.  There is no CPU path:
if the library is missing or fails to load, every call raises.

    plan = pack_plan([(text_len, height_px, width_px), ...], token_budget=32768)
    o, lse = attn_fwd(q, k, v, plan)               # bf16 [T, heads, head_dim]
    dq, dk, dv = attn_bwd(q, k, v, o, lse, do, plan)
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["MfError", "Plan", "pack_plan", "attn_fwd", "attn_bwd", "check", "record_main_kernel", "lib",
           "library_path", "fwd_workspace_bytes", "bwd_workspace_bytes", "debug_inject", "cfg_combine", "norm_modulate", "gate_residual", "attn_fwd_qkv",
           "DEBUG_DROP_FWD_KV", "DEBUG_DROP_BWD_QDO", "EXPORTED_SYMBOLS", "STATUS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmf.so")

STATUS = {0: "MF_OK", 1: "MF_ERR_INVALID_ARG", 2: "MF_ERR_UNSUPPORTED", 3: "MF_ERR_BUDGET",
          4: "MF_ERR_CUDA", 5: "MF_ERR_TIMEOUT", 6: "MF_ERR_RANGE"}

EXPORTED_SYMBOLS = ["mf_pack_plan_workspace_size", "mf_pack_plan", "mf_attn_fwd_workspace_size", "mf_attn_fwd",
                    "mf_attn_bwd_workspace_size", "mf_attn_bwd", "mf_attn_bwd_noalloc", "mf_check",
                    "mf_record_main_kernel", "mf_debug_inject", "mf_cfg_combine", "mf_norm_modulate",
                    "mf_gate_residual", "mf_attn_fwd_qkv", "mf_status_string", "mf_last_cuda_error"]

TILE = 128


class MfSample(ctypes.Structure):
    _fields_ = [("text_len", ctypes.c_int32), ("height", ctypes.c_int32), ("width", ctypes.c_int32),
                ("frames", ctypes.c_int32)]


class MfPlan(ctypes.Structure):
    _fields_ = [("n_samples", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("max_seqlen", ctypes.c_int32), ("max_grid", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_tiles", ctypes.c_int32),
                ("n_pairs", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("frame", ctypes.c_void_p),
                ("rope_axes", ctypes.c_int32), ("rope_cs", ctypes.c_void_p), ("rope_f", ctypes.c_void_p),
                ("order", ctypes.c_void_p), ("status", ctypes.c_void_p)]


class MfError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        self.code = STATUS.get(status, str(status))
        msg = f"{where}: {self.code}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


_lib = None


def lib():
    """Load libmf.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError(f"libmf.so not found at {library_path}: build it with "
                           "`python -m packed_resolution_diffusion_plan_b300.build`")
    L = ctypes.CDLL(library_path)
    c_i32, c_vp, c_sz = ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    L.mf_pack_plan_workspace_size.argtypes = [ctypes.POINTER(MfSample), c_i32, c_i32, c_i32, c_i32,
                                              ctypes.POINTER(c_sz)]
    L.mf_pack_plan.argtypes = [ctypes.POINTER(MfSample), c_i32, c_i32, c_i32, c_i32, ctypes.c_float, c_vp,
                               c_sz, ctypes.POINTER(MfPlan), c_vp]
    L.mf_attn_fwd_workspace_size.argtypes = [c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)]
    L.mf_attn_fwd.argtypes = [c_vp, c_vp, c_vp, ctypes.POINTER(MfPlan), c_i32, c_i32, ctypes.c_float,
                              c_vp, c_sz, c_vp, c_vp, c_vp]
    L.mf_attn_bwd_workspace_size.argtypes = [c_i32, c_i32, c_i32, ctypes.POINTER(c_sz)]
    L.mf_attn_bwd.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.POINTER(MfPlan), c_i32, c_i32,
                              ctypes.c_float, c_vp, c_sz, c_vp, c_vp, c_vp, c_vp]
    L.mf_check.argtypes = [ctypes.POINTER(MfPlan), c_vp]
    L.mf_record_main_kernel.argtypes = [c_vp, c_vp]
    L.mf_debug_inject.argtypes = [c_i32]
    L.mf_cfg_combine.argtypes = [c_vp, ctypes.POINTER(MfPlan), c_i32, c_i32, ctypes.c_float, c_vp, c_vp]
    L.mf_norm_modulate.argtypes = [c_vp, ctypes.POINTER(MfPlan), c_i32, c_vp, c_vp, ctypes.c_float, c_vp, c_vp]
    L.mf_gate_residual.argtypes = [c_vp, c_vp, ctypes.POINTER(MfPlan), c_i32, c_vp, c_vp, c_vp]
    L.mf_attn_fwd_qkv.argtypes = [c_vp, ctypes.POINTER(MfPlan), c_i32, c_i32, ctypes.c_float, c_vp, c_sz, c_vp,
                                  c_vp, c_vp]
    L.mf_status_string.argtypes = [c_i32]
    L.mf_status_string.restype = ctypes.c_char_p
    L.mf_last_cuda_error.argtypes = []
    L.mf_last_cuda_error.restype = ctypes.c_char_p
    for name in ("mf_pack_plan_workspace_size", "mf_pack_plan", "mf_attn_fwd_workspace_size", "mf_attn_fwd",
                 "mf_attn_bwd_workspace_size", "mf_attn_bwd", "mf_check", "mf_record_main_kernel",
                 "mf_debug_inject", "mf_cfg_combine", "mf_norm_modulate", "mf_gate_residual", "mf_attn_fwd_qkv"):
        getattr(L, name).restype = c_i32
    _lib = L
    return L


def _raise(status: int, where: str):
    if status != 0:
        detail = lib().mf_last_cuda_error().decode() if status in (4, 5) else ""
        raise MfError(status, where, detail)


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _workspace(nbytes: int, device, stream):
    """A device scratch buffer for a call enqueued on `stream`.  It is
    allocated on torch's current stream; when the call runs on another one,
    the buffer is tied to that stream too, so that the caching allocator does
    not hand it out again while the call's kernels may still use it."""
    ws = torch.empty(max(256, int(nbytes)), dtype=torch.uint8, device=device)
    if stream is not None and stream != torch.cuda.current_stream(ws.device):
        ws.record_stream(stream)
    return ws


def _samples_array(samples):
    arr = (MfSample * max(1, len(samples)))()
    for i, smp in enumerate(samples):
        t, h, w = smp[:3]
        arr[i] = MfSample(int(t), int(h), int(w), int(smp[3]) if len(smp) > 3 else 1)
    return arr


class Plan:
    """A pack plan living in a device workspace owned by this object."""

    def __init__(self, raw: MfPlan, workspace: torch.Tensor, samples, token_budget):
        self.raw = raw
        self.workspace = workspace
        self.samples = list(samples)
        self.token_budget = token_budget

    n_samples = property(lambda self: self.raw.n_samples)
    total_tokens = property(lambda self: self.raw.total_tokens)
    max_seqlen = property(lambda self: self.raw.max_seqlen)
    max_grid = property(lambda self: self.raw.max_grid)
    head_dim = property(lambda self: self.raw.head_dim)
    rope_axes = property(lambda self: self.raw.rope_axes)
    n_tiles = property(lambda self: self.raw.n_tiles)
    n_pairs = property(lambda self: self.raw.n_pairs)

    @property
    def device(self):
        return self.workspace.device

    def _view(self, ptr, count, dtype):
        off = ptr - self.workspace.data_ptr()
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype)

    def cu_seqlens(self) -> torch.Tensor:
        return self._view(self.raw.cu_seqlens, self.n_samples + 1, torch.int32)

    def pos(self) -> torch.Tensor:
        return self._view(self.raw.pos, 2 * self.total_tokens, torch.int32).view(-1, 2)

    def frame(self) -> torch.Tensor:
        """Latent frame of each token (-1 for text)."""
        return self._view(self.raw.frame, self.total_tokens, torch.int32)

    def rope_table_frame(self) -> torch.Tensor:
        """The frame slice's table of a 3-axis plan: [2, head_dim/16, 2] (cos, sin)."""
        assert self.rope_axes == 3
        n = 2 * (self.head_dim // 16) * 2
        return self._view(self.raw.rope_f, n, torch.float32).view(2, self.head_dim // 16, 2)

    def rope_table(self) -> torch.Tensor:
        """The row/col table: [max_grid, a/2, 2] (cos, sin), a = the row/col slice width."""
        nh = self.head_dim // 4 if self.rope_axes == 2 else 7 * self.head_dim // 32
        n = self.max_grid * nh * 2
        return self._view(self.raw.rope_cs, n, torch.float32).view(self.max_grid, nh, 2)

    def order(self) -> torch.Tensor:
        return self._view(self.raw.order, 4 * self.n_samples, torch.int32).view(-1, 4)


def pack_plan(samples, token_budget: int = 0, head_dim: int = 128, rope_theta: float = 10000.0,
              device=None, stream=None, rope_axes: int = 2) -> Plan:
    """Plan a pack of (text_len, height_px, width_px[, frames]) samples on the
    GPU; rope_axes 3 selects the (frame, row, col) rotation of edit packs."""
    L = lib()
    device = torch.device(device if device is not None else "cuda")
    arr = _samples_array(samples)
    nbytes = ctypes.c_size_t(0)
    _raise(L.mf_pack_plan_workspace_size(arr, len(samples), int(token_budget), int(head_dim), int(rope_axes),
                                         ctypes.byref(nbytes)), "mf_pack_plan_workspace_size")
    ws = _workspace(nbytes.value, device, stream)
    raw = MfPlan()
    _raise(L.mf_pack_plan(arr, len(samples), int(token_budget), int(head_dim), int(rope_axes), float(rope_theta),
                          ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.byref(raw),
                          _stream_ptr(stream, device)), "mf_pack_plan")
    return Plan(raw, ws, samples, token_budget)


def _check_qkv(plan: Plan, *ts):
    for t in ts:
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous bf16 CUDA tensors [T, heads, head_dim]")
        if t.dim() != 3 or t.shape[0] != plan.total_tokens or t.shape[2] != plan.head_dim:
            raise ValueError(f"expected [{plan.total_tokens}, heads, {plan.head_dim}], got {tuple(t.shape)}")
        if t.shape != ts[0].shape:
            raise ValueError("shape mismatch")


def fwd_workspace_bytes(total_tokens: int, heads: int, head_dim: int) -> int:
    n = ctypes.c_size_t(0)
    _raise(lib().mf_attn_fwd_workspace_size(total_tokens, heads, head_dim, ctypes.byref(n)),
           "mf_attn_fwd_workspace_size")
    return n.value


def attn_fwd(q, k, v, plan: Plan, softmax_scale: float = 0.0, out=None, lse=None, workspace=None,
             stream=None):
    """O, LSE of packed 2D-RoPE joint attention (see mf_attn_fwd)."""
    _check_qkv(plan, q, k, v)
    T, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(fwd_workspace_bytes(T, H, D), q.device, stream)
    _raise(lib().mf_attn_fwd(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                             ctypes.c_void_p(v.data_ptr()), ctypes.byref(plan.raw), H, D,
                             float(softmax_scale), ctypes.c_void_p(workspace.data_ptr()),
                             workspace.numel(), ctypes.c_void_p(out.data_ptr()),
                             ctypes.c_void_p(lse.data_ptr()), _stream_ptr(stream, q.device)),
           "mf_attn_fwd")
    return out, lse


def bwd_workspace_bytes(total_tokens: int, heads: int, head_dim: int) -> int:
    n = ctypes.c_size_t(0)
    _raise(lib().mf_attn_bwd_workspace_size(total_tokens, heads, head_dim, ctypes.byref(n)),
           "mf_attn_bwd_workspace_size")
    return n.value


def attn_bwd(q, k, v, o, lse, do, plan: Plan, softmax_scale: float = 0.0, workspace=None,
             dq=None, dk=None, dv=None, stream=None):
    """dQ, dK, dV of packed 2D-RoPE joint attention (see mf_attn_bwd)."""
    _check_qkv(plan, q, k, v, o, do)
    T, H, D = q.shape
    nbytes = bwd_workspace_bytes(T, H, D)
    if workspace is None:
        workspace = _workspace(nbytes, q.device, stream)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    _raise(lib().mf_attn_bwd(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                             ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                             ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(do.data_ptr()),
                             ctypes.byref(plan.raw), H, D, float(softmax_scale),
                             ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                             ctypes.c_void_p(dq.data_ptr()), ctypes.c_void_p(dk.data_ptr()),
                             ctypes.c_void_p(dv.data_ptr()), _stream_ptr(stream, q.device)),
           "mf_attn_bwd")
    return dq, dk, dv


def record_main_kernel(start=None, stop=None, stream=None):
    """Have the next attn_fwd / attn_bwd call record torch.cuda.Event `start`
    right before and `stop` right after its main tensor-core kernel.

    Both events are first recorded here on `stream` so that torch considers
    them recorded (it refuses elapsed_time otherwise); the library's own
    record during the attention call then supersedes that placeholder."""
    if start is not None and stop is not None:
        st = stream if stream is not None else torch.cuda.current_stream()
        start.record(st)
        stop.record(st)
        a, b = ctypes.c_void_p(start.cuda_event), ctypes.c_void_p(stop.cuda_event)
    else:
        a = b = None
    _raise(lib().mf_record_main_kernel(a, b), "mf_record_main_kernel")


def _check_rows(plan: Plan, *ts):
    for t in ts:
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError("expected contiguous bf16 CUDA tensors [rows, hidden]")


def norm_modulate(x, plan: Plan, shift, scale, eps: float = 1e-6, out=None, stream=None):
    """LN(x) (1 + scale_s) + shift_s per sample s (see mf_norm_modulate)."""
    _check_rows(plan, x, shift, scale)
    T, C = x.shape
    if T != plan.total_tokens or shift.shape != (plan.n_samples, C) or scale.shape != shift.shape:
        raise ValueError("x is [total_tokens, hidden], shift/scale are [n_samples, hidden]")
    out = torch.empty_like(x) if out is None else out
    _raise(lib().mf_norm_modulate(ctypes.c_void_p(x.data_ptr()), ctypes.byref(plan.raw), C,
                                  ctypes.c_void_p(shift.data_ptr()), ctypes.c_void_p(scale.data_ptr()), float(eps),
                                  ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream, x.device)), "mf_norm_modulate")
    return out


def gate_residual(x, z, plan: Plan, gate, out=None, stream=None):
    """x + gate_s * z per sample s (see mf_gate_residual)."""
    _check_rows(plan, x, z, gate)
    T, C = x.shape
    if z.shape != x.shape or T != plan.total_tokens or gate.shape != (plan.n_samples, C):
        raise ValueError("x, z are [total_tokens, hidden], gate is [n_samples, hidden]")
    out = torch.empty_like(x) if out is None else out
    _raise(lib().mf_gate_residual(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(z.data_ptr()), ctypes.byref(plan.raw),
                                  C, ctypes.c_void_p(gate.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                  _stream_ptr(stream, x.device)), "mf_gate_residual")
    return out


def attn_fwd_qkv(qkv, plan: Plan, heads: int, softmax_scale: float = 0.0, out=None, lse=None, workspace=None,
                 stream=None):
    """O, LSE from a QKV projection's output [T, 3 * heads * head_dim] (see mf_attn_fwd_qkv)."""
    _check_rows(plan, qkv)
    T, C3 = qkv.shape
    D = plan.head_dim
    if T != plan.total_tokens or C3 != 3 * heads * D:
        raise ValueError(f"expected [{plan.total_tokens}, {3 * heads * D}], got {tuple(qkv.shape)}")
    out = torch.empty((T, heads, D), dtype=torch.bfloat16, device=qkv.device) if out is None else out
    lse = torch.empty((heads, T), dtype=torch.float32, device=qkv.device) if lse is None else lse
    if workspace is None:
        workspace = _workspace(fwd_workspace_bytes(T, heads, D), qkv.device, stream)
    _raise(lib().mf_attn_fwd_qkv(ctypes.c_void_p(qkv.data_ptr()), ctypes.byref(plan.raw), heads, D,
                                 float(softmax_scale), ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                 ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                 _stream_ptr(stream, qkv.device)), "mf_attn_fwd_qkv")
    return out, lse


def cfg_combine(o, plan: Plan, guidance: float, out=None, stream=None):
    """Classifier-free guidance over (cond, uncond) sample pairs (see
    mf_cfg_combine): out's conditional image rows = u + guidance (c - u)."""
    _check_qkv(plan, o)
    T, H, D = o.shape
    if out is None:
        out = o.clone()
    _check_qkv(plan, out)
    _raise(lib().mf_cfg_combine(ctypes.c_void_p(o.data_ptr()), ctypes.byref(plan.raw), H, D, float(guidance),
                                ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream, o.device)), "mf_cfg_combine")
    return out


DEBUG_DROP_FWD_KV = 1
DEBUG_DROP_BWD_QDO = 2


def debug_inject(flags: int = 0):
    """Timeout-path test aid (see mf_debug_inject): while set, the attention
    calls of this thread drop their streamed-tile loads so that their bounded
    waits run out and check() raises MF_ERR_TIMEOUT.  0 restores normal use."""
    _raise(lib().mf_debug_inject(int(flags)), "mf_debug_inject")


def check(plan: Plan, stream=None):
    """Synchronize and raise MfError(MF_ERR_TIMEOUT) if a kernel gave up a wait."""
    _raise(lib().mf_check(ctypes.byref(plan.raw), _stream_ptr(stream, plan.device)), "mf_check")
