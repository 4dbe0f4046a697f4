"""GB300-native decode-step front of a Gated DeltaNet layer.

`GdnDecode` wraps the C ABI of libgdn_decode.so (include/gdn_decode.h) for
torch CUDA tensors: it allocates the workspace with torch, marshals pointers
and streams, and launches one persistent CUDA kernel per step. It computes
nothing itself and has no fallback: without the built library it raises.
"""
from __future__ import annotations

import ctypes

from . import _native
from ._native import (GDN_ENGINE_AUTO, GDN_ENGINE_CUDA_CORE, GDN_ENGINE_TCGEN05, GDN_OK,
                      GDN_STATE_BF16, GDN_STATE_F32, GDN_W_BF16, GDN_W_MXFP4, GDN_W_MXFP6, GdnError)

_FORMATS = {"bf16": GDN_W_BF16, "mxfp4": GDN_W_MXFP4, "mxfp6": GDN_W_MXFP6}

__all__ = ["GdnDecode", "GdnError", "ENGINES", "step_static"]

ENGINES = {"auto": GDN_ENGINE_AUTO, "cuda_core": GDN_ENGINE_CUDA_CORE, "tcgen05": GDN_ENGINE_TCGEN05}
_WEIGHT_KEYS = ("input_norm_w", "qkvz", "qkvz_scales", "ba", "conv_w", "A_log", "dt_bias", "gated_norm_w",
                "out_proj")


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def make_config(shape, *, engine: str = "auto", deadline_us: int = 0, num_ctas: int = 0,
                debug_flags: int = 0, max_rows: int | None = None, launch_flags: int = 0) -> _native.Config:
    """C config from a layer description (any object with the LayerShape fields)."""
    q_scale = shape.q_scale if shape.q_scale is not None else float(shape.head_k_dim) ** -0.5
    return _native.Config(
        hidden=shape.hidden, num_k_heads=shape.num_k_heads, num_v_heads=shape.num_v_heads,
        head_k_dim=shape.head_k_dim, head_v_dim=shape.head_v_dim, conv_kernel=shape.conv_kernel,
        num_slots=shape.num_slots, max_rows=max_rows or shape.max_rows,
        ssm_dtype=GDN_STATE_BF16 if shape.ssm_dtype == "bf16" else GDN_STATE_F32,
        qkvz_format=_FORMATS[shape.qkvz_format],
        engine=ENGINES[engine], norm_eps=shape.norm_eps, gated_norm_eps=shape.gated_norm_eps,
        l2_eps=shape.l2_eps, q_scale=q_scale, deadline_us=deadline_us, num_ctas=num_ctas,
        debug_flags=debug_flags, launch_flags=launch_flags)


class GdnDecode:
    """A GDN layer front's decode step, bound to one workspace on one device."""

    def __init__(self, shape, *, engine: str = "auto", deadline_us: int = 0, num_ctas: int = 0,
                 debug_flags: int = 0, max_rows: int | None = None, launch_flags: int = 0, stream=None):
        import torch
        L = _native.lib()
        self.shape = shape
        self.cfg = make_config(shape, engine=engine, deadline_us=deadline_us, num_ctas=num_ctas,
                               debug_flags=debug_flags, max_rows=max_rows, launch_flags=launch_flags)
        n = L.gdn_decode_workspace_bytes(ctypes.byref(self.cfg))
        if n == 0:
            raise GdnError("gdn_decode_workspace_bytes", _native.GDN_ERR_UNSUPPORTED)
        self.workspace = torch.empty(n, dtype=torch.uint8, device="cuda")
        h = ctypes.c_void_p()
        st = L.gdn_decode_create(ctypes.byref(self.cfg), _ptr(self.workspace), n, _stream_ptr(stream),
                                 ctypes.byref(h))
        if st != GDN_OK:
            raise GdnError("gdn_decode_create", st)
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _native.lib().gdn_decode_destroy(h)
            self._h = None

    def launch_info(self, rows: int):
        n, e = ctypes.c_int32(), ctypes.c_int32()
        st = _native.lib().gdn_decode_launch_info(self._h, rows, ctypes.byref(n), ctypes.byref(e))
        if st != GDN_OK:
            raise GdnError("gdn_decode_launch_info", st)
        return n.value, e.value

    @staticmethod
    def weights_struct(weights: dict) -> _native.Weights:
        return _native.Weights(**{k: (weights[k].data_ptr() if weights.get(k) is not None else None)
                                  for k in _WEIGHT_KEYS})

    def step(self, x, residual, weights: dict, state_indices, conv_state, ssm_state,
             core_out=None, residual_out=None, stream=None, weights_struct=None):
        """One decode step. Tensors must be contiguous CUDA tensors in the
        layouts of include/gdn_decode.h. Returns (core_out, residual_out)."""
        import torch
        rows = x.shape[0]
        if core_out is None:
            core_out = torch.empty(rows, self.shape.num_v_heads * self.shape.head_v_dim,
                                   dtype=torch.bfloat16, device=x.device)
        if residual_out is None:
            residual_out = torch.empty_like(x)
        for t in (x, residual, state_indices, conv_state, ssm_state, core_out, residual_out):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("tensors must be contiguous CUDA tensors")
        ws = weights_struct if weights_struct is not None else self.weights_struct(weights)
        st = _native.lib().gdn_decode_step(
            self._h, rows, _ptr(x), _ptr(residual), ctypes.byref(ws), _ptr(state_indices),
            _ptr(conv_state), _ptr(ssm_state), _ptr(core_out), _ptr(residual_out), _stream_ptr(stream))
        if st != GDN_OK:
            raise GdnError("gdn_decode_step", st)
        return core_out, residual_out

    def step_out(self, x, residual, weights: dict, state_indices, conv_state, ssm_state,
                 core_out=None, residual_out=None, out=None, stream=None, weights_struct=None):
        """A decode step followed by out_proj in the same launch (weights must
        hold "out_proj" [H, Hv*dv] bf16). Returns (core_out, residual_out, out)."""
        import torch
        rows = x.shape[0]
        if core_out is None:
            core_out = torch.empty(rows, self.shape.num_v_heads * self.shape.head_v_dim,
                                   dtype=torch.bfloat16, device=x.device)
        if residual_out is None:
            residual_out = torch.empty_like(x)
        if out is None:
            out = torch.empty_like(x)
        for t in (x, residual, state_indices, conv_state, ssm_state, core_out, residual_out, out):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("tensors must be contiguous CUDA tensors")
        ws = weights_struct if weights_struct is not None else self.weights_struct(weights)
        st = _native.lib().gdn_decode_step_out(
            self._h, rows, _ptr(x), _ptr(residual), ctypes.byref(ws), _ptr(state_indices),
            _ptr(conv_state), _ptr(ssm_state), _ptr(core_out), _ptr(residual_out), _ptr(out), _stream_ptr(stream))
        if st != GDN_OK:
            raise GdnError("gdn_decode_step_out", st)
        return core_out, residual_out, out

    def verify(self, x, residual, weights: dict, state_in, state_out, conv_state, ssm_state,
               core_out=None, residual_out=None, stream=None, weights_struct=None):
        """A verify step: state_in [S] int32, state_out [S, T] int32 (one slot
        per token), x [S*T, H] (sequence-major). Returns (core_out, residual_out)."""
        import torch
        S, T = state_out.shape
        rows = x.shape[0]
        if rows != S * T or state_in.shape[0] != S:
            raise ValueError("x must have S*T rows and state_in S entries")
        if core_out is None:
            core_out = torch.empty(rows, self.shape.num_v_heads * self.shape.head_v_dim,
                                   dtype=torch.bfloat16, device=x.device)
        if residual_out is None:
            residual_out = torch.empty_like(x)
        for t in (x, residual, state_in, state_out, conv_state, ssm_state, core_out, residual_out):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("tensors must be contiguous CUDA tensors")
        ws = weights_struct if weights_struct is not None else self.weights_struct(weights)
        st = _native.lib().gdn_decode_verify(
            self._h, S, T, _ptr(x), _ptr(residual), ctypes.byref(ws), _ptr(state_in), _ptr(state_out),
            _ptr(conv_state), _ptr(ssm_state), _ptr(core_out), _ptr(residual_out), _stream_ptr(stream))
        if st != GDN_OK:
            raise GdnError("gdn_decode_verify", st)
        return core_out, residual_out

    def timeline(self, stream=None):
        """Phase stamps of the last step (handle made with GDN_DEBUG_TIMELINE):
        per-CTA [G][48] nanosecond stamps as nested lists."""
        L = _native.lib()
        cap_c = 256 * 48
        cs = (ctypes.c_uint64 * cap_c)()
        g = ctypes.c_int32()
        st = L.gdn_decode_debug_timeline(self._h, _stream_ptr(stream), cs, cap_c, ctypes.byref(g))
        if st != GDN_OK:
            raise GdnError("gdn_decode_debug_timeline", st)
        return [list(cs[i * 48:(i + 1) * 48]) for i in range(g.value)]

    def check(self, stream=None):
        """(status, detail word) of the sticky device error word; synchronises."""
        d = ctypes.c_uint32()
        st = _native.lib().gdn_decode_check(self._h, _stream_ptr(stream), ctypes.byref(d))
        return st, d.value

    def reset(self, stream=None):
        st = _native.lib().gdn_decode_reset(self._h, _stream_ptr(stream))
        if st != GDN_OK:
            raise GdnError("gdn_decode_reset", st)


def step_static(shape, x, residual, weights, state_indices, conv_state, ssm_state, core_out, residual_out,
                *, stream=None, check: bool = False, engine: str = "auto", deadline_us: int = 0,
                num_ctas: int = 0, debug_flags: int = 0, max_rows: int | None = None, launch_flags: int = 0):
    """One decode step through gdn_decode_step_static, for callers that cannot
    allocate device memory: the library's fixed device scratch stands in for
    the workspace and there is no handle. Every tensor, outputs included, is
    the caller's; this call allocates nothing. `weights` is a dict of tensors
    or a prepared `_native.Weights`. With check=True the call waits for the
    launch and returns (status, detail word) of the device error word (read
    and cleared); else it returns None."""
    for t in (x, residual, state_indices, conv_state, ssm_state, core_out, residual_out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    cfg = make_config(shape, engine=engine, deadline_us=deadline_us, num_ctas=num_ctas,
                      debug_flags=debug_flags, max_rows=max_rows, launch_flags=launch_flags)
    ws = weights if isinstance(weights, _native.Weights) else GdnDecode.weights_struct(weights)
    d = ctypes.c_uint32()
    st = _native.lib().gdn_decode_step_static(
        ctypes.byref(cfg), x.shape[0], _ptr(x), _ptr(residual), ctypes.byref(ws), _ptr(state_indices),
        _ptr(conv_state), _ptr(ssm_state), _ptr(core_out), _ptr(residual_out), _stream_ptr(stream),
        ctypes.byref(d) if check else None)
    if check and st in (GDN_OK, _native.GDN_ERR_DEADLINE, _native.GDN_ERR_INDEX, _native.GDN_ERR_FAILED):
        return st, d.value
    if st != GDN_OK:
        raise GdnError("gdn_decode_step_static", st)
    return None
