"""ctypes binding of the C ABI in include/gdn_decode.h (argument marshalling only).

Every step of the decode path runs in the CUDA library libgdn_decode.so. If the
library is missing this module raises; there is no other implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgdn_decode.so")

GDN_OK, GDN_ERR_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEADLINE, GDN_ERR_INDEX, GDN_ERR_FAILED = range(7)
GDN_STATE_F32, GDN_STATE_BF16 = 0, 1
GDN_W_BF16, GDN_W_MXFP4, GDN_W_MXFP6 = 0, 1, 2
GDN_ENGINE_AUTO, GDN_ENGINE_CUDA_CORE, GDN_ENGINE_TCGEN05 = 0, 1, 2
GDN_DEBUG_SKIP_NORM_PUBLISH = 0x1
GDN_DEBUG_TIMELINE = 0x2
GDN_LAUNCH_COOPERATIVE = 0x1
GDN_LAUNCH_NO_EARLY_WEIGHTS = 0x2

# Every symbol the headers declare (include/gdn_decode.h and the diagnostics
# in include/gdn_decode_diag.h).
EXPORTS = (
    "gdn_decode_workspace_bytes", "gdn_decode_create", "gdn_decode_step", "gdn_decode_check",
    "gdn_decode_reset", "gdn_decode_destroy", "gdn_status_string", "gdn_decode_launch_info",
    "gdn_decode_plan", "gdn_decode_debug_timeline", "gdn_decode_step_static", "gdn_decode_verify",
    "gdn_decode_step_out",
)

# Size of the library's fixed device scratch (gdn_decode_step_static).
GDN_STATIC_SCRATCH_BYTES = 8 << 20


class Config(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int32), ("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
        ("head_k_dim", ctypes.c_int32), ("head_v_dim", ctypes.c_int32), ("conv_kernel", ctypes.c_int32),
        ("num_slots", ctypes.c_int32), ("max_rows", ctypes.c_int32), ("ssm_dtype", ctypes.c_int32),
        ("qkvz_format", ctypes.c_int32), ("engine", ctypes.c_int32),
        ("norm_eps", ctypes.c_float), ("gated_norm_eps", ctypes.c_float), ("l2_eps", ctypes.c_float),
        ("q_scale", ctypes.c_float), ("deadline_us", ctypes.c_uint32), ("num_ctas", ctypes.c_int32),
        ("debug_flags", ctypes.c_int32), ("launch_flags", ctypes.c_int32),
    ]


class Weights(ctypes.Structure):
    _fields_ = [
        ("input_norm_w", ctypes.c_void_p), ("qkvz", ctypes.c_void_p), ("qkvz_scales", ctypes.c_void_p),
        ("ba", ctypes.c_void_p), ("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
        ("dt_bias", ctypes.c_void_p), ("gated_norm_w", ctypes.c_void_p), ("out_proj", ctypes.c_void_p),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libgdn_decode.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    import torch  # noqa: F401  (loads the CUDA runtime first, so both share it)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u32p = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
    cfgp = ctypes.POINTER(Config)
    L.gdn_decode_workspace_bytes.argtypes = [cfgp]
    L.gdn_decode_workspace_bytes.restype = ctypes.c_size_t
    L.gdn_decode_create.argtypes = [cfgp, vp, ctypes.c_size_t, vp, ctypes.POINTER(vp)]
    L.gdn_decode_create.restype = ctypes.c_int
    L.gdn_decode_step.argtypes = [vp, i32, vp, vp, ctypes.POINTER(Weights), vp, vp, vp, vp, vp, vp]
    L.gdn_decode_step.restype = ctypes.c_int
    L.gdn_decode_step_out.argtypes = [vp, i32, vp, vp, ctypes.POINTER(Weights), vp, vp, vp, vp, vp, vp, vp]
    L.gdn_decode_step_out.restype = ctypes.c_int
    L.gdn_decode_verify.argtypes = [vp, i32, i32, vp, vp, ctypes.POINTER(Weights), vp, vp, vp, vp, vp, vp, vp]
    L.gdn_decode_verify.restype = ctypes.c_int
    L.gdn_decode_check.argtypes = [vp, vp, u32p]
    L.gdn_decode_check.restype = ctypes.c_int
    L.gdn_decode_reset.argtypes = [vp, vp]
    L.gdn_decode_reset.restype = ctypes.c_int
    L.gdn_decode_destroy.argtypes = [vp]
    L.gdn_decode_destroy.restype = None
    L.gdn_status_string.argtypes = [ctypes.c_int]
    L.gdn_status_string.restype = ctypes.c_char_p
    L.gdn_decode_launch_info.argtypes = [vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.gdn_decode_launch_info.restype = ctypes.c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    i32p = ctypes.POINTER(ctypes.c_int32)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    L.gdn_decode_plan.argtypes = [cfgp, i32, i32p, i32p, u8p, u16p, u8p, u32p, u8p, i32, i32p, i32p, i32p]
    L.gdn_decode_plan.restype = ctypes.c_int
    u64p = ctypes.POINTER(ctypes.c_uint64)
    L.gdn_decode_debug_timeline.argtypes = [vp, vp, u64p, i32, i32p]
    L.gdn_decode_debug_timeline.restype = ctypes.c_int
    L.gdn_decode_step_static.argtypes = [cfgp, i32, vp, vp, ctypes.POINTER(Weights), vp, vp, vp, vp, vp, vp,
                                         u32p]
    L.gdn_decode_step_static.restype = ctypes.c_int
    _lib = L
    return L


def plan(cfg: Config, num_ctas: int) -> dict:
    """Stream-K plan of the projection units (host-only diagnostics)."""
    L = lib()
    eng = ctypes.c_int32()
    ub = (ctypes.c_int32 * (num_ctas + 1))()
    seg = (ctypes.c_uint8 * (num_ctas * 16))()
    ksf = (ctypes.c_uint16 * num_ctas)()
    nbs = (ctypes.c_uint8 * num_ctas)()
    own = (ctypes.c_uint32 * num_ctas)()
    cap = 4096
    tc = (ctypes.c_uint8 * cap)()
    nt, ks, kb = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = L.gdn_decode_plan(ctypes.byref(cfg), num_ctas, ctypes.byref(eng), ub, seg, ksf, nbs, own, tc, cap,
                           ctypes.byref(nt), ctypes.byref(ks), ctypes.byref(kb))
    if st != GDN_OK:
        raise GdnError("gdn_decode_plan", st)
    return {"engine": eng.value, "unit_begin": list(ub),
            "seg_slot": [list(seg[c * 16:(c + 1) * 16]) for c in range(num_ctas)],
            "ks_first": list(ksf), "nb_slots": list(nbs), "own_mask": list(own), "tile_count": list(tc[:nt.value]),
            "num_tiles": nt.value, "ksteps": ks.value, "kblock": kb.value}


def status_string(code: int) -> str:
    return lib().gdn_status_string(code).decode()


class GdnError(RuntimeError):
    def __init__(self, where: str, code: int, detail: int = 0):
        self.code, self.detail = code, detail
        super().__init__(f"{where}: {status_string(code)} (status {code}, detail 0x{detail:08x})")
