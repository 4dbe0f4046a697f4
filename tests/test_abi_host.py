"""Host-only checks of the C ABI: the library builds, loads and exports every
symbol the header declares; argument errors come back before any launch.
No kernel runs here (no GPU is needed)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from gated_deltanet_layer_gb300 import _native, build as B, make_config
from gated_deltanet_layer_gb300 import workloads as WL

HEADERS = [os.path.join(B.ROOT, "include", h) for h in sorted(os.listdir(os.path.join(B.ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _native.lib()


def declared_functions():
    """Every function any header under include/ declares."""
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(gdn_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_what_the_binding_binds():
    assert declared_functions() == sorted(_native.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _native.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code in range(7):
        assert lib.gdn_status_string(code)
    assert lib.gdn_status_string(99) == b"unknown status"


def _cfg(**kw):
    c = make_config(WL.SHARD)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value", [
    ("max_rows", 0), ("max_rows", 65), ("hidden", 0), ("num_slots", 0), ("ssm_dtype", 7),
    ("engine", 9), ("num_ctas", -1), ("norm_eps", float("nan")), ("launch_flags", 4), ("launch_flags", -1),
])
def test_invalid_config_has_no_workspace(lib, field, value):
    c = _cfg(**{field: value})
    assert lib.gdn_decode_workspace_bytes(ctypes.byref(c)) == 0


@pytest.mark.parametrize("field,value", [
    ("conv_kernel", 3), ("head_k_dim", 96), ("hidden", 8192 + 32), ("num_k_heads", 3),
])
def test_unsupported_shapes_refused_at_create(lib, field, value):
    c = _cfg(**{field: value})
    h = ctypes.c_void_p()
    st = lib.gdn_decode_create(ctypes.byref(c), ctypes.c_void_p(256), 1 << 30, None, ctypes.byref(h))
    assert st in (_native.GDN_ERR_UNSUPPORTED, _native.GDN_ERR_ARG)
    assert not h.value


def test_create_and_step_argument_errors(lib):
    c = _cfg()
    assert lib.gdn_decode_create(ctypes.byref(c), None, 0, None, None) == _native.GDN_ERR_ARG
    h = ctypes.c_void_p()
    assert lib.gdn_decode_create(ctypes.byref(c), None, 1 << 20, None, ctypes.byref(h)) == _native.GDN_ERR_ARG
    w = _native.Weights()
    assert lib.gdn_decode_step(None, 1, None, None, ctypes.byref(w), None, None, None, None, None,
                               None) == _native.GDN_ERR_ARG
    assert lib.gdn_decode_check(None, None, None) == _native.GDN_ERR_ARG
    assert lib.gdn_decode_reset(None, None) == _native.GDN_ERR_ARG
    lib.gdn_decode_destroy(None)  # no-op


def test_static_step_argument_errors_return_before_any_cuda_call(lib):
    # every case fails host-side validation, so no pointer below is ever used
    c = _cfg()
    P = ctypes.c_void_p
    ok, odd = P(0x10000), P(0x10001)  # placeholders: aligned / misaligned
    w = _native.Weights()
    for f in ("input_norm_w", "qkvz", "ba", "conv_w", "A_log", "dt_bias", "gated_norm_w"):
        setattr(w, f, ok.value)  # each case below has exactly one defect
    args = lambda x, idx: (1, x, None, ctypes.byref(w), idx, ok, ok, ok, ok, None, None)
    assert lib.gdn_decode_step_static(None, *args(ok, ok)) == _native.GDN_ERR_ARG       # no config
    assert lib.gdn_decode_step_static(ctypes.byref(c), 1, ok, None, None, ok, ok, ok, ok, ok, None,
                                      None) == _native.GDN_ERR_ARG                     # no weights
    assert lib.gdn_decode_step_static(ctypes.byref(c), 0, ok, None, ctypes.byref(w), ok, ok, ok, ok, ok,
                                      None, None) == _native.GDN_ERR_ARG               # rows < 1
    assert lib.gdn_decode_step_static(ctypes.byref(c), c.max_rows + 1, ok, None, ctypes.byref(w), ok, ok,
                                      ok, ok, ok, None, None) == _native.GDN_ERR_ARG   # rows > max_rows
    assert lib.gdn_decode_step_static(ctypes.byref(c), *args(None, ok)) == _native.GDN_ERR_ARG  # no x
    assert lib.gdn_decode_step_static(ctypes.byref(c), *args(ok, None)) == _native.GDN_ERR_ARG  # no indices
    assert lib.gdn_decode_step_static(ctypes.byref(c), *args(odd, ok)) == _native.GDN_ERR_ARG   # misaligned x
    mx = _cfg(qkvz_format=_native.GDN_W_MXFP4)
    assert lib.gdn_decode_step_static(ctypes.byref(mx), *args(ok, ok)) == _native.GDN_ERR_ARG  # MXFP4, no scales


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(B.ROOT, "gated_deltanet_layer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, flags=re.M), f
            if f.endswith((".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text, f


@pytest.mark.parametrize("engine", ["cuda_core", "auto"])
@pytest.mark.parametrize("shape,G", [(s, g) for s in (WL.TINY, WL.SHARD, WL.FULL, WL.SHARD_BF16)
                                     for g in (1, 7, 33, 148, 152, 160)] +
                         [(s, g) for s in (WL.DENSE_MXFP4, WL.DENSE_MXFP6) for g in (148, 152, 160)])
def test_stream_k_plan_invariants(lib, shape, G, engine):
    """The units partition [0, U) in CTA order with equal counts (within one);
    walking each CTA's units the way the kernels do (group g = u // kblock,
    tile g % T, k-step (g // T) * kblock + u % kblock) gives per tile the
    slots 0..count-1 exactly once; every unit's normed-input slot lies inside
    the CTA's window of at most 32 k-steps (24 with coded weights). A grid of
    a GB300's SMs (or near it) plans every workload; a small grid may leave a
    CTA more k-steps than its window holds, and is refused."""
    cfg = make_config(shape, engine=engine)
    if engine == "cuda_core" and shape.qkvz_format != "bf16":
        with pytest.raises(_native.GdnError):
            _native.plan(cfg, G)
        return
    try:
        P = _native.plan(cfg, G)
    except _native.GdnError:
        assert G < 148
        return
    ub, nt, KS, KB = P["unit_begin"], P["num_tiles"], P["ksteps"], P["kblock"]
    U = nt * KS
    assert ub[0] == 0 and ub[G] == U and all(a <= b for a, b in zip(ub, ub[1:]))
    counts = [ub[c + 1] - ub[c] for c in range(G)]
    assert max(counts) - min(counts) <= 1
    assert P["engine"] == (1 if engine == "cuda_core" else 2)
    slots = {t: [] for t in range(nt)}
    for c in range(G):
        seg, g_prev = -1, None
        for u in range(ub[c], ub[c + 1]):
            g = u // KB
            t, ks = g % nt, (g // nt) * KB + u % KB
            if g != g_prev:
                seg += 1
                assert seg < 16
                slots[t].append(P["seg_slot"][c][seg])
                g_prev = g
            j = (ks - P["ks_first"][c]) % KS
            assert j < P["nb_slots"][c] <= (24 if cfg.qkvz_format != _native.GDN_W_BF16 else 32)
    for t in range(nt):
        assert P["tile_count"][t] == len(slots[t]) >= 1
        assert sorted(slots[t]) == list(range(P["tile_count"][t]))


@pytest.mark.parametrize("shape", [WL.TINY, WL.SHARD, WL.FULL, WL.SHARD_BF16, WL.DENSE_MXFP4, WL.DENSE_MXFP6])
@pytest.mark.parametrize("G", [148, 152, 160])
def test_every_k_step_has_one_owner(lib, shape, G):
    """Each k-step is owned (its norm partial published, its residual_out
    written) by exactly one CTA, the first whose window holds it."""
    P = _native.plan(make_config(shape), G)
    KS, own = P["ksteps"], P["own_mask"]
    owners = [0] * KS
    for c in range(G):
        for j in range(32):
            if (own[c] >> j) & 1:
                assert j < P["nb_slots"][c]
                owners[(P["ks_first"][c] + j) % KS] += 1
    assert owners == [1] * KS
    for ks in range(KS):
        first = next(c for c in range(G) if (ks - P["ks_first"][c]) % KS < P["nb_slots"][c])
        assert (own[first] >> ((ks - P["ks_first"][first]) % KS)) & 1


@pytest.mark.parametrize("shape", [WL.TINY, WL.SHARD, WL.FULL, WL.SHARD_BF16])
def test_engines_share_the_plan(lib, shape):
    """The CUDA-core and tensor-core engines run the same units, partial slots
    and normed-input windows: they differ only in what multiplies."""
    a = _native.plan(make_config(shape, engine="cuda_core"), 152)
    b = _native.plan(make_config(shape, engine="tcgen05"), 152)
    assert (a["engine"], b["engine"]) == (1, 2)
    for k in a:
        if k != "engine":
            assert list(np.ravel(a[k])) == list(np.ravel(b[k])), k


@pytest.mark.parametrize("G", [148, 152])
def test_mxfp4_plan_is_tensor_core_only(lib, G):
    """MXFP4 in_proj_qkvz runs on the tensor-core engine (auto picks it; the
    CUDA-core engine refuses it)."""
    P = _native.plan(make_config(WL.DENSE_MXFP4), G)
    assert P["engine"] == 2
    assert P["num_tiles"] == WL.DENSE_MXFP4.n_qkvz // 256 + 1
    with pytest.raises(_native.GdnError):
        _native.plan(make_config(WL.DENSE_MXFP4, engine="cuda_core"), G)
    with pytest.raises(_native.GdnError):  # the scale loads need H % 512 == 0
        _native.plan(make_config(WL.DENSE_MXFP4.with_(hidden=5120 + 64)), G)
