"""Helpers shared by the parity tests: seeded inputs on host and device, the
CUDA path through the C ABI, the CPU oracle on the same inputs, and the
comparisons with the tolerances of the method's own checks (core cosine >=
0.9999 as in sgl-amd-mono #89 "check mode": NUMERICS k1.core.cosine).

Why not bit-exact: the kernel sums the 8192-term projections in f32 in its own
order, the oracle in float64. The absolute f32 accumulation error (~1e-5 at
these magnitudes) can exceed one bf16 ulp of a near-zero projection output, so
bf16 outputs are compared with absolute bars, and only order-free results
(residual_out, pad rows, copied conv taps, untouched slots) bit for bit."""
from __future__ import annotations

import numpy as np
import torch

from gated_deltanet_layer_gb300 import workloads as WL

# Tolerances (core: cosine and max-abs; states: max-abs; residual_out and pad
# handling: bit-exact).
CORE_COS = 0.9999
CORE_MAX_ABS = 2e-2
STATE_F32_MAX_ABS = 1e-3
STATE_BF16_MAX_ABS = 1e-2
# The conv state's new tap is the bf16 projection output: within one bf16 ulp
# of the oracle's value (one rounding step either way), plus an absolute floor
# that covers the f32 accumulation error of an 8192-term dot product near zero
# (typical size 1e-5, floor 2e-3); and at most 2% of the taps may differ.
CONV_NEW_TAP_FLOOR = 2e-3


def f64(t):
    if t is None:
        return None
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.to(torch.float64).cpu().numpy()


class Case:
    """One layer + state + step on the host, and their device copies."""

    def __init__(self, shape, rows, seed, *, first_layer=False, pad_rows=0, weights=None, state=None,
                 step=None, **wkw):
        self.shape, self.rows = shape, rows
        self.w = weights if weights is not None else WL.make_weights(shape, seed, **wkw)
        self.st = state if state is not None else WL.make_state(shape, seed + 1)
        self.step = step if step is not None else WL.make_step(shape, rows, seed + 2,
                                                               first_layer=first_layer, pad_rows=pad_rows)

    def to_device(self):
        self.dw = {k: (v.cuda() if v is not None else None) for k, v in self.w.items()}
        self.dconv = self.st["conv_state"].cuda()
        self.dssm = self.st["ssm_state"].cuda()
        self.dx = self.step["x"].cuda()
        self.dres = self.step["residual"].cuda() if self.step["residual"] is not None else None
        self.didx = self.step["state_indices"].cuda()
        return self

    def run_gpu(self, layer):
        core, res_out = layer.step(self.dx, self.dres, self.dw, self.didx, self.dconv, self.dssm)
        torch.cuda.synchronize()
        return core, res_out

    def run_oracle(self):
        from oracle import gdn_oracle as O
        wn = {k: f64(v) for k, v in self.w.items()}
        return O.gdn_step(self.shape, f64(self.step["x"]), f64(self.step["residual"]), wn,
                          self.step["state_indices"].numpy(), f64(self.st["conv_state"]),
                          f64(self.st["ssm_state"]))


def cosine(a, b):
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def bf16_ulp(v):
    v = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(np.where(v == 0, 1.0, v))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def compare(case, ref, core, res_out, *, state_tol=None):
    """Assert the GPU outputs of `case` (already run) against the oracle `ref`."""
    shape = case.shape
    idx = case.step["state_indices"].numpy()
    live = [(r, int(s)) for r, s in enumerate(idx) if 0 < s < shape.num_slots]
    np.testing.assert_array_equal(f64(res_out), ref["residual_out"], err_msg="residual_out")
    gcore = f64(core)
    for r, s in enumerate(idx):
        if not (0 < s < shape.num_slots):
            assert np.all(gcore[r] == 0.0), f"pad row {r} core not zero"
    if live:
        rows = [r for r, _ in live]
        c = cosine(gcore[rows], ref["core"][rows])
        m = float(np.max(np.abs(gcore[rows] - ref["core"][rows])))
        assert c >= CORE_COS, f"core cosine {c}"
        assert m <= CORE_MAX_ABS, f"core max-abs {m}"
    gconv, gssm = f64(case.dconv), f64(case.dssm)
    conv0, ssm0 = f64(case.st["conv_state"]), f64(case.st["ssm_state"])
    touched = sorted(s for _, s in live)
    untouched = [s for s in range(shape.num_slots) if s not in touched]
    np.testing.assert_array_equal(gconv[untouched], conv0[untouched], err_msg="untouched conv slots")
    np.testing.assert_array_equal(gssm[untouched], ssm0[untouched], err_msg="untouched ssm slots")
    if touched:
        # the two older taps are copies of the previous state: bit-exact; the
        # new tap is the bf16 projection output: within the bf16-state bar
        np.testing.assert_array_equal(gconv[touched][..., :-1], ref["conv_state"][touched][..., :-1],
                                      err_msg="shifted conv taps")
        g_new, r_new = gconv[touched][..., -1], ref["conv_state"][touched][..., -1]
        excess = np.abs(g_new - r_new) - (bf16_ulp(r_new) + CONV_NEW_TAP_FLOOR)
        assert np.all(excess <= 0), f"conv state new tap beyond 1 ulp + floor by {float(excess.max())}"
        assert np.mean(g_new != r_new) <= 0.02, f"conv new tap mismatch rate {np.mean(g_new != r_new)}"
        tol = state_tol if state_tol is not None else (
            STATE_BF16_MAX_ABS if shape.ssm_dtype == "bf16" else STATE_F32_MAX_ABS)
        m = float(np.max(np.abs(gssm[touched] - ref["ssm_state"][touched])))
        assert m <= tol, f"ssm state max-abs {m}"
    return True
