"""CPU oracle for the decode-step front of a Gated DeltaNet (GDN) layer.

TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import or run this module. The library's
product path (the CUDA kernels behind the C ABI and their Python binding)
never calls it, and this module shares no code with that path: it imports
numpy only.

What one step computes, row by row (the step list of sgl-amd-mono #89
"Run each GDN layer's front as one K1 launch", Modifications table, gdn.py
row; vLLM #60833 "Qwen3.8-2.4T specialized decode on MI355X", Details,
Launches; SGLang #43558 "Qwen3.8-27B dense mono decode", Modifications, K1):

  1. residual add                       r  = x + residual     (first layer: r = x)
  2. Gemma RMSNorm                      xn = r * rstd * (1 + w_in),
                                        rstd = 1 / sqrt(mean(r^2) + eps)
  3. in_proj_qkvz, in_proj_ba           p  = W xn   (bf16, MXFP4 or MXFP6 weights)
  4. split                              p -> q | k | v | z   and  b | a
  5. causal depthwise conv1d + SiLU     over the q, k, v channels, state update
  6. L2 norm of q and k per key head    (q also times q_scale)
  7. gates                              g = -exp(A_log) softplus(a + dt_bias),
                                        beta = sigmoid(b)
  8. gated delta rule on the slot state S <- e^g S;  S += k (x) beta (v - S^T k);
                                        o = S^T q
  9. gated RMSNorm over the head        core = rmsnorm(o) * w_g * silu(z)
  10. (with out_proj weights) out_proj   out = W_o core   over the Hv*dv core columns
  Pad rows (state index <= 0) write a zero core row and no state.

Arithmetic: float64 throughout. Values are rounded to their storage type
exactly where the layer stores them: bf16 for residual_out, the normed input
xn, the projection outputs (they also enter the bf16 conv state), a bf16 SSM
state and the core output; f32 for an f32 SSM state. The conv output, q, k,
v, the gates and the recurrence stay in float64. Each rounding is a single
round-to-nearest-even of the float64 value.

Layouts (the library's documented layouts):
  W_qkvz rows  [q (Hk*dk) | k (Hk*dk) | v (Hv*dv) | z (Hv*dv)]
  W_ba rows    [b (Hv) | a (Hv)]
  conv state   [slot][channel][tap], oldest tap first; conv weight [channel][tap],
               the last tap multiplies the new input; channels are q | k | v
  SSM state    [slot][value head][v][k]   (S[v][k], k innermost)
  value head h reads key head h // (Hv / Hk)

Parity status: every function below is pinned by the CPU tests against
closed forms, hand-worked values, brute force or library routines (see
tests/test_oracle_pins.py); the split's slices are pinned index by index
against the documented row layout and through whole steps whose core and
state depend on z and a alone.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_round", "f32_round", "silu", "softplus", "sigmoid",
    "residual_add", "gemma_rmsnorm", "project_bf16", "e2m1_value",
    "mxfp4_unpack_codes", "mxfp4_quantize_block", "mxfp4_quantize_row",
    "project_mxfp4", "e2m3_value", "mxfp6_quantize_block", "mxfp6_quantize_matrix",
    "mxfp6_pack", "mxfp6_unpack", "project_mxfp6", "split_projection", "conv_update", "l2norm",
    "gates", "delta_rule", "gated_rmsnorm", "out_proj", "gdn_step", "gdn_verify",
]

# --------------------------------------------------------------------------
# Rounding to storage types
# --------------------------------------------------------------------------

_BF16_MAX = float.fromhex("0x1.fep127")  # largest finite bf16


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits (1 implicit + 7 stored) with the f32
    exponent range; below 2^-126 the spacing is fixed at 2^-133. The result
    is returned as float64 holding the exact bf16 value.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    m, e = np.frexp(x[nz])  # x = m * 2^e with 0.5 <= |m| < 1
    quantum_exp = np.maximum(e - 8, -133)  # spacing of bf16 values near x
    q = np.ldexp(np.ones_like(m), quantum_exp)
    r = np.rint(x[nz] / q) * q  # np.rint rounds halves to even
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, r), r)
    out[nz] = r
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    out[x == 0] = x[x == 0]
    return out


def f32_round(x) -> np.ndarray:
    """Round float64 values to the nearest float32, ties to even."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def silu(t):
    t = np.asarray(t, dtype=np.float64)
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def sigmoid(t):
    t = np.asarray(t, dtype=np.float64)
    with np.errstate(over="ignore"):  # exp overflow to inf gives the exact limit 0
        return 1.0 / (1.0 + np.exp(-t))


def softplus(t, threshold: float = 20.0):
    """log(1 + e^t), taken as t itself above the threshold."""
    t = np.asarray(t, dtype=np.float64)
    return np.where(t > threshold, t, np.log1p(np.exp(np.minimum(t, threshold))))


# --------------------------------------------------------------------------
# Steps 1-2: residual add and Gemma RMSNorm
# (sgl-amd-mono #89, "Kernels before and after" table: the residual add and
#  the input norm, a Gemma fused add + RMSNorm, plain Gemma RMSNorm on the
#  first layer; SGLang #43558 commit text: rstd = 1 / sqrt(sum / n + eps))
# --------------------------------------------------------------------------

def residual_add(x, residual):
    """r = bf16(x + residual); the first layer (residual None) passes x on."""
    x = np.asarray(x, dtype=np.float64)
    if residual is None:
        return x.copy()
    return bf16_round(x + np.asarray(residual, dtype=np.float64))


def gemma_rmsnorm(r, w_in, eps: float):
    """xn = bf16(r * rstd * (1 + w_in)) with rstd = 1/sqrt(mean(r^2) + eps),
    the mean taken over the last axis."""
    r = np.asarray(r, dtype=np.float64)
    ms = np.mean(r * r, axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(ms + eps)
    return bf16_round(r * rstd * (1.0 + np.asarray(w_in, dtype=np.float64)))


# --------------------------------------------------------------------------
# Step 3: projections
# (sgl-amd-mono #89, Modifications: in_proj_qkvz and in_proj_ba; SGLang
#  #43558, Exact by construction / the fp4 argument: an fp4 x fp4 product
#  scaled by e8m0 codes is exact, and the stock result is bf16 of the exact
#  sum -- the oracle takes the exact sum and rounds it once)
# --------------------------------------------------------------------------

def project_bf16(xn, W):
    """p[w, n] = bf16(sum_h W[n, h] * xn[w, h]); products of bf16 values are
    exact in float64 and the float64 sum is rounded once to bf16."""
    xn = np.asarray(xn, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    return bf16_round(xn @ W.T)


def e2m1_value(code):
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1, mantissa
    bit 0, exponent bias 1; exponent field 0 is subnormal (0 or 0.5)."""
    code = np.asarray(code, dtype=np.int64)
    s = np.where((code >> 3) & 1, -1.0, 1.0)
    e = (code >> 1) & 3
    m = code & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return s * mag


def mxfp4_unpack_codes(packed):
    """[..., K/2] bytes -> [..., K] codes; element 2i is the low nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0x0F
    hi = packed >> 4
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def _e2m1_round_magnitude(a):
    """Round non-negative magnitudes to the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6},
    ties to even code, saturating at 6."""
    a = np.asarray(a, dtype=np.float64)
    # grid spacing: 0.5 below 2, 1 in [2, 4), 2 in [4, 6]
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    q = np.rint(a / step) * step  # ties to even multiple of the step = even code
    return np.minimum(q, 6.0)


def _magnitude_to_code(q):
    table = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
    return np.vectorize(lambda v: table[float(v)], otypes=[np.int64])(q)


def mxfp4_quantize_block(v):
    """Dynamic MXFP4 quantisation of one block of 32 values.

    Scale (by analogy with the E2M3 rule of vLLM #60833, review comment "How
    to make the MXFP6 weights", step 2, which follows the same dynamic MXFP
    quantiser with the element type's maximum): take the block maximum |v|,
    round its f32 mantissa to 1 bit (half up: a carry moves the exponent),
    keep only the exponent E, and use 2^(E - 2) as the scale, E - 2 clamped
    to [-126, 127] so that the scale is always a normal f32 (an all-zero
    block, whose maximum has exponent field 0, gets 2^-126); E2M1's largest
    exponent is 2. Elements: |v| / scale rounded to the E2M1 grid, ties to
    even, saturating at 6.

    Returns (codes [32] uint8, scale exponent int, e8m0 byte).
    """
    v = np.asarray(v, dtype=np.float64)
    amax = np.float32(np.max(np.abs(v)))
    bits = int(amax.view(np.uint32))
    # half-up rounding of the mantissa to 1 bit: add half of the kept bit's
    # weight (2^21 in the 23-bit field); a carry moves into the exponent.
    e_field = ((bits + (1 << 21)) >> 23) & 0xFF
    exp = e_field - 127 - 2
    exp = int(min(max(exp, -126), 127))
    scale = math.ldexp(1.0, exp)
    mag = _e2m1_round_magnitude(np.abs(v) / scale)
    codes = _magnitude_to_code(mag)
    codes = np.where(np.signbit(v) & (mag > 0), codes | 8, codes).astype(np.uint8)
    return codes, exp, exp + 127


def mxfp4_quantize_row(x):
    """Quantise a row (length a multiple of 32) block by block.
    Returns (codes [K] uint8, exponents [K/32] int)."""
    x = np.asarray(x, dtype=np.float64)
    K = x.shape[-1]
    codes = np.empty(K, dtype=np.uint8)
    exps = np.empty(K // 32, dtype=np.int64)
    for b in range(K // 32):
        c, e, _ = mxfp4_quantize_block(x[32 * b:32 * b + 32])
        codes[32 * b:32 * b + 32] = c
        exps[b] = e
    return codes, exps


def project_mxfp4(xn, w_packed, w_scales):
    """W4A4 MXFP4 projection (vLLM #60833, Details, "x without an LDS tile" and
    "MXFP4 layouts"; SGLang #43558, the fp4 exactness argument).

    Each row of xn is quantised per block of 32 (mxfp4_quantize_row); the
    weight codes carry one e8m0 scale byte per 32 elements (2^(byte - 127)).
    p[w, n] = bf16(sum over blocks of 2^(sw + sx) * sum_j e2m1(w) e2m1(x)),
    the sum exact in float64.
    """
    xn = np.asarray(xn, dtype=np.float64)
    wc = e2m1_value(mxfp4_unpack_codes(w_packed))  # [N, K]
    ws = np.ldexp(1.0, np.asarray(w_scales, dtype=np.int64) - 127)  # [N, K/32]
    W = wc * np.repeat(ws, 32, axis=1)
    out = np.empty((xn.shape[0], W.shape[0]))
    for w in range(xn.shape[0]):
        c, e = mxfp4_quantize_row(xn[w])
        xq = e2m1_value(c) * np.repeat(np.ldexp(1.0, e), 32)
        out[w] = W @ xq
    return bf16_round(out)


# --------------------------------------------------------------------------
# MXFP6 E2M3 weights with bf16 activations (W6A16): vLLM #60833, review
# comment "How to make the MXFP6 weights". Step 2 there rounds each bf16
# weight, one block of 32 along K at a time, to its E2M3 value times a
# power-of-two block scale; step 3 packs the codes (sign at bit 5, then two
# exponent and three mantissa bits) 32 to 24 bytes, code i at bits 6i to
# 6i + 5 in little-endian order, with one e8m0 byte per block. The
# activations stay bf16; decoded weights are exact in bf16.
# --------------------------------------------------------------------------

def e2m3_value(code):
    """Value of a 6-bit E2M3 code: sign bit 5, exponent bits 4..3 with bias
    1, mantissa bits 2..0; exponent field 0 is subnormal (m / 8)."""
    code = np.asarray(code, dtype=np.int64)
    s = np.where((code >> 5) & 1, -1.0, 1.0)
    e = (code >> 3) & 3
    m = code & 7
    mag = np.where(e == 0, m / 8.0, np.ldexp(1.0 + m / 8.0, e - 1))
    return s * mag


def _e2m3_round_magnitude(a):
    """Round non-negative magnitudes to the E2M3 grid (steps of 1/8 below 2,
    1/4 in [2, 4), 1/2 from 4), ties to even, saturating at 7.5."""
    a = np.asarray(a, dtype=np.float64)
    step = np.where(a < 2.0, 0.125, np.where(a < 4.0, 0.25, 0.5))
    return np.minimum(np.rint(a / step) * step, 7.5)


def _e2m3_code(q):
    """Code of a non-negative E2M3 grid value q."""
    q = np.asarray(q, dtype=np.float64)
    sub = q < 1.0
    e = np.where(sub, 0, np.floor(np.log2(np.where(sub, 1.0, q))).astype(np.int64) + 1)
    m = np.where(sub, np.rint(q * 8.0), np.rint((q / np.ldexp(1.0, e - 1) - 1.0) * 8.0))
    return (e << 3 | m.astype(np.int64)).astype(np.int64)


def mxfp6_quantize_block(v):
    """One block of 32 values to E2M3 codes and a block scale.

    Scale: the block maximum |v| as f32, its mantissa rounded at the third
    bit (2^19 added to its bits: a carry moves the exponent), exponent E kept;
    the scale is 2^(E - 2), E - 2 clamped to [-126, 127] so an all-zero
    block keeps a normal scale. Elements: |v| / scale rounded to the E2M3
    grid, ties to even, saturating at 7.5.

    Returns (codes [32] uint8, scale exponent int, e8m0 byte)."""
    v = np.asarray(v, dtype=np.float64)
    amax = np.float32(np.max(np.abs(v)))
    bits = int(amax.view(np.uint32))
    e_field = ((bits + (1 << 19)) >> 23) & 0xFF
    exp = int(min(max(e_field - 127 - 2, -126), 127))
    mag = _e2m3_round_magnitude(np.abs(v) / math.ldexp(1.0, exp))
    codes = _e2m3_code(mag)
    codes = np.where(np.signbit(v) & (mag > 0), codes | 32, codes).astype(np.uint8)
    return codes, exp, exp + 127


def mxfp6_quantize_matrix(W):
    """[N, K] weights (K a multiple of 32) to E2M3 codes [N, K] and e8m0
    scale bytes [N, K/32]: mxfp6_quantize_block's steps applied to every
    block of 32 along K at once."""
    W = np.asarray(W, dtype=np.float64)
    N, K = W.shape
    v = W.reshape(N, K // 32, 32)
    amax = np.max(np.abs(v), axis=-1).astype(np.float32)
    bits = amax.view(np.uint32).astype(np.int64)
    e_field = ((bits + (1 << 19)) >> 23) & 0xFF
    exp = np.clip(e_field - 127 - 2, -126, 127)
    mag = _e2m3_round_magnitude(np.abs(v) / np.ldexp(1.0, exp)[..., None])
    codes = _e2m3_code(mag)
    codes = np.where(np.signbit(v) & (mag > 0), codes | 32, codes).astype(np.uint8)
    return codes.reshape(N, K), (exp + 127).astype(np.uint8)


def mxfp6_pack(codes):
    """[..., K] 6-bit codes to [..., 3K/4] bytes: each block of 32 codes
    is a 192-bit little-endian number with code i at bits 6i..6i+5."""
    codes = np.asarray(codes, dtype=np.uint64)
    lead, K = codes.shape[:-1], codes.shape[-1]
    blocks = codes.reshape(-1, K // 32, 32)
    out = np.zeros(blocks.shape[:2] + (24,), dtype=np.uint8)
    for i in range(32):
        for bit in range(6):
            pos = 6 * i + bit
            out[..., pos // 8] |= (((blocks[..., i] >> np.uint64(bit)) & np.uint64(1)) << np.uint64(pos % 8)).astype(np.uint8)
    return out.reshape(lead + (K // 32 * 24,))


def mxfp6_unpack(packed):
    """Inverse of mxfp6_pack: [..., 3K/4] bytes to [..., K] codes."""
    packed = np.asarray(packed, dtype=np.uint8)
    lead, nb = packed.shape[:-1], packed.shape[-1]
    groups = packed.reshape(-1, nb // 24, 24)
    codes = np.zeros(groups.shape[:2] + (32,), dtype=np.uint8)
    for i in range(32):
        for bit in range(6):
            pos = 6 * i + bit
            codes[..., i] |= ((groups[..., pos // 8] >> (pos % 8)) & 1).astype(np.uint8) << bit
    return codes.reshape(lead + (nb // 24 * 32,))


def project_mxfp6(xn, w_packed, w_scales):
    """W6A16 projection: p[w, n] = bf16(sum_h e2m3(W[n, h]) 2^(s[n, h/32] - 127)
    xn[w, h]) with bf16 activations, the sum taken in float64 and rounded once."""
    xn = np.asarray(xn, dtype=np.float64)
    wv = e2m3_value(mxfp6_unpack(w_packed))  # [N, K]
    ws = np.ldexp(1.0, np.asarray(w_scales, dtype=np.int64) - 127)
    W = wv * np.repeat(ws, 32, axis=1)
    return bf16_round(xn @ W.T)


# --------------------------------------------------------------------------
# Step 4: split of the projection outputs (sgl-amd-mono #89, "Kernels before
# and after": the split of the projection output is its own stock kernel)
# --------------------------------------------------------------------------

def split_projection(p_qkvz, p_ba, Hk, Hv, dk, dv):
    """Planar split: q, k [W, Hk, dk]; v, z [W, Hv, dv]; b, a [W, Hv]."""
    Wr = p_qkvz.shape[0]
    o = 0
    q = p_qkvz[:, o:o + Hk * dk].reshape(Wr, Hk, dk); o += Hk * dk
    k = p_qkvz[:, o:o + Hk * dk].reshape(Wr, Hk, dk); o += Hk * dk
    v = p_qkvz[:, o:o + Hv * dv].reshape(Wr, Hv, dv); o += Hv * dv
    z = p_qkvz[:, o:o + Hv * dv].reshape(Wr, Hv, dv)
    b = p_ba[:, :Hv]
    a = p_ba[:, Hv:2 * Hv]
    return q, k, v, z, b, a


# --------------------------------------------------------------------------
# Step 5: causal depthwise conv1d update + SiLU (sgl-amd-mono #89: the conv
# update is a stock kernel; refusals: no conv bias, SiLU required; conv state
# bf16)
# --------------------------------------------------------------------------

def conv_update(conv_state_slot, conv_w, u):
    """One decode step of a causal depthwise conv of kernel K over channels.

    conv_state_slot [C, K-1] holds the previous K-1 inputs, oldest first;
    conv_w [C, K]; u [C] the new input. Output y[c] = silu(sum_j w[c, j] *
    window[c, j]) with window = [state, u]; the new state drops the oldest
    input and appends u. Returns (y float64 [C], new state [C, K-1])."""
    s = np.asarray(conv_state_slot, dtype=np.float64)
    w = np.asarray(conv_w, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    window = np.concatenate([s, u[:, None]], axis=1)  # [C, K]
    y = silu(np.sum(w * window, axis=1))
    return y, window[:, 1:].copy()


# --------------------------------------------------------------------------
# Steps 6-7: L2 norm and gates
# --------------------------------------------------------------------------

def l2norm(t, eps: float):
    """t / sqrt(sum(t^2) + eps) over the last axis."""
    t = np.asarray(t, dtype=np.float64)
    return t / np.sqrt(np.sum(t * t, axis=-1, keepdims=True) + eps)


def gates(a, b, A_log, dt_bias):
    """g = -exp(A_log) * softplus(a + dt_bias); beta = sigmoid(b).
    (sgl-amd-mono #89 refusals: A_log f32, dt_bias bf16.)"""
    a = np.asarray(a, dtype=np.float64)
    g = -np.exp(np.asarray(A_log, dtype=np.float64)) * softplus(a + np.asarray(dt_bias, dtype=np.float64))
    beta = sigmoid(b)
    return g, beta


# --------------------------------------------------------------------------
# Step 8: gated delta rule (sgl-amd-mono #89, Modifications: the recurrence in
# f32 on the cached state, stored in f32 or bf16 in place; Kernel checks:
# a bf16 state is widened, the recurrence runs on it, the result rounded)
# --------------------------------------------------------------------------

def delta_rule(S, k, v, q, g, beta):
    """One step of the gated delta rule on one value head.

    S [dv, dk] with S[v][k] (the stored layout); in matrix terms with
    M = S^T ([dk, dv]): M <- e^g M; M += k (x) beta (v - M^T k); o = M^T q.
    Written out per value row v:
      S[v, :] <- e^g S[v, :]
      u[v]     = beta * (v[v] - sum_k S[v, k] k[k])
      S[v, :] += u[v] k
      o[v]     = sum_k S[v, k] q[k]
    Returns (new S float64, o float64 [dv])."""
    S = np.asarray(S, dtype=np.float64) * math.exp(float(g))
    k = np.asarray(k, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    u = float(beta) * (np.asarray(v, dtype=np.float64) - S @ k)
    S = S + np.outer(u, k)
    o = S @ q
    return S, o


# --------------------------------------------------------------------------
# Step 9: gated RMSNorm x SiLU(z) (sgl-amd-mono #89 refusals: the gated norm is
# over the head, with SiLU, the norm before the gate; vLLM #60833 Tests:
# RMSNormGated)
# --------------------------------------------------------------------------

def gated_rmsnorm(o, z, w_g, eps: float):
    """core = bf16(o / sqrt(mean(o^2) + eps) * w_g * silu(z)) over the head."""
    o = np.asarray(o, dtype=np.float64)
    rstd = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return bf16_round(o * rstd * np.asarray(w_g, dtype=np.float64) * silu(z))


# --------------------------------------------------------------------------
# out_proj folded into the launch (SGLang #43558, commit text of the
# SGLANG_QWEN3_8_DENSE_MONO_OPROJ fold, "dense_gdn (K1Build.oproj)": every
# CTA publishes its core rows, then each runs its hidden columns of
# out_proj over the K share and the launch writes the out_proj result)
# --------------------------------------------------------------------------

def out_proj(core, W_o):
    """out[w, n] = bf16(sum_j W_o[n, j] core[w, j]) over the Hv*dv core
    columns of the bf16 core rows; the float64 sum is rounded once."""
    return bf16_round(np.asarray(core, dtype=np.float64) @ np.asarray(W_o, dtype=np.float64).T)


# --------------------------------------------------------------------------
# The whole step
# --------------------------------------------------------------------------

def gdn_step(shape, x, residual, weights, state_indices, conv_state, ssm_state):
    """One decode step of the GDN layer front for all rows.

    Arguments are numpy arrays (float64 holding the stored values exactly,
    int32 indices, uint8 for MXFP4 codes and scales); `shape` carries the
    sizes and constants (hidden, heads, dims, eps values, q_scale, state
    dtype, weight format, slot count). conv_state and ssm_state hold all
    slots and are NOT modified; updated copies are returned.

    Returns a dict: residual_out [W, H], core [W, Hv*dv], conv_state,
    ssm_state, index_error (True when a state index >= num_slots was seen;
    such a row is treated as a pad row) and the intermediates xn, p_qkvz,
    p_ba for diagnostics.
    """
    H, Hk, Hv = shape.hidden, shape.num_k_heads, shape.num_v_heads
    dk, dv = shape.head_k_dim, shape.head_v_dim
    G = Hv // Hk
    idx = np.asarray(state_indices, dtype=np.int64)
    Wr = idx.shape[0]
    conv_new = np.array(conv_state, dtype=np.float64, copy=True)
    ssm_new = np.array(ssm_state, dtype=np.float64, copy=True)

    r = residual_add(x, residual)
    xn = gemma_rmsnorm(r, weights["input_norm_w"], shape.norm_eps)
    if shape.qkvz_format == "mxfp4":
        p_qkvz = project_mxfp4(xn, weights["qkvz"], weights["qkvz_scales"])
    elif shape.qkvz_format == "mxfp6":
        p_qkvz = project_mxfp6(xn, weights["qkvz"], weights["qkvz_scales"])
    else:
        p_qkvz = project_bf16(xn, weights["qkvz"])
    p_ba = project_bf16(xn, weights["ba"])
    q, k, v, z, b, a = split_projection(p_qkvz, p_ba, Hk, Hv, dk, dv)

    core = np.zeros((Wr, Hv * dv))
    index_error = False
    for w in range(Wr):
        slot = int(idx[w])
        if slot >= shape.num_slots:
            index_error = True
            continue
        if slot <= 0:
            continue  # pad row: zero core, no state read or write
        u = np.concatenate([q[w].reshape(-1), k[w].reshape(-1), v[w].reshape(-1)])
        y, conv_new[slot] = conv_update(conv_state[slot], weights["conv_w"], u)
        yq = y[:Hk * dk].reshape(Hk, dk)
        yk = y[Hk * dk:2 * Hk * dk].reshape(Hk, dk)
        yv = y[2 * Hk * dk:].reshape(Hv, dv)
        qn = l2norm(yq, shape.l2_eps) * shape.scale_q
        kn = l2norm(yk, shape.l2_eps)
        g, beta = gates(a[w], b[w], weights["A_log"], weights["dt_bias"])
        for h in range(Hv):
            kh = h // G
            S, o = delta_rule(ssm_state[slot, h], kn[kh], yv[h], qn[kh], g[h], beta[h])
            ssm_new[slot, h] = bf16_round(S) if shape.ssm_dtype == "bf16" else f32_round(S)
            core[w, h * dv:(h + 1) * dv] = gated_rmsnorm(o, z[w, h], weights["gated_norm_w"],
                                                         shape.gated_norm_eps)
    out = {
        "residual_out": r, "core": core, "conv_state": conv_new, "ssm_state": ssm_new,
        "index_error": index_error, "xn": xn, "p_qkvz": p_qkvz, "p_ba": p_ba,
    }
    if weights.get("out_proj") is not None:
        out["out"] = out_proj(core, weights["out_proj"])
    return out


# --------------------------------------------------------------------------
# Multi-token verify with a state per token (the follow-up the pages name:
# sgl-amd-mono #89, Motivation, "keeps no state for each draft token, so a
# rejected draft token cannot roll back"; vLLM #60833, Details,
# "Limitations / follow-ups": MTP verify steps). Reading: sequence s has T
# tokens, rows s*T .. s*T + T - 1; it starts from slot state_in[s], and after
# token t its conv and SSM state go to their own slot state_out[s, t]. Each
# token continues from the state as stored (f32 or bf16), so the T tokens
# give what T decode steps would, and accepting the first a tokens means
# taking slot state_out[s, a - 1]. A sequence with state_in <= 0 is padding.
# --------------------------------------------------------------------------

def gdn_verify(shape, x, residual, weights, state_in, state_out, conv_state, ssm_state):
    """One verify step: len(state_in) sequences of T = state_out.shape[1]
    tokens. Arguments as for gdn_step, plus state_in [S] and state_out [S, T]
    int32 slots. Returns a dict as gdn_step's (residual_out, core, conv_state,
    ssm_state, index_error); the input state arrays are not modified."""
    H, Hk, Hv = shape.hidden, shape.num_k_heads, shape.num_v_heads
    dk, dv = shape.head_k_dim, shape.head_v_dim
    G = Hv // Hk
    sin = np.asarray(state_in, dtype=np.int64)
    sout = np.asarray(state_out, dtype=np.int64)
    S, T = sout.shape
    conv_new = np.array(conv_state, dtype=np.float64, copy=True)
    ssm_new = np.array(ssm_state, dtype=np.float64, copy=True)

    r = residual_add(x, residual)
    xn = gemma_rmsnorm(r, weights["input_norm_w"], shape.norm_eps)
    if shape.qkvz_format == "mxfp4":
        p_qkvz = project_mxfp4(xn, weights["qkvz"], weights["qkvz_scales"])
    elif shape.qkvz_format == "mxfp6":
        p_qkvz = project_mxfp6(xn, weights["qkvz"], weights["qkvz_scales"])
    else:
        p_qkvz = project_bf16(xn, weights["qkvz"])
    p_ba = project_bf16(xn, weights["ba"])
    q, k, v, z, b, a = split_projection(p_qkvz, p_ba, Hk, Hv, dk, dv)

    core = np.zeros((S * T, Hv * dv))
    index_error = False
    for s in range(S):
        slot = int(sin[s])
        outs = [int(o) for o in sout[s]]
        if slot >= shape.num_slots or any(o <= 0 or o >= shape.num_slots for o in outs):
            index_error = True
            continue
        if slot <= 0:
            continue  # a padding sequence: zero core rows, no state read or written
        conv_prev = conv_state[slot]
        ssm_prev = ssm_state[slot]
        for t in range(T):
            w = s * T + t
            u = np.concatenate([q[w].reshape(-1), k[w].reshape(-1), v[w].reshape(-1)])
            y, conv_t = conv_update(conv_prev, weights["conv_w"], u)
            yq = y[:Hk * dk].reshape(Hk, dk)
            yk = y[Hk * dk:2 * Hk * dk].reshape(Hk, dk)
            yv = y[2 * Hk * dk:].reshape(Hv, dv)
            qn = l2norm(yq, shape.l2_eps) * shape.scale_q
            kn = l2norm(yk, shape.l2_eps)
            g, beta = gates(a[w], b[w], weights["A_log"], weights["dt_bias"])
            ssm_t = np.empty_like(ssm_prev, dtype=np.float64)
            for h in range(Hv):
                kh = h // G
                St, o = delta_rule(ssm_prev[h], kn[kh], yv[h], qn[kh], g[h], beta[h])
                ssm_t[h] = bf16_round(St) if shape.ssm_dtype == "bf16" else f32_round(St)
                core[w, h * dv:(h + 1) * dv] = gated_rmsnorm(o, z[w, h], weights["gated_norm_w"],
                                                             shape.gated_norm_eps)
            conv_new[outs[t]] = conv_t
            ssm_new[outs[t]] = ssm_t
            conv_prev, ssm_prev = conv_t, ssm_t
    out = {"residual_out": r, "core": core, "conv_state": conv_new, "ssm_state": ssm_new,
           "index_error": index_error, "xn": xn, "p_qkvz": p_qkvz, "p_ba": p_ba}
    if weights.get("out_proj") is not None:
        out["out"] = out_proj(core, weights["out_proj"])
    return out
