"""Seeded synthetic workloads for the GDN decode-step front.

This module only describes layer shapes and draws seeded random numbers in
the storage types the layer uses (bf16, f32, int32, packed fp4 bytes). It
holds none of the layer's arithmetic, so both the CPU oracle's tests and the
CUDA path can take their inputs from it without sharing any of the method.

Value distributions (one recipe for every shape):
  in_proj_qkvz, in_proj_ba, conv weight   bf16 ~ N(0, 0.02)
  input norm weight, gated norm weight    bf16 ~ N(0, 0.1)
  x, residual                             bf16 ~ N(0, 1)
  A_log                                   f32  ~ U(-2, 0)
  dt_bias                                 bf16 ~ N(0, 0.5)
  conv state                              bf16 ~ N(0, 1)
  SSM state                               f32 or bf16 ~ N(0, 0.1)
  state indices                           distinct, drawn from 1..slots-1;
                                          pad rows get 0 or -1
  MXFP4 in_proj_qkvz                      e2m1 codes uniform over all 16
                                          codes, block exponents ~ U{-8..-4}
                                          (e8m0 byte = 127 + exponent)
  MXFP6 in_proj_qkvz                      packed code bytes uniform (so the
                                          e2m3 codes are uniform over all 64),
                                          block exponents ~ U{-10..-6} (weight
                                          std ~0.03, the bf16 layers' scale)
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class LayerShape:
    """Shapes and constants of one GDN layer front (one rank's share)."""

    name: str
    hidden: int
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    num_slots: int
    conv_kernel: int = 4
    ssm_dtype: str = "f32"  # "f32" or "bf16"
    qkvz_format: str = "bf16"  # "bf16", "mxfp4" or "mxfp6"
    max_rows: int = 16
    norm_eps: float = 1e-6
    gated_norm_eps: float = 1e-6
    l2_eps: float = 1e-6
    q_scale: float | None = None  # None: 1/sqrt(head_k_dim)

    @property
    def n_qkvz(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + 2 * self.num_v_heads * self.head_v_dim

    @property
    def n_ba(self) -> int:
        return 2 * self.num_v_heads

    @property
    def conv_channels(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim

    @property
    def group(self) -> int:
        return self.num_v_heads // self.num_k_heads

    @property
    def scale_q(self) -> float:
        return self.q_scale if self.q_scale is not None else float(self.head_k_dim) ** -0.5

    def with_(self, **kw) -> "LayerShape":
        return replace(self, **kw)

    # ---- byte counts (algorithmic traffic of one launch) ----
    def weight_bytes(self) -> int:
        H = self.hidden
        if self.qkvz_format == "mxfp4":
            qkvz = self.n_qkvz * (H // 2) + self.n_qkvz * (H // 32)
        elif self.qkvz_format == "mxfp6":
            qkvz = self.n_qkvz * (H * 3 // 4) + self.n_qkvz * (H // 32)
        else:
            qkvz = self.n_qkvz * H * 2
        ba = self.n_ba * H * 2
        small = (H + self.conv_channels * self.conv_kernel + self.num_v_heads
                 + self.head_v_dim) * 2 + self.num_v_heads * 4
        return qkvz + ba + small

    def state_bytes_per_row(self) -> int:
        """SSM + conv state read+write bytes of one non-pad row."""
        s = 4 if self.ssm_dtype == "f32" else 2
        ssm = self.num_v_heads * self.head_v_dim * self.head_k_dim * s
        conv = self.conv_channels * (self.conv_kernel - 1) * 2
        return 2 * (ssm + conv)

    def activation_bytes_per_row(self, first_layer: bool = False) -> int:
        """x (+ residual) in, residual_out and core out, the state index."""
        H = self.hidden
        return H * 2 * (1 if first_layer else 2) + H * 2 + self.num_v_heads * self.head_v_dim * 2 + 4

    def out_proj_bytes(self, rows: int) -> int:
        """What out_proj adds to a step: its weights and the rows' output."""
        return self.hidden * self.num_v_heads * self.head_v_dim * 2 + rows * self.hidden * 2

    def verify_bytes(self, seqs: int, tokens: int) -> int:
        """A verify step: the weights, each sequence's input state read once,
        one conv + SSM state written per token, and the rows' activations."""
        return (self.weight_bytes() + seqs * self.state_bytes_per_row() // 2
                + seqs * tokens * (self.state_bytes_per_row() // 2 + self.activation_bytes_per_row()))

    def launch_bytes(self, rows: int, live_rows: int | None = None, first_layer: bool = False) -> int:
        live = rows if live_rows is None else live_rows
        return (self.weight_bytes() + live * self.state_bytes_per_row()
                + rows * self.activation_bytes_per_row(first_layer))


# The workloads: a tiny correctness layer, one tensor-parallel rank's shard
# of a large layer, the same large layer unsharded, the shard with a bf16
# state (first-layer variant and pad rows in its cases), and a dense layer
# with an MXFP4 or an MXFP6 in_proj_qkvz.
TINY = LayerShape("tiny", hidden=1024, num_k_heads=4, num_v_heads=8,
                  head_k_dim=64, head_v_dim=64, num_slots=16)
SHARD = LayerShape("shard", hidden=8192, num_k_heads=2, num_v_heads=8,
                   head_k_dim=128, head_v_dim=128, num_slots=256)
FULL = LayerShape("full", hidden=8192, num_k_heads=16, num_v_heads=64,
                  head_k_dim=128, head_v_dim=128, num_slots=512)
SHARD_BF16 = SHARD.with_(name="shard_bf16", ssm_dtype="bf16")
DENSE_MXFP4 = LayerShape("dense_mxfp4", hidden=5120, num_k_heads=16, num_v_heads=48,
                         head_k_dim=128, head_v_dim=128, num_slots=20,
                         qkvz_format="mxfp4")

DENSE_MXFP6 = DENSE_MXFP4.with_(name="dense_mxfp6", qkvz_format="mxfp6")

SHAPES = {s.name: s for s in (TINY, SHARD, FULL, SHARD_BF16, DENSE_MXFP4, DENSE_MXFP6)}


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def _bf16(a: np.ndarray) -> torch.Tensor:
    """Store float32 draws as bf16 (a storage cast of random numbers)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng, shape, std, mean=0.0):
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std) + np.float32(mean)


def make_weights(shape: LayerShape, seed: int, *, weight_std: float = 0.02,
                 conv_std: float = 0.02, norm_std: float = 0.1) -> dict:
    """One layer's weights as CPU tensors in their storage types."""
    rng = _rng(seed)
    H, Hv, C, K = shape.hidden, shape.num_v_heads, shape.conv_channels, shape.conv_kernel
    w = {}
    w["input_norm_w"] = _bf16(_normal(rng, (H,), norm_std))
    if shape.qkvz_format == "mxfp4":
        n = shape.n_qkvz
        codes = rng.integers(0, 16, size=(n, H), dtype=np.uint8)
        packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
        exps = rng.integers(-8, -3, size=(n, H // 32))
        w["qkvz"] = torch.from_numpy(np.ascontiguousarray(packed))
        w["qkvz_scales"] = torch.from_numpy((127 + exps).astype(np.uint8))
    elif shape.qkvz_format == "mxfp6":
        n = shape.n_qkvz
        packed = rng.integers(0, 256, size=(n, H * 3 // 4), dtype=np.uint8)
        exps = rng.integers(-10, -5, size=(n, H // 32))
        w["qkvz"] = torch.from_numpy(packed)
        w["qkvz_scales"] = torch.from_numpy((127 + exps).astype(np.uint8))
    else:
        w["qkvz"] = _bf16(_normal(rng, (shape.n_qkvz, H), weight_std))
        w["qkvz_scales"] = None
    w["ba"] = _bf16(_normal(rng, (shape.n_ba, H), weight_std))
    w["conv_w"] = _bf16(_normal(rng, (C, K), conv_std))
    w["A_log"] = torch.from_numpy(rng.uniform(-2.0, 0.0, size=(Hv,)).astype(np.float32))
    w["dt_bias"] = _bf16(_normal(rng, (Hv,), 0.5))
    w["gated_norm_w"] = _bf16(_normal(rng, (shape.head_v_dim,), norm_std))
    return w


def make_out_proj(shape: LayerShape, seed: int, *, std: float = 0.02) -> torch.Tensor:
    """The layer's out_proj [H, Hv*dv] as a bf16 CPU tensor ~N(0, std)."""
    rng = _rng(seed)
    return _bf16(_normal(rng, (shape.hidden, shape.num_v_heads * shape.head_v_dim), std))


def make_state(shape: LayerShape, seed: int, *, ssm_std: float = 0.1) -> dict:
    """Per-slot conv and SSM state as CPU tensors."""
    rng = _rng(seed)
    S, C, K = shape.num_slots, shape.conv_channels, shape.conv_kernel
    conv = _bf16(_normal(rng, (S, C, K - 1), 1.0))
    ssm_np = _normal(rng, (S, shape.num_v_heads, shape.head_v_dim, shape.head_k_dim), ssm_std)
    ssm = _bf16(ssm_np) if shape.ssm_dtype == "bf16" else torch.from_numpy(ssm_np)
    return {"conv_state": conv, "ssm_state": ssm}


def make_step(shape: LayerShape, rows: int, seed: int, *, first_layer: bool = False,
              pad_rows: int = 0) -> dict:
    """One decode step's inputs: x, residual (None on the first layer) and
    the int32 state indices (distinct slots; `pad_rows` of them set to 0 or -1)."""
    if rows > shape.num_slots - 1:
        raise ValueError("more rows than distinct non-zero slots")
    rng = _rng(seed)
    H = shape.hidden
    x = _bf16(_normal(rng, (rows, H), 1.0))
    res = None if first_layer else _bf16(_normal(rng, (rows, H), 1.0))
    idx = rng.permutation(np.arange(1, shape.num_slots, dtype=np.int64))[:rows].astype(np.int32)
    if pad_rows:
        where = rng.permutation(rows)[:pad_rows]
        idx[where] = np.where(rng.integers(0, 2, size=pad_rows) == 0, 0, -1).astype(np.int32)
    return {"x": x, "residual": res, "state_indices": torch.from_numpy(idx)}


def default_pad_rows(rows: int) -> int:
    """About a quarter of the rows are pad rows in the mixed-pad cases."""
    return int(round(0.25 * rows))
