"""Seeded synthetic inputs for MM-DiT joint attention (QK-RMSNorm + softmax attention).

This module holds no attention arithmetic.  It only draws random numbers and
rounds them to bfloat16-representable float32 values, so the same arrays can
feed both the CUDA path and the CPU oracle.

Shapes follow the re-diffusion README (MM-DiT backbone): 768 hidden = 12 heads
x 64 ("architecture flowchart" and the 12-layer table of the "attention fix"
section), 1024 image tokens at 512 px (4x64x64 latent, patchify stride 2) plus
77 CLIP caption tokens, concatenated text-first as ``[c; x]``.

Draw order (numpy PCG64 ``default_rng(seed)``, float32 draws): q, k, v, dout
from N(0, 1) with shape ``[B, H, N, d]``, then the gains gq, gk from
U(0.5, 1.5) with shape ``[d]``.  Every array is rounded to bf16 (round to
nearest, ties to even) and kept as float32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

EPS = 1e-6


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


@dataclass(frozen=True)
class JointConfig:
    """One joint-attention workload: batch, heads, image/text token counts, head dim."""

    name: str
    B: int
    H: int
    N_img: int
    N_txt: int
    d: int
    seed: int
    value_scale: float = 1.0
    mode: str = "fwdbwd"  # "fwdbwd" or "cfg_fwd"
    steps: int = 1
    n_uncond: int = 0  # CFG: trailing batch items that are the unconditional branch

    @property
    def N(self) -> int:
        return self.N_img + self.N_txt

    @property
    def BH(self) -> int:
        return self.B * self.H


# The five workloads.  Sizes: latent side = image side / 8 (frozen SD VAE),
# patch 2 -> (side/16)^2 image tokens; 77 CLIP text tokens.
CONFIGS = {
    "tiny": JointConfig("tiny", B=1, H=2, N_img=16, N_txt=8, d=64, seed=0),
    "256px": JointConfig("256px", B=64, H=12, N_img=256, N_txt=77, d=64, seed=1),
    "512px": JointConfig("512px", B=16, H=12, N_img=1024, N_txt=77, d=64, seed=2),
    "768px_d128": JointConfig("768px_d128", B=4, H=24, N_img=2304, N_txt=77, d=128, seed=3, value_scale=0.5),
    "cfg_512px": JointConfig("cfg_512px", B=16, H=12, N_img=1024, N_txt=77, d=64, seed=4, mode="cfg_fwd",
                             steps=50, n_uncond=8),
}


@dataclass
class JointInputs:
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dout: np.ndarray | None
    gq: np.ndarray
    gk: np.ndarray
    meta: dict = field(default_factory=dict)


def _normal(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        x = x * np.float32(scale)
    return to_bf16_values(x)


def _gain(rng: np.random.Generator, d: int, lo: float = 0.5, hi: float = 1.5) -> np.ndarray:
    g = rng.random(d, dtype=np.float32) * np.float32(hi - lo) + np.float32(lo)
    return to_bf16_values(g)


def make_inputs(B: int, H: int, N: int, d: int, seed: int, value_scale: float = 1.0,
                with_dout: bool = True, gain_range=(0.5, 1.5)) -> JointInputs:
    """Draw q, k, v, dout ~ N(0,1)*value_scale and gq, gk ~ U(gain_range), bf16-rounded."""
    rng = np.random.default_rng(seed)
    shape = (B, H, N, d)
    q = _normal(rng, shape, value_scale)
    k = _normal(rng, shape, value_scale)
    v = _normal(rng, shape, value_scale)
    dout = _normal(rng, shape, value_scale) if with_dout else None
    gq = _gain(rng, d, *gain_range)
    gk = _gain(rng, d, *gain_range)
    return JointInputs(q, k, v, dout, gq, gk, {"B": B, "H": H, "N": N, "d": d, "seed": seed})


def make_config_inputs(cfg: JointConfig) -> JointInputs:
    """Inputs of a fwd+bwd workload (the CFG workload uses :class:`CfgStream`)."""
    if cfg.mode != "fwdbwd":
        raise ValueError("use CfgStream for the CFG sampling workload")
    out = make_inputs(cfg.B, cfg.H, cfg.N, cfg.d, cfg.seed, cfg.value_scale)
    out.meta.update(name=cfg.name, N_img=cfg.N_img, N_txt=cfg.N_txt)
    return out


class CfgStream:
    """Per-step inputs of classifier-free-guidance sampling (forward only).

    The batch is ``[cond; uncond]``.  For the unconditional items the caption
    is the zero embedding, so every text row of q, k and v is the same vector
    per (tensor, head): one N(0,1) vector per head, shared by all unconditional
    items and all N_txt text rows.  Image rows are fresh every step.  Gains
    are drawn once, before the first step; each step then draws q, k, v (full
    shape) followed by the three shared text vectors ``[H, d]``.
    """

    def __init__(self, cfg: JointConfig):
        self.cfg = cfg
        self.rng = np.random.default_rng(cfg.seed)
        self.gq = _gain(self.rng, cfg.d)
        self.gk = _gain(self.rng, cfg.d)
        self.step_index = 0

    def next_step(self) -> JointInputs:
        c = self.cfg
        shape = (c.B, c.H, c.N, c.d)
        q = _normal(self.rng, shape, c.value_scale)
        k = _normal(self.rng, shape, c.value_scale)
        v = _normal(self.rng, shape, c.value_scale)
        u0 = c.B - c.n_uncond
        for arr in (q, k, v):
            shared = _normal(self.rng, (c.H, c.d), c.value_scale)
            arr[u0:, :, : c.N_txt, :] = shared[None, :, None, :]
        out = JointInputs(q, k, v, None, self.gq, self.gk,
                          {"name": c.name, "step": self.step_index, "N_img": c.N_img, "N_txt": c.N_txt})
        self.step_index += 1
        return out


@dataclass
class QkvInputs:
    """Tokens and weights of the two streams' QKV projections."""

    x_img: np.ndarray  # [B, N_img, C]
    w_img: np.ndarray  # [3 H d, C]
    b_img: np.ndarray | None  # [3 H d]
    x_txt: np.ndarray  # [B, N_txt, C]
    w_txt: np.ndarray
    b_txt: np.ndarray | None
    gq: np.ndarray
    gk: np.ndarray
    meta: dict = field(default_factory=dict)


def make_qkv_inputs(B: int, H: int, N_img: int, N_txt: int, d: int, C: int, seed: int,
                    bias: bool = True) -> QkvInputs:
    """Draw the projection inputs of both streams.

    Tokens ~ N(0, 1) (the adaLN-modulated hidden states feeding the
    projection are of unit scale), weights ~ N(0, 1/C) (a linear layer's usual
    initial scale, so each projected value is of unit scale), all
    bf16-rounded; biases ~ N(0, 0.1^2) float32 (not rounded); gains
    ~ U(0.5, 1.5) bf16-rounded.  Draw order (PCG64, float32): x_img, x_txt,
    w_img, w_txt, then (if bias) b_img, b_txt, then gq, gk.
    """
    rng = np.random.default_rng(seed)
    x_img = _normal(rng, (B, N_img, C), 1.0)
    x_txt = _normal(rng, (B, N_txt, C), 1.0)
    ws = float(1.0 / np.sqrt(C))
    w_img = _normal(rng, (3 * H * d, C), ws)
    w_txt = _normal(rng, (3 * H * d, C), ws)
    b_img = b_txt = None
    if bias:
        b_img = rng.standard_normal(3 * H * d, dtype=np.float32) * np.float32(0.1)
        b_txt = rng.standard_normal(3 * H * d, dtype=np.float32) * np.float32(0.1)
    gq = _gain(rng, d)
    gk = _gain(rng, d)
    return QkvInputs(x_img, w_img, b_img, x_txt, w_txt, b_txt, gq, gk,
                     {"B": B, "H": H, "N_img": N_img, "N_txt": N_txt, "d": d, "C": C, "seed": seed})
