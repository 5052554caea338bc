"""Seeded synthetic inputs for Attn-QAT workloads.

This module only draws random numbers and rounds them to BF16; it holds none
of the method's arithmetic, so both the CPU oracle tests and the CUDA path can
take their inputs from it without sharing any computation.

Every tensor is drawn per (tensor, batch, head) from
``numpy.random.default_rng([seed, b, h])``, so one head of a large workload can
be regenerated on its own (the sampled-head parity checks rely on that).

Workloads (BHSD, BF16 activations):

* ``c1``  B=1  H=2  S=256   D=64  non-causal, iid N(0,1), scale 1/8.
* ``c2``  B=1  H=16 S=4096  D=128 non-causal, iid N(0,1), scale 1/sqrt(128).
* ``c3``  B=2  H=32 S=8192  D=128 causal; Q and K N(0,1) with 4 of 128
  channels per head scaled x20 (the same channels for Q and K of a head);
  V and dO N(0,1).
* ``c4``  B=1  H=40 S=32760 D=128 non-causal (21x30x52 video latents, not a
  multiple of 64), iid N(0,1).
* ``c5``  B=1  H=64 S=16384 D=128 causal; Q, K, V N(0,1) with 1 % of the
  entries scaled x10 (heavy tail); dO N(0, 0.01), i.e. std 0.1.
* ``peaked`` B=1 H=2 S=256 D=64 non-causal with logits sharpened (Q x4) so
  that most probability groups survive quantization.
* ``ctx32k`` B=1 H=16 S=32768 D=128 non-causal, iid N(0,1): the long-context
  shape the FP4 inference forward is quoted on (dO unused there).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_Q, SEED_K, SEED_V, SEED_DO, SEED_OUTLIER, SEED_HEAVY = 1, 2, 3, 4, 5, 6


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    scale: float
    structure: str = "iid"     # iid | outlier | heavy | peaked
    q_gain: float = 1.0

    @property
    def shape_q(self):
        return (self.B, self.H, self.Sq, self.D)

    @property
    def shape_k(self):
        return (self.B, self.H, self.Sk, self.D)

    def fwd_flops(self) -> float:
        f = 4.0 * self.B * self.H * self.Sq * self.Sk * self.D
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        f = 10.0 * self.B * self.H * self.Sq * self.Sk * self.D
        return f / 2 if self.causal else f


WORKLOADS = {
    "c1": Workload("c1", 1, 2, 256, 256, 64, False, 1 / 8),
    "c2": Workload("c2", 1, 16, 4096, 4096, 128, False, 1 / math.sqrt(128)),
    "c3": Workload("c3", 2, 32, 8192, 8192, 128, True, 1 / math.sqrt(128), "outlier"),
    "c4": Workload("c4", 1, 40, 32760, 32760, 128, False, 1 / math.sqrt(128)),
    "c5": Workload("c5", 1, 64, 16384, 16384, 128, True, 1 / math.sqrt(128), "heavy"),
    "peaked": Workload("peaked", 1, 2, 256, 256, 64, False, 1 / 8, "peaked", 4.0),
    "ctx32k": Workload("ctx32k", 1, 16, 32768, 32768, 128, False, 1 / math.sqrt(128)),
}


def workload(name: str, **override) -> Workload:
    """A named workload, optionally with fields replaced (e.g. a smaller H)."""
    w = WORKLOADS[name]
    return dataclasses.replace(w, **override) if override else w


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest BF16 (ties to even); float32 out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _normal(seed: int, b: int, h: int, rows: int, d: int) -> np.ndarray:
    return np.random.default_rng([seed, b, h]).standard_normal((rows, d), dtype=np.float32)


def head_inputs(w: Workload, b: int, h: int) -> dict:
    """Q, K, V, dO of one (b, h) head as BF16-exact float32 arrays."""
    q = _normal(SEED_Q, b, h, w.Sq, w.D)
    k = _normal(SEED_K, b, h, w.Sk, w.D)
    v = _normal(SEED_V, b, h, w.Sk, w.D)
    do = _normal(SEED_DO, b, h, w.Sq, w.D)
    if w.structure == "outlier":
        ch = np.random.default_rng([SEED_OUTLIER, b, h]).choice(w.D, size=4, replace=False)
        q[:, ch] *= 20.0
        k[:, ch] *= 20.0
    elif w.structure == "heavy":
        for i, t in enumerate((q, k, v)):
            m = np.random.default_rng([SEED_HEAVY, b, h, i]).random(t.shape) < 0.01
            t[m] *= 10.0
        do *= 0.1
    if w.q_gain != 1.0:
        q *= np.float32(w.q_gain)
    return {n: bf16_round(t) for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}


def inputs(w: Workload, heads=None) -> dict:
    """All heads (or the listed (b, h) pairs, stacked on axis 0) as float32 BHSD."""
    if heads is None:
        out = {n: np.empty(w.shape_q if n in ("q", "do") else w.shape_k, np.float32)
               for n in ("q", "k", "v", "do")}
        for b in range(w.B):
            for h in range(w.H):
                for n, t in head_inputs(w, b, h).items():
                    out[n][b, h] = t
        return out
    per = [head_inputs(w, b, h) for (b, h) in heads]
    return {n: np.stack([p[n] for p in per])[:, None] for n in ("q", "k", "v", "do")}


def random_bf16(shape, seed: int, scale: float = 1.0) -> np.ndarray:
    """Generic seeded N(0, scale^2) BF16-exact array (for quantizer tests)."""
    x = np.random.default_rng(seed).standard_normal(shape, dtype=np.float32) * np.float32(scale)
    return bf16_round(x)
