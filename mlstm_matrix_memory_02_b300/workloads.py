"""Seeded synthetic inputs for the mLSTM cell, shared by the GPU path's tests/benchmark and
by the CPU oracle.

This module draws random numbers and rounds them to the storage type; it holds none of
the method's arithmetic (no gates, no stabiliser, no state update).

The shapes stand in for the language-model layers that "xLSTM: How Exponential Gating and
Matrix Memory Scale Recurrent Neural Networks" (llms.blog) describes (section 4 "mLSTM Block
Structure": up-projection factor 2 in front of the cell; section 6: 125M to 1.3B parameter
models).  No dataset is read: q, k, v and the gate pre-activations are drawn directly.

Generator: numpy PCG64 ``default_rng(seed)``, drawn in the order q, k, v, i~, f~ as
float32; bf16 workloads round q, k, v to bfloat16 with round-to-nearest-even and keep them
in float32 containers (exactly representable), so both sides see identical values.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    NH: int
    S: int
    DQK: int
    DV: int
    chunk: int
    dtype: str  # "f32" or "bf16": storage type of q, k, v and h
    ig: tuple = ("normal", 0.0, 1.0)  # input-gate pre-activation distribution
    fg: tuple = ("normal", 3.0, 1.0)  # forget-gate pre-activation distribution
    seed: int = 0
    # decode workloads: number of prior tokens that build the starting state
    prior: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return self.B * self.S

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY_F32 = Workload("tiny fp32", B=1, NH=2, S=64, DQK=32, DV=32, chunk=16, dtype="f32",
                    ig=("normal", 0.0, 1.0), fg=("normal", 3.0, 1.0))
LAYER_350M = Workload("350M-style layer", B=8, NH=4, S=1024, DQK=256, DV=256, chunk=64,
                      dtype="bf16", ig=("normal", 0.0, 1.0), fg=("normal", 3.0, 1.5))
LAYER_1P3B = Workload("1.3B-style layer", B=4, NH=4, S=2048, DQK=512, DV=512, chunk=64,
                      dtype="bf16", ig=("normal", 0.0, 1.0), fg=("normal", 3.0, 1.5))
STRESS_16K = Workload("long-context stabiliser stress", B=1, NH=8, S=16384, DQK=256, DV=256,
                      chunk=128, dtype="bf16", ig=("student_t", 4.0, 3.0),
                      fg=("normal", 0.0, 2.0))
# Decode: S is the number of timed single-token steps; `prior` tokens (seed 0) build the
# starting state, the timed steps draw from seed 1.
DECODE = Workload("recurrent decode", B=256, NH=8, S=64, DQK=256, DV=256, chunk=64,
                  dtype="bf16", ig=("normal", 0.0, 1.0), fg=("normal", 3.0, 1.0), seed=1,
                  prior=512)

WORKLOADS = {
    "tiny": TINY_F32,
    "350m": LAYER_350M,
    "1p3b": LAYER_1P3B,
    "stress": STRESS_16K,
    "decode": DECODE,
}


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); float32 container."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32)


def _draw(rng: np.random.Generator, spec: tuple, size) -> np.ndarray:
    kind = spec[0]
    if kind == "normal":
        _, mu, sigma = spec
        return (rng.standard_normal(size, dtype=np.float32) * np.float32(sigma)
                + np.float32(mu)).astype(np.float32)
    if kind == "student_t":
        _, scale, dof = spec
        return (np.float32(scale) * rng.standard_t(dof, size).astype(np.float32)).astype(
            np.float32)
    raise ValueError(f"unknown distribution {spec!r}")


def make_inputs(w: Workload, seed: int | None = None, S: int | None = None) -> dict:
    """Draw q, k, v [B,NH,S,D] and the gate pre-activations ig, fg [B,NH,S] (float32).

    ``S`` overrides the workload's sequence length (decode: ``prior`` for the starting
    state).  bf16 workloads return q, k, v already rounded to bfloat16 values.
    """
    seed = w.seed if seed is None else seed
    S = w.S if S is None else S
    rng = np.random.default_rng(seed)
    qk_shape = (w.B, w.NH, S, w.DQK)
    v_shape = (w.B, w.NH, S, w.DV)
    q = rng.standard_normal(qk_shape, dtype=np.float32)
    k = rng.standard_normal(qk_shape, dtype=np.float32)
    v = rng.standard_normal(v_shape, dtype=np.float32)
    ig = _draw(rng, w.ig, (w.B, w.NH, S))
    fg = _draw(rng, w.fg, (w.B, w.NH, S))
    if w.dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    return {"q": q, "k": k, "v": v, "ig": ig, "fg": fg}


def make_decode_inputs(w: Workload = DECODE) -> tuple[dict, dict]:
    """(prior, steps): ``prior`` holds w.prior tokens drawn with seed 0 that build the
    starting state; ``steps`` holds w.S single-token steps drawn with w.seed."""
    prior = make_inputs(w, seed=0, S=w.prior)
    steps = make_inputs(w, seed=w.seed, S=w.S)
    return prior, steps
