"""Seeded synthetic inputs for the attention forward pass.

This module is the only code shared by the CUDA path's callers and the oracle's
callers. It draws random numbers and rounds them to bf16; it holds none of the
attention arithmetic.

Recipe (all workloads):

* numpy ``Generator(PCG64)`` seeded from ``SeedSequence(seed).spawn(4)``; the
  four child streams draw Q, K, V and the spike key indices, in that order.
* Samples are drawn in fp64, rounded to fp32 (round to nearest even), then to
  bf16 (round to nearest even on the fp32 bits). This is the same two-step
  rounding ``torch.Tensor.to(torch.bfloat16)`` applies to fp64 data.
* The GPU receives those bf16 bytes; the oracle receives the same values
  widened exactly to fp64 (``bf16_to_f64``).

The five named workloads are the shapes of the attention forward pass on the
pages: a single 128-token head, a ragged causal batch whose length is not a
tile multiple, an LLM-prefill shape, a long sequence, and a "max-shift"
stress case whose scores are large and spiked so that the running maximum
moves by a lot ("How Did I Write My First FlashAttention Kernel in CUDA?",
N = 16,384 long-sequence paragraph; "Mini FlashAttention", §2 "Why fuse it",
the 4096-token example).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

SEED_BASE = 20260000


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    values: str          # "normal" or "maxshift"
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Algorithmic flops: 4·B·H·N²·d (QKᵀ and PV), halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM bytes: read Q, K, V and write O (bf16), write LSE (fp32)."""
        return self.B * self.H * self.N * (4 * self.d * 2 + 4)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 128, 64, False, "normal", SEED_BASE + 0),
    "ragged_causal": Workload("ragged_causal", 2, 4, 1000, 64, True, "normal", SEED_BASE + 1),
    "llm_prefill": Workload("llm_prefill", 4, 32, 4096, 128, True, "normal", SEED_BASE + 2),
    "long_sequence": Workload("long_sequence", 1, 8, 16384, 64, False, "normal", SEED_BASE + 3),
    "max_shift": Workload("max_shift", 16, 16, 1024, 128, False, "maxshift", SEED_BASE + 4),
}


def custom(B: int, H: int, N: int, d: int, causal: bool, seed: int,
           values: str = "normal") -> Workload:
    return Workload(f"custom_{B}x{H}x{N}x{d}{'_causal' if causal else ''}",
                    B, H, N, d, causal, values, seed)


# ---------------------------------------------------------------- bf16 bits

def bf16_from_f64(x: np.ndarray) -> np.ndarray:
    """fp64 → fp32 (RNE) → bf16 (RNE); returns the bf16 bit patterns (uint16)."""
    f32 = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    bits = f32.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f32)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    out = rounded.astype(np.uint16)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- generators

@dataclasses.dataclass
class Inputs:
    workload: Workload
    q: np.ndarray            # uint16 bf16 bits [B, H, N, d]
    k: np.ndarray
    v: np.ndarray
    spike_keys: np.ndarray | None = None   # [B, H, N] int64 (max-shift only)

    def f64(self):
        return bf16_to_f64(self.q), bf16_to_f64(self.k), bf16_to_f64(self.v)


def make_inputs(w: Workload) -> Inputs:
    """Draw the seeded bf16 inputs of workload ``w``.

    * ``normal``: Q, K, V iid N(0, 1).
    * ``maxshift``: Q, K iid N(0, 3²); V iid U(-1, 1); then one spike per
      query row: a key index j_i ~ U{0..N-1} is drawn and Q[i] moves by
      (20/scale)·K[j_i]/‖K[j_i]‖² (fp64, K already rounded to bf16), so that
      the scaled score of that key rises by about +20; Q is rounded to bf16
      after the move.
    """
    shape = (w.B, w.H, w.N, w.d)
    gq, gk, gv, gs = [np.random.Generator(np.random.PCG64(s))
                      for s in np.random.SeedSequence(w.seed).spawn(4)]
    if w.values == "normal":
        q = bf16_from_f64(gq.standard_normal(shape))
        k = bf16_from_f64(gk.standard_normal(shape))
        v = bf16_from_f64(gv.standard_normal(shape))
        return Inputs(w, q, k, v)
    if w.values == "maxshift":
        q64 = 3.0 * gq.standard_normal(shape)
        k = bf16_from_f64(3.0 * gk.standard_normal(shape))
        v = bf16_from_f64(gv.uniform(-1.0, 1.0, shape))
        spike = gs.integers(0, w.N, size=(w.B, w.H, w.N), dtype=np.int64)
        k64 = bf16_to_f64(k)
        kj = np.take_along_axis(k64, spike[..., None], axis=2)       # [B,H,N,d]
        norm2 = np.maximum(np.sum(kj * kj, axis=-1, keepdims=True), 1e-30)
        q64 = q64 + (20.0 / w.scale) * kj / norm2
        q = bf16_from_f64(q64)
        return Inputs(w, q, k, v, spike)
    raise ValueError(f"unknown value recipe {w.values!r}")


@dataclasses.dataclass
class VarlenInputs:
    seqlens_q: tuple
    seqlens_k: tuple
    cu_q: np.ndarray         # int32 [B + 1]
    cu_k: np.ndarray
    q: np.ndarray            # uint16 bf16 bits [total_q, H, d]
    k: np.ndarray            # [total_k, H, d]
    v: np.ndarray

    def f64(self):
        return bf16_to_f64(self.q), bf16_to_f64(self.k), bf16_to_f64(self.v)


def make_varlen_inputs(seqlens_q, seqlens_k, H: int, d: int, seed: int) -> VarlenInputs:
    """A batch of sequences of their own query and key counts, token-major
    [total, H, d] bf16 with Q, K, V iid N(0, 1), and the int32 offsets."""
    if len(seqlens_q) != len(seqlens_k) or len(seqlens_q) < 1:
        raise ValueError("one query count and one key count per sequence")
    cu_q = np.concatenate([[0], np.cumsum(seqlens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seqlens_k)]).astype(np.int32)
    gq, gk, gv = [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(3)]
    q = bf16_from_f64(gq.standard_normal((int(cu_q[-1]), H, d)))
    k = bf16_from_f64(gk.standard_normal((int(cu_k[-1]), H, d)))
    v = bf16_from_f64(gv.standard_normal((int(cu_k[-1]), H, d)))
    return VarlenInputs(tuple(seqlens_q), tuple(seqlens_k), cu_q, cu_k, q, k, v)
