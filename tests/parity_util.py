"""Helpers for the GPU parity tests: upload the seeded bf16 inputs, run the
CUDA path through the C ABI, and compare with the fp64 oracle.

Tolerances (bf16 inputs and output, fp32 accumulation): O max |Δ| ≤ 1e-2 and
mean |Δ| ≤ 1e-3 over the compared elements; LSE max |Δ| ≤ 1e-3.

A query row that sees at most FEW_KEYS keys (N ≤ 8, or the first rows under
the causal mask) is an average of a handful of V rows, so |O| is O(1) and the
bf16 rounding of the exact O alone costs up to half a bf16 ulp of |O| (7.8e-3
at |O| in [2, 4)) and about 1e-3 on average. For those rows alone the max bar
is 1e-2 on top of the half-ulp of each exact element, and the mean bar holds
for the distance to the exact O rounded to bf16 (the result the output type
can hold). Every other row is held to the plain bars against the fp64
oracle.
"""
from __future__ import annotations

import numpy as np

from exact_attention_91_gb300 import inputs as fin

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def to_device(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def o_to_numpy(o) -> np.ndarray:
    """bf16 device tensor -> fp64 numpy (exact)."""
    import torch
    bits = o.view(torch.int16).cpu().numpy().view(np.uint16)
    return fin.bf16_to_f64(bits)


def run_gpu(x: fin.Inputs, *, causal: bool | None = None, scale: float | None = None,
            with_lse: bool = True):
    import exact_attention_91_gb300 as fa
    w = x.workload
    q, k, v = to_device(x.q), to_device(x.k), to_device(x.v)
    o, lse = fa.attention_forward(q, k, v, causal=w.causal if causal is None else causal,
                                  scale=w.scale if scale is None else scale, return_lse=True)
    if not with_lse:
        return o, None
    return o, lse


FEW_KEYS = 8


def visible_keys(N: int, causal: bool, i: np.ndarray) -> np.ndarray:
    """Keys that query row i (0-based within its head) sees."""
    i = np.asarray(i)
    return (i + 1) if causal else np.full(i.shape, N)


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits): the most
    that rounding x to bf16 can cost."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8.0)


def compare(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray,
            label: str = "", keys: np.ndarray | None = None) -> dict:
    """Error statistics of GPU O/LSE against the oracle. ``keys`` (shaped like
    the LSE) gives each row's visible key count; rows with at most FEW_KEYS
    keys get the rounding allowance described above."""
    few = np.zeros(lse_ref.shape, bool) if keys is None else (np.asarray(keys) <= FEW_KEYS)
    many = ~few
    d_exact = np.abs(o_gpu - o_ref)
    d_l = np.abs(lse_gpu.astype(np.float64) - lse_ref)
    o_ref_bf16 = fin.bf16_to_f64(fin.bf16_from_f64(o_ref))
    stats = {
        # rows that see more than FEW_KEYS keys: the plain bars against the fp64 oracle
        "o_max_abs": float(d_exact[many].max()) if many.any() else 0.0,
        "o_mean_abs": float(d_exact[many].mean()) if many.any() else 0.0,
        # rows that see at most FEW_KEYS keys
        "few_key_rows": int(few.sum()),
        "few_max_over_allowance": float((d_exact[few] - half_ulp_bf16(o_ref[few])).max()) if few.any() else 0.0,
        "few_mean_vs_rounded": float(np.abs(o_gpu[few] - o_ref_bf16[few]).mean()) if few.any() else 0.0,
        # what bf16 rounding of the exact O alone costs (for the record)
        "o_mean_abs_rounding_only": float(np.abs(o_ref_bf16 - o_ref).mean()),
        "lse_max_abs": float(d_l.max()),
        "finite": bool(np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all()),
    }
    print(label, stats)
    return stats


def assert_within(stats: dict) -> None:
    assert stats["finite"], stats
    assert stats["o_max_abs"] <= O_MAX_ABS, stats
    assert stats["o_mean_abs"] <= O_MEAN_ABS, stats
    assert stats["few_max_over_allowance"] <= O_MAX_ABS, stats
    assert stats["few_mean_vs_rounded"] <= O_MEAN_ABS, stats
    assert stats["lse_max_abs"] <= LSE_MAX_ABS, stats


def sample_rows(B: int, H: int, N: int, n_random: int, seed: int) -> np.ndarray:
    """Flat row ids ((b*H + h)*N + i): the first and last heads' edge rows,
    rows on both sides of every 128-row tile boundary of a few heads, and
    uniformly random rows."""
    g = np.random.Generator(np.random.PCG64(seed))
    BH = B * H
    heads = sorted({0, BH - 1, BH // 2, int(g.integers(0, BH))})
    picks = []
    for h in heads:
        edge = [0, 1, N - 2, N - 1]
        for t in range(128, N, 128):
            edge += [t - 1, t]
        picks += [h * N + i for i in edge if 0 <= i < N]
    picks += list(g.integers(0, BH * N, n_random))
    return np.unique(np.array(picks, dtype=np.int64))


def oracle_rows(oracle_mod, x: fin.Inputs, rows: np.ndarray, causal: bool, scale: float):
    """Oracle O/LSE for flat rows, widening only the heads those rows touch."""
    w = x.workload
    B, H, N, d = w.B, w.H, w.N, w.d
    heads = np.unique(rows // N)
    qh = x.q.reshape(B * H, N, d)[heads]
    kh = x.k.reshape(B * H, N, d)[heads]
    vh = x.v.reshape(B * H, N, d)[heads]
    remap = {int(h): n for n, h in enumerate(heads)}
    local = np.array([remap[int(r // N)] * N + int(r % N) for r in rows], dtype=np.int64)
    q64, k64, v64 = (fin.bf16_to_f64(a)[None] for a in (qh, kh, vh))
    return oracle_mod.attn_rows(q64, k64, v64, local, scale, causal)
