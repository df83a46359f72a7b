"""fp64 CPU oracle for exact softmax attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The product path (``include/fa.h``, the CUDA
library and its Python binding) never imports, links or calls it, and the two
share no code.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, POSIX threads over
independent query rows); this module only compiles it with the host compiler
and marshals numpy arrays through ``ctypes``.

* ``attn_fwd``   -- every row, by the definition S = scale·QKᵀ (+ causal
  mask), P = row softmax(S), O = P·V, LSE = ln Σ exp(S) ("Mini
  FlashAttention", §1 "What attention is").
* ``attn_rows``  -- the same for a chosen list of rows (sampled parity on
  large workloads, bounded CPU-baseline timing).
* ``attn_online`` -- the chunked online-softmax loop ("Mini FlashAttention",
  §4 "The flash trick: online softmax"), to check that streaming equals the
  definition.
* ``attn_probs`` -- the probability matrix P of one head, for small N.

Parity of every function here is pinned by ``tests/test_oracle.py`` against
closed forms, invariants, a library routine and a worked example; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` beside it (gcc, -O2).

    Portable flags only (no -march=native), so x86 and Arm builds give the
    same numbers. Returns the library path.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cc = os.environ.get("CC", "gcc")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-shared",
           "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_long)
    L, D, I = ctypes.c_long, ctypes.c_double, ctypes.c_int
    lib.oracle_attn_fwd_f64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, D, I, I]
    lib.oracle_attn_rows_f64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, D, I, lp, L, I]
    lib.oracle_attn_online_f64.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, D, I, L, I]
    lib.oracle_attn_probs_f64.argtypes = [dp, dp, dp, L, L, D, I]
    lib.oracle_attn_varlen_f64.argtypes = [dp, dp, dp, dp, dp, lp, lp, L, L, L, D, I, I]
    lib.oracle_host_threads.argtypes = []
    for fn in (lib.oracle_attn_fwd_f64, lib.oracle_attn_rows_f64,
               lib.oracle_attn_online_f64, lib.oracle_attn_probs_f64,
               lib.oracle_attn_varlen_f64, lib.oracle_host_threads):
        fn.restype = ctypes.c_int
    _lib = lib
    return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _shape4(q: np.ndarray):
    if q.ndim != 4:
        raise ValueError("expected [B, H, N, d]")
    return q.shape


def host_threads() -> int:
    """Threads the oracle uses when ``nthreads=0`` (all online host cores)."""
    return int(_load().oracle_host_threads())


def attn_fwd(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """O [B,H,N,d] and LSE [B,H,N] (fp64) by the definition."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape4(q)
    assert k.shape == q.shape and v.shape == q.shape
    o = np.empty((B, H, N, d), np.float64)
    lse = np.empty((B, H, N), np.float64)
    _check(_load().oracle_attn_fwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                       B, H, N, d, float(scale), int(bool(causal)),
                                       int(nthreads)), "attn_fwd")
    return o, lse


def attn_rows(q, k, v, rows, scale: float, causal: bool, nthreads: int = 0):
    """O [R,d] and LSE [R] for flat row indices ``rows`` ((b*H + h)*N + i)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape4(q)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    o = np.empty((R, d), np.float64)
    lse = np.empty((R,), np.float64)
    _check(_load().oracle_attn_rows_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
        int(bool(causal)), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), R,
        int(nthreads)), "attn_rows")
    return o, lse


def attn_online(q, k, v, scale: float, causal: bool, chunk: int, nthreads: int = 0):
    """O and LSE by the chunked online-softmax loop (``chunk`` keys per step)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = _shape4(q)
    o = np.empty((B, H, N, d), np.float64)
    lse = np.empty((B, H, N), np.float64)
    _check(_load().oracle_attn_online_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                          B, H, N, d, float(scale), int(bool(causal)),
                                          int(chunk), int(nthreads)), "attn_online")
    return o, lse


def attn_probs(q, k, scale: float, causal: bool):
    """P = softmax(scale·QKᵀ) of one head (q, k: [N, d]) as an [N, N] array."""
    q, k = _f64(q), _f64(k)
    N, d = q.shape
    p = np.empty((N, N), np.float64)
    _check(_load().oracle_attn_probs_f64(_ptr(q), _ptr(k), _ptr(p), N, d, float(scale),
                                         int(bool(causal))), "attn_probs")
    return p


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))


def attn_varlen(q, k, v, cu_q, cu_k, scale: float, causal: bool, nthreads: int = 0):
    """Variable-length batch by the definition: q [total_q, H, d], k and v
    [total_k, H, d], sequence b = query tokens cu_q[b]:cu_q[b+1] and key
    tokens cu_k[b]:cu_k[b+1]; the causal mask aligns each sequence's last
    query with its last key. Returns O [total_q, H, d] and LSE [H, total_q]
    (fp64); a query that sees no key gives O = 0 and LSE = -inf."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 3 or k.ndim != 3 or v.shape != k.shape or q.shape[1:] != k.shape[1:]:
        raise ValueError("expected q [total_q, H, d], k and v [total_k, H, d]")
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int64)
    cu_k = np.ascontiguousarray(cu_k, dtype=np.int64)
    B = cu_q.shape[0] - 1
    if cu_k.shape[0] != B + 1 or cu_q[-1] != q.shape[0] or cu_k[-1] != k.shape[0]:
        raise ValueError("cu_seqlens do not match the token counts")
    H, d = q.shape[1], q.shape[2]
    o = np.empty(q.shape, np.float64)
    lse = np.empty((H, q.shape[0]), np.float64)
    lp = ctypes.POINTER(ctypes.c_long)
    _check(_load().oracle_attn_varlen_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), cu_q.ctypes.data_as(lp),
        cu_k.ctypes.data_as(lp), B, H, d, float(scale), int(bool(causal)), int(nthreads)),
        "attn_varlen")
    return o, lse
