"""Python binding of libfa.so, the GB300 (sm_103a) exact-attention forward.

The C entry points (``include/fa.h``) are exposed under the same names and
take raw device pointers (ints), exactly like the C ABI. ``attention_forward``
is a convenience wrapper for torch tensors: it checks dtypes and layout,
allocates the outputs with torch and calls ``fa_fwd`` on the current stream.
Every step of the computation runs in the CUDA library; if the library is
missing this module raises instead of computing anything elsewhere.
"""
from __future__ import annotations

import ctypes
import math
import os

from .build import LIB_PATH

__all__ = ["FaError", "load_library", "fa_fwd", "fa_fwd_noalloc", "fa_strerror", "fa_device_status",
           "fa_set_wait_limit_ns", "fa_abi_version", "fa_selftest_wait_timeout", "fa_fwd_varlen",
           "fa_varlen_num_splits", "fa_selftest_exp2", "fa_selftest_ex2_rate", "EX2_RATE_THREADS",
           "EX2_RATE_CHAINS", "attention_forward", "attention_forward_varlen",
           "head_shards", "attention_forward_heads", "EXPORTED_SYMBOLS"]

EXPORTED_SYMBOLS = ("fa_fwd", "fa_fwd_noalloc", "fa_fwd_varlen", "fa_strerror", "fa_device_status",
                    "fa_set_wait_limit_ns", "fa_abi_version", "fa_selftest_wait_timeout", "fa_varlen_num_splits",
                    "fa_selftest_exp2", "fa_selftest_ex2_rate")

FA_OK = 0
FA_ERR_DEVICE_TIMEOUT = -8

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = "fa_fwd"):
        self.status = status
        super().__init__(f"{what} failed: {status} ({fa_strerror(status)})")


def load_library(path: str | None = None):
    """Loads libfa.so (built in-tree by ``exact_attention_91_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    lib.fa_fwd_noalloc.restype = i
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_strerror.argtypes = [i]
    lib.fa_strerror.restype = ctypes.c_char_p
    lib.fa_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.fa_device_status.restype = i
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_set_wait_limit_ns.restype = None
    lib.fa_abi_version.argtypes = []
    lib.fa_abi_version.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [vp, ctypes.c_ulonglong]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_varlen_num_splits.argtypes = [i, i, i, i, i]
    lib.fa_varlen_num_splits.restype = i
    lib.fa_selftest_exp2.argtypes = [vp, vp, vp, i, vp]
    lib.fa_selftest_exp2.restype = i
    lib.fa_selftest_ex2_rate.argtypes = [vp, vp, i, i, vp]
    lib.fa_selftest_ex2_rate.restype = i
    if path is None:
        _lib = lib
    return lib


def fa_fwd(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, N: int, d: int,
           scale: float, causal: bool, stream: int | None) -> int:
    """The C ``fa_fwd``: device pointers as ints, returns the status code."""
    return load_library().fa_fwd(q, k, v, o, lse or None, B, H, N, d, scale, int(bool(causal)),
                                 stream or None)


def fa_fwd_noalloc(q: int, k: int, v: int, o: int, lse: int | None, B: int, H: int, N: int, d: int,
                   scale: float, causal: bool, stream: int | None) -> int:
    """The C ``fa_fwd_noalloc``: ``fa_fwd`` for callers that cannot let the
    library allocate device memory (its scratch is a fixed array inside the
    library). Calls whose kernels overlap on the GPU share that scratch and
    must not be issued. Returns the status code."""
    return load_library().fa_fwd_noalloc(q, k, v, o, lse or None, B, H, N, d, scale, int(bool(causal)),
                                         stream or None)


def fa_fwd_varlen(q: int, k: int, v: int, o: int, lse: int | None, cu_q: int, cu_k: int, B: int, H: int,
                  total_q: int, total_k: int, max_seqlen_q: int, d: int, scale: float, causal: bool,
                  stream: int | None) -> int:
    """The C ``fa_fwd_varlen``: device pointers as ints, returns the status code."""
    return load_library().fa_fwd_varlen(q, k, v, o, lse or None, cu_q, cu_k, B, H, total_q, total_k,
                                        max_seqlen_q, d, scale, int(bool(causal)), stream or None)


def fa_varlen_num_splits(B: int, H: int, total_k: int, max_seqlen_q: int, sm_count: int) -> int:
    """The C ``fa_varlen_num_splits`` (host only): work items per unit's key
    range that ``fa_fwd_varlen`` uses for these sizes, or a negative status."""
    return load_library().fa_varlen_num_splits(B, H, total_k, max_seqlen_q, sm_count)


def fa_strerror(status: int) -> str:
    return load_library().fa_strerror(status).decode()


def fa_device_status(stream: int | None = None) -> tuple[int, int]:
    """Synchronises ``stream``, reads and clears the device status word."""
    bits = ctypes.c_uint(0)
    rc = load_library().fa_device_status(stream or None, ctypes.byref(bits))
    return rc, bits.value


def fa_set_wait_limit_ns(ns: int) -> None:
    load_library().fa_set_wait_limit_ns(ns)


def fa_abi_version() -> int:
    return load_library().fa_abi_version()


def fa_selftest_wait_timeout(limit_ns: int, stream: int | None = None) -> int:
    """The C ``fa_selftest_wait_timeout``: one warp waits on a barrier that
    nothing completes until ``limit_ns`` passes, then records the timeout in
    the device status word. Returns the launch status."""
    return load_library().fa_selftest_wait_timeout(stream or None, limit_ns)


def fa_selftest_exp2(x: int, y_approx: int, y_exp2f: int, n: int, stream: int | None = None) -> int:
    """The C ``fa_selftest_exp2``: 2^x on the device by the softmax's
    ex2.approx.ftz.f32 and by CUDA's exp2f, for n fp32 arguments (device
    pointers as ints). Returns the status code."""
    return load_library().fa_selftest_exp2(x, y_approx, y_exp2f, n, stream or None)


# fa_selftest_ex2_rate: threads per block and chains per thread
EX2_RATE_THREADS = 1024
EX2_RATE_CHAINS = 8


def fa_selftest_ex2_rate(cycles: int, sink: int, blocks: int, iters: int, stream: int | None = None) -> int:
    """The C ``fa_selftest_ex2_rate``: ``blocks`` blocks (one per SM) each
    run EX2_RATE_THREADS x EX2_RATE_CHAINS chains of ``iters`` dependent
    ex2.approx; ``cycles`` (device int64 [blocks]) receives each block's span
    in SM clocks, ``sink`` (device fp32 [blocks * EX2_RATE_THREADS]) the
    chains' last values. Returns the status code."""
    return load_library().fa_selftest_ex2_rate(cycles, sink, blocks, iters, stream or None)


def _current_stream_handle(torch, device) -> int:
    """The raw cudaStream_t of the current stream on `device` (without
    building a Stream object when torch offers the raw handle)."""
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(device.index if device.index is not None else torch.cuda.current_device())
    return torch.cuda.current_stream(device).cuda_stream


def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                      return_lse: bool = True, stream=None):
    """O (bf16) and LSE (fp32) for bf16 CUDA tensors q, k, v of shape [B, H, N, d].

    ``out`` / ``lse`` may be given to reuse buffers. Runs on ``stream`` (a
    torch.cuda.Stream) or the current stream.
    """
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bf16")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B, H, N, d]")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    sp = stream.cuda_stream if stream is not None else _current_stream_handle(torch, q.device)
    rc = (_lib or load_library()).fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         lse.data_ptr() if lse is not None else None, B, H, N, d, float(scale),
                                         1 if causal else 0, sp or None)
    if rc != FA_OK:
        raise FaError(rc)
    return (out, lse) if return_lse else out


def attention_forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal: bool = False,
                             scale: float | None = None, out=None, lse=None, return_lse: bool = True,
                             stream=None):
    """O [total_q, H, d] (bf16) and LSE [H, total_q] (fp32) for a batch of
    sequences of different lengths: q [total_q, H, d], k and v [total_k, H, d]
    (bf16, CUDA, contiguous), int32 CUDA offsets ``cu_seqlens_q`` /
    ``cu_seqlens_k`` of B + 1 entries. Under ``causal`` each sequence's last
    query is aligned with its last key."""
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bf16")
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or q.shape[1:] != k.shape[1:]:
        raise ValueError("q must be [total_q, H, d] and k, v [total_k, H, d]")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if cu_seqlens_q.dim() != 1 or cu_seqlens_k.shape != cu_seqlens_q.shape or cu_seqlens_q.numel() < 2:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 offsets")
    for t in (q, k, v, cu_seqlens_q, cu_seqlens_k):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all inputs must be contiguous CUDA tensors")
    total_q, H, d = q.shape
    total_k = k.shape[0]
    B = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    sp = stream.cuda_stream if stream is not None else _current_stream_handle(torch, q.device)
    rc = fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                       lse.data_ptr() if lse is not None else None, cu_seqlens_q.data_ptr(),
                       cu_seqlens_k.data_ptr(), B, H, total_q, total_k, int(max_seqlen_q), d, float(scale),
                       causal, sp)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_varlen")
    return (out, lse) if return_lse else out


def head_shards(num_heads_total: int, world: int) -> list[tuple[int, int]]:
    """Contiguous ranges (start, count) of the flattened B*H head axis for
    ``world`` ranks, in rank order, sizes differing by at most one (the first
    ``num_heads_total % world`` ranks take one more). Heads are independent
    (each head's O and LSE depend only on its own Q, K, V), so a rank that
    holds its range's Q, K, V computes its O and LSE alone: the head-sharded
    multi-GPU forward needs no exchange between ranks."""
    if num_heads_total < 0 or world < 1:
        raise ValueError("need num_heads_total >= 0 and world >= 1")
    base, extra = divmod(num_heads_total, world)
    out, start = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((start, n))
        start += n
    return out


def attention_forward_heads(q, k, v, head_start: int, head_count: int, causal: bool = False,
                            scale: float | None = None, out=None, lse=None, stream=None):
    """fa_fwd on heads [head_start, head_start + head_count) of the flattened
    B*H axis of contiguous bf16 CUDA tensors [B, H, N, d]: the C call gets
    pointers into q, k, v (and into ``out`` / ``lse``, allocated whole when
    not given), nothing is copied, and the other heads of ``out`` and ``lse``
    are left as they were. Returns (out, lse) for the whole [B, H, N, d] /
    [B, H, N] shape. Each rank of a head-sharded job calls this on the range
    ``head_shards(B*H, world)[rank]`` of tensors in its own device memory."""
    import torch
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k, v must be bf16")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B, H, N, d]")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, H, N, d = q.shape
    if head_start < 0 or head_count < 0 or head_start + head_count > B * H:
        raise ValueError("head range outside [0, B*H)")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if head_count == 0:
        return out, lse
    eo, el = N * d * q.element_size(), N * 4   # bytes per head of q/k/v/out and of lse
    sp = stream.cuda_stream if stream is not None else _current_stream_handle(torch, q.device)
    rc = fa_fwd(q.data_ptr() + head_start * eo, k.data_ptr() + head_start * eo, v.data_ptr() + head_start * eo,
                out.data_ptr() + head_start * eo, lse.data_ptr() + head_start * el, 1, head_count, N, d,
                float(scale), causal, sp)
    if rc != FA_OK:
        raise FaError(rc)
    return out, lse
