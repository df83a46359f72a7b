"""PyTorch custom operators over the C ABI.

``torch.ops.fa91.attention_forward(q, k, v, causal, scale)`` returns
``(O, LSE)`` for bf16 CUDA tensors ``[B, H, N, d]``, computed by ``fa_fwd``
(the same kernels as :func:`exact_attention_91_gb300.attention_forward`).
``torch.ops.fa91.attention_forward_varlen(q, k, v, cu_seqlens_q,
cu_seqlens_k, max_seqlen_q, causal, scale)`` returns ``(O [total_q, H, d],
LSE [H, total_q])`` for packed sequences, computed by ``fa_fwd_varlen``. The
operators are forward-only: the attention backward pass is not part of this
library. Their fake (meta) implementations give output shapes and dtypes
without a GPU, so the operators can be traced.
"""
from __future__ import annotations

import torch

from . import attention_forward, attention_forward_varlen


@torch.library.custom_op("fa91::attention_forward", mutates_args=())
def attention_forward_op(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                         scale: float | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    o, lse = attention_forward(q, k, v, causal=causal, scale=scale, return_lse=True)
    return o, lse


@attention_forward_op.register_fake
def _attention_forward_fake(q, k, v, causal=False, scale=None):
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B, H, N, d]")
    B, H, N, _ = q.shape
    return torch.empty_like(q), q.new_empty((B, H, N), dtype=torch.float32)


@torch.library.custom_op("fa91::attention_forward_varlen", mutates_args=())
def attention_forward_varlen_op(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                                cu_seqlens_k: torch.Tensor, max_seqlen_q: int, causal: bool = False,
                                scale: float | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    o, lse = attention_forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, causal=causal,
                                      scale=scale, return_lse=True)
    return o, lse


@attention_forward_varlen_op.register_fake
def _attention_forward_varlen_fake(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, causal=False, scale=None):
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or q.shape[1:] != k.shape[1:]:
        raise ValueError("q must be [total_q, H, d] and k, v [total_k, H, d]")
    total_q, H, _ = q.shape
    return torch.empty_like(q), q.new_empty((H, total_q), dtype=torch.float32)
