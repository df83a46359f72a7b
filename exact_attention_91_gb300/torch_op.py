"""PyTorch custom operator over the C ABI.

``torch.ops.fa91.attention_forward(q, k, v, causal, scale)`` returns
``(O, LSE)`` for bf16 CUDA tensors ``[B, H, N, d]``, computed by ``fa_fwd``
(the same kernels as :func:`exact_attention_91_gb300.attention_forward`). The
operator is forward-only: the attention backward pass is not part of this
library. Its fake (meta) implementation gives output shapes and dtypes
without a GPU, so the operator can be traced.
"""
from __future__ import annotations

import torch

from . import attention_forward


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
