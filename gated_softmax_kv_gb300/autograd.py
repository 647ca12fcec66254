"""A thin torch.autograd wrapper over the two C-ABI calls.

`compressor(...)` returns `out` and, on backward, calls csa_compress_bwd for
dkv, dscore and dape (cuDNN-frontend "CSA Fused Compressor", sections
"High-level wrappers" and "Semantics"). Both directions run in
libcsa_compress.so; this module only routes tensors.
"""
from __future__ import annotations

from typing import Optional

import torch

from .binding import csa_compress_bwd, csa_compress_fwd


class CompressorFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, kv, score, ape, cu_seqlens, cu_seqlens_comp, capacity: int, ratio: int,
                coff: int, head_dim: int, exact: bool = False):
        out = csa_compress_fwd(kv, score, ape, cu_seqlens, cu_seqlens_comp, capacity, ratio, coff,
                               head_dim, exact=exact)
        ctx.save_for_backward(kv, score, ape, cu_seqlens, cu_seqlens_comp)
        ctx.meta = (capacity, ratio, coff, head_dim, exact)
        return out

    @staticmethod
    def backward(ctx, grad_out):
        kv, score, ape, cu, cuc = ctx.saved_tensors
        capacity, ratio, coff, head_dim, exact = ctx.meta
        dkv, dscore, dape = csa_compress_bwd(kv, score, ape, cu, cuc, capacity, ratio, coff, head_dim,
                                             grad_out.contiguous(), exact=exact)
        return dkv, dscore, dape, None, None, None, None, None, None, None


def compressor(kv: torch.Tensor, score: torch.Tensor, ape: torch.Tensor, cu_seqlens: torch.Tensor,
               cu_seqlens_comp: torch.Tensor, ratio: int, coff: int, head_dim: int,
               capacity: Optional[int] = None, exact: bool = False) -> torch.Tensor:
    """Differentiable fused Compressor. `capacity` defaults to cu_seqlens_comp[-1],
    which reads the device (a host synchronisation); pass a static capacity to
    keep the call free of synchronisation (e.g. for CUDA-graph capture).
    exact=True runs both directions in the exact mode (windows of at most 8
    slots)."""
    if capacity is None:
        capacity = int(cu_seqlens_comp[-1].item())
    return CompressorFunction.apply(kv, score, ape, cu_seqlens, cu_seqlens_comp, capacity, ratio,
                                    coff, head_dim, exact)
