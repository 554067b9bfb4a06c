"""Fused scaled-dot-product attention (forward and backward) for GB300.

The compute lives in a CUDA library built for sm_103a (``build.build()``)
behind the C ABI of ``include/attn_gb300.h``; this package is its binding.
"""
from .ops import (attn_bwd, attn_fwd, attn_fwd_fp8, attn_score_recompute,  # noqa: F401
                  attn_sparse_bwd, bwd_workspace_bytes, fwd_fp8_workspace_bytes, get_error,
                  score_workspace_bytes, sparse_bwd_workspace_bytes)

__all__ = ["attn_fwd", "attn_fwd_fp8", "attn_bwd", "attn_score_recompute", "attn_sparse_bwd",
           "bwd_workspace_bytes", "fwd_fp8_workspace_bytes", "score_workspace_bytes",
           "sparse_bwd_workspace_bytes", "get_error"]
