"""Python binding of the attention library: argument marshalling only.

Torch is used for device memory and streams.  Every output and the backward
workspace is allocated inside ``torch.cuda.stream(s)`` for the stream ``s``
that the library launches on, so allocation, zero-fill and kernels are
ordered on one stream (NVIDIA/cudnn-frontend PR #429, first fix).  All
arithmetic runs in the CUDA library; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib

_DT = {torch.bfloat16: _lib.ATTN_BF16, torch.float16: _lib.ATTN_F16,
       torch.float32: _lib.ATTN_F32, torch.int32: _lib.ATTN_I32,
       torch.uint8: _lib.ATTN_U8, torch.bool: _lib.ATTN_U8,
       torch.float8_e4m3fn: _lib.ATTN_E4M3}


def tensor_desc(t):
    """attn_tensor_t for a torch tensor (or None -> NULL)."""
    if t is None:
        return None
    if t.dim() > 4:
        raise ValueError("rank > 4 not supported")
    d = _lib.AttnTensor()
    d.data = t.data_ptr() if t.numel() > 0 else 0
    d.dtype = _DT.get(t.dtype, 0)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    d.device = t.device.index if t.is_cuda else -1
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _stream(stream, device):
    return stream if stream is not None else torch.cuda.current_stream(device)


def _max_seqlen(cu_seqlens, max_seqlen):
    if cu_seqlens is None:
        return 0
    if max_seqlen is None:   # convenience: one device->host read
        lens = cu_seqlens[1:] - cu_seqlens[:-1]
        return int(lens.max().item()) if lens.numel() else 0
    return int(max_seqlen)


def attn_fwd(q, k, v, mask=None, cu_seqlens=None, max_seqlen=None, causal=False, scale=None,
             out=None, lse=None, eager_rescale=False, stream=None):
    """Forward pass.  Returns (out, lse).

    q, k, v: bf16 or fp16 (all the same); out has their type, lse is fp32.
    Dense: q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] -> out like q, lse [B,Hq,Sq] fp32.
    Varlen (cu_seqlens int32 [n+1]): q [T,Hq,D], k/v [T,Hkv,D], lse [Hq,T].
    mask: bool (True = visible) or additive fp32/bf16/fp16, broadcastable to
    [B,Hq,Sq,Sk].  scale=None means 1/sqrt(D).
    """
    lib = _lib.load()
    s = _stream(stream, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    msl = _max_seqlen(cu_seqlens, max_seqlen)
    if mask is not None and mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    with torch.cuda.device(q.device), torch.cuda.stream(s):
        if out is None:
            out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
        if lse is None:
            if cu_seqlens is None:
                lse = torch.empty(q.shape[0], q.shape[2], q.shape[1], dtype=torch.float32,
                                  device=q.device)
            else:
                lse = torch.empty(q.shape[1], q.shape[0], dtype=torch.float32, device=q.device)
        descs = [tensor_desc(x) for x in (q, k, v, mask, cu_seqlens, out, lse)]
        rc = lib.attn_fwd(*[_ref(d) for d in descs[:5]], msl, 1 if causal else 0, float(scale),
                          _ref(descs[5]), _ref(descs[6]),
                          _lib.ATTN_EAGER_RESCALE if eager_rescale else 0,
                          ctypes.c_void_p(s.cuda_stream))
    _lib.check(rc, "attn_fwd")
    return out, lse


def fwd_fp8_workspace_bytes(k):
    lib = _lib.load()
    return int(lib.attn_fwd_fp8_workspace_bytes(ctypes.byref(tensor_desc(k))))


def attn_fwd_fp8(q, k, v, descale_q, descale_k, descale_v, causal=False, scale=None, out=None,
                 lse=None, workspace=None, eager_rescale=False, stream=None):
    """Forward on fp8 inputs.  Returns (out, lse).

    q [B,Sq,Hq,128], k/v [B,Sk,Hkv,128]: torch.float8_e4m3fn; real value =
    element * descale (one float per tensor).  out is bf16 like q's shape,
    lse fp32 [B,Hq,Sq].  scale=None means 1/sqrt(D).
    """
    lib = _lib.load()
    s = _stream(stream, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    with torch.cuda.device(q.device), torch.cuda.stream(s):
        if out is None:
            out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
        if lse is None:
            lse = torch.empty(q.shape[0], q.shape[2], q.shape[1], dtype=torch.float32,
                              device=q.device)
        nbytes = fwd_fp8_workspace_bytes(k)
        if workspace is None or workspace.numel() < nbytes:
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        descs = [tensor_desc(x) for x in (q, k, v, out, lse)]
        rc = lib.attn_fwd_fp8(*[_ref(d) for d in descs[:3]], float(descale_q), float(descale_k),
                              float(descale_v), 1 if causal else 0, float(scale),
                              _ref(descs[3]), _ref(descs[4]),
                              ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                              _lib.ATTN_EAGER_RESCALE if eager_rescale else 0,
                              ctypes.c_void_p(s.cuda_stream))
    _lib.check(rc, "attn_fwd_fp8")
    return out, lse


def score_workspace_bytes(q, k, cu_seqlens=None, max_seqlen=None):
    lib = _lib.load()
    msl = _max_seqlen(cu_seqlens, max_seqlen)
    descs = [tensor_desc(x) for x in (q, k, cu_seqlens)]
    return int(lib.attn_score_workspace_bytes(*[_ref(d) for d in descs], msl))


def attn_score_recompute(q, k, lse, cu_seqlens=None, max_seqlen=None, causal=False, scale=None,
                         score=None, l1=None, workspace=None, stream=None):
    """Attention targets recomputed from the forward's lse, summed over the
    query heads, and each row's L1 norm.  Returns (score, l1), both fp32.

    Dense: q [B,Sq,Hq,D], k [B,Sk,Hkv,D], lse [B,Hq,Sq] -> score [B,Sq,Sk],
    l1 [B,Sq].  Varlen: q [T,Hq,D], k [T,Hkv,D], lse [Hq,T] -> score
    [T,max_seqlen], l1 [T].  scale=None means 1/sqrt(D).
    """
    lib = _lib.load()
    s = _stream(stream, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    msl = _max_seqlen(cu_seqlens, max_seqlen)
    with torch.cuda.device(q.device), torch.cuda.stream(s):
        if cu_seqlens is None:
            sshape, lshape = (q.shape[0], q.shape[1], k.shape[1]), (q.shape[0], q.shape[1])
        else:
            sshape, lshape = (q.shape[0], msl), (q.shape[0],)
        if score is None:
            score = torch.empty(sshape, dtype=torch.float32, device=q.device)
        if l1 is None:
            l1 = torch.empty(lshape, dtype=torch.float32, device=q.device)
        nbytes = score_workspace_bytes(q, k, cu_seqlens, msl)
        if workspace is None or workspace.numel() < nbytes:
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        descs = [tensor_desc(x) for x in (q, k, lse, cu_seqlens, score, l1)]
        rc = lib.attn_score_recompute(*[_ref(d) for d in descs[:4]], msl, 1 if causal else 0,
                                      float(scale), _ref(descs[4]), _ref(descs[5]),
                                      ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), 0,
                                      ctypes.c_void_p(s.cuda_stream))
    _lib.check(rc, "attn_score_recompute")
    return score, l1


def sparse_bwd_workspace_bytes(q, kv, with_sink):
    lib = _lib.load()
    q_, kv_ = tensor_desc(q), tensor_desc(kv)
    return int(lib.attn_sparse_bwd_workspace_bytes(ctypes.byref(q_), ctypes.byref(kv_),
                                                   1 if with_sink else 0))


def attn_sparse_bwd(q, kv, out, dout, lse, topk_idxs, topk_length=None, attn_sink=None,
                    scale=None, dq=None, dkv=None, d_sink=None, workspace=None, stream=None):
    """Backward of sparse top-k attention with an attention sink.

    q [B,S,64,Dqk] (Dqk 512 or 576), kv [B,S_kv,Dqk], out / dout [B,S,64,512],
    lse [B,S,64] fp32, topk_idxs int32 [B,S,K], topk_length int32 [B,S] or
    None, attn_sink fp32 [64] or None.  Returns (dq, dkv, d_sink); d_sink is
    None without a sink.  scale=None means 1/sqrt(Dqk).
    """
    lib = _lib.load()
    s = _stream(stream, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    with torch.cuda.device(q.device), torch.cuda.stream(s):
        dq = torch.empty(q.shape, dtype=q.dtype, device=q.device) if dq is None else dq
        dkv = torch.empty(kv.shape, dtype=kv.dtype, device=kv.device) if dkv is None else dkv
        if attn_sink is not None and d_sink is None:
            d_sink = torch.empty(attn_sink.shape, dtype=torch.float32, device=q.device)
        nbytes = sparse_bwd_workspace_bytes(q, kv, attn_sink is not None)
        if workspace is None or workspace.numel() < nbytes:
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        descs = [tensor_desc(x) for x in (q, kv, out, dout, lse, attn_sink, topk_idxs,
                                          topk_length, dq, dkv, d_sink)]
        rc = lib.attn_sparse_bwd(*[_ref(d) for d in descs[:8]], float(scale),
                                 *[_ref(d) for d in descs[8:]],
                                 ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), 0,
                                 ctypes.c_void_p(s.cuda_stream))
    _lib.check(rc, "attn_sparse_bwd")
    return dq, dkv, d_sink


def bwd_workspace_bytes(q, k, deterministic=False):
    lib = _lib.load()
    dq_, dk_ = tensor_desc(q), tensor_desc(k)
    return int(lib.attn_bwd_workspace_bytes(ctypes.byref(dq_), ctypes.byref(dk_),
                                            _lib.ATTN_DETERMINISTIC if deterministic else 0))


def attn_bwd(q, k, v, out, dout, lse, mask=None, cu_seqlens=None, max_seqlen=None, causal=False,
             scale=None, deterministic=False, dq=None, dk=None, dv=None, workspace=None,
             stream=None):
    """Backward pass.  Returns (dq, dk, dv) in the shapes of q, k, v."""
    lib = _lib.load()
    s = _stream(stream, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    msl = _max_seqlen(cu_seqlens, max_seqlen)
    if mask is not None and mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    flags = _lib.ATTN_DETERMINISTIC if deterministic else 0
    with torch.cuda.device(q.device), torch.cuda.stream(s):
        dq = torch.empty(q.shape, dtype=q.dtype, device=q.device) if dq is None else dq
        dk = torch.empty(k.shape, dtype=k.dtype, device=k.device) if dk is None else dk
        dv = torch.empty(v.shape, dtype=v.dtype, device=v.device) if dv is None else dv
        nbytes = bwd_workspace_bytes(q, k, deterministic)
        if workspace is None or workspace.numel() < nbytes:
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
        descs = [tensor_desc(x) for x in (q, k, v, out, dout, lse, mask, cu_seqlens)]
        outs = [tensor_desc(x) for x in (dq, dk, dv)]
        rc = lib.attn_bwd(*[_ref(d) for d in descs], msl, 1 if causal else 0, float(scale),
                          *[_ref(d) for d in outs], ctypes.c_void_p(workspace.data_ptr()),
                          workspace.numel(), flags, ctypes.c_void_p(s.cuda_stream))
    _lib.check(rc, "attn_bwd")
    return dq, dk, dv


def get_error(stream=None):
    """Synchronise the stream and return-and-clear the device error word."""
    lib = _lib.load()
    s = torch.cuda.current_stream() if stream is None else stream
    return lib.attn_get_error(ctypes.c_void_p(s.cuda_stream))
