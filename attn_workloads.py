"""Seeded synthetic inputs for the attention workloads.

Shared by the tests, the smoke check and the benchmark, on both sides of a
parity check (the fp64 oracle and the CUDA library).  This module only draws
random numbers and lays them out: it holds none of the attention arithmetic.

Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)``
in fp32 and rounded to bf16 (or to fp16 when ``dtype=torch.float16``), in the
fixed order q, k, v, dO, then extras, so both sides see the same 16-bit
values.

Workloads (sizes and value distributions as the pages give them):

* ``causal_small``   B=1, H=1, S=256, D=64, causal, dO = ones
  (flash-dmattn PR #122, "Problem": seed 42, loss = out.sum()).
* ``low_lse_row``    B=2, H=4, D=64/128, (Sq, Sk) in {392x392, 360x64,
  100x77, 392x512}, bool / additive / no key-padding mask hiding the last
  ceil(0.1 Sk) keys; every key gets c u added (u a random unit vector) and
  one query row is -c u, so that row's LSE sits far below -88.7
  (OpenWAM PR #64, "Validation": one query row anti-aligned with keys that
  share a large component, row logsumexp about -111 to -120).  c = 37.5
  puts that row at -112..-118 for D = 128 on every shape and mask kind
  (c = 36 would leave it at -103..-109); D = 64 keeps the same c (its row
  then sits at -150..-167).
* ``wide_spread``    B=2, S=8192, H=32, D=128, k = N(0,1) * s for s in
  {8, 16, 24, 32, 48, 64} (FlyDSL PR #1033, "Repro").
* ``varlen_gqa``     16 packed sequences, lengths uniform in [128, 4096],
  Hq=32, Hkv=8, D=128, causal, 512 trailing rows that belong to no sequence.
* ``long_seq``       B=1, H=16, D=128, S in {16384, 65536, 131072}.
* ``fp8_qkv``        fp8 (E4M3) q, k, v with one descale factor per tensor:
  q, k = N(0,1) with k scaled by 1000 / 5000 / 20000 and V = ones at
  B=1, H=16, S=12288, D=128 (FlyDSL PR #1033, "The fp8 helper, second
  commit"); each tensor is divided by amax/448 and rounded to E4M3 by
  PyTorch's float8 conversion.
* ``dsa_case``       sparse top-k attention with a sink (NVIDIA/cudnn-frontend
  PR #429: S = 512 queries, S_kv = 2048 kv rows, H = 64, D = 576 with values
  in the first 512 columns, or D = 512, top-k = 128, with and without
  topk_length): q, kv, dout = N(0,1); every token lists K distinct kv rows
  drawn uniformly; with ``length`` each token's topk_length is uniform in
  [1, K] and the entries past it are -1; the sink per head is N(0,1).
"""
from __future__ import annotations

import math

import torch

BF16 = torch.bfloat16


def _gen(seed):
    return torch.Generator().manual_seed(seed)


def _randn(g, shape):
    return torch.randn(*shape, generator=g, dtype=torch.float32)


def dense_qkvdo(B, Sq, Sk, Hq, Hkv, D, seed=42, dout="randn", k_scale=1.0, dtype=BF16):
    """q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D], dO like q; 16-bit on the CPU."""
    g = _gen(seed)
    q = _randn(g, (B, Sq, Hq, D)).to(dtype)
    k = (_randn(g, (B, Sk, Hkv, D)) * k_scale).to(dtype)
    v = _randn(g, (B, Sk, Hkv, D)).to(dtype)
    if dout == "ones":
        do = torch.ones(B, Sq, Hq, D, dtype=dtype)
    else:
        do = _randn(g, (B, Sq, Hq, D)).to(dtype)
    return q, k, v, do


def causal_small(seed=42, dtype=BF16):
    """B=1, Hq=Hkv=1, S=256, D=64, causal, dO = ones."""
    q, k, v, do = dense_qkvdo(1, 256, 256, 1, 1, 64, seed=seed, dout="ones", dtype=dtype)
    return dict(q=q, k=k, v=v, do=do, causal=True, scale=1.0 / 8.0, mask=None)


def padding_mask(B, Sq, Sk, kind, Hq=1, per_row=False, seed=7):
    """Key-padding mask that hides the last ceil(0.1 Sk) keys.

    kind: "bool" (uint8 1 = visible), "additive" (fp32 0 / -inf) or "none".
    Shape [B,1,1,Sk] expanded (stride 0) to [B,Hq,Sq,Sk]; with per_row=True a
    materialised [B,Hq,Sq,Sk] mask that additionally hides random keys.
    """
    if kind == "none":
        return None
    n_hidden = math.ceil(0.1 * Sk)
    vis = torch.ones(B, 1, 1, Sk, dtype=torch.bool)
    if n_hidden:
        vis[..., Sk - n_hidden:] = False
    if per_row:
        g = _gen(seed)
        extra = torch.rand(B, Hq, Sq, Sk, generator=g) < 0.2
        vis = vis.expand(B, Hq, Sq, Sk) & ~extra
        vis = vis.contiguous()
    else:
        vis = vis.expand(B, Hq, Sq, Sk)
    if kind == "bool":
        return vis.to(torch.uint8) if not per_row else vis.to(torch.uint8)
    add = torch.zeros(vis.shape, dtype=torch.float32)
    add = add.masked_fill(~vis, float("-inf"))
    if not per_row:
        add = add[:, :1, :1, :].expand(B, Hq, Sq, Sk)
    return add


LOW_ROW_SHARED = 37.5


def low_lse_row(Sq, Sk, mask_kind, D=128, row="first", seed=42, B=2, H=4, dtype=BF16,
                shared=LOW_ROW_SHARED):
    """Keys share `shared` * u; one query row is -`shared` * u (row LSE far
    below -88.7)."""
    g = _gen(seed)
    q = _randn(g, (B, Sq, H, D))
    k = _randn(g, (B, Sk, H, D))
    v = _randn(g, (B, Sk, H, D))
    do = _randn(g, (B, Sq, H, D))
    u = _randn(g, (D,))
    u = u / u.norm()
    k = k + shared * u
    r = 0 if row == "first" else Sq - 1
    q[:, r, :, :] = -shared * u
    mask = padding_mask(B, Sq, Sk, mask_kind, Hq=H)
    return dict(q=q.to(dtype), k=k.to(dtype), v=v.to(dtype), do=do.to(dtype),
                causal=False, scale=1.0 / math.sqrt(D), mask=mask, low_row=r)


def wide_spread(s, B=2, S=8192, H=32, D=128, seed=42, dtype=BF16):
    """q, v ~ N(0,1); k = bf16(N(0,1) * s); dO ~ N(0,1); non-causal."""
    q, k, v, do = dense_qkvdo(B, S, S, H, H, D, seed=seed, k_scale=float(s), dtype=dtype)
    return dict(q=q, k=k, v=v, do=do, causal=False, scale=1.0 / math.sqrt(D), mask=None)


def varlen_lengths(n=16, lo=128, hi=4096, seed=42):
    g = _gen(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def varlen_gqa(n=16, lo=128, hi=4096, Hq=32, Hkv=8, D=128, trailing=512, seed=42, dtype=BF16):
    """Packed THD: q/dO [T,Hq,D], k/v [T,Hkv,D], cu_seqlens int32 [n+1]."""
    lens = varlen_lengths(n, lo, hi, seed)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    T = cu[-1] + trailing
    g = _gen(seed + 1)
    q = _randn(g, (T, Hq, D)).to(dtype)
    k = _randn(g, (T, Hkv, D)).to(dtype)
    v = _randn(g, (T, Hkv, D)).to(dtype)
    do = _randn(g, (T, Hq, D)).to(dtype)
    return dict(q=q, k=k, v=v, do=do, cu_seqlens=torch.tensor(cu, dtype=torch.int32),
                max_seqlen=max(lens), causal=True, scale=1.0 / math.sqrt(D), lens=lens)


def long_seq(S, causal, B=1, H=16, D=128, seed=42, dtype=BF16):
    q, k, v, do = dense_qkvdo(B, S, S, H, H, D, seed=seed, dtype=dtype)
    return dict(q=q, k=k, v=v, do=do, causal=causal, scale=1.0 / math.sqrt(D), mask=None)


def sample_rows(B, H, S, n=64, seed=5):
    """n seeded query rows per (b, h), always including 0 and S-1."""
    g = _gen(seed)
    rows = []
    for b in range(B):
        for h in range(H):
            idx = torch.randperm(S, generator=g)[: max(n - 2, 0)].tolist()
            pick = sorted(set([0, S - 1] + idx))[:n]
            rows += [(b, h, i) for i in pick]
    return rows


def _to_e4m3(x):
    """fp32 tensor -> (E4M3 codes as uint8, descale) with descale = amax / 448."""
    amax = float(x.abs().max()) if x.numel() else 0.0
    d = amax / 448.0 if amax > 0 else 1.0
    d = float(torch.tensor(d, dtype=torch.float32))          # an fp32 value
    codes = (x / d).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, d


def fp8_qkv(B=1, S=12288, H=16, D=128, k_scale=1000.0, v="ones", causal=False, seed=42):
    """E4M3 codes q, k, v [B,S,H,D] (uint8) and their descale factors."""
    g = _gen(seed)
    q = _randn(g, (B, S, H, D))
    k = _randn(g, (B, S, H, D)) * k_scale
    vv = torch.ones(B, S, H, D) if v == "ones" else _randn(g, (B, S, H, D))
    (qc, dq), (kc, dk), (vc, dv) = _to_e4m3(q), _to_e4m3(k), _to_e4m3(vv)
    return dict(q=qc, k=kc, v=vc, descale_q=dq, descale_k=dk, descale_v=dv, causal=causal,
                scale=1.0 / math.sqrt(D))


def dsa_case(B=1, S=512, Skv=2048, H=64, D=576, K=128, sink=True, length=True, seed=42,
             dtype=BF16):
    """Inputs of the sparse top-k backward (the forward's out and lse come
    from whichever side runs it).  Returns q [B,S,H,D], kv [B,Skv,D], dout
    [B,S,H,512] (16-bit), topk_idxs int32 [B,S,K], topk_length int32 [B,S]
    or None, attn_sink fp32 [H] or None."""
    g = _gen(seed)
    q = _randn(g, (B, S, H, D)).to(dtype)
    kv = _randn(g, (B, Skv, D)).to(dtype)
    dout = _randn(g, (B, S, H, 512)).to(dtype)
    keys = torch.rand(B, S, Skv, generator=g)
    idx = keys.argsort(dim=2)[:, :, :K].to(torch.int32)       # K distinct rows per token
    ln = None
    if length:
        ln = torch.randint(1, K + 1, (B, S), generator=g, dtype=torch.int32)
        pos = torch.arange(K, dtype=torch.int32)
        idx = torch.where(pos[None, None, :] < ln[:, :, None], idx, torch.full_like(idx, -1))
    sk = _randn(g, (H,)) if sink else None
    return dict(q=q, kv=kv, dout=dout, topk_idxs=idx.contiguous(), topk_length=ln, attn_sink=sk)
