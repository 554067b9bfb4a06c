"""fp64 CPU oracle for scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE, NOT PART OF THE LIBRARY.  Only the test-suite, the smoke
check of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
this module.  It shares no code with the CUDA path: it computes the plain
definition, one (batch, head) at a time, with numpy fp64 matrix products.

What it computes (the definition that every page relies on):

* scores   s_ij = scale * q_i . k_j + bias_ij, where bias is the user's
  additive mask, -inf for a bool mask entry that is False, -inf for a causal
  pair j > i (top-left alignment), and keys outside a sequence do not exist.
  Sources: flash-dmattn PR #122, "Problem" (causal call with ``scale=None``);
  OpenWAM PR #64, "Summary" and "Fix" (bool mask False = hidden, additive
  -inf = hidden, zero keys hidden in the mask get exactly zero attention).
* forward  P = softmax_j(s), out = P v, lse_i = m_i + log sum_j exp(s_ij - m_i)
  in natural log (OpenWAM PR #64, "Summary": the row log-sum-exp and
  exp(0 - lse)).  The oracle takes the exact row max m_i once; the GPU's
  online max / lazy rescale (FlyDSL PR #1033, "Root cause" and "The fix")
  must reach the same numbers.
* a row with no visible key (m_i = -inf) has out_i = 0 and lse_i = 0, and it
  contributes no gradient.  The pages do not define this row; 0 rather than
  -inf follows the reasoning of PFCCLab/cudnn-frontend PR #9, section 2
  (a -inf statistic turns into -inf - (-inf) = NaN downstream).
* backward (the standard analytic gradient of out = softmax(s) v with
  upstream gradient dO):
      dP = dO v^T,  Delta_i = sum_j P_ij dP_ij (= rowsum(dO * out)),
      dS = P * (dP - Delta),  dQ = scale dS K,  dK = scale dS^T Q,
      dV = P^T dO;
  with grouped-query attention (GQA) dK and dV of a kv head are summed over
  the q heads that share it (flash-dmattn PR #122 names num_heads and
  num_kv_heads).
* varlen packed sequences: rows [cu[s], cu[s+1]) form sequence s; rows past
  cu[-1] belong to no sequence and come back as out = 0, lse = 0 and zero
  gradients (PFCCLab/cudnn-frontend PR #9, section 2: rows the scheduler
  never visits must still be written).

* fp8 inputs: E4M3 codes with one descale factor per tensor are decoded
  from the format's definition and the forward is the same definition on
  the decoded values (FlyDSL PR #1033, "The fp8 helper, second commit").
* attention targets recomputed from the forward's lse and summed over the
  query heads, with the exponent clamped at 120, and each row's L1 norm
  (PFCCLab/cudnn-frontend PR #9, sections 2 and 3: the dense score
  recompute that produces the targets of a sparse-attention indexer).

Layouts follow the library: q/out/dout [B, Sq, Hq, D]; k/v [B, Sk, Hkv, D];
lse [B, Hq, Sq]; varlen q [T, Hq, D], k/v [T, Hkv, D], lse [Hq, T].
Masks are broadcastable to [B, Hq, Sq, Sk]: a bool array (True = visible) or a
float array (additive).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "attn_score_recompute",
    "attn_fwd",
    "attn_fwd_fp8",
    "e4m3_decode",
    "attn_bwd",
    "attn_varlen",
    "attn_rows",
    "bias_for",
]


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def bias_for(mask, b, h, Sq, Sk, causal, rows=None):
    """Additive fp64 bias for one (batch, q head): [Sq, Sk], or [len(rows), Sk].

    bool mask: True = visible (0), False = hidden (-inf).  Float mask: added
    as is.  Causal: key j > query i is hidden (top-left alignment).
    ``rows`` selects query rows (default: all Sq of them).
    """
    ri = np.arange(Sq) if rows is None else np.asarray(rows)
    bias = np.zeros((len(ri), Sk), dtype=np.float64)
    if mask is not None:
        m = np.asarray(mask)
        while m.ndim < 4:
            m = m[None]
        mb = m[b if m.shape[0] > 1 else 0, h if m.shape[1] > 1 else 0]
        mb = np.broadcast_to(mb, (Sq, Sk))[ri]
        if mb.dtype == np.bool_:
            bias = np.where(mb, 0.0, -np.inf)
        else:
            bias = bias + mb.astype(np.float64)
    if causal:
        j = np.arange(Sk)[None, :]
        bias = np.where(j > ri[:, None], -np.inf, bias)
    return bias


def _fwd_head(qh, kh, vh, bias, scale):
    """One (batch, head): returns P [Sq,Sk], out [Sq,D], lse [Sq].

    Softmax over the scores with the exact row max; rows with no visible key
    give P = 0, out = 0, lse = 0.
    """
    s = scale * (qh @ kh.T) + bias
    Sq, Sk = s.shape
    if Sk == 0:
        m = np.full(Sq, -np.inf)
    else:
        m = s.max(axis=1)
    live = m > -np.inf
    m_safe = np.where(live, m, 0.0)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for hidden keys
    e[~live] = 0.0
    l = e.sum(axis=1)
    P = np.zeros_like(e)
    P[live] = e[live] / l[live, None]
    out = P @ vh
    lse = np.zeros(Sq)
    lse[live] = m[live] + np.log(l[live])
    return P, out, lse


def _bwd_head(qh, kh, vh, P, dOh, scale):
    """Analytic gradients of one (batch, q head) given its P and dO."""
    dP = dOh @ vh.T
    delta = (P * dP).sum(axis=1)
    dS = P * (dP - delta[:, None])
    dq = scale * (dS @ kh)
    dk = scale * (dS.T @ qh)
    dv = P.T @ dOh
    return dq, dk, dv


def _default_scale(D, scale):
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def attn_fwd(q, k, v, mask=None, causal=False, scale=None):
    """Dense forward.  q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] -> out, lse [B,Hq,Sq]."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    sc = _default_scale(D, scale)
    out = np.zeros((B, Sq, Hq, v.shape[-1]))
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        for h in range(Hq):
            bias = bias_for(mask, b, h, Sq, Sk, causal)
            _, o, l = _fwd_head(q[b, :, h], k[b, :, h // G], v[b, :, h // G], bias, sc)
            out[b, :, h] = o
            lse[b, h] = l
    return out, lse


def attn_bwd(q, k, v, dout, mask=None, causal=False, scale=None):
    """Dense forward + backward.  Returns out, lse, dq, dk, dv (fp64)."""
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    sc = _default_scale(D, scale)
    out = np.zeros_like(q)
    lse = np.zeros((B, Hq, Sq))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            bias = bias_for(mask, b, h, Sq, Sk, causal)
            P, o, l = _fwd_head(q[b, :, h], k[b, :, hk], v[b, :, hk], bias, sc)
            out[b, :, h] = o
            lse[b, h] = l
            gq, gk, gv = _bwd_head(q[b, :, h], k[b, :, hk], v[b, :, hk], P, dout[b, :, h], sc)
            dq[b, :, h] = gq
            dk[b, :, hk] += gk
            dv[b, :, hk] += gv
    return out, lse, dq, dk, dv


def attn_varlen(q, k, v, dout, cu_seqlens, causal=False, scale=None, heads=None):
    """Packed varlen (THD) forward + backward.

    q/dout [T,Hq,D], k/v [T,Hkv,D]; sequence s owns rows [cu[s], cu[s+1]) of
    all four, so Sq = Sk per sequence.  Rows >= cu[-1] get zeros everywhere.
    ``heads`` optionally restricts the work to a subset of q heads (their
    kv heads' dK/dV then hold only those q heads' contributions).
    Returns out, lse [Hq,T], dq, dk, dv.
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = _default_scale(D, scale)
    cu = [int(x) for x in cu_seqlens]
    out = np.zeros_like(q)
    lse = np.zeros((Hq, T))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    hs = range(Hq) if heads is None else heads
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        L = e - a
        if L == 0:
            continue
        for h in hs:
            hk = h // G
            bias = bias_for(None, 0, 0, L, L, causal)
            P, o, l = _fwd_head(q[a:e, h], k[a:e, hk], v[a:e, hk], bias, sc)
            out[a:e, h] = o
            lse[h, a:e] = l
            gq, gk, gv = _bwd_head(q[a:e, h], k[a:e, hk], v[a:e, hk], P, dout[a:e, h], sc)
            dq[a:e, h] = gq
            dk[a:e, hk] += gk
            dv[a:e, hk] += gv
    return out, lse, dq, dk, dv


def attn_rows(q, k, v, dout, rows, mask=None, causal=False, scale=None):
    """Selected query rows of a dense problem.

    ``rows`` is a list of (b, h, i).  For each, returns out_i [D], lse_i and
    dq_i [D].  Row i's dq needs only its own P, dP and Delta, so the cost is
    O(Sk * D) per row; rows of one (b, h) are stacked into one matrix product.
    """
    q, k, v, dout = _as64(q), _as64(k), _as64(v), _as64(dout)
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    sc = _default_scale(D, scale)
    n = len(rows)
    outs = np.zeros((n, v.shape[-1]))
    lses = np.zeros(n)
    dqs = np.zeros((n, D))
    groups = {}
    for idx, (b, h, i) in enumerate(rows):
        groups.setdefault((b, h), []).append((idx, i))
    for (b, h), items in groups.items():
        hk = h // G
        idxs = [t[0] for t in items]
        ii = [t[1] for t in items]
        bias = bias_for(mask, b, h, Sq, Sk, causal, rows=ii)
        P, o, l = _fwd_head(q[b, ii, h], k[b, :, hk], v[b, :, hk], bias, sc)
        gq, _, _ = _bwd_head(q[b, ii, h], k[b, :, hk], v[b, :, hk], P, dout[b, ii, h], sc)
        outs[idxs] = o
        lses[idxs] = l
        dqs[idxs] = gq
    return outs, lses, dqs


# ---------------------------------------------------------------- fp8 inputs

def e4m3_decode(codes):
    """Value of each 8-bit E4M3 code (the OCP 8-bit floating-point format's
    finite-only E4M3: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent field 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN
    and there is no infinity, so the largest finite magnitude is
    1.75 * 2^8 = 448)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def attn_fwd_fp8(q_codes, k_codes, v_codes, descale_q, descale_k, descale_v, causal=False,
                 scale=None):
    """Forward on fp8 inputs: q, k, v are E4M3 codes with one descale factor
    per tensor (real value = decoded code * descale).  The fp8 forward of
    FlyDSL PR #1033 ("The fp8 helper, second commit") still computes
    softmax(scale * q k^T) v; only its route there (P rounded to fp8 for the
    P V product, a lazily rebased running max) is fp8-specific, so the oracle
    is the fp64 definition on the decoded inputs."""
    q = e4m3_decode(q_codes) * float(descale_q)
    k = e4m3_decode(k_codes) * float(descale_k)
    v = e4m3_decode(v_codes) * float(descale_v)
    return attn_fwd(q, k, v, causal=causal, scale=scale)


# ---------------------------------------------------------------- score recompute

SCORE_CLAMP_LOG2 = 120.0


def _score_terms(qh, kh, lse_h, bias, scale):
    """One (batch or sequence, q head): exp2(min(log2(e) (s - lse), 120)),
    [rows, keys]; hidden pairs (bias -inf) give exactly 0."""
    s = scale * (qh @ kh.T) + bias
    t = np.log2(np.e) * (s - lse_h[:, None])
    return np.exp2(np.minimum(t, SCORE_CLAMP_LOG2))


def attn_score_recompute(q, k, lse, causal=False, scale=None, cu_seqlens=None, max_seqlen=None):
    """Attention targets recomputed from the forward's lse, summed over heads.

    PFCCLab/cudnn-frontend PR #9, section 3 (the dense score recompute): for a
    query row i and a key j of its sequence,
        score_ij = sum over q heads h of exp2(min(log2(e) (s_hij - lse_hi), 120))
    with s_hij = scale q_hi . k_j (k of h's kv head; hidden pairs - causal
    j > i - contribute 0), and the row's L1 norm l1_i = sum_j score_ij; the
    consumer's target is score_ij / l1_i.  The clamp bounds every term by
    2^120 so that the sum over heads stays finite (2^120 * 64 < FLT_MAX) even
    when an lse is far too small; with the forward's own lse each head's
    terms over j sum to 1, so l1_i is the number of heads with a visible key.
    Section 2: rows that no tile visits (varlen rows past cu[-1]) come back
    as 0, not -inf, in both outputs.

    dense:  q [B,Sq,Hq,D], k [B,Sk,Hkv,D], lse [B,Hq,Sq] -> score [B,Sq,Sk], l1 [B,Sq]
    varlen: q [T,Hq,D], k [T,Hkv,D], lse [Hq,T], cu_seqlens [n+1] ->
            score [T, max_seqlen] (row cu[s] + i holds keys 0.. of sequence s;
            columns past the sequence are 0), l1 [T]
    """
    q, k, lse = _as64(q), _as64(k), _as64(lse)
    if cu_seqlens is None:
        B, Sq, Hq, D = q.shape
        Sk, Hkv = k.shape[1], k.shape[2]
        G = Hq // Hkv
        sc = _default_scale(D, scale)
        score = np.zeros((B, Sq, Sk))
        for b in range(B):
            bias = bias_for(None, 0, 0, Sq, Sk, causal)
            for h in range(Hq):
                score[b] += _score_terms(q[b, :, h], k[b, :, h // G], lse[b, h], bias, sc)
        return score, score.sum(axis=2)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = _default_scale(D, scale)
    cu = [int(x) for x in cu_seqlens]
    W = int(max_seqlen) if max_seqlen is not None else max(
        [cu[i + 1] - cu[i] for i in range(len(cu) - 1)] + [0])
    score = np.zeros((T, W))
    for si in range(len(cu) - 1):
        a, e = cu[si], cu[si + 1]
        L = e - a
        if L == 0:
            continue
        bias = bias_for(None, 0, 0, L, L, causal)
        for h in range(Hq):
            score[a:e, :L] += _score_terms(q[a:e, h], k[a:e, h // G], lse[h, a:e], bias, sc)
    return score, score.sum(axis=1)

