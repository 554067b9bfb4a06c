"""fp64 CPU oracle for sparse top-k attention with an attention sink (the DSA
forward and backward).

TEST INFRASTRUCTURE, NOT PART OF THE LIBRARY.  Only the test-suite, the smoke
check of ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
this module.  It shares no code with the CUDA path: it computes the plain
definition, one (batch, token) at a time, with numpy fp64 products.

Source: NVIDIA/cudnn-frontend PR #429, "Fix stream-ordering and
input-validation holes in the SM100 DSA backward interface" (Summary; API and
compatibility impact; the two review findings).  The page fixes the interface
of the backward: inputs q, kv, out, dout, lse, attn_sink, topk_idxs and an
optional topk_length; outputs dq, dkv and d_sink; head_dim 512, or 576 in the
MLA form where the query-key product uses all 576 columns and the values are
the first 512 columns of the same kv rows; one kv row set shared by all query
heads; the page's check runs S = 512 queries against S_kv = 2048 kv rows with
H = 64 heads and top-k = 128.  It does not print the formula; the readings
below are the plainest ones the interface supports:

* token i of batch b attends to the kv rows listed in topk_idxs[b, i, :]; an
  entry e takes part when e < topk_length[b, i] (all entries when no length
  is given) and 0 <= idx < S_kv; other entries (padding such as -1) take no
  part.  Each listed entry is one term (the generator never repeats a row).
* scores s_he = scale * q[b, i, h] . kv[b, idx_e]; the sink is one more logit
  per head, attn_sink[h], with no value:
      lse_h = log(exp(attn_sink[h]) + sum_e exp(s_he))   (natural log),
      P_he  = exp(s_he - lse_h),   P_sink,h = exp(attn_sink[h] - lse_h),
      out_h = sum_e P_he v_e,      v_e = kv[b, idx_e, :Dv].
  Without a sink the exp(attn_sink) term is absent; a token with no valid
  entry and no sink has out = 0, lse = 0 and no gradient (the convention of
  the dense oracle).
* backward, given dout: dP_he = dout_h . v_e, Delta_h = sum_e P_he dP_he
  (= dout_h . out_h), dS_he = P_he (dP_he - Delta_h),
      dq_h   = scale sum_e dS_he kv[idx_e],
      dkv[idx_e]       += scale sum_h dS_he q_h       (all Dqk columns),
      dkv[idx_e, :Dv]  += sum_h P_he dout_h          (the value part),
      d_sink[h]         = - sum_(b,i) P_sink,h Delta_h.
  The last line is the derivative of the loss through the normaliser alone:
  the sink has no value, so its only effect on out is to scale every P_he.

Layouts: q [B, S, H, Dqk]; kv [B, S_kv, Dqk]; topk_idxs [B, S, K] (int);
topk_length [B, S] (int) or None; attn_sink [H] or None; out / dout
[B, S, H, Dv]; lse [B, S, H]; dq like q, dkv like kv, d_sink [H].
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["dsa_fwd", "dsa_bwd", "valid_entries"]


def _as64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def valid_entries(idx_row, length, s_kv):
    """Positions e of one token's index list that take part, in list order."""
    K = len(idx_row)
    n = K if length is None else max(0, min(int(length), K))
    return [e for e in range(n) if 0 <= int(idx_row[e]) < s_kv]


def _token_fwd(qt, kv_b, rows, sink, scale, dv):
    """One (batch, token): qt [H, Dqk], kv rows `rows` -> P [H, n], Psink [H],
    out [H, Dv], lse [H]."""
    H = qt.shape[0]
    ksel = kv_b[rows]                                   # [n, Dqk]
    s = scale * (qt @ ksel.T)                           # [H, n]
    if sink is None:
        if len(rows) == 0:
            return np.zeros((H, 0)), np.zeros(H), np.zeros((H, dv)), np.zeros(H)
        m = s.max(axis=1)
        tot = np.exp(s - m[:, None]).sum(axis=1)
    else:
        m = np.maximum(sink, s.max(axis=1)) if len(rows) else sink.copy()
        tot = np.exp(sink - m) + np.exp(s - m[:, None]).sum(axis=1)
    lse = m + np.log(tot)
    P = np.exp(s - lse[:, None])
    psink = np.zeros(H) if sink is None else np.exp(sink - lse)
    out = P @ ksel[:, :dv]
    return P, psink, out, lse


def _token_bwd(qt, ksel, P, psink, dout_t, scale, dv):
    """Analytic gradients of one (batch, token) given its P, P_sink and dout:
    dq_t [H, Dqk], the dkv rows of its listed entries [n, Dqk], and its
    d_sink terms [H]."""
    dP = dout_t @ ksel[:, :dv].T                           # [H, n]
    delta = (P * dP).sum(axis=1)                            # [H]
    dS = P * (dP - delta[:, None])
    dq_t = scale * (dS @ ksel)
    gk = scale * (dS.T @ qt)                                # [n, Dqk]
    gk[:, :dv] += P.T @ dout_t
    return dq_t, gk, -psink * delta


def _prep(q, kv, topk_idxs, topk_length, attn_sink, scale, dv):
    q, kv, sink = _as64(q), _as64(kv), _as64(attn_sink)
    B, S, H, D = q.shape
    dv = D if dv is None else int(dv)
    assert kv.shape[0] == B and kv.shape[2] == D and dv <= D
    sc = 1.0 / math.sqrt(D) if scale is None else float(scale)
    idx = np.asarray(topk_idxs)
    ln = None if topk_length is None else np.asarray(topk_length)
    return q, kv, sink, idx, ln, B, S, H, D, dv, sc


def dsa_fwd(q, kv, topk_idxs, topk_length=None, attn_sink=None, scale=None, dv=None):
    """Sparse top-k forward.  Returns out [B,S,H,Dv], lse [B,S,H] (fp64)."""
    q, kv, sink, idx, ln, B, S, H, D, dv, sc = _prep(q, kv, topk_idxs, topk_length, attn_sink,
                                                      scale, dv)
    out = np.zeros((B, S, H, dv))
    lse = np.zeros((B, S, H))
    for b in range(B):
        for i in range(S):
            rows = [int(idx[b, i, e]) for e in
                    valid_entries(idx[b, i], None if ln is None else ln[b, i], kv.shape[1])]
            _, _, o, l = _token_fwd(q[b, i], kv[b], rows, sink, sc, dv)
            out[b, i], lse[b, i] = o, l
    return out, lse


def dsa_bwd(q, kv, dout, topk_idxs, topk_length=None, attn_sink=None, scale=None, dv=None):
    """Sparse top-k forward + backward.  Returns out, lse, dq, dkv, d_sink
    (fp64; d_sink is None without a sink)."""
    q, kv, sink, idx, ln, B, S, H, D, dv, sc = _prep(q, kv, topk_idxs, topk_length, attn_sink,
                                                      scale, dv)
    dout = _as64(dout)
    out = np.zeros((B, S, H, dv))
    lse = np.zeros((B, S, H))
    dq = np.zeros_like(q)
    dkv = np.zeros_like(kv)
    dsink = np.zeros(H)
    for b in range(B):
        for i in range(S):
            rows = [int(idx[b, i, e]) for e in
                    valid_entries(idx[b, i], None if ln is None else ln[b, i], kv.shape[1])]
            P, psink, o, l = _token_fwd(q[b, i], kv[b], rows, sink, sc, dv)
            out[b, i], lse[b, i] = o, l
            dq[b, i], gk, ds_t = _token_bwd(q[b, i], kv[b][rows], P, psink, dout[b, i], sc, dv)
            for e, r in enumerate(rows):
                dkv[b, r] += gk[e]
            dsink += ds_t
    return out, lse, dq, dkv, (dsink if sink is not None else None)
