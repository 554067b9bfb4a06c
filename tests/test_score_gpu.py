"""GPU parity of the head-summed score recompute against the fp64 oracle
(PFCCLab/cudnn-frontend PR #9, sections 2 and 3).

The library's own forward provides lse; both sides then take the same fp32
lse values, so the only differences are the fp32 score products on the
tensor cores and the hardware exp2: a few 1e-6 relative per term.  Bar:
score rel-L2 <= 1e-4 and every row's L1 norm within 1e-4 relative, zero NaN,
exact zeros where the oracle has them (causal pairs, columns past a varlen
sequence, unvisited rows), and bit-identical outputs on a second call (the
L1 partial sums are added in a fixed order).
"""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
from oracle import attn_oracle as O
from parity_utils import rel_l2, to64

pytestmark = pytest.mark.gpu

TOL_SCORE_REL = 1e-4
TOL_L1_REL = 1e-4


def _run(q, k, cu=None, max_seqlen=None, causal=False, scale=None):
    from softmax_attention_numerics_gb300 import attn_fwd, attn_score_recompute
    qd, kd = q.cuda(), k.cuda()
    cud = None if cu is None else torch.tensor(cu, dtype=torch.int32, device="cuda")
    _, lse = attn_fwd(qd, kd, kd, cu_seqlens=cud, max_seqlen=max_seqlen, causal=causal,
                      scale=scale)
    score, l1 = attn_score_recompute(qd, kd, lse, cu_seqlens=cud, max_seqlen=max_seqlen,
                                     causal=causal, scale=scale)
    torch.cuda.synchronize()
    return lse, score, l1


def _check(score, l1, ref_s, ref_l1, ctx):
    s, l = to64(score), to64(l1)
    assert np.isfinite(s).all() and np.isfinite(l).all(), ctx
    assert rel_l2(s, ref_s) <= TOL_SCORE_REL, (ctx, rel_l2(s, ref_s))
    assert (s[ref_s == 0] == 0).all(), ctx                       # hidden pairs exactly 0
    den = np.maximum(np.abs(ref_l1), 1e-30)
    assert (np.abs(l - ref_l1) / den)[ref_l1 != 0].max(initial=0) <= TOL_L1_REL, ctx
    assert (l[ref_l1 == 0] == 0).all(), ctx


DENSE = [  # (B, Sq, Sk, Hq, Hkv, D, causal, dtype)
    (2, 300, 300, 8, 2, 128, False, torch.bfloat16),
    (2, 384, 384, 4, 4, 64, True, torch.bfloat16),
    (1, 200, 333, 4, 1, 128, False, torch.bfloat16),
    (1, 256, 256, 64, 1, 128, True, torch.bfloat16),       # 64 heads sharing one kv head
    (2, 130, 130, 6, 3, 64, False, torch.float16),
    (1, 1, 77, 2, 1, 64, False, torch.bfloat16),
]


@pytest.mark.parametrize("cfg", DENSE, ids=[str(c[:7]) for c in DENSE])
def test_score_dense_matches_oracle(cfg):
    B, Sq, Sk, Hq, Hkv, D, causal, dt = cfg
    q, k, _, _ = W.dense_qkvdo(B, Sq, Sk, Hq, Hkv, D, seed=51, dtype=dt)
    sc = 1.0 / math.sqrt(D)
    lse, score, l1 = _run(q, k, causal=causal, scale=sc)
    ref_s, ref_l1 = O.attn_score_recompute(to64(q), to64(k), to64(lse), causal=causal, scale=sc)
    _check(score, l1, ref_s, ref_l1, "dense %s" % (cfg,))
    # the forward's own lse: every row's L1 norm is the number of heads
    assert np.allclose(to64(l1), Hq, rtol=TOL_L1_REL)


def test_score_varlen_with_trailing_rows():
    case = W.varlen_gqa(n=5, lo=100, hi=700, Hq=8, Hkv=2, D=128, trailing=61)
    cu = case["cu_seqlens"].tolist()
    lse, score, l1 = _run(case["q"], case["k"], cu=cu, max_seqlen=case["max_seqlen"], causal=True,
                          scale=case["scale"])
    ref_s, ref_l1 = O.attn_score_recompute(to64(case["q"]), to64(case["k"]), to64(lse), causal=True,
                                           scale=case["scale"], cu_seqlens=cu,
                                           max_seqlen=case["max_seqlen"])
    _check(score, l1, ref_s, ref_l1, "varlen")
    assert torch.count_nonzero(score[cu[-1]:]) == 0 and torch.count_nonzero(l1[cu[-1]:]) == 0


def test_score_varlen_unvisited_rows_are_overwritten():
    """PFCCLab PR #9, section 2: rows no tile visits must come back as 0, not
    whatever the buffer held (the leaked 64.0 of that page)."""
    from softmax_attention_numerics_gb300 import attn_fwd, attn_score_recompute
    case = W.varlen_gqa(n=3, lo=64, hi=200, Hq=4, Hkv=4, D=64, trailing=40)
    cu = case["cu_seqlens"].cuda()
    q, k = case["q"].cuda(), case["k"].cuda()
    _, lse = attn_fwd(q, k, k, cu_seqlens=cu, max_seqlen=case["max_seqlen"], causal=False)
    score = torch.full((q.shape[0], case["max_seqlen"]), 64.0, device="cuda")
    l1 = torch.full((q.shape[0],), 64.0, device="cuda")
    attn_score_recompute(q, k, lse, cu_seqlens=cu, max_seqlen=case["max_seqlen"], score=score, l1=l1)
    torch.cuda.synchronize()
    end = int(case["cu_seqlens"][-1])
    assert torch.count_nonzero(score[end:]) == 0 and torch.count_nonzero(l1[end:]) == 0
    lens = case["lens"]
    cuh = case["cu_seqlens"].tolist()
    for s, L in enumerate(lens):
        assert torch.count_nonzero(score[cuh[s]:cuh[s + 1], L:]) == 0   # columns past the sequence


def test_score_clamp_keeps_a_degenerate_lse_finite():
    """PFCCLab PR #9, section 3, the degenerate-lse probe: an lse far too
    small on a row makes every term exp2(+huge); the clamp keeps each term at
    2^120 and the score finite (the page: 37888 +inf score elements before the
    fix, none after); the row's L1 norm may saturate to +inf, which the page
    calls benign."""
    from softmax_attention_numerics_gb300 import attn_fwd, attn_score_recompute
    q, k, _, _ = W.dense_qkvdo(1, 200, 200, 64, 1, 128, seed=52)
    qd, kd = q.cuda(), k.cuda()
    _, lse = attn_fwd(qd, kd, kd, causal=True)
    lse[0, :, 150] = -1e30
    score, l1 = attn_score_recompute(qd, kd, lse, causal=True)
    torch.cuda.synchronize()
    assert not torch.isnan(score).any() and not torch.isinf(score).any()
    row = score[0, 150].double()
    assert torch.allclose(row[:151], torch.full_like(row[:151], 64 * 2.0 ** 120), rtol=1e-5)
    assert torch.count_nonzero(row[151:]) == 0
    assert torch.isinf(l1[0, 150])                        # 151 * 64 * 2^120 > FLT_MAX
    others = torch.cat([l1[0, :150], l1[0, 151:]])
    assert torch.allclose(others, torch.full_like(others, 64.0), rtol=TOL_L1_REL)


def test_score_is_bit_reproducible():
    q, k, _, _ = W.dense_qkvdo(2, 517, 517, 8, 2, 128, seed=53)
    lse, s1, l1a = _run(q, k, causal=True)
    from softmax_attention_numerics_gb300 import attn_score_recompute
    s2, l1b = attn_score_recompute(q.cuda(), k.cuda(), lse, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(s1, s2) and torch.equal(l1a, l1b)
