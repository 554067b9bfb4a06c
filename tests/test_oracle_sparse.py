"""Pins for the sparse top-k (DSA) oracle, independent of its own formulas.

Each check ties ``oracle/sparse_oracle.py`` to something it does not compute
itself: central finite differences of L = sum(out * dout) with respect to q,
kv and the sink; the attention sink written as one more kv row (an extra
column carries the sink logit, the row's value is zero) and run through the
no-sink path; the dense fp64 oracle when every key is listed; PyTorch fp64
autograd of a gather + softmax written independently here; closed forms and
invariants.  The mutation tests at the end plant plausible mistakes in the
oracle (on the CPU) and check that the pins catch them.

Source: NVIDIA/cudnn-frontend PR #429 (the DSA backward interface: q, kv,
out, dout, lse, attn_sink, topk_idxs, topk_length -> dq, dkv, d_sink; head
dim 512 or 576 with values in the first 512 columns).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attn_oracle as DO
from oracle import sparse_oracle as O


def sparse_case(seed, B=2, S=3, H=2, D=6, Dv=4, Skv=9, K=5, sink=True, length=True, pad=True):
    """Random inputs; each token lists distinct kv rows, some entries are -1
    padding and (with `length`) some lie past the token's topk_length."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, S, H, D))
    kv = rng.standard_normal((B, Skv, D))
    dout = rng.standard_normal((B, S, H, Dv))
    idx = np.stack([np.stack([rng.permutation(Skv)[:K] for _ in range(S)]) for _ in range(B)])
    if pad:
        idx[:, :, -1] = -1
    ln = rng.integers(1, K + 1, size=(B, S)) if length else None
    sk = rng.standard_normal(H) if sink else None
    return dict(q=q, kv=kv, dout=dout, topk_idxs=idx, topk_length=ln, attn_sink=sk, dv=Dv)


def fd_error(c, scale=0.43, h=1e-6, bwd=None):
    """max |analytic - central FD| / max(1, |FD|) over q, kv and the sink."""
    bwd = bwd or O.dsa_bwd
    args = dict(topk_idxs=c["topk_idxs"], topk_length=c["topk_length"], scale=scale, dv=c["dv"])
    _, _, dq, dkv, ds = bwd(c["q"], c["kv"], c["dout"], attn_sink=c["attn_sink"], **args)

    def loss(q, kv, sk):
        out, _ = O.dsa_fwd(q, kv, attn_sink=sk, **args)
        return float((out * c["dout"]).sum())

    worst = 0.0
    names = [("q", dq), ("kv", dkv)] + ([("attn_sink", ds)] if c["attn_sink"] is not None else [])
    for name, g in names:
        x = c[name]
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            ix = it.multi_index
            vals = {"q": c["q"], "kv": c["kv"], "attn_sink": c["attn_sink"]}
            xp = x.copy(); xp[ix] += h
            xm = x.copy(); xm[ix] -= h
            vals[name] = xp
            lp = loss(vals["q"], vals["kv"], vals["attn_sink"])
            vals[name] = xm
            lm = loss(vals["q"], vals["kv"], vals["attn_sink"])
            fd = (lp - lm) / (2 * h)
            worst = max(worst, abs(fd - g[ix]) / max(1.0, abs(fd)))
    return worst


def torch_reference(c, scale):
    """PyTorch fp64 autograd of the plain gather + softmax (the sink as one
    more logit with no value).  Returns out, lse, dq, dkv, d_sink."""
    q = torch.tensor(c["q"], requires_grad=True)
    kv = torch.tensor(c["kv"], requires_grad=True)
    sink = None if c["attn_sink"] is None else torch.tensor(c["attn_sink"], requires_grad=True)
    B, S, H, D = q.shape
    Skv, Dv = kv.shape[1], c["dv"]
    outs, lses = [], []
    for b in range(B):
        for i in range(S):
            n = c["topk_idxs"].shape[2] if c["topk_length"] is None else int(c["topk_length"][b, i])
            rows = [int(r) for r in c["topk_idxs"][b, i, :n] if 0 <= int(r) < Skv]
            ksel = kv[b, rows]
            logits = scale * q[b, i] @ ksel.T
            if sink is not None:
                logits = torch.cat([logits, sink[:, None]], dim=1)
            if logits.shape[1] == 0:
                outs.append(torch.zeros(H, Dv, dtype=q.dtype))
                lses.append(torch.zeros(H, dtype=q.dtype))
                continue
            w = torch.softmax(logits, dim=1)[:, :len(rows)]
            outs.append(w @ ksel[:, :Dv])
            lses.append(torch.logsumexp(logits, dim=1))
    out = torch.stack(outs).reshape(B, S, H, Dv)
    lse = torch.stack(lses).reshape(B, S, H)
    (out * torch.tensor(c["dout"])).sum().backward()
    return (out.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), kv.grad.numpy(),
            None if sink is None else sink.grad.numpy())


def torch_error(c, scale=0.29, bwd=None):
    bwd = bwd or O.dsa_bwd
    got = bwd(c["q"], c["kv"], c["dout"], c["topk_idxs"], topk_length=c["topk_length"],
              attn_sink=c["attn_sink"], scale=scale, dv=c["dv"])
    ref = torch_reference(c, scale)
    worst = 0.0
    for g, r in zip(got, ref):
        if r is None:
            assert g is None
            continue
        worst = max(worst, float(np.abs(g - r).max() / max(1.0, np.abs(r).max())))
    return worst


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("sink,length", [(True, True), (False, True), (True, False), (False, False)])
def test_fd_sparse(sink, length):
    assert fd_error(sparse_case(1, sink=sink, length=length)) < 1e-7


def test_fd_mla_shape_and_large_sink():
    c = sparse_case(2, H=3, D=8, Dv=4, Skv=11, K=6)
    c["attn_sink"] = np.array([3.0, -2.0, 0.5])       # a sink that dominates one head
    assert fd_error(c, scale=0.6) < 1e-7


# ---------------------------------------------------------------- library routine

@pytest.mark.parametrize("seed,sink,length", [(3, True, True), (4, False, True), (5, True, False)])
def test_matches_torch_autograd(seed, sink, length):
    c = sparse_case(seed, B=2, S=8, H=4, D=40, Dv=32, Skv=50, K=12, sink=sink, length=length)
    assert torch_error(c) < 1e-12


def test_matches_torch_autograd_page_like_shape():
    """H = 64 heads, Dqk = 72 / Dv = 64 (the 576 / 512 split scaled by 1/8),
    top-k = 16 of 64 kv rows."""
    c = sparse_case(6, B=1, S=4, H=64, D=72, Dv=64, Skv=64, K=16)
    assert torch_error(c, scale=1 / math.sqrt(72)) < 1e-12


# ---------------------------------------------------------------- other paths

def test_sink_is_a_zero_value_kv_row():
    """The sink logit of head h equals the score of one extra kv row whose
    extra column is 1 (the query's extra column is sink_h / scale) and whose
    value columns are 0.  The no-sink path on the extended problem then gives
    the same out, lse, dq, dkv, and d_sink = sum_i dq'[i, h, extra] / scale."""
    c = sparse_case(7, B=2, S=4, H=3, D=6, Dv=4, Skv=9, K=5)
    sc = 0.37
    out, lse, dq, dkv, ds = O.dsa_bwd(c["q"], c["kv"], c["dout"], c["topk_idxs"], c["topk_length"],
                                      c["attn_sink"], scale=sc, dv=4)
    B, S, H, D = c["q"].shape
    Skv, K = c["kv"].shape[1], c["topk_idxs"].shape[2]
    q2 = np.concatenate([c["q"], np.broadcast_to(c["attn_sink"] / sc, (B, S, H))[..., None]], -1)
    kv2 = np.zeros((B, Skv + 1, D + 1))
    kv2[:, :Skv, :D] = c["kv"]
    kv2[:, Skv, D] = 1.0
    # the extra row goes first in every list, so the length grows by one
    idx2 = np.concatenate([np.full((B, S, 1), Skv), c["topk_idxs"]], axis=2)
    ln2 = c["topk_length"] + 1
    out2, lse2, dq2, dkv2, ds2 = O.dsa_bwd(q2, kv2, c["dout"], idx2, ln2, None, scale=sc, dv=4)
    assert ds2 is None and K + 1 == idx2.shape[2]
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq2[..., :D], dq, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dkv2[:, :Skv, :D], dkv, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dq2[..., D].sum(axis=(0, 1)) / sc, ds, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("mla", [False, True])
def test_all_keys_listed_equals_dense_oracle(mla):
    """Every kv row listed, no sink: the dense fp64 oracle with one kv head
    (k = kv, v = kv's value columns padded with zeros to D) gives the same
    out, lse, dq, and dk + dv = dkv."""
    rng = np.random.default_rng(8)
    B, S, H, D, Skv = 2, 5, 3, 8, 7
    Dv = 6 if mla else D
    q = rng.standard_normal((B, S, H, D))
    kv = rng.standard_normal((B, Skv, D))
    dout = rng.standard_normal((B, S, H, Dv))
    idx = np.broadcast_to(np.arange(Skv)[::-1], (B, S, Skv)).copy()
    out, lse, dq, dkv, _ = O.dsa_bwd(q, kv, dout, idx, scale=0.5, dv=Dv)
    v = np.zeros((B, Skv, 1, D))
    v[..., :Dv] = kv[:, :, None, :Dv]
    dpad = np.zeros((B, S, H, D))
    dpad[..., :Dv] = dout
    o_d, l_d, dq_d, dk_d, dv_d = DO.attn_bwd(q, kv[:, :, None, :], v, dpad, scale=0.5)
    np.testing.assert_allclose(out, o_d[..., :Dv], rtol=1e-12, atol=1e-13)
    assert np.abs(o_d[..., Dv:]).max(initial=0) == 0
    np.testing.assert_allclose(lse, l_d.transpose(0, 2, 1), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, dq_d, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dkv, dk_d[:, :, 0] + dv_d[:, :, 0], rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- closed forms

def test_single_entry_without_sink():
    """One valid entry: P = 1, out = v, lse = s, no score gradient (dS = 0),
    so dq = 0 and dkv of that row = (sum_h dout_h, 0 in the extra columns)."""
    c = sparse_case(9, B=1, S=2, H=3, D=6, Dv=4, Skv=5, K=3, sink=False)
    c["topk_length"] = np.ones((1, 2), dtype=np.int64)
    c["topk_idxs"][0, :, 0] = [2, 4]
    out, lse, dq, dkv, _ = O.dsa_bwd(c["q"], c["kv"], c["dout"], c["topk_idxs"], c["topk_length"],
                                     scale=0.7, dv=4)
    for i, r in enumerate([2, 4]):
        np.testing.assert_allclose(out[0, i], np.broadcast_to(c["kv"][0, r, :4], (3, 4)), rtol=1e-14)
        np.testing.assert_allclose(lse[0, i], 0.7 * c["q"][0, i] @ c["kv"][0, r], rtol=1e-13)
        np.testing.assert_allclose(dkv[0, r, :4], c["dout"][0, i].sum(axis=0), rtol=1e-13)
        assert np.abs(dkv[0, r, 4:]).max() < 1e-14
    assert np.abs(dq).max() < 1e-14
    assert np.abs(dkv[0, [0, 1, 3]]).max() == 0


def test_no_entry_with_sink():
    """No valid entry: lse = sink, out = 0, zero gradients (Delta = 0)."""
    c = sparse_case(10, B=1, S=2, H=3, D=6, Dv=4, Skv=5, K=3)
    c["topk_idxs"][:] = -1
    out, lse, dq, dkv, ds = O.dsa_bwd(c["q"], c["kv"], c["dout"], c["topk_idxs"], None,
                                      c["attn_sink"], scale=0.7, dv=4)
    np.testing.assert_array_equal(lse[0], np.broadcast_to(c["attn_sink"], (2, 3)))
    assert not out.any() and not dq.any() and not dkv.any() and not ds.any()


def test_equal_logits_share_with_the_sink():
    """q = 0 and sink = 0: every entry and the sink weigh 1 / (n + 1), so
    out = n / (n + 1) * mean of the listed values, lse = log(n + 1)."""
    c = sparse_case(11, B=1, S=1, H=2, D=6, Dv=4, Skv=8, K=5, length=False, pad=False)
    c["q"][:] = 0
    c["attn_sink"] = np.zeros(2)
    out, lse = O.dsa_fwd(c["q"], c["kv"], c["topk_idxs"], attn_sink=c["attn_sink"], dv=4)
    rows = c["topk_idxs"][0, 0]
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(c["kv"][0, rows, :4].sum(0) / 6, (2, 4)),
                               rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(6), rtol=1e-14)


# ---------------------------------------------------------------- invariants

def _run(c, **kw):
    return O.dsa_bwd(c["q"], c["kv"], c["dout"], kw.get("idx", c["topk_idxs"]),
                     kw.get("ln", c["topk_length"]), c["attn_sink"], scale=0.5, dv=c["dv"])


def _close(a, b):
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)


def test_entry_order_does_not_matter():
    c = sparse_case(12, length=False)
    perm = np.random.default_rng(0).permutation(c["topk_idxs"].shape[2])
    _close(_run(c), _run(c, idx=c["topk_idxs"][:, :, perm]))


def test_entries_past_the_length_are_ignored():
    c = sparse_case(13, Skv=20, K=6)
    idx2 = c["topk_idxs"].copy()
    for b in range(idx2.shape[0]):
        for i in range(idx2.shape[1]):
            idx2[b, i, c["topk_length"][b, i]:] = 19 - b        # any valid row
    _close(_run(c), _run(c, idx=idx2))


def test_padding_equals_a_shorter_length():
    c = sparse_case(14, length=False)                          # last entry is -1
    _close(_run(c), _run(c, ln=np.full(c["topk_idxs"].shape[:2], c["topk_idxs"].shape[2] - 1)))


def test_sink_at_minus_infinity_is_no_sink():
    c = sparse_case(15)
    none = _run(dict(c, attn_sink=None))
    b = _run(dict(c, attn_sink=np.full(c["attn_sink"].shape, -np.inf)))
    assert not np.allclose(_run(c)[0], none[0])               # a finite sink matters
    _close(b[:4], none[:4])
    assert not b[4].any()


def test_dsink_is_minus_sink_weight_times_delta():
    """d_sink_h = -sum_i P_sink,ih (dout_ih . out_ih), with P_sink from lse."""
    c = sparse_case(16, S=5)
    out, lse, _, _, ds = _run(c)
    psink = np.exp(c["attn_sink"][None, None, :] - lse)
    np.testing.assert_allclose(ds, -(psink * (c["dout"] * out).sum(-1)).sum(axis=(0, 1)),
                               rtol=1e-12)


# ---------------------------------------------------------------- mutation tests

ORIG_BWD = O.dsa_bwd
ORIG_TOKEN_FWD = O._token_fwd
ORIG_TOKEN_BWD = O._token_bwd


def _bwd_dsink_sign(*a, **k):
    r = list(ORIG_BWD(*a, **k))
    r[4] = -r[4]
    return tuple(r)


def _token_bwd_no_value_part(qt, ksel, P, psink, dout_t, scale, dv):
    """dkv rows without sum_h P_he dout_h (only the score part)."""
    dq_t, gk, ds = ORIG_TOKEN_BWD(qt, ksel, P, psink, dout_t, scale, dv)
    gk[:, :dv] -= P.T @ dout_t
    return dq_t, gk, ds


def _token_bwd_unscaled_dq(qt, ksel, P, psink, dout_t, scale, dv):
    dq_t, gk, ds = ORIG_TOKEN_BWD(qt, ksel, P, psink, dout_t, scale, dv)
    return dq_t / scale, gk, ds


def _token_bwd_value_part_on_last_columns(qt, ksel, P, psink, dout_t, scale, dv):
    """The value gradient added to the last Dv columns instead of the first."""
    dq_t, gk, ds = ORIG_TOKEN_BWD(qt, ksel, P, psink, dout_t, scale, dv)
    vp = P.T @ dout_t
    gk[:, :dv] -= vp
    gk[:, gk.shape[1] - dv:] += vp
    return dq_t, gk, ds


def _token_fwd_lse_without_sink(qt, kv_b, rows, sink, scale, dv):
    P, psink, out, lse = ORIG_TOKEN_FWD(qt, kv_b, rows, None, scale, dv)
    if sink is not None:
        psink = np.exp(sink - lse) if len(rows) else np.ones_like(sink)
    return P, psink, out, lse


def _valid_entries_ignoring_length(idx_row, length, s_kv):
    return [e for e in range(len(idx_row)) if 0 <= int(idx_row[e]) < s_kv]


def test_pins_catch_wrong_dsink_sign():
    c = sparse_case(20)
    assert fd_error(c, bwd=_bwd_dsink_sign) > 1e-3
    assert torch_error(c, bwd=_bwd_dsink_sign) > 1e-3


@pytest.mark.parametrize("mutant", [_token_bwd_no_value_part, _token_bwd_unscaled_dq,
                                    _token_bwd_value_part_on_last_columns])
def test_pins_catch_planted_token_bwd_mistakes(monkeypatch, mutant):
    c = sparse_case(21)
    monkeypatch.setattr(O, "_token_bwd", mutant)
    assert fd_error(c) > 1e-3
    assert torch_error(c) > 1e-3


def test_pins_catch_sink_missing_from_lse(monkeypatch):
    c = sparse_case(22)
    monkeypatch.setattr(O, "_token_fwd", _token_fwd_lse_without_sink)
    assert fd_error(c) > 1e-3
    assert torch_error(c) > 1e-3


def test_pins_catch_ignored_length(monkeypatch):
    c = sparse_case(23, pad=False)
    monkeypatch.setattr(O, "valid_entries", _valid_entries_ignoring_length)
    assert torch_error(c) > 1e-3
