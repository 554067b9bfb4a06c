"""Pins for the fp64 oracle, independent of the oracle's own formulas.

Each check ties the oracle to something it does not compute itself:
central finite differences of L = sum(out * dO), closed forms, invariants,
the textbook CPU fp64 attention of PyTorch, and a hand-derived worked example
stored under tests/golden/.  The mutation tests at the end plant plausible
mistakes in the oracle (on the CPU) and check that the pins catch them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attn_oracle as O
from parity_utils import oracle_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _rand(*shape, rng=None):
    return (rng or RNG).standard_normal(shape)


# ---------------------------------------------------------------- pins as functions

def fd_grad_error(q, k, v, dout, mask=None, causal=False, scale=0.37, h=1e-6):
    """max |analytic - central FD| / max(1, |FD|) over every input element of
    L = sum(out * dO)."""
    _, _, dq, dk, dv = O.attn_bwd(q, k, v, dout, mask=mask, causal=causal, scale=scale)

    def loss(qq, kk, vv):
        out, _ = O.attn_fwd(qq, kk, vv, mask=mask, causal=causal, scale=scale)
        return float((out * dout).sum())

    worst = 0.0
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {"q": q, "k": k, "v": v}
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"])
            fd = (lp - lm) / (2 * h)
            worst = max(worst, abs(fd - g[idx]) / max(1.0, abs(fd)))
    return worst


def fd_varlen_error(q, k, v, dout, cu, causal, scale=0.41, h=1e-6):
    _, _, dq, dk, dv = O.attn_varlen(q, k, v, dout, cu, causal=causal, scale=scale)

    def loss(qq, kk, vv):
        out, _, _, _, _ = O.attn_varlen(qq, kk, vv, dout, cu, causal=causal, scale=scale)
        return float((out * dout).sum())

    worst = 0.0
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {"q": q, "k": k, "v": v}
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args[name] = xp
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm
            lm = loss(args["q"], args["k"], args["v"])
            worst = max(worst, abs((lp - lm) / (2 * h) - g[idx]) / max(1.0, abs((lp - lm) / (2 * h))))
    return worst


def lse_vs_weights_error(q, k, mask=None, causal=False, scale=0.5, h=1e-6):
    """d lse_i / d bias_ij (central FD through an additive mask) must equal the
    attention weight P_ij, which the oracle's out exposes when V holds one-hot
    rows (out_i = sum_j P_ij e_j).  Ties lse to out without reusing either
    formula."""
    B, Sq, Hq, D = q.shape
    Sk, Hkv = k.shape[1], k.shape[2]
    assert Sk <= 64
    v = np.zeros((B, Sk, Hkv, Sk))
    for j in range(Sk):
        v[:, j, :, j] = 1.0
    base = np.zeros((B, Hq, Sq, Sk)) if mask is None else mask.astype(np.float64).copy()
    base = np.broadcast_to(base, (B, Hq, Sq, Sk)).copy()
    out, lse = O.attn_fwd(q, k, v, mask=base, causal=causal, scale=scale)
    worst = 0.0
    for b in range(B):
        for hh in range(Hq):
            for i in range(Sq):
                for j in range(Sk):
                    if not np.isfinite(base[b, hh, i, j]) or (causal and j > i):
                        continue
                    bp = base.copy(); bp[b, hh, i, j] += h
                    bm = base.copy(); bm[b, hh, i, j] -= h
                    _, lp = O.attn_fwd(q, k, v, mask=bp, causal=causal, scale=scale)
                    _, lm = O.attn_fwd(q, k, v, mask=bm, causal=causal, scale=scale)
                    fd = (lp[b, hh, i] - lm[b, hh, i]) / (2 * h)
                    worst = max(worst, abs(fd - out[b, i, hh, j]))
    return worst


def tiny_case(seed, B=1, Sq=5, Sk=7, Hq=2, Hkv=1, D=4):
    rng = np.random.default_rng(seed)
    return (_rand(B, Sq, Hq, D, rng=rng), _rand(B, Sk, Hkv, D, rng=rng),
            _rand(B, Sk, Hkv, D, rng=rng), _rand(B, Sq, Hq, D, rng=rng))


FD_TOL = 1e-7

# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("causal", [False, True])
def test_fd_dense_gqa(causal):
    q, k, v, do = tiny_case(1, Sq=5, Sk=5 if causal else 7)
    assert fd_grad_error(q, k, v, do, causal=causal) < FD_TOL


def test_fd_bool_mask():
    q, k, v, do = tiny_case(2)
    mask = np.ones((1, 2, 5, 7), dtype=bool)
    mask[..., 5:] = False            # key padding
    mask[0, 1, 2, 1] = False         # one extra hidden pair
    assert fd_grad_error(q, k, v, do, mask=mask) < FD_TOL


def test_fd_additive_mask_finite_values():
    q, k, v, do = tiny_case(3)
    add = _rand(1, 1, 5, 7) * 0.7
    add[..., -1] = -np.inf
    assert fd_grad_error(q, k, v, do, mask=add) < FD_TOL


def test_fd_sq_ne_sk_and_batch():
    q, k, v, do = tiny_case(4, B=2, Sq=3, Sk=6, Hq=3, Hkv=3, D=3)
    assert fd_grad_error(q, k, v, do, causal=True) < FD_TOL


def test_fd_varlen_with_trailing_rows():
    rng = np.random.default_rng(5)
    cu = [0, 3, 7]
    T = 9                              # rows 7, 8 belong to no sequence
    q = _rand(T, 2, 3, rng=rng); k = _rand(T, 1, 3, rng=rng)
    v = _rand(T, 1, 3, rng=rng); do = _rand(T, 2, 3, rng=rng)
    assert fd_varlen_error(q, k, v, do, cu, causal=True) < FD_TOL
    out, lse, dq, dk, dv = O.attn_varlen(q, k, v, do, cu, causal=True)
    for t in (out, dq, dk, dv):
        assert np.all(t[7:] == 0.0)
    assert np.all(lse[:, 7:] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_lse_derivative_is_attention_weight(causal):
    rng = np.random.default_rng(6)
    q = _rand(1, 4, 2, 3, rng=rng)
    k = _rand(1, 4, 1, 3, rng=rng)
    assert lse_vs_weights_error(q, k, causal=causal) < 1e-8


# ---------------------------------------------------------------- closed forms

def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(7)
    B, Sq, Sk, H, D = 1, 3, 6, 1, 5
    q = np.zeros((B, Sq, H, D)); k = _rand(B, Sk, H, D, rng=rng); v = _rand(B, Sk, H, D, rng=rng)
    vis = np.array([True, False, True, True, False, True])
    mask = np.broadcast_to(vis, (B, H, Sq, Sk))
    out, lse = O.attn_fwd(q, k, v, mask=mask, scale=0.3)
    expect = v[0, vis, 0].mean(axis=0)
    assert np.allclose(out[0, :, 0], expect, atol=1e-14)
    assert np.allclose(lse, math.log(vis.sum()), atol=1e-14)


def test_single_visible_key():
    rng = np.random.default_rng(8)
    B, Sq, Sk, H, D = 1, 2, 5, 1, 4
    q, k, v, do = (_rand(B, Sq, H, D, rng=rng), _rand(B, Sk, H, D, rng=rng),
                   _rand(B, Sk, H, D, rng=rng), _rand(B, Sq, H, D, rng=rng))
    j = 3
    mask = np.zeros((B, H, Sq, Sk), dtype=bool); mask[..., j] = True
    sc = 0.45
    out, lse, dq, dk, dv = O.attn_bwd(q, k, v, do, mask=mask, scale=sc)
    assert np.allclose(out[0, :, 0], v[0, j, 0][None], atol=1e-14)
    assert np.allclose(lse[0, 0], sc * q[0, :, 0] @ k[0, j, 0], atol=1e-13)
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    assert np.allclose(dv[0, j, 0], do[0, :, 0].sum(axis=0), atol=1e-14)
    others = [i for i in range(Sk) if i != j]
    assert np.all(dv[0, others] == 0.0)


def test_equal_value_rows():
    rng = np.random.default_rng(9)
    q, k, _, do = tiny_case(9)
    c = _rand(4, rng=rng)
    v = np.broadcast_to(c, (1, 7, 1, 4)).copy()
    out, lse, dq, dk, dv = O.attn_bwd(q, k, v, do, causal=False, scale=0.6)
    assert np.allclose(out, c, atol=1e-14)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


def test_constant_logit_shift():
    q, k, v, do = tiny_case(10)
    c = 3.25
    out0, lse0 = O.attn_fwd(q, k, v, scale=0.5)
    out1, lse1 = O.attn_fwd(q, k, v, mask=np.full((1, 1, 1, 7), c), scale=0.5)
    assert np.allclose(out0, out1, atol=1e-14)
    assert np.allclose(lse1 - lse0, c, atol=1e-13)


def test_causal_first_row_sees_only_first_key():
    q, k, v, do = tiny_case(11, Sq=6, Sk=6)
    out, lse = O.attn_fwd(q, k, v, causal=True, scale=0.7)
    assert np.allclose(out[0, 0, :], v[0, 0, 0][None], atol=1e-14)
    assert np.allclose(lse[0, :, 0], 0.7 * np.einsum("hd,d->h", q[0, 0], k[0, 0, 0]), atol=1e-14)


def test_fully_masked_row_is_zero():
    q, k, v, do = tiny_case(12)
    mask = np.ones((1, 2, 5, 7), dtype=bool)
    mask[0, 1, 3, :] = False
    out, lse, dq, dk, dv = O.attn_bwd(q, k, v, do, mask=mask, scale=0.5)
    assert np.all(out[0, 3, 1] == 0) and lse[0, 1, 3] == 0 and np.all(dq[0, 3, 1] == 0)
    for t in (out, lse, dq, dk, dv):
        assert np.isfinite(t).all()


# ---------------------------------------------------------------- invariants

def test_weights_rows_sum_to_one():
    rng = np.random.default_rng(13)
    q = _rand(1, 6, 2, 3, rng=rng); k = _rand(1, 8, 2, 3, rng=rng)
    v = np.zeros((1, 8, 2, 8))
    for j in range(8):
        v[:, j, :, j] = 1.0
    out, _ = O.attn_fwd(q, k, v, causal=True, scale=1.3)
    assert np.all(out >= 0)
    assert np.allclose(out.sum(axis=-1), 1.0, atol=1e-14)


def test_dk_sums_to_zero_per_head():
    q, k, v, do = tiny_case(14, Hq=4, Hkv=2)
    _, _, _, dk, _ = O.attn_bwd(q, k, v, do, causal=False, scale=0.5)
    assert np.abs(dk.sum(axis=1)).max() < 1e-13


def test_masked_keys_get_zero_grad():
    q, k, v, do = tiny_case(15)
    mask = np.ones((1, 1, 1, 7), dtype=bool); mask[..., 2] = False; mask[..., 6] = False
    _, _, _, dk, dv = O.attn_bwd(q, k, v, do, mask=mask, scale=0.5)
    assert np.all(dk[:, [2, 6]] == 0.0) and np.all(dv[:, [2, 6]] == 0.0)


@pytest.mark.parametrize("kind", ["bool", "additive", "none"])
def test_appending_masked_zero_keys_changes_nothing(kind):
    """OpenWAM PR #64, "Fix" / "Tests": zero keys hidden in the mask get exactly
    zero attention, so outputs and gradients are unchanged."""
    q, k, v, do = tiny_case(16, Sq=4, Sk=5)
    pad = 3
    k2 = np.concatenate([k, np.zeros((1, pad, 1, 4))], axis=1)
    v2 = np.concatenate([v, np.zeros((1, pad, 1, 4))], axis=1)
    if kind == "bool":
        m1 = np.ones((1, 1, 1, 5), dtype=bool); m1[..., 1] = False
        m2 = np.concatenate([m1, np.zeros((1, 1, 1, pad), dtype=bool)], axis=-1)
    elif kind == "additive":
        m1 = np.zeros((1, 1, 1, 5)); m1[..., 1] = -np.inf
        m2 = np.concatenate([m1, np.full((1, 1, 1, pad), -np.inf)], axis=-1)
    else:
        m1 = None
        m2 = np.concatenate([np.ones((1, 1, 1, 5), bool), np.zeros((1, 1, 1, pad), bool)], -1)
    a = O.attn_bwd(q, k, v, do, mask=m1, scale=0.5)
    b = O.attn_bwd(q, k2, v2, do, mask=m2, scale=0.5)
    for x, y in zip(a[:3], b[:3]):
        assert np.allclose(x, y, rtol=0, atol=1e-14)
    assert np.allclose(a[3], b[3][:, :5], rtol=0, atol=1e-14)
    assert np.allclose(a[4], b[4][:, :5], rtol=0, atol=1e-14)
    assert np.all(b[3][:, 5:] == 0) and np.all(b[4][:, 5:] == 0)


def test_key_permutation_equivariance():
    q, k, v, do = tiny_case(17)
    perm = np.array([3, 0, 6, 1, 5, 2, 4])
    mask = np.ones((1, 1, 1, 7), dtype=bool); mask[..., 4] = False
    a = O.attn_bwd(q, k, v, do, mask=mask, scale=0.5)
    b = O.attn_bwd(q, k[:, perm], v[:, perm], do, mask=mask[..., perm], scale=0.5)
    for x, y in zip(a[:3], b[:3]):
        assert np.allclose(x, y, atol=1e-13)
    assert np.allclose(a[3][:, perm], b[3], atol=1e-13)
    assert np.allclose(a[4][:, perm], b[4], atol=1e-13)


def test_gqa_equals_repeated_kv():
    q, k, v, do = tiny_case(18, Hq=4, Hkv=2)
    a = O.attn_bwd(q, k, v, do, causal=True, scale=0.5) if q.shape[1] == k.shape[1] else \
        O.attn_bwd(q, k, v, do, scale=0.5)
    kr = np.repeat(k, 2, axis=2); vr = np.repeat(v, 2, axis=2)
    b = O.attn_bwd(q, kr, vr, do, scale=0.5)
    for x, y in zip(a[:3], b[:3]):
        assert np.allclose(x, y, atol=1e-13)
    assert np.allclose(a[3], b[3].reshape(1, 7, 2, 2, 4).sum(axis=3), atol=1e-13)
    assert np.allclose(a[4], b[4].reshape(1, 7, 2, 2, 4).sum(axis=3), atol=1e-13)


def test_varlen_equals_separate_dense_problems():
    rng = np.random.default_rng(19)
    cu = [0, 4, 9]
    T = 11
    q = _rand(T, 2, 3, rng=rng); k = _rand(T, 1, 3, rng=rng)
    v = _rand(T, 1, 3, rng=rng); do = _rand(T, 2, 3, rng=rng)
    out, lse, dq, dk, dv = O.attn_varlen(q, k, v, do, cu, causal=True, scale=0.5)
    for a, e in zip(cu[:-1], cu[1:]):
        r = O.attn_bwd(q[None, a:e], k[None, a:e], v[None, a:e], do[None, a:e], causal=True, scale=0.5)
        assert np.allclose(out[a:e], r[0][0], atol=1e-14)
        assert np.allclose(lse[:, a:e], r[1][0], atol=1e-14)
        assert np.allclose(dq[a:e], r[2][0], atol=1e-14)
        assert np.allclose(dk[a:e], r[3][0], atol=1e-14)


def test_rows_match_full_problem():
    q, k, v, do = tiny_case(20, B=2, Sq=6, Sk=9, Hq=4, Hkv=2, D=5)
    mask = np.ones((2, 1, 1, 9), dtype=bool); mask[..., -2:] = False
    full = O.attn_bwd(q, k, v, do, mask=mask, scale=0.5)
    rows = [(0, 0, 0), (1, 3, 5), (1, 2, 2), (0, 1, 4)]
    out, lse, dq = O.attn_rows(q, k, v, do, rows, mask=mask, scale=0.5)
    for n, (b, h, i) in enumerate(rows):
        assert np.allclose(out[n], full[0][b, i, h], atol=1e-14)
        assert np.allclose(lse[n], full[1][b, h, i], atol=1e-14)
        assert np.allclose(dq[n], full[2][b, i, h], atol=1e-14)


# ---------------------------------------------------------------- library special case

def _torch_sdpa(q, k, v, do, mask, causal, scale):
    G = q.shape[2] // k.shape[2]
    tq = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_()
    tk = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_()
    tv = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_()
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    m = None if mask is None else torch.tensor(np.ascontiguousarray(mask))
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=m,
                                                           is_causal=causal, scale=scale)
    out.backward(torch.tensor(do).permute(0, 2, 1, 3))
    f = lambda t: t.detach().permute(0, 2, 1, 3).numpy()
    return f(out), tq.grad.permute(0, 2, 1, 3).numpy(), tk.grad.permute(0, 2, 1, 3).numpy(), \
        tv.grad.permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("case", ["plain", "causal", "bool", "additive", "gqa"])
def test_matches_torch_fp64_sdpa(case):
    rng = np.random.default_rng(21)
    B, Sq, Sk, Hq, Hkv, D = 2, 17, 23, 4, 4, 8
    if case == "gqa":
        Hkv = 2
    if case == "causal":
        Sk = Sq
    q = _rand(B, Sq, Hq, D, rng=rng); k = _rand(B, Sk, Hkv, D, rng=rng)
    v = _rand(B, Sk, Hkv, D, rng=rng); do = _rand(B, Sq, Hq, D, rng=rng)
    mask = None
    if case == "bool":
        mask = rng.random((B, Hq, Sq, Sk)) > 0.3
        mask[..., 0] = True
    if case == "additive":
        mask = rng.standard_normal((B, 1, Sq, Sk))
        mask[..., 3] = -np.inf
    ours = O.attn_bwd(q, k, v, do, mask=mask, causal=case == "causal", scale=0.3)
    ref = _torch_sdpa(q, k, v, do, mask, case == "causal", 0.3)
    for a, b in zip((ours[0], ours[2], ours[3], ours[4]), ref):
        assert np.allclose(a, b, atol=1e-12, rtol=1e-10)


# ---------------------------------------------------------------- golden worked example

def test_golden_two_key_example():
    with open(os.path.join(GOLDEN, "two_key_example.json")) as f:
        g = json.load(f)
    q = np.array(g["q"], dtype=np.float64).reshape(1, 1, 1, -1)
    k = np.array(g["k"], dtype=np.float64).reshape(1, -1, 1, q.shape[-1])
    v = np.array(g["v"], dtype=np.float64).reshape(1, -1, 1, q.shape[-1])
    do = np.array(g["dout"], dtype=np.float64).reshape(1, 1, 1, -1)
    out, lse, dq, dk, dv = O.attn_bwd(q, k, v, do, scale=g["scale"])
    assert np.allclose(out.ravel(), g["out"], atol=1e-12)
    assert abs(lse.item() - g["lse"]) < 1e-12
    assert np.allclose(dq.ravel(), g["dq"], atol=1e-12)
    assert np.allclose(dk.ravel(), g["dk"], atol=1e-12)
    assert np.allclose(dv.ravel(), g["dv"], atol=1e-12)


def test_golden_overflow_threshold():
    """The failure condition of OpenWAM PR #64, "Summary": exp(0 - lse)
    overflows fp32 once lse < -ln(FLT_MAX) (about -88.7)."""
    with open(os.path.join(GOLDEN, "fp32_exp_overflow.json")) as f:
        g = json.load(f)
    flt_max = float(np.finfo(np.float32).max)
    assert abs(-math.log(flt_max) - g["lse_threshold"]) < 1e-3
    with np.errstate(over="ignore"):
        assert np.isinf(np.exp(np.float32(-g["lse_threshold"] + 0.01)))
        assert np.isfinite(np.exp(np.float32(-g["lse_threshold"] - 0.01)))


def _unpredicated_tile_dq_fp32(case, lse, delta, key_tile):
    """dQ of the backward as OpenWAM PR #64 ("Summary") describes the broken
    kernel, in fp32: the key axis is padded to a multiple of the key tile
    with zero keys and zero values, and the padded columns of the last tile
    see neither the mask nor any predicate (score 0, P = exp(0 - lse)).
    The real columns use the oracle's statistics and are finite."""
    q, k, v, do = (np.asarray(case[n].float().numpy(), np.float32) for n in ("q", "k", "v", "do"))
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    pad = (-Sk) % key_tile
    scale = np.float32(case["scale"])
    mask = oracle_mask(case["mask"])
    dq = np.zeros_like(q)
    with np.errstate(over="ignore", invalid="ignore"):
        for b in range(B):
            for h in range(H):
                qh, kh, vh, doh = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
                s = scale * (qh @ kh.T)
                if mask is not None:
                    mb = np.broadcast_to(mask, (B, H, Sq, Sk))[b, h]
                    s = np.where(mb, s, -np.inf) if mb.dtype == bool else s + mb.astype(np.float32)
                kp = np.concatenate([kh, np.zeros((pad, D), np.float32)])
                vp = np.concatenate([vh, np.zeros((pad, D), np.float32)])
                sp = np.concatenate([s, np.zeros((Sq, pad), np.float32)], axis=1)   # unmasked zeros
                P = np.exp(sp - lse[b, h][:, None].astype(np.float32))
                dP = doh @ vp.T
                dS = P * (dP - delta[b, h][:, None].astype(np.float32))
                dq[b, :, h] = scale * (dS @ kp)
    return dq


def test_golden_openwam_partial_tile_counts():
    """The page's table of non-finite dQ elements: the workload's anti-aligned
    row has an lse below -ln(FLT_MAX), and computing the last partial key tile
    without predicates turns exactly that row of dQ (B*H*D elements) non-finite
    for each mask kind, nothing when the key count is a multiple of the tile,
    and the oracle's own (predicated) gradients are finite everywhere."""
    import attn_workloads as W
    with open(os.path.join(GOLDEN, "openwam_partial_tile_nonfinite.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        for kind, want in c["nonfinite_dq_unpredicated"].items():
            case = W.low_lse_row(c["sq"], c["skv"], kind, D=g["D"], B=g["B"], H=g["H"])
            q, k, v, do = (case[n].double().numpy() for n in ("q", "k", "v", "do"))
            m = oracle_mask(case["mask"])
            out, lse, dq, dk, dv = O.attn_bwd(q, k, v, do, mask=m, scale=case["scale"])
            r = case["low_row"]
            assert (lse[:, :, r] < g["lse_overflow_below"]).all()
            others = np.delete(lse, r, axis=2)
            assert (others > g["lse_overflow_below"]).all()
            for x in (out, lse, dq, dk, dv):
                assert np.isfinite(x).all()
            delta = np.einsum("bshd,bshd->bhs", do, out)
            bad = _unpredicated_tile_dq_fp32(case, lse, delta, g["key_tile"])
            assert int((~np.isfinite(bad)).sum()) == want, (c, kind)
            if want:                              # only the anti-aligned row
                assert list(np.unique(np.nonzero(~np.isfinite(bad))[1])) == [r]


# ---------------------------------------------------------------- fp8 inputs

def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    mine = O.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert list(np.nonzero(np.isnan(mine))[0]) == [0x7F, 0xFF]
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_e4m3_decode_worked_values():
    # straight from the format: bias 7, 3 mantissa bits, subnormals m/8 * 2^-6
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0,
             0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    got = O.e4m3_decode(np.array(list(table), dtype=np.uint8))
    assert list(got) == list(table.values())


def test_fp8_generator_maps_each_amax_to_448():
    import attn_workloads as W
    c = W.fp8_qkv(S=512, H=2, D=64, k_scale=5000.0, v="randn")
    for n in ("q", "k", "v"):
        x = O.e4m3_decode(c[n].numpy())
        assert np.isfinite(x).all()
        assert np.abs(x).max() == 448.0


def test_fp8_forward_with_unit_values_returns_the_value():
    """Softmax weights sum to one, so with V = ones (one E4M3 code, 448 after
    the amax scaling) every output is 448 * descale_v, at any logit spread."""
    import attn_workloads as W
    for ks in (1.0, 1000.0, 20000.0):
        c = W.fp8_qkv(S=384, H=2, D=128, k_scale=ks, v="ones")
        out, lse = O.attn_fwd_fp8(c["q"].numpy(), c["k"].numpy(), c["v"].numpy(), c["descale_q"],
                                  c["descale_k"], c["descale_v"], scale=c["scale"])
        assert np.all(np.abs(out - 448.0 * c["descale_v"]) < 1e-12)
        assert np.isfinite(lse).all()


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_matches_torch_sdpa_on_decoded_inputs(causal):
    import attn_workloads as W
    c = W.fp8_qkv(B=2, S=200, H=2, D=64, k_scale=8.0, v="randn", causal=causal)
    dec = {n: torch.from_numpy(c[n].numpy()).view(torch.float8_e4m3fn).to(torch.float64)
              * c["descale_" + n] for n in ("q", "k", "v")}
    ref = torch.nn.functional.scaled_dot_product_attention(
        dec["q"].transpose(1, 2), dec["k"].transpose(1, 2), dec["v"].transpose(1, 2),
        is_causal=causal, scale=c["scale"]).transpose(1, 2).numpy()
    out, _ = O.attn_fwd_fp8(c["q"].numpy(), c["k"].numpy(), c["v"].numpy(), c["descale_q"],
                            c["descale_k"], c["descale_v"], causal=causal, scale=c["scale"])
    assert np.abs(out - ref).max() < 1e-10


# ---------------------------------------------------------------- mutation tests

ORIG_BWD = O._bwd_head


def _bwd_no_delta(qh, kh, vh, P, dOh, scale):
    dP = dOh @ vh.T
    dS = P * dP
    return scale * dS @ kh, scale * dS.T @ qh, P.T @ dOh


def _bwd_no_scale_dq(qh, kh, vh, P, dOh, scale):
    dq, dk, dv = ORIG_BWD(qh, kh, vh, P, dOh, scale)
    return dq / scale, dk, dv


def _bwd_dv_from_dS(qh, kh, vh, P, dOh, scale):
    dq, dk, _ = ORIG_BWD(qh, kh, vh, P, dOh, scale)
    dP = dOh @ vh.T
    delta = (P * dP).sum(axis=1)
    return dq, dk, (P * (dP - delta[:, None])).T @ dOh


def _bwd_dk_untransposed(qh, kh, vh, P, dOh, scale):
    dq, _, dv = ORIG_BWD(qh, kh, vh, P, dOh, scale)
    dP = dOh @ vh.T
    dS = P * (dP - (P * dP).sum(axis=1)[:, None])
    return dq, scale * (dS @ qh), dv          # needs Sq == Sk to be shape-valid


@pytest.mark.parametrize("mutant", [_bwd_no_delta, _bwd_no_scale_dq, _bwd_dv_from_dS,
                                    _bwd_dk_untransposed])
def test_fd_pin_catches_planted_bwd_mistakes(monkeypatch, mutant):
    q, k, v, do = tiny_case(30, Sq=6, Sk=6)
    monkeypatch.setattr(O, "_bwd_head", mutant)
    assert fd_grad_error(q, k, v, do, scale=0.37) > 1e-3


def test_pins_catch_flipped_causal_direction(monkeypatch):
    orig = O.bias_for

    def flipped(mask, b, h, Sq, Sk, causal, rows=None):
        bias = orig(mask, b, h, Sq, Sk, False, rows)
        if causal:
            ri = np.arange(Sq) if rows is None else np.asarray(rows)
            bias = np.where(np.arange(Sk)[None, :] < ri[:, None], -np.inf, bias)
        return bias

    monkeypatch.setattr(O, "bias_for", flipped)
    with pytest.raises(AssertionError):
        test_causal_first_row_sees_only_first_key()


def test_pins_catch_missing_max_in_lse(monkeypatch):
    orig = O._fwd_head

    def bad(qh, kh, vh, bias, scale):
        P, out, lse = orig(qh, kh, vh, bias, scale)
        s = scale * (qh @ kh.T) + bias
        return P, out, np.where(lse != 0, lse - s.max(axis=1), 0.0)

    monkeypatch.setattr(O, "_fwd_head", bad)
    with pytest.raises(AssertionError):
        test_constant_logit_shift()


# ---------------------------------------------------------------- score recompute

def _score_case(seed, B=2, Sq=9, Sk=11, Hq=4, Hkv=2, D=8):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Sq, Hq, D)), rng.standard_normal((B, Sk, Hkv, D)))


@pytest.mark.parametrize("causal", [False, True])
def test_score_l1_norm_is_the_head_count(causal):
    """With the forward's own lse every head's terms of a row sum to 1, so
    the L1 norm of the head-summed scores is the number of heads
    (PFCCLab/cudnn-frontend PR #9, How it was verified: a leaked 64.0 is a
    previous attn_l1norm of 64 heads)."""
    q, k = _score_case(40)
    _, lse = O.attn_fwd(q, k, k, causal=causal, scale=0.3)
    score, l1 = O.attn_score_recompute(q, k, lse, causal=causal, scale=0.3)
    assert np.allclose(l1, q.shape[2], rtol=1e-12, atol=0)
    assert (score >= 0).all()


def test_score_is_the_head_sum_of_attention_weights():
    """score_ij equals the sum over heads of the softmax weights the forward
    computes (a different route: exact row max, then normalise)."""
    q, k = _score_case(41, Sq=7, Sk=7)
    _, lse = O.attn_fwd(q, k, k, causal=True, scale=0.45)
    score, _ = O.attn_score_recompute(q, k, lse, causal=True, scale=0.45)
    ref = np.zeros_like(score)
    G = q.shape[2] // k.shape[2]
    for b in range(q.shape[0]):
        bias = O.bias_for(None, 0, 0, 7, 7, True)
        for h in range(q.shape[2]):
            P, _, _ = O._fwd_head(q[b, :, h], k[b, :, h // G], k[b, :, h // G], bias, 0.45)
            ref[b] += P
    assert np.allclose(score, ref, rtol=1e-12, atol=1e-15)
    j, i = np.meshgrid(np.arange(7), np.arange(7))
    assert (score[:, j > i] == 0).all()                # causal pairs get exactly 0


def test_score_clamp_keeps_a_degenerate_lse_finite():
    """PFCCLab/cudnn-frontend PR #9, section 3: an lse far too small (the
    -1e30 mask constant) makes every term exp2(+huge); the clamp at 120 keeps
    each at 2^120 and the sum over heads finite (2^120 * 64 < FLT_MAX)."""
    q, k = _score_case(42, Hq=64, Hkv=1)
    _, lse = O.attn_fwd(q, k, k, scale=0.3)
    lse[0, :, 3] = -1e30                              # one degenerate row, every head
    score, l1 = O.attn_score_recompute(q, k, lse, scale=0.3)
    assert np.isfinite(score).all() and np.isfinite(l1).all()
    assert (score[0, 3] == 64 * 2.0 ** 120).all()
    assert np.float32(64 * 2.0 ** 120) < np.finfo(np.float32).max
    others = np.delete(l1, 3, axis=1)
    assert np.allclose(others, 64, rtol=1e-12)


def test_score_varlen_layout_and_unvisited_rows():
    """Varlen: row cu[s] + i holds sequence s's keys in columns 0..len-1 and
    0 beyond; rows past cu[-1] are 0 in both outputs (section 2: 0, not
    -inf); each sequence equals the dense problem on its own rows."""
    rng = np.random.default_rng(43)
    cu = [0, 5, 5, 12]
    T, Hq, Hkv, D = 15, 4, 2, 8
    q, k = rng.standard_normal((T, Hq, D)), rng.standard_normal((T, Hkv, D))
    out, lse, *_ = O.attn_varlen(q, k, k, np.zeros_like(q), cu, causal=True, scale=0.4)
    score, l1 = O.attn_score_recompute(q, k, lse, causal=True, scale=0.4, cu_seqlens=cu,
                                       max_seqlen=8)
    assert score.shape == (T, 8) and l1.shape == (T,)
    assert (score[12:] == 0).all() and (l1[12:] == 0).all()
    assert (score[0:5, 5:] == 0).all()
    assert np.allclose(l1[:12], Hq, rtol=1e-12)
    a, e = 5, 12
    _, lse_d = O.attn_fwd(q[None, a:e], k[None, a:e], k[None, a:e], causal=True, scale=0.4)
    sd, _ = O.attn_score_recompute(q[None, a:e], k[None, a:e], lse_d, causal=True, scale=0.4)
    assert np.allclose(score[a:e, :7], sd[0], rtol=1e-12)


def test_score_pins_catch_planted_mistakes(monkeypatch):
    """A missing clamp, a dropped lse or exp in place of exp2 each fail a pin."""
    orig = O._score_terms

    def no_clamp(qh, kh, lse_h, bias, scale):
        s = scale * (qh @ kh.T) + bias
        return np.exp2(np.log2(np.e) * (s - lse_h[:, None]))

    def no_lse(qh, kh, lse_h, bias, scale):
        return orig(qh, kh, np.zeros_like(lse_h), bias, scale)

    def exp_not_exp2(qh, kh, lse_h, bias, scale):
        s = scale * (qh @ kh.T) + bias
        return np.exp(np.minimum(np.log2(np.e) * (s - lse_h[:, None]), 120.0))

    with np.errstate(over="ignore"):
        monkeypatch.setattr(O, "_score_terms", no_clamp)
        with pytest.raises(AssertionError):
            test_score_clamp_keeps_a_degenerate_lse_finite()
    for bad in (no_lse, exp_not_exp2):
        monkeypatch.setattr(O, "_score_terms", bad)
        with pytest.raises(AssertionError):
            test_score_l1_norm_is_the_head_count(False)
