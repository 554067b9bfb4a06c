"""GPU parity of the fp16 path (the kernels templated on the element type)
against the fp64 oracle, with the same acceptance bar and zero NaN/Inf.

The workloads are the bf16 ones of the pages drawn in fp16 instead: the
causal S=256 D=64 call (flash-dmattn PR #122), rows whose lse is far below
-88.7 next to a partial last key tile with bool / additive / no mask
(OpenWAM PR #64), a wide logit spread (FlyDSL PR #1033), packed varlen with
GQA and trailing rows, and a long sequence.  fp16 keeps 11 significant bits
against bf16's 8, so the bar is met with more room; its range (65504) is far
above every value these workloads produce.
"""
import math

import pytest
import torch

import attn_workloads as W
from oracle import attn_oracle as O
from parity_utils import assert_finite, compare, gpu_run, oracle_dense, to64

pytestmark = pytest.mark.gpu
F16 = torch.float16


@pytest.fixture(scope="session", autouse=True)
def _built():
    from softmax_attention_numerics_gb300 import build
    build.build()
    yield


def _is_f16(res):
    for n in ("out", "dq", "dk", "dv"):
        assert res[n].dtype == F16, n
    assert res["lse"].dtype == torch.float32


@pytest.mark.parametrize("mode", ["default", "eager", "deterministic"])
def test_f16_causal_small(mode):
    case = W.causal_small(dtype=F16)
    res = gpu_run(case, deterministic=mode == "deterministic", eager=mode == "eager")
    _is_f16(res)
    assert_finite(res)
    compare(res, oracle_dense(case), ctx="f16 causal_small/" + mode)


SHAPES = [(392, 392), (100, 77)]


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("mask", ["bool", "additive", "additive_f16", "none"])
@pytest.mark.parametrize("shape", SHAPES, ids=["%dx%d" % s for s in SHAPES])
def test_f16_low_lse_row(shape, mask, D):
    Sq, Sk = shape
    case = W.low_lse_row(Sq, Sk, "additive" if mask == "additive_f16" else mask, D=D,
                         row="last", dtype=F16)
    if mask == "additive_f16":
        case["mask"] = case["mask"].to(F16)       # 0 / -inf are exact in fp16
    res = gpu_run(case)
    _is_f16(res)
    assert_finite(res)
    ref = oracle_dense(case)
    assert ref["lse"][:, :, case["low_row"]].max() < -88.73
    compare(res, ref, ctx="f16 low_lse %s %s D=%d" % (shape, mask, D))
    if mask != "none":
        hidden = Sk - math.ceil(0.1 * Sk)
        assert torch.count_nonzero(res["dk"][:, hidden:]) == 0
        assert torch.count_nonzero(res["dv"][:, hidden:]) == 0


@pytest.mark.parametrize("s", [8, 32])
def test_f16_wide_spread(s):
    case = W.wide_spread(s, dtype=F16)
    res = gpu_run(case)
    _is_f16(res)
    assert_finite(res)
    for (b, h) in [(0, 3), (1, 17)]:
        qh, kh, vh, dh = (to64(case[n][b, :, h]) for n in ("q", "k", "v", "do"))
        import numpy as np
        P, out, lse = O._fwd_head(qh, kh, vh, np.zeros((qh.shape[0], kh.shape[0])), case["scale"])
        dq, dk, dv = O._bwd_head(qh, kh, vh, P, dh, case["scale"])
        del P
        got = {n: res[n][b, :, h] for n in ("out", "dq", "dk", "dv")}
        got["lse"] = res["lse"][b, h]
        compare(got, dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv), ctx="f16 wide s=%d" % s)


def test_f16_varlen_gqa():
    case = W.varlen_gqa(dtype=F16)
    res = gpu_run(case)
    _is_f16(res)
    assert_finite(res)
    cu = case["cu_seqlens"].tolist()
    end = cu[-1]
    for n in ("out", "dq", "dk", "dv"):
        assert torch.count_nonzero(res[n][end:]) == 0, n
    assert torch.count_nonzero(res["lse"][:, end:]) == 0
    lens = case["lens"]
    sidx = max(range(len(lens)), key=lambda i: lens[i])
    a, e = cu[sidx], cu[sidx + 1]
    heads = [0, 1, 2, 3, 28, 29, 30, 31]
    sub = {n: case[n][a:e] for n in ("q", "k", "v", "do")}
    out, lse, dq, dk, dv = O.attn_varlen(to64(sub["q"]), to64(sub["k"]), to64(sub["v"]),
                                         to64(sub["do"]), [0, e - a], causal=True,
                                         scale=case["scale"], heads=heads)
    got = dict(out=res["out"][a:e, heads], lse=res["lse"][heads, a:e], dq=res["dq"][a:e, heads],
               dk=res["dk"][a:e][:, [0, 7]], dv=res["dv"][a:e][:, [0, 7]])
    ref = dict(out=out[:, heads], lse=lse[heads], dq=dq[:, heads], dk=dk[:, [0, 7]],
               dv=dv[:, [0, 7]])
    compare(got, ref, ctx="f16 varlen seq %d (len %d)" % (sidx, e - a))


@pytest.mark.parametrize("deterministic", [False, True])
def test_f16_long_seq(deterministic):
    S = 16384
    case = W.long_seq(S, True, dtype=F16)
    res = gpu_run(case, deterministic=deterministic)
    _is_f16(res)
    assert_finite(res)
    rows = W.sample_rows(1, 16, S, n=32)
    out, lse, dq = O.attn_rows(to64(case["q"]), to64(case["k"]), to64(case["v"]),
                               to64(case["do"]), rows, causal=True, scale=case["scale"])
    bi = [r[0] for r in rows]
    hi = [r[1] for r in rows]
    ii = [r[2] for r in rows]
    got = dict(out=res["out"][bi, ii, hi], lse=res["lse"][bi, hi, ii], dq=res["dq"][bi, ii, hi])
    compare(got, dict(out=out, lse=lse, dq=dq), names=("out", "lse", "dq"),
            ctx="f16 long S=%d det=%s" % (S, deterministic))


def test_f16_deterministic_bitwise():
    case = W.causal_small(dtype=F16)
    a = gpu_run(case, deterministic=True)
    b = gpu_run(case, deterministic=True)
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[n], b[n]), n
