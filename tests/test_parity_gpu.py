"""GPU parity of the CUDA attention path against the fp64 oracle.

Every case feeds the same seeded bf16 inputs (attn_workloads) to the library
(through the C ABI) and to the oracle, and checks the acceptance bar in
parity_utils plus zero NaN/Inf.  Workloads follow the pages:
flash-dmattn PR #122 (causal S=256 D=64, loss = out.sum()), OpenWAM PR #64
(partial last key tile with a row whose lse is far below -88.7), FlyDSL
PR #1033 (wide logit spread), packed varlen with GQA and trailing rows
(PFCCLab/cudnn-frontend PR #9, section 2), and long sequences.
"""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
from oracle import attn_oracle as O
from parity_utils import (assert_finite, compare, gpu_run, nonfinite, oracle_dense,
                          oracle_mask, rel_l2, to64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session", autouse=True)
def _built():
    from softmax_attention_numerics_gb300 import build
    build.build()
    yield


# ------------------------------------------------------------- causal S=256 D=64

@pytest.mark.parametrize("mode", ["default", "eager", "deterministic"])
def test_causal_small(mode):
    case = W.causal_small()
    res = gpu_run(case, deterministic=mode == "deterministic", eager=mode == "eager")
    assert_finite(res)
    compare(res, oracle_dense(case), ctx="causal_small/" + mode)


# ------------------------------------------------------------- low-lse row + key padding

SHAPES = [(392, 392), (360, 64), (100, 77), (392, 512)]


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("row", ["first", "last"])
@pytest.mark.parametrize("mask", ["bool", "additive", "none"])
@pytest.mark.parametrize("shape", SHAPES, ids=["%dx%d" % s for s in SHAPES])
def test_low_lse_row(shape, mask, row, D):
    Sq, Sk = shape
    case = W.low_lse_row(Sq, Sk, mask, D=D, row=row)
    res = gpu_run(case)
    assert_finite(res)
    ref = oracle_dense(case)
    r = case["low_row"]
    # the case really exercises the failure condition: exp(0 - lse) overflows fp32,
    # and at D = 128 the row sits where OpenWAM PR #64 (Validation) puts it
    assert ref["lse"][:, :, r].max() < -88.73
    if D == 128:
        assert -120.0 <= ref["lse"][:, :, r].min() and ref["lse"][:, :, r].max() <= -110.0
    compare(res, ref, ctx="low_lse %s %s %s D=%d" % (shape, mask, row, D))
    if mask != "none":
        hidden = Sk - math.ceil(0.1 * Sk)
        assert torch.count_nonzero(res["dk"][:, hidden:]) == 0
        assert torch.count_nonzero(res["dv"][:, hidden:]) == 0


# ------------------------------------------------------------- wide logit spread

# FlyDSL PR #1033 (Result) reports the output's rel-L2 per K scale for the lazy
# and the eager rescale; this test measures the same quantities against the fp64
# oracle (plus the gradients, the lse error and NaN / Inf counted separately
# over the full tensors) and, when ATTN_REPORT_DIR is set, appends one JSON
# record per (scale, mode) to wide_spread_report.jsonl there.
_WIDE_ORACLE = {}


def _wide_pairs(s):
    g = torch.Generator().manual_seed(100 + s)
    return [(int(torch.randint(0, 2, (1,), generator=g)), int(torch.randint(0, 32, (1,), generator=g)))
            for _ in range(4)]


def _wide_oracle(case, s, b, h):
    key = (s, b, h)
    if key not in _WIDE_ORACLE:
        qh, kh, vh, dh = (to64(case[n][b, :, h]) for n in ("q", "k", "v", "do"))
        P, out, lse = O._fwd_head(qh, kh, vh, np.zeros((qh.shape[0], kh.shape[0])), case["scale"])
        dq, dk, dv = O._bwd_head(qh, kh, vh, P, dh, case["scale"])
        del P
        _WIDE_ORACLE[key] = dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv)
    return _WIDE_ORACLE[key]


@pytest.mark.parametrize("mode", ["lazy", "eager"])
@pytest.mark.parametrize("s", [8, 16, 24, 32, 48, 64])
def test_wide_spread(s, mode):
    import json
    import os
    case = W.wide_spread(s)
    res = gpu_run(case, eager=mode == "eager")
    torch.cuda.synchronize()
    record = {"k_scale": s, "mode": mode, "workload": "B=2 S=8192 H=32 D=128 non-causal bf16",
              "nan": {}, "inf": {}, "pairs": []}
    for n in ("out", "lse", "dq", "dk", "dv"):
        record["nan"][n], record["inf"][n] = nonfinite(res[n])
    for (b, h) in _wide_pairs(s):
        ref = _wide_oracle(case, s, b, h)
        got = {n: to64(res[n][b, :, h]) for n in ("out", "dq", "dk", "dv")}
        got["lse"] = to64(res["lse"][b, h])
        record["pairs"].append({
            "b": b, "h": h,
            "out_rel_l2": rel_l2(got["out"], ref["out"]),
            "out_max_abs": float(np.abs(got["out"] - ref["out"]).max()),
            "lse_max_abs": float(np.abs(got["lse"] - ref["lse"]).max()),
            **{n + "_rel_l2": rel_l2(got[n], ref[n]) for n in ("dq", "dk", "dv")}})
        record["pairs"][-1] = {k: (float(v) if isinstance(v, (float, np.floating)) else v)
                               for k, v in record["pairs"][-1].items()}
    rdir = os.environ.get("ATTN_REPORT_DIR")
    if rdir:
        os.makedirs(rdir, exist_ok=True)
        with open(os.path.join(rdir, "wide_spread_report.jsonl"), "a") as f:
            f.write(json.dumps(record) + "\n")
    print("wide_spread", json.dumps(record))
    assert_finite(res)
    for (b, h) in _wide_pairs(s):
        got = {n: res[n][b, :, h] for n in ("out", "dq", "dk", "dv")}
        got["lse"] = res["lse"][b, h]
        compare(got, _wide_oracle(case, s, b, h), ctx="wide s=%d %s (b=%d,h=%d)" % (s, mode, b, h))


# ------------------------------------------------------------- varlen + GQA + trailing rows

def test_varlen_gqa():
    case = W.varlen_gqa()
    res = gpu_run(case)
    assert_finite(res)
    cu = case["cu_seqlens"].tolist()
    end = cu[-1]
    for n in ("out", "dq", "dk", "dv"):
        assert torch.count_nonzero(res[n][end:]) == 0, n
    assert torch.count_nonzero(res["lse"][:, end:]) == 0
    lens = case["lens"]
    order = sorted(range(len(lens)), key=lambda i: lens[i])
    # every head of four whole sequences: the shortest, two in the middle, the longest
    pick = [order[0], order[len(order) // 3], order[2 * len(order) // 3], order[-1]]
    for sidx in pick:
        a, e = cu[sidx], cu[sidx + 1]
        sub = {n: case[n][a:e] for n in ("q", "k", "v", "do")}
        out, lse, dq, dk, dv = O.attn_varlen(to64(sub["q"]), to64(sub["k"]), to64(sub["v"]),
                                             to64(sub["do"]), [0, e - a], causal=True,
                                             scale=case["scale"])
        got = dict(out=res["out"][a:e], lse=res["lse"][:, a:e], dq=res["dq"][a:e],
                   dk=res["dk"][a:e], dv=res["dv"][a:e])
        ref = dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv)
        compare(got, ref, ctx="varlen seq %d (len %d)" % (sidx, e - a))


# ------------------------------------------------------------- long sequences (sampled)

LONG = [(S, 128) for S in (16384, 65536, 131072)] + [(16384, 64), (131072, 64)]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("S,D", LONG, ids=["S%d_D%d" % c for c in LONG])
def test_long_seq(S, D, causal):
    """Sampled rows of out, lse and dq at the long lengths (the benchmark's
    S = 131072 among them, at both head dims: hundreds of query tiles per key
    tile, so every buffer rotation of the backward's pipeline is exercised),
    and one head's full dK / dV at S = 16384."""
    case = W.long_seq(S, causal, D=D)
    res = gpu_run(case)
    assert_finite(res)
    rows = W.sample_rows(1, 16, S, n=64)
    out, lse, dq = O.attn_rows(to64(case["q"]), to64(case["k"]), to64(case["v"]),
                               to64(case["do"]), rows, causal=causal, scale=case["scale"])
    bi = [r[0] for r in rows]
    hi = [r[1] for r in rows]
    ii = [r[2] for r in rows]
    got = dict(out=res["out"][bi, ii, hi], lse=res["lse"][bi, hi, ii], dq=res["dq"][bi, ii, hi])
    compare(got, dict(out=out, lse=lse, dq=dq), names=("out", "lse", "dq"),
            ctx="long S=%d D=%d causal=%s" % (S, D, causal))
    if S == 16384:
        h = 5
        qh, kh, vh, dh = (to64(case[n][0, :, h]) for n in ("q", "k", "v", "do"))
        bias = O.bias_for(None, 0, 0, S, S, causal)
        P, _, _ = O._fwd_head(qh, kh, vh, bias, case["scale"])
        del bias
        _, dk, dv = O._bwd_head(qh, kh, vh, P, dh, case["scale"])
        del P
        compare(dict(dk=res["dk"][0, :, h], dv=res["dv"][0, :, h]), dict(dk=dk, dv=dv),
                names=("dk", "dv"), ctx="long S=%d D=%d dk/dv head %d" % (S, D, h))


# ------------------------------------------------------------- edge cases

EDGE = [
    # (B, Sq, Sk, Hq, Hkv, D, causal, mask)
    (1, 1, 1, 1, 1, 64, False, "none"),
    (1, 129, 65, 2, 1, 64, False, "none"),
    (2, 129, 129, 4, 2, 128, True, "none"),
    (1, 300, 700, 8, 2, 128, False, "bool_rows"),
    (2, 200, 333, 4, 4, 64, False, "additive_random"),
    (1, 190, 190, 2, 2, 128, False, "bf16_additive"),
    (1, 100, 260, 2, 1, 128, True, "none"),          # Sq < Sk, top-left causal
    (1, 260, 100, 2, 1, 64, True, "none"),           # Sq > Sk
    (1, 64, 0, 2, 1, 64, False, "none"),             # no keys at all
    (1, 0, 64, 2, 1, 128, False, "none"),            # no queries
    (1, 1000, 1000, 16, 2, 128, True, "none"),       # GQA G=8: dK/dV summed over 8 q heads
    (1, 1000, 1000, 16, 2, 64, False, "none"),
    (1, 1000, 1000, 16, 2, 64, True, "none"),        # causal GQA: key tiles with 1..8 query tiles per head
    (4, 130, 130, 32, 32, 64, False, "none"),        # many small (batch, head) problems
    (2, 257, 383, 8, 4, 128, False, "bool_rows"),    # ragged in both dimensions, per-row mask
    (1, 513, 513, 4, 1, 128, True, "additive_random"),  # causal + additive mask, G=4
]


def _edge_case(B, Sq, Sk, Hq, Hkv, D, causal, mask):
    q, k, v, do = W.dense_qkvdo(B, Sq, Sk, Hq, Hkv, D, seed=11)
    m = None
    if mask == "bool_rows":
        m = W.padding_mask(B, Sq, Sk, "bool", Hq=Hq, per_row=True)
        m[0, 1, 5, :] = 0                           # a fully masked row
    elif mask == "additive_random":
        g = torch.Generator().manual_seed(3)
        m = torch.randn(B, 1, Sq, Sk, generator=g) * 2.0
        m[..., -7:] = float("-inf")
    elif mask == "bf16_additive":
        g = torch.Generator().manual_seed(4)
        m = (torch.randn(1, Hq, 1, Sk, generator=g) * 3.0).to(torch.bfloat16)
    return dict(q=q, k=k, v=v, do=do, causal=causal, scale=1.0 / math.sqrt(D), mask=m)


@pytest.mark.parametrize("cfg", EDGE, ids=[str(c) for c in EDGE])
def test_edge_cases(cfg):
    case = _edge_case(*cfg)
    for det in (False, True):
        res = gpu_run(case, deterministic=det)
        assert_finite(res)
        compare(res, oracle_dense(case), ctx="edge %s det=%s" % (cfg, det))


def test_fully_masked_row_is_zero():
    case = _edge_case(1, 300, 700, 8, 2, 128, False, "bool_rows")
    res = gpu_run(case)
    assert torch.count_nonzero(res["out"][0, 5, 1]) == 0
    assert res["lse"][0, 1, 5].item() == 0.0
    assert torch.count_nonzero(res["dq"][0, 5, 1]) == 0


def test_strided_bhsd_inputs():
    """BHSD buffers viewed as BSHD (OpenWAM PR #64, Tests: layout preservation)."""
    B, S, H, D = 2, 200, 4, 128
    g = torch.Generator().manual_seed(9)
    base = [torch.randn(B, H, S, D, generator=g).to(torch.bfloat16) for _ in range(4)]
    case = dict(q=base[0].transpose(1, 2), k=base[1].transpose(1, 2), v=base[2].transpose(1, 2),
                do=base[3].transpose(1, 2), causal=True, scale=0.1, mask=None)
    gcase = dict(case)
    for n in ("q", "k", "v", "do"):
        gcase[n] = base[["q", "k", "v", "do"].index(n)].cuda().transpose(1, 2)
    res = gpu_run(gcase)
    assert_finite(res)
    compare(res, oracle_dense(case), ctx="strided")


def test_varlen_empty_and_short_sequences():
    lens = [0, 1, 130, 0, 257, 64]
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    T = cu[-1] + 37
    g = torch.Generator().manual_seed(12)
    q = torch.randn(T, 4, 64, generator=g).to(torch.bfloat16)
    k = torch.randn(T, 2, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(T, 2, 64, generator=g).to(torch.bfloat16)
    do = torch.randn(T, 4, 64, generator=g).to(torch.bfloat16)
    for causal in (False, True):
        case = dict(q=q, k=k, v=v, do=do, cu_seqlens=torch.tensor(cu, dtype=torch.int32),
                    max_seqlen=max(lens), causal=causal, scale=0.125)
        res = gpu_run(case)
        assert_finite(res)
        out, lse, dq, dk, dv = O.attn_varlen(to64(q), to64(k), to64(v), to64(do), cu,
                                             causal=causal, scale=0.125)
        compare(res, dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv), ctx="varlen short")


# ------------------------------------------------------------- determinism

def test_deterministic_path_is_bitwise_stable():
    case = W.varlen_gqa(n=4, lo=300, hi=900)
    first = gpu_run(case, deterministic=True)
    for _ in range(7):
        again = gpu_run(case, deterministic=True)
        for n in ("dq", "dk", "dv", "out", "lse"):
            assert torch.equal(first[n], again[n]), n


def test_atomic_path_spread_within_fp32_reassociation_bound():
    """PFCCLab/cudnn-frontend PR #9, How it was verified: a sum of N fp32 terms
    in any order differs run to run by at most (N-1) 2^-24 sum|t_i|.  Each
    dq_acc element receives one partial per 128-key tile (N = 4 here); after
    the final rounding to bf16 two runs may differ by that bound plus one bf16
    ulp (at most 2^-7 of the magnitude).  sum|t_i| is estimated in fp64 from
    the oracle's probabilities, with a factor 2 of slack for bf16 dS."""
    case = W.low_lse_row(392, 512, "bool", D=128)
    runs = np.stack([to64(gpu_run(case)["dq"]) for _ in range(8)])
    spread = runs.max(0) - runs.min(0)
    q, k, v, do = (to64(case[n]) for n in ("q", "k", "v", "do"))
    mask = oracle_mask(case["mask"])
    sc = case["scale"]
    sabs = np.zeros_like(q)
    for b in range(q.shape[0]):
        for h in range(q.shape[2]):
            bias = O.bias_for(mask, b, h, q.shape[1], k.shape[1], False)
            P, _, _ = O._fwd_head(q[b, :, h], k[b, :, h], v[b, :, h], bias, sc)
            dP = do[b, :, h] @ v[b, :, h].T
            dS = P * (dP - (P * dP).sum(1)[:, None])
            for t0 in range(0, k.shape[1], 128):
                sabs[b, :, h] += np.abs(sc * dS[:, t0:t0 + 128] @ k[b, t0:t0 + 128, h])
    n_terms = math.ceil(k.shape[1] / 128)
    bound = 2 * (n_terms - 1) * 2.0 ** -24 * sabs + 2.0 ** -7 * np.abs(runs).max(0)
    assert np.all(spread <= bound + 1e-30)


def test_atomic_spread_bound_holds_under_concurrent_load():
    """The same reassociation bound with another stream keeping the GPU busy
    (PFCCLab/cudnn-frontend PR #9: the spread criterion also under concurrent
    load): the reduction order may change, the bound may not be exceeded."""
    case = W.low_lse_row(392, 512, "bool", D=128)
    ref = to64(gpu_run(case)["dq"])
    side = torch.cuda.Stream()
    a = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    runs = []
    for _ in range(8):
        with torch.cuda.stream(side):
            for _ in range(4):
                a = (a @ a).clamp_(-1, 1)           # busy work on another stream
        runs.append(to64(gpu_run(case)["dq"]))
    torch.cuda.synchronize()
    runs = np.stack(runs + [ref])
    spread = runs.max(0) - runs.min(0)
    # the bound of the test above, computed the same way
    q, k, v, do = (to64(case[n]) for n in ("q", "k", "v", "do"))
    mask = oracle_mask(case["mask"])
    sc = case["scale"]
    sabs = np.zeros_like(q)
    for b in range(q.shape[0]):
        for h in range(q.shape[2]):
            bias = O.bias_for(mask, b, h, q.shape[1], k.shape[1], False)
            P, _, _ = O._fwd_head(q[b, :, h], k[b, :, h], v[b, :, h], bias, sc)
            dP = do[b, :, h] @ v[b, :, h].T
            dS = P * (dP - (P * dP).sum(1)[:, None])
            for t0 in range(0, k.shape[1], 128):
                sabs[b, :, h] += np.abs(sc * dS[:, t0:t0 + 128] @ k[b, t0:t0 + 128, h])
    n_terms = math.ceil(k.shape[1] / 128)
    bound = 2 * (n_terms - 1) * 2.0 ** -24 * sabs + 2.0 ** -7 * np.abs(runs).max(0)
    assert np.all(spread <= bound + 1e-30)


def test_dq_strategy_leaves_other_outputs_bit_identical():
    """Switching the dQ path (fp32 reductions vs the per-query-tile kernel)
    changes only dq: out, lse, dk and dv come from the same kernels in the same
    order and must be bit-identical (the "untouched outputs" check of
    PFCCLab/cudnn-frontend PR #9)."""
    for case in (W.low_lse_row(392, 512, "additive", D=64), W.varlen_gqa(n=4, hi=1024)):
        a = gpu_run(case, deterministic=False)
        b = gpu_run(case, deterministic=True)
        for n in ("out", "lse", "dk", "dv"):
            assert torch.equal(a[n], b[n]), n
        assert_finite(a)
        assert_finite(b)


@pytest.mark.parametrize("mask", ["bool", "additive", "none"])
@pytest.mark.parametrize("shape", [(392, 392), (100, 77)], ids=["392x392", "100x77"])
def test_low_lse_row_bhsd_layout(shape, mask):
    """The low-lse / partial-tile workload with BHSD buffers viewed as BSHD
    (OpenWAM PR #64, Tests: the layout axis of the GPU matrix)."""
    Sq, Sk = shape
    case = W.low_lse_row(Sq, Sk, mask, D=128, row="last")
    gcase = dict(case)
    for n in ("q", "k", "v", "do"):
        gcase[n] = case[n].transpose(1, 2).contiguous().cuda().transpose(1, 2)
        assert not gcase[n].is_contiguous()
    res = gpu_run(gcase)
    assert_finite(res)
    compare(res, oracle_dense(case), ctx="low_lse bhsd %s %s" % (shape, mask))


# ------------------------------------------------------------- stream discipline

def test_side_stream_with_busy_ambient_stream():
    """NVIDIA/cudnn-frontend PR #429, first fix: allocations and zero-fills are
    ordered with the launch stream even while the ambient stream is busy."""
    case = W.low_lse_row(392, 392, "bool", D=128)
    ref = gpu_run(case, deterministic=True)
    dev = {n: (case[n].cuda() if torch.is_tensor(case[n]) else case[n]) for n in case}
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    torch.cuda._sleep(400_000_000)        # keep the ambient stream busy
    res = gpu_run(dev, deterministic=True, stream=side)
    side.synchronize()
    for n in ("out", "lse", "dq", "dk", "dv"):
        assert torch.equal(res[n], ref[n]), n
    torch.cuda.synchronize()


# ------------------------------------------------------------- device-side errors

def test_malformed_cu_seqlens_sets_error_word():
    from softmax_attention_numerics_gb300 import attn_fwd, get_error
    T = 256
    q = torch.randn(T, 2, 64, device="cuda").to(torch.bfloat16)
    k = torch.randn(T, 2, 64, device="cuda").to(torch.bfloat16)
    cu = torch.tensor([0, 100, 50, 300], dtype=torch.int32, device="cuda")   # decreasing, past T
    assert get_error() == 0
    out, lse = attn_fwd(q, k, k, cu_seqlens=cu, max_seqlen=128)
    assert get_error() == -9          # rows of skipped sequences are undefined
    assert get_error() == 0


def test_varlen_max_seqlen_zero_still_checks_sequences():
    """With max_seqlen = 0 no attention block runs; a non-empty sequence must
    still be reported (its rows would otherwise be left unwritten), and with
    every sequence empty all rows are trailing rows: zero, no error."""
    from softmax_attention_numerics_gb300 import attn_bwd, attn_fwd, get_error
    T, H, D = 300, 2, 64
    g = torch.Generator().manual_seed(3)
    q, k, do = (torch.randn(T, H, D, generator=g).to(torch.bfloat16).cuda() for _ in range(3))
    cu = torch.tensor([0, 100, 250], dtype=torch.int32, device="cuda")
    assert get_error() == 0
    out, lse = attn_fwd(q, k, k, cu_seqlens=cu, max_seqlen=0)
    assert get_error() == -9
    attn_bwd(q, k, k, q, do, torch.zeros(H, T, device="cuda"), cu_seqlens=cu, max_seqlen=0)
    assert get_error() == -9
    empty = torch.zeros(3, dtype=torch.int32, device="cuda")
    out, lse = attn_fwd(q, k, k, cu_seqlens=empty, max_seqlen=0)
    dq, dk, dv = attn_bwd(q, k, k, out, do, lse, cu_seqlens=empty, max_seqlen=0)
    assert get_error() == 0
    for x in (out, lse, dq, dk, dv):
        assert not x.float().abs().gt(0).any()


def test_cpu_tensors_rejected():
    from softmax_attention_numerics_gb300 import _lib, attn_fwd
    q = torch.randn(1, 8, 1, 64).to(torch.bfloat16)
    with pytest.raises((_lib.AttnError, RuntimeError)):
        attn_fwd(q.cuda(), q, q.cuda())
