"""GPU parity of the sparse top-k (DSA) backward against the fp64 oracle
(NVIDIA/cudnn-frontend PR #429: q, kv, out, dout, lse, attn_sink, topk_idxs,
topk_length -> dq, dkv, d_sink; head dim 576 (MLA, values in the first 512
columns) or 512; the page's check: S = 512, S_kv = 2048, H = 64, top-k = 128,
with and without topk_length).

The oracle's forward supplies out (rounded to the 16-bit type) and lse
(fp32), as a training step's forward would; both sides then take the same
16-bit q, kv, dout.  Bar, as for the dense backward: dq, dkv, d_sink rel-L2
<= 2e-2 for bf16 (P and dS are rounded to bf16 before the products), 5e-3
for fp16; zero NaN / Inf; dq and d_sink bit-identical on a second call.
"""
import math

import numpy as np
import pytest
import torch

import attn_workloads as W
from oracle import sparse_oracle as OS
from parity_utils import nonfinite, rel_l2, to64

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float16: 5e-3}


def _np(x):
    return None if x is None else (to64(x) if x.dtype.is_floating_point else x.numpy())


def _oracle(c, scale):
    return OS.dsa_bwd(_np(c["q"]), _np(c["kv"]), _np(c["dout"]), _np(c["topk_idxs"]),
                      _np(c["topk_length"]), _np(c["attn_sink"]), scale=scale, dv=512)


def _gpu(c, out64, lse64, scale, stream=None):
    from softmax_attention_numerics_gb300 import attn_sparse_bwd
    dt = c["q"].dtype
    cu = {k: (None if v is None else v.cuda()) for k, v in c.items()}
    out = torch.from_numpy(out64).to(dt).cuda()
    lse = torch.from_numpy(lse64).float().cuda()
    return attn_sparse_bwd(cu["q"], cu["kv"], out, cu["dout"], lse, cu["topk_idxs"],
                           topk_length=cu["topk_length"], attn_sink=cu["attn_sink"], scale=scale,
                           stream=stream)


def _check(got, ref, tol, ctx):
    dq, dkv, ds = got
    _, _, rdq, rdkv, rds = ref
    for name, t in (("dq", dq), ("dkv", dkv), ("d_sink", ds)):
        if t is not None:
            assert nonfinite(t) == (0, 0), (ctx, name)
    e = {"dq": rel_l2(to64(dq), rdq), "dkv": rel_l2(to64(dkv), rdkv)}
    if rds is not None:
        e["d_sink"] = rel_l2(to64(ds), rds)
    else:
        assert ds is None
    for k, v in e.items():
        assert v <= tol, (ctx, k, v)
    return e


CASES = {  # name: (dsa_case kwargs)
    "page_mla_length": dict(B=1, S=512, Skv=2048, D=576, K=128, sink=True, length=True),
    "page_mla_full": dict(B=1, S=512, Skv=2048, D=576, K=128, sink=True, length=False),
    "d512_length": dict(B=1, S=512, Skv=2048, D=512, K=128, sink=True, length=True),
    "no_sink": dict(B=2, S=96, Skv=700, D=576, K=128, sink=False, length=True),
    "two_items_ragged": dict(B=2, S=80, Skv=900, D=576, K=200, sink=True, length=True),
    "three_items_full": dict(B=1, S=40, Skv=1000, D=512, K=384, sink=True, length=False),
}


@pytest.mark.parametrize("name", list(CASES))
def test_sparse_bwd_matches_oracle(name):
    kw = CASES[name]
    c = W.dsa_case(seed=61, **kw)
    sc = 1.0 / math.sqrt(kw["D"])
    ref = _oracle(c, sc)
    got = _gpu(c, ref[0], ref[1], sc)
    torch.cuda.synchronize()
    e = _check(got, ref, TOL[torch.bfloat16], name)
    print(name, {k: "%.2e" % v for k, v in e.items()})


@pytest.mark.parametrize("D", [512, 576])
def test_sparse_bwd_fp16(D):
    """The page's fp16 check (a real fp16 path, not bf16 bits read as fp16)."""
    c = W.dsa_case(S=256, Skv=1024, D=D, seed=62, dtype=torch.float16)
    sc = 1.0 / math.sqrt(D)
    ref = _oracle(c, sc)
    got = _gpu(c, ref[0], ref[1], sc)
    torch.cuda.synchronize()
    _check(got, ref, TOL[torch.float16], "fp16 D=%d" % D)


def test_sparse_bwd_invalid_and_repeated_entries():
    """Entries past the length, -1, rows >= S_kv and a token with length 0
    take no part; a row listed twice counts twice; dq of a token with no
    valid entry is exactly 0."""
    c = W.dsa_case(B=2, S=64, Skv=300, D=576, K=128, seed=63)
    idx, ln = c["topk_idxs"], c["topk_length"]
    ln[0, 3] = 0
    ln[1, 5] = 128
    idx[1, 5, 7] = 300 + 11                                      # past S_kv
    idx[1, 5, 9] = -7
    idx[1, 5, 20] = idx[1, 5, 21]                                # repeated row
    idx[0, 9, :] = -1
    ln[0, 9] = 128
    sc = 0.05
    ref = _oracle(c, sc)
    got = _gpu(c, ref[0], ref[1], sc)
    torch.cuda.synchronize()
    _check(got, ref, TOL[torch.bfloat16], "invalid entries")
    assert torch.count_nonzero(got[0][0, 3]) == 0 and torch.count_nonzero(got[0][0, 9]) == 0


def test_sparse_bwd_no_kv_rows_gives_zero_dq():
    from softmax_attention_numerics_gb300 import attn_sparse_bwd
    q = torch.randn(1, 4, 64, 512, device="cuda").bfloat16()
    kv = torch.empty(1, 0, 512, device="cuda", dtype=torch.bfloat16)
    out = torch.randn(1, 4, 64, 512, device="cuda").bfloat16()
    lse = torch.zeros(1, 4, 64, device="cuda")
    idx = torch.zeros(1, 4, 8, dtype=torch.int32, device="cuda")
    sink = torch.zeros(64, device="cuda")
    dq, dkv, ds = attn_sparse_bwd(q, kv, out, out, lse, idx, attn_sink=sink)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dq) == 0 and dkv.numel() == 0
    # d_sink = -sum exp(sink - lse) (dout . out) with lse = sink = 0
    ref = -(out.double() * out.double()).sum(dim=(0, 1, 3))
    assert torch.allclose(ds.double(), ref, rtol=1e-3)


def test_sparse_bwd_strided_inputs():
    """q, out and dout as views with padded rows (strides that are multiples
    of 8 elements but not contiguous)."""
    c = W.dsa_case(B=1, S=128, Skv=512, D=576, K=128, seed=64)
    sc = 1.0 / 24
    ref = _oracle(c, sc)
    from softmax_attention_numerics_gb300 import attn_sparse_bwd
    qb = torch.zeros(1, 128, 64, 640, dtype=torch.bfloat16, device="cuda")
    qb[..., :576] = c["q"].cuda()
    ob = torch.zeros(1, 128, 64, 520, dtype=torch.bfloat16, device="cuda")
    ob[..., :512] = torch.from_numpy(ref[0]).bfloat16().cuda()
    db = torch.zeros(1, 128, 64, 520, dtype=torch.bfloat16, device="cuda")
    db[..., :512] = c["dout"].cuda()
    got = attn_sparse_bwd(qb[..., :576], c["kv"].cuda(), ob[..., :512], db[..., :512],
                          torch.from_numpy(ref[1]).float().cuda(), c["topk_idxs"].cuda(),
                          topk_length=c["topk_length"].cuda(), attn_sink=c["attn_sink"].cuda(),
                          scale=sc)
    torch.cuda.synchronize()
    _check(got, ref, TOL[torch.bfloat16], "strided")


def test_sparse_bwd_reproducible_and_stream_ordered():
    """dq and d_sink are bit-identical on a second call; a call on a side
    stream while the ambient stream is busy (NVIDIA/cudnn-frontend PR #429's
    regression: the zero-fills must be ordered with the kernels on the launch
    stream) gives the same dq and d_sink and a dkv within the fp32 reduction
    reordering bound."""
    c = W.dsa_case(B=1, S=256, Skv=1024, D=576, K=128, seed=65)
    sc = 1.0 / 24
    ref = _oracle(c, sc)
    a = _gpu(c, ref[0], ref[1], sc)
    b = _gpu(c, ref[0], ref[1], sc)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])
    side = torch.cuda.Stream()
    torch.cuda._sleep(200_000_000)                                   # busy ambient stream
    s = _gpu(c, ref[0], ref[1], sc, stream=side)
    torch.cuda.synchronize()
    assert torch.equal(a[0], s[0]) and torch.equal(a[2], s[2])
    assert rel_l2(to64(s[1]), to64(a[1])) < 1e-2
    _check(s, ref, TOL[torch.bfloat16], "side stream")


def test_sparse_bwd_bench_size_sampled():
    """The benchmark's workload (16 sequences of S = 512 over S_kv = 2048,
    H = 64, D = 576, top-k = 128, sink and lengths) in the launch
    configuration the benchmark times, checked on sampled outputs: dq of 24
    tokens and dkv of 12 rows against the oracle token by token (a row's dkv
    collects the terms of every token that lists it), and d_sink against
    -sum exp(sink - lse) dout . out over all tokens."""
    kw = dict(B=16, S=512, Skv=2048, D=576, K=128, sink=True, length=True)
    c = W.dsa_case(seed=66, **kw)
    sc = 1.0 / math.sqrt(576)
    # forward statistics from the oracle, token by token
    q64, kv64, do64 = _np(c["q"]), _np(c["kv"]), _np(c["dout"])
    idx, ln, sink = c["topk_idxs"].numpy(), c["topk_length"].numpy(), c["attn_sink"].double().numpy()
    B, S = idx.shape[:2]
    out64 = np.zeros((B, S, 64, 512))
    lse64 = np.zeros((B, S, 64))
    toks = {}
    for b in range(B):
        for i in range(S):
            rows = [int(idx[b, i, e]) for e in OS.valid_entries(idx[b, i], ln[b, i], kw["Skv"])]
            P, psink, o, l = OS._token_fwd(q64[b, i], kv64[b], rows, sink, sc, 512)
            out64[b, i], lse64[b, i] = o, l
            toks[(b, i)] = (rows, P, psink)
    dq, dkv, ds = _gpu(c, out64, lse64, sc)
    torch.cuda.synchronize()
    for t in (dq, dkv, ds):
        assert nonfinite(t) == (0, 0)
    # the inputs the kernel saw: out rounded to bf16
    out_r = to64(torch.from_numpy(out64).bfloat16())
    rng = np.random.default_rng(0)
    dq64 = to64(dq)
    for n in rng.choice(B * S, 24, replace=False):
        b, i = divmod(int(n), S)
        rows, P, psink = toks[(b, i)]
        g, _, _ = OS._token_bwd(q64[b, i], kv64[b][rows], P, psink, do64[b, i], sc, 512)
        assert rel_l2(dq64[b, i], g) <= 2e-2, (b, i)
    dkv64 = to64(dkv)
    for n in rng.choice(B * kw["Skv"], 12, replace=False):
        b, r = divmod(int(n), kw["Skv"])
        acc = np.zeros(576)
        for i in range(S):
            rows, P, psink = toks[(b, i)]
            if r not in rows:
                continue
            _, gk, _ = OS._token_bwd(q64[b, i], kv64[b][rows], P, psink, do64[b, i], sc, 512)
            for e, rr in enumerate(rows):
                if rr == r:
                    acc += gk[e]
        assert rel_l2(dkv64[b, r], acc) <= 2e-2, (b, r)
    delta = (out_r * do64).sum(-1)
    ref_ds = -(np.exp(sink[None, None, :] - lse64) * delta).sum(axis=(0, 1))
    assert rel_l2(to64(ds), ref_ds) <= 1e-4
