"""The bounds-check / stall-injection debug build (ATTN_DEBUG_CHECKS).

1. Run through the debug build, the parity workloads give the same bits as
   the product build (the checks only read indices; the fp32 dQ reductions
   may land in another order) with a clean error word: no per-tile bounds
   check fired.
2. attn_debug_inject_stall makes one bounded wait of block (0, 0, 0)'s MMA
   issuer run out on a barrier that nothing completes at that point.  The
   kernel then unwinds through its own paths: the abort flag, the TMA
   producer waiting for its copies in flight, the MMA issuer draining its
   MMAs, TMEM freed, ATTN_E_TIMEOUT in the device error word
   (PFCCLab/cudnn-frontend PR #9: a wait that would hang reports instead).
   Nothing faults or hangs, and a full forward + backward through the
   product build right after matches the fp64 oracle: the context stays
   usable.
"""
import ctypes

import pytest
import torch

import attn_workloads as W
from parity_utils import assert_finite, compare, gpu_run, oracle_dense

pytestmark = pytest.mark.gpu

E_TIMEOUT = -8


@pytest.fixture(scope="module")
def checked_lib():
    from softmax_attention_numerics_gb300 import build as _build
    _build.build()
    return _build.build(variant="checked")


def _cases():
    q, k, v, do = W.dense_qkvdo(2, 700, 700, 8, 2, 128, seed=31)
    yield "causal_gqa_ragged", dict(q=q, k=k, v=v, do=do, causal=True, scale=0.088)
    q, k, v, do = W.dense_qkvdo(1, 1100, 1100, 4, 4, 64, seed=32)
    yield "d64_ragged", dict(q=q, k=k, v=v, do=do, causal=False, scale=0.125)
    yield "low_lse_bool_mask", W.low_lse_row(392, 392, "bool")
    yield "varlen_gqa_trailing", W.varlen_gqa(n=4, lo=130, hi=900, Hq=8, Hkv=2, trailing=77)
    yield "fp16_low_lse_additive", W.low_lse_row(100, 77, "additive", row="last",
                                                 dtype=torch.float16)


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("name", [n for n, _ in _cases()])
def test_checked_build_matches_product_build(checked_lib, name, deterministic):
    from softmax_attention_numerics_gb300 import _lib, get_error
    case = dict(_cases())[name]
    ref = gpu_run(case, deterministic=deterministic)
    torch.cuda.synchronize()
    with _lib.use_library(checked_lib):
        got = gpu_run(case, deterministic=deterministic)
        torch.cuda.synchronize()
        assert get_error() == 0, "a bounds check fired"
    assert_finite(got)
    for n in ("out", "lse", "dq", "dk", "dv"):
        if n == "dq" and not deterministic:          # fp32 reduction order may differ
            assert torch.allclose(got[n].float(), ref[n].float(), rtol=2e-2, atol=2e-3), n
        else:
            assert torch.equal(got[n], ref[n]), (name, n)


def test_checked_build_fp8_forward_matches_product_build(checked_lib):
    from softmax_attention_numerics_gb300 import _lib, attn_fwd_fp8, get_error
    c = W.fp8_qkv(B=2, S=300, H=4, D=128, k_scale=8.0, v="randn", causal=True, seed=7)
    q, k, v = (c[n].cuda().view(torch.float8_e4m3fn) for n in ("q", "k", "v"))
    args = (q, k, v, c["descale_q"], c["descale_k"], c["descale_v"])
    ref = attn_fwd_fp8(*args, causal=True, scale=c["scale"])
    with _lib.use_library(checked_lib):
        got = attn_fwd_fp8(*args, causal=True, scale=c["scale"])
        torch.cuda.synchronize()
        assert get_error() == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_checked_build_score_recompute_matches_product_build(checked_lib):
    from softmax_attention_numerics_gb300 import _lib, attn_fwd, attn_score_recompute, get_error
    q, k, _, _ = (t.cuda() for t in W.dense_qkvdo(2, 300, 300, 8, 2, 128, seed=34))
    _, lse = attn_fwd(q, k, k, causal=True)
    ref = attn_score_recompute(q, k, lse, causal=True)
    with _lib.use_library(checked_lib):
        got = attn_score_recompute(q, k, lse, causal=True)
        torch.cuda.synchronize()
        assert get_error() == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def _sparse_inputs(S=8, Skv=600, K=512, seed=36, length=False):
    c = W.dsa_case(B=1, S=S, Skv=Skv, D=576, K=K, seed=seed, length=length)
    d = {k: (None if v is None else v.cuda()) for k, v in c.items()}
    d["out"] = torch.randn(1, S, 64, 512, device="cuda").bfloat16()
    d["lse"] = torch.randn(1, S, 64, device="cuda") + 8.0
    return d


def test_checked_build_sparse_bwd_matches_product_build(checked_lib):
    from softmax_attention_numerics_gb300 import _lib, attn_sparse_bwd, get_error
    d = _sparse_inputs(S=40, Skv=700, K=300, length=True)
    args = (d["q"], d["kv"], d["out"], d["dout"], d["lse"], d["topk_idxs"])
    kw = dict(topk_length=d["topk_length"], attn_sink=d["attn_sink"], scale=0.04)
    ref = attn_sparse_bwd(*args, **kw)
    with _lib.use_library(checked_lib):
        got = attn_sparse_bwd(*args, **kw)
        torch.cuda.synchronize()
        assert get_error() == 0
    assert torch.equal(got[0], ref[0]) and torch.equal(got[2], ref[2])       # dq, d_sink
    assert torch.allclose(got[1].float(), ref[1].float(), rtol=2e-2, atol=1e-3)   # fp32 add order


# (kernel, iteration of its MMA issuer's loop): 1 forward, 2 backward main,
# 3 deterministic dQ, 4 fp8 forward, 5 score recompute (the loop runs over heads),
# 6 sparse backward (the loop runs over work items: token 0 has four of them).
STALLS = [(1, 0), (1, 3), (2, 0), (2, 5), (3, 0), (3, 2), (4, 0), (4, 2), (5, 0), (5, 3),
          (6, 0), (6, 3)]


def _stalled_call(kernel):
    """The call whose kernel the stall targets, on a problem where block
    (0, 0, 0) runs more than three iterations of its loop."""
    from softmax_attention_numerics_gb300 import attn_bwd, attn_fwd, attn_fwd_fp8
    from softmax_attention_numerics_gb300 import attn_score_recompute
    if kernel == 6:
        from softmax_attention_numerics_gb300 import attn_sparse_bwd
        d = _sparse_inputs()
        attn_sparse_bwd(d["q"], d["kv"], d["out"], d["dout"], d["lse"], d["topk_idxs"],
                        attn_sink=d["attn_sink"], scale=0.04)
        return
    if kernel == 5:
        q, k, _, _ = (t.cuda() for t in W.dense_qkvdo(1, 300, 300, 8, 2, 128, seed=35))
        lse = torch.zeros(1, 8, 300, device="cuda")
        attn_score_recompute(q, k, lse)
        return
    if kernel == 4:
        c = W.fp8_qkv(B=1, S=700, H=2, D=128, k_scale=1.0, v="randn", seed=9)
        q, k, v = (c[n].cuda().view(torch.float8_e4m3fn) for n in ("q", "k", "v"))
        attn_fwd_fp8(q, k, v, c["descale_q"], c["descale_k"], c["descale_v"], scale=c["scale"])
        return
    q, k, v, do = (t.cuda() for t in W.dense_qkvdo(1, 700, 700, 4, 2, 128, seed=33))
    out, lse = attn_fwd(q, k, v, scale=0.088)
    if kernel in (2, 3):
        attn_bwd(q, k, v, out, do, lse, scale=0.088, deterministic=kernel == 3)


@pytest.mark.parametrize("kernel,iteration", STALLS, ids=["k%d_it%d" % s for s in STALLS])
def test_injected_stall_unwinds_and_reports_timeout(checked_lib, kernel, iteration):
    from softmax_attention_numerics_gb300 import _lib, get_error
    with _lib.use_library(checked_lib) as lib:
        lib.attn_debug_inject_stall.restype = ctypes.c_int
        lib.attn_debug_inject_stall.argtypes = [ctypes.c_int, ctypes.c_int]
        assert get_error() == 0
        assert lib.attn_debug_inject_stall(kernel, iteration) == 0
        try:
            _stalled_call(kernel)
            torch.cuda.synchronize()
            err = get_error()
        finally:
            lib.attn_debug_inject_stall(0, 0)
        assert err == E_TIMEOUT
        assert get_error() == 0                       # reading cleared it
    # the context is intact: the product build still matches the oracle
    case = W.causal_small()
    res = gpu_run(case)
    assert_finite(res)
    compare(res, oracle_dense(case), ctx="after stall %d/%d" % (kernel, iteration))
