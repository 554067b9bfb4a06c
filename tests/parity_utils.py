"""Shared helpers of the GPU parity tests: run a workload through the CUDA
library and through the fp64 oracle, and compare them with the acceptance
bar of the attention path:

    out   rel-L2 <= 1e-2 and max-abs <= 2e-2
    dq, dk, dv  rel-L2 <= 2e-2
    lse   abs error <= 1e-3
    zero NaN / Inf anywhere (counted separately, FlyDSL PR #1033 review)
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import attn_oracle as O

TOL_OUT_REL = 1e-2
TOL_OUT_ABS = 2e-2
TOL_GRAD_REL = 2e-2
TOL_LSE_ABS = 1e-3


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_mask(mask):
    """torch mask (uint8/bool visible flags or additive float) -> oracle form."""
    if mask is None:
        return None
    m = mask.detach().cpu()
    if m.dtype in (torch.uint8, torch.bool):
        return m.bool().numpy()
    return m.to(torch.float64).numpy()


def rel_l2(a, b):
    den = np.linalg.norm(b.ravel())
    num = np.linalg.norm((a - b).ravel())
    return num / den if den > 0 else num


def nonfinite(x):
    x = x.detach() if torch.is_tensor(x) else torch.as_tensor(x)
    return int(torch.isnan(x).sum()), int(torch.isinf(x).sum())


def gpu_run(case, deterministic=False, eager=False, dev="cuda", stream=None):
    """fwd + bwd through the library; returns torch tensors on the device."""
    from softmax_attention_numerics_gb300 import attn_bwd, attn_fwd
    q, k, v, do = (case[n].to(dev) for n in ("q", "k", "v", "do"))
    mask = case.get("mask")
    mask = None if mask is None else mask.to(dev)
    cu = case.get("cu_seqlens")
    cu = None if cu is None else cu.to(dev)
    kw = dict(mask=mask, cu_seqlens=cu, max_seqlen=case.get("max_seqlen"),
              causal=case["causal"], scale=case["scale"], stream=stream)
    out, lse = attn_fwd(q, k, v, eager_rescale=eager, **kw)
    dq, dk, dv = attn_bwd(q, k, v, out, do, lse, deterministic=deterministic, **kw)
    return dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv)


def assert_finite(res):
    for name, t in res.items():
        nan, inf = nonfinite(t)
        assert nan == 0 and inf == 0, "%s: %d NaN, %d Inf" % (name, nan, inf)


def compare(got, ref, names=("out", "lse", "dq", "dk", "dv"), ctx=""):
    """got: dict of torch (GPU) tensors; ref: dict of fp64 numpy arrays."""
    report = {}
    for n in names:
        g = to64(got[n]) if torch.is_tensor(got[n]) else got[n]
        r = ref[n]
        # the reference itself must be finite before it can serve as one
        # (FlyDSL PR #1033, review: NaN and Inf reported on both sides)
        assert np.isfinite(r).all(), "%s: oracle %s not finite" % (ctx, n)
        if n == "lse":
            err = float(np.abs(g - r).max()) if r.size else 0.0
            report[n] = err
            assert err <= TOL_LSE_ABS, "%s lse abs err %.3g" % (ctx, err)
        elif n == "out":
            rl = rel_l2(g, r)
            ma = float(np.abs(g - r).max()) if r.size else 0.0
            report[n] = (rl, ma)
            assert rl <= TOL_OUT_REL and ma <= TOL_OUT_ABS, "%s out rel %.3g abs %.3g" % (ctx, rl, ma)
        else:
            rl = rel_l2(g, r)
            report[n] = rl
            assert rl <= TOL_GRAD_REL, "%s %s rel-L2 %.3g" % (ctx, n, rl)
    return report


def oracle_dense(case):
    out, lse, dq, dk, dv = O.attn_bwd(to64(case["q"]), to64(case["k"]), to64(case["v"]),
                                      to64(case["do"]), mask=oracle_mask(case.get("mask")),
                                      causal=case["causal"], scale=case["scale"])
    return dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv)
