"""GPU parity of the fp8 (E4M3) forward against the fp64 oracle on the decoded
inputs (FlyDSL PR #1033, "The fp8 helper, second commit").

Bar (from a numerics model of the kernel's arithmetic: P rounded to E4M3
before P V, out normalised by the sum of the rounded P): out rel-L2 <= 5e-2
and max-abs <= 0.15, lse abs <= 1e-3, zero NaN/Inf; on the pages' own test,
K scaled x1000 / x5000 / x20000 with V = ones at B=1 H=16 S=12288 D=128,
mean |out - 1| <= 2e-3 and no non-finite value."""
import numpy as np
import pytest
import torch

import attn_workloads as W
from oracle import attn_oracle as O
from parity_utils import rel_l2

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS, TOL_LSE = 5e-2, 0.15, 1e-3


def _run(c, dev="cuda", eager=False):
    from softmax_attention_numerics_gb300 import attn_fwd_fp8
    q, k, v = (c[n].to(dev).view(torch.float8_e4m3fn) for n in ("q", "k", "v"))
    out, lse = attn_fwd_fp8(q, k, v, c["descale_q"], c["descale_k"], c["descale_v"],
                            causal=c["causal"], scale=c["scale"], eager_rescale=eager)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def _oracle(c):
    return O.attn_fwd_fp8(c["q"].numpy(), c["k"].numpy(), c["v"].numpy(), c["descale_q"],
                          c["descale_k"], c["descale_v"], causal=c["causal"], scale=c["scale"])


CASES = [  # (B, S, H, k_scale, causal)
    (1, 128, 2, 1.0, False),
    (2, 300, 4, 1.0, False),      # ragged: partial last key and query tiles
    (2, 300, 4, 1.0, True),
    (1, 1000, 2, 8.0, False),
    (1, 1000, 2, 32.0, True),
    (1, 77, 3, 1.0, False),       # fewer keys than a tile
]


@pytest.mark.parametrize("cfg", CASES, ids=[str(c) for c in CASES])
@pytest.mark.parametrize("eager", [False, True])
def test_fp8_forward_matches_oracle(cfg, eager):
    B, S, H, ks, causal = cfg
    c = W.fp8_qkv(B=B, S=S, H=H, D=128, k_scale=ks, v="randn", causal=causal, seed=7)
    out, lse = _run(c, eager=eager)
    ref_out, ref_lse = _oracle(c)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert rel_l2(out, ref_out) <= TOL_REL
    assert np.abs(out - ref_out).max() <= TOL_ABS
    assert np.abs(lse - ref_lse).max() <= TOL_LSE


@pytest.mark.parametrize("ks", [1000.0, 5000.0, 20000.0])
def test_fp8_unit_values_at_the_pages_spreads(ks):
    c = W.fp8_qkv(B=1, S=12288, H=16, D=128, k_scale=ks, v="ones")
    out, lse = _run(c)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    one = 448.0 * c["descale_v"]
    assert np.abs(out / one - 1.0).mean() <= 2e-3
