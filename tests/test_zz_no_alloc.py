"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory when they run it (a plugin inside a framework that owns all device
memory, a real-time caller with a fixed memory budget).  Its scratch is an
array compiled into the library instead of a caller-provided workspace.

The test calls it through the C ABI, twice in a row for each case and dQ
mode and all of them back to back, and checks every result against the
regular attn_bwd entry point (which takes a workspace): bit-identical where
the same kernels run in the same order, within the gradient tolerance of the
parity tests for the atomic dQ.  The outputs are filled with NaN
before every call, so a row the call forgot to write would show up.  It also
checks that a problem too large for the built-in array is refused before
anything is launched.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import attn_workloads as W
from parity_utils import TOL_GRAD_REL, assert_finite, rel_l2, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from softmax_attention_numerics_gb300 import _lib, build
    build.build()
    return _lib.load()


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _cases():
    """A dense masked case (OpenWAM PR #64's low-lse row) and a packed varlen
    GQA case with trailing rows: the workspace layout differs between them
    (dense B*Sq rows against T rows) and with ATTN_DETERMINISTIC (no dQ
    accumulator)."""
    dense = W.low_lse_row(392, 392, "bool", D=128)
    dense["mask"] = dense["mask"].cuda()
    var = W.varlen_gqa(n=4, lo=130, hi=700, Hq=8, Hkv=2, trailing=77)
    var["cu_seqlens"] = var["cu_seqlens"].cuda()
    for c in (dense, var):
        for n in ("q", "k", "v", "do"):
            c[n] = c[n].cuda()
    return [("dense", dense), ("varlen", var)]


def _noalloc(lib, c, out, lse, flags):
    from softmax_attention_numerics_gb300.ops import tensor_desc
    q, k, v, do = c["q"], c["k"], c["v"], c["do"]
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    mask = c.get("mask")
    cu = c.get("cu_seqlens")
    ins = [tensor_desc(x) for x in (q, k, v, out, do, lse)]
    md = None if mask is None else tensor_desc(mask.view(torch.uint8))
    cd = None if cu is None else tensor_desc(cu)
    outs = [tensor_desc(x) for x in (dq, dk, dv)]
    stream = torch.cuda.current_stream()
    rc = lib.attn_bwd_noalloc(*[_ref(d) for d in ins], _ref(md), _ref(cd),
                              int(c.get("max_seqlen") or 0), 1 if c["causal"] else 0,
                              c["scale"], *[_ref(d) for d in outs], flags,
                              ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, lib.attn_strerror(rc)
    torch.cuda.synchronize()
    return dict(dq=dq, dk=dk, dv=dv)


def test_noalloc_matches_attn_bwd_on_two_calls(lib):
    """Every (case, dQ mode) pair runs twice in a row, and the pairs run back to
    back, so each call starts from what the previous one left in the shared
    array.  dk and dv come from the same kernels as attn_bwd's and must be
    bit-identical; so must dq on the deterministic path, while the fp32
    reductions of the atomic path only promise the gradient tolerance."""
    from softmax_attention_numerics_gb300 import attn_bwd, attn_fwd
    det = _lib_flags()
    runs = []
    for name, c in _cases():
        kw = dict(mask=c.get("mask"), cu_seqlens=c.get("cu_seqlens"),
                  max_seqlen=c.get("max_seqlen"), causal=c["causal"], scale=c["scale"])
        out, lse = attn_fwd(c["q"], c["k"], c["v"], **kw)
        for flags in (0, det):
            ref = attn_bwd(c["q"], c["k"], c["v"], out, c["do"], lse,
                           deterministic=flags == det, **kw)
            runs.append((name, c, out, lse, flags, dict(zip(("dq", "dk", "dv"), ref))))
    for name, c, out, lse, flags, ref in runs + runs[:1]:
        for _ in range(2):
            got = _noalloc(lib, c, out, lse, flags)
            assert_finite(got)
            for n in ("dk", "dv"):
                assert torch.equal(got[n], ref[n]), (name, flags, n)
            if flags == det:
                assert torch.equal(got["dq"], ref["dq"]), (name, "dq")
            else:
                assert rel_l2(to64(got["dq"]), to64(ref["dq"])) <= TOL_GRAD_REL, (name, "dq")


def _lib_flags():
    from softmax_attention_numerics_gb300 import _lib
    return _lib.ATTN_DETERMINISTIC


def test_noalloc_refuses_problems_beyond_its_array(lib):
    from softmax_attention_numerics_gb300 import _lib

    def desc(shape, dtype=_lib.ATTN_BF16):
        d = _lib.AttnTensor()
        d.data = 1 << 20          # never dereferenced: the call returns first
        d.dtype = dtype
        d.ndim = len(shape)
        s = 1
        for i in reversed(range(len(shape))):
            d.shape[i] = shape[i]
            d.stride[i] = s
            s *= shape[i]
        d.device = 0
        return d

    big_q = desc([1, 65536, 16, 128])      # workspace ~ 545 MB
    big_k = desc([1, 65536, 16, 128])
    lse = desc([1, 16, 65536], _lib.ATTN_F32)
    rc = lib.attn_bwd_noalloc(_ref(big_q), _ref(big_k), _ref(big_k), _ref(big_q), _ref(big_q),
                              _ref(lse), None, None, 0, 0, 0.1, _ref(big_q), _ref(big_k),
                              _ref(big_k), 0, None)
    assert rc == -12       # ATTN_E_TOO_LARGE
