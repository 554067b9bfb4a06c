"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory when they run it (a plugin inside a framework that owns all device
memory, a real-time caller with a fixed memory budget).  Its scratch is an
array compiled into the library instead of a caller-provided workspace.

The test calls it through the C ABI twice in a row and checks both results
against the regular attn_bwd entry point (which takes a workspace), with the
gradient tolerance of the parity tests.  The outputs are filled with NaN
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


def test_noalloc_matches_attn_bwd_on_two_calls(lib):
    from softmax_attention_numerics_gb300 import attn_bwd, attn_fwd
    from softmax_attention_numerics_gb300.ops import tensor_desc
    case = W.low_lse_row(392, 392, "bool", D=128)
    q, k, v, do = (case[n].cuda() for n in ("q", "k", "v", "do"))
    mask = case["mask"].cuda()
    scale = case["scale"]
    out, lse = attn_fwd(q, k, v, mask=mask, scale=scale)
    ref = attn_bwd(q, k, v, out, do, lse, mask=mask, scale=scale)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        dq = torch.full_like(q, float("nan"))
        dk = torch.full_like(k, float("nan"))
        dv = torch.full_like(v, float("nan"))
        ins = [tensor_desc(x) for x in (q, k, v, out, do, lse, mask.view(torch.uint8))]
        outs = [tensor_desc(x) for x in (dq, dk, dv)]
        rc = lib.attn_bwd_noalloc(*[_ref(d) for d in ins], None, 0, 0, scale,
                                  *[_ref(d) for d in outs], 0, ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, lib.attn_strerror(rc)
        torch.cuda.synchronize()
        got = dict(dq=dq, dk=dk, dv=dv)
        assert_finite(got)
        for name, r in zip(("dq", "dk", "dv"), ref):
            assert rel_l2(to64(got[name]), to64(r)) <= TOL_GRAD_REL, name


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
