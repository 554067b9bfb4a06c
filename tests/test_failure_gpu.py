"""Failure detection on the GPU without a fault: a bounded device wait that
nothing satisfies gives up, the error word reports ATTN_E_TIMEOUT on the
host, and the context stays usable for the next attention call.  The wait is
the same loop that bounds every wait of the attention kernels; here its
budget is 20 ms instead of 2 s."""
import time

import pytest
import torch

import attn_workloads as W
from parity_utils import assert_finite, compare, gpu_run, oracle_dense
from softmax_attention_numerics_gb300 import _lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    lib = _lib.load()
    s = torch.cuda.Stream()
    assert lib.attn_get_error(ctypes_stream(s)) == 0          # clean start
    t0 = time.perf_counter()
    assert lib.attn_selftest_wait_timeout(20000, ctypes_stream(s)) == 0
    code = lib.attn_get_error(ctypes_stream(s))                # synchronises s
    waited = time.perf_counter() - t0
    timeout_code = {name: c for c, name in _lib.ERRORS.items()}["ATTN_E_TIMEOUT"]
    assert code == timeout_code, code
    assert waited >= 0.02
    assert lib.attn_get_error(ctypes_stream(s)) == 0          # read and cleared
    # the context is still usable: a full fwd + bwd matches the oracle
    case = W.causal_small()
    res = gpu_run(case)
    assert_finite(res)
    compare(res, oracle_dense(case), ctx="after timeout probe")
    assert lib.attn_get_error(None) == 0


def ctypes_stream(s):
    import ctypes
    return ctypes.c_void_p(s.cuda_stream)
