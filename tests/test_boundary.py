"""Host-side tests of the C ABI: the library builds, loads and exports every
symbol the header declares, and malformed calls are rejected before any
launch (NVIDIA/cudnn-frontend PR #429: dtype gate, shape contract including a
transposed dout or lse, contiguous out-parameters; PFCCLab/cudnn-frontend
PR #9, section 4: unsupported head_dim).  The descriptors here point at fake
device addresses: every call under test returns before touching the GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from softmax_attention_numerics_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_gb300.h")

E = {v: k for k, v in _lib.ERRORS.items()}
FAKE = 1 << 20   # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_expected_api():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True).stdout
    for name in declared_functions():
        assert re.search(r"\bT %s\b" % name, out), name


def test_version_and_strerror(lib):
    assert lib.attn_version() >= 100
    for code in _lib.ERRORS:
        assert lib.attn_strerror(code)


def desc(shape, dtype=_lib.ATTN_BF16, stride=None, data=FAKE, device=-1):
    """Descriptor of a fake buffer.  The default device -1 (host memory) makes
    a call that passes every host-side check stop at the device check, so no
    call in this file can reach a launch, even where a GPU is present."""
    d = _lib.AttnTensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    if stride is None:
        stride, s = [], 1
        for n in reversed(shape):
            stride.insert(0, s)
            s *= n
    for i, n in enumerate(shape):
        d.shape[i] = n
        d.stride[i] = stride[i]
    d.device = device
    return d


def dense(B=2, Sq=100, Sk=77, Hq=4, Hkv=2, D=128):
    return dict(q=desc([B, Sq, Hq, D]), k=desc([B, Sk, Hkv, D]), v=desc([B, Sk, Hkv, D]),
                out=desc([B, Sq, Hq, D]), lse=desc([B, Hq, Sq], _lib.ATTN_F32),
                dout=desc([B, Sq, Hq, D]), dq=desc([B, Sq, Hq, D]), dk=desc([B, Sk, Hkv, D]),
                dv=desc([B, Sk, Hkv, D]))


def R(x):
    return None if x is None else ctypes.byref(x)


def call_fwd(lib, t, mask=None, cu=None, max_seqlen=0, scale=0.1):
    return lib.attn_fwd(R(t["q"]), R(t["k"]), R(t["v"]), R(mask), R(cu), max_seqlen, 0, scale,
                        R(t["out"]), R(t["lse"]), 0, None)


def call_bwd(lib, t, mask=None, cu=None, max_seqlen=0, ws=FAKE, ws_bytes=1 << 40, flags=0):
    return lib.attn_bwd(R(t["q"]), R(t["k"]), R(t["v"]), R(t["out"]), R(t["dout"]), R(t["lse"]),
                        R(mask), R(cu), max_seqlen, 0, 0.1, R(t["dq"]), R(t["dk"]), R(t["dv"]),
                        ctypes.c_void_p(ws), ws_bytes, flags, None)


def test_rejects_mixed_or_unsupported_element_types(lib):
    # fp16 is computed, but every 16-bit tensor must have q's type
    t = dense()
    t["q"] = desc([2, 100, 4, 128], _lib.ATTN_F16)
    assert call_fwd(lib, t) == E["ATTN_E_DTYPE"]                 # k, v still bf16
    t = dense()
    for n in ("q", "k", "v"):
        t[n] = desc(t[n].shape[:4], _lib.ATTN_F16)
    assert call_fwd(lib, t) == E["ATTN_E_DTYPE"]                 # out still bf16
    t = dense()
    t["dout"] = desc([2, 100, 4, 128], _lib.ATTN_F16)
    assert call_bwd(lib, t) == E["ATTN_E_DTYPE"]
    t = dense()
    t["dq"] = desc([2, 100, 4, 128], _lib.ATTN_F16)
    assert call_bwd(lib, t) == E["ATTN_E_DTYPE"]
    for bad in (_lib.ATTN_F32, _lib.ATTN_I32, _lib.ATTN_U8):
        t = dense()
        for n in ("q", "k", "v"):
            t[n] = desc(t[n].shape[:4], bad)
        assert call_fwd(lib, t) == E["ATTN_E_DTYPE"]


def test_accepts_all_fp16(lib):
    """All-fp16 tensors pass the element-type gate; the descriptors say host
    memory (device -1), so the call stops at the device check and nothing is
    launched even where a GPU is present."""
    t = dense()
    for n in t:
        t[n] = desc(t[n].shape[:t[n].ndim],
                    _lib.ATTN_F32 if n == "lse" else _lib.ATTN_F16, device=-1)
    # ATTN_E_CUDA where no GPU is present (the device query itself fails)
    stop = (E["ATTN_E_DEVICE"], E["ATTN_E_CUDA"])
    assert call_fwd(lib, t) in stop
    assert call_bwd(lib, t) in stop


@pytest.mark.parametrize("D", [32, 96, 100, 112, 192, 256])
def test_rejects_unsupported_head_dim(lib, D):
    assert call_fwd(lib, dense(D=D)) == E["ATTN_E_UNSUPPORTED"]


def test_rejects_bad_gqa_ratio(lib):
    assert call_fwd(lib, dense(Hq=6, Hkv=4)) == E["ATTN_E_SHAPE"]


def test_rejects_mismatched_companions(lib):
    t = dense()
    t["v"] = desc([2, 76, 2, 128])
    assert call_fwd(lib, t) == E["ATTN_E_SHAPE"]
    t = dense()
    t["k"] = desc([1, 77, 2, 128]); t["v"] = desc([1, 77, 2, 128])
    assert call_fwd(lib, t) == E["ATTN_E_SHAPE"]


def test_rejects_transposed_dout_and_lse(lib):
    t = dense(Sq=100, Hq=4)
    t["dout"] = desc([2, 4, 100, 128])     # BHSD passed where BSHD is expected
    assert call_bwd(lib, t) == E["ATTN_E_SHAPE"]
    t = dense(Sq=100, Hq=4)
    t["lse"] = desc([2, 100, 4], _lib.ATTN_F32)
    assert call_bwd(lib, t) == E["ATTN_E_SHAPE"]
    t = dense()
    t["lse"] = desc([2, 4, 100], _lib.ATTN_BF16)
    assert call_bwd(lib, t) == E["ATTN_E_DTYPE"]


def test_rejects_layout_violations(lib):
    t = dense()
    t["q"] = desc([2, 100, 4, 128], stride=[100 * 4 * 128, 4 * 128, 128, 2])
    assert call_fwd(lib, t) == E["ATTN_E_LAYOUT"]
    t = dense()
    t["k"] = desc([2, 77, 2, 128], stride=[77 * 2 * 132, 2 * 132, 132, 1])   # 264-byte rows
    assert call_fwd(lib, t) == E["ATTN_E_LAYOUT"]
    t = dense()
    t["q"] = desc([2, 100, 4, 128], data=FAKE + 8)
    assert call_fwd(lib, t) == E["ATTN_E_LAYOUT"]


def test_strided_inputs_pass_validation(lib):
    # A BHSD buffer viewed as BSHD is a legal input (OpenWAM PR #64, Tests:
    # BSHD buffers viewed as BHSD); it reaches the device stage.
    t = dense()
    t["q"] = desc([2, 100, 4, 128], stride=[4 * 100 * 128, 128, 100 * 128, 1])
    rc = call_fwd(lib, t)
    assert rc in (E["ATTN_E_CUDA"], E["ATTN_E_DEVICE"])


def test_rejects_strided_out_params(lib):
    t = dense()
    t["out"] = desc([2, 100, 4, 128], stride=[4 * 100 * 128, 128, 100 * 128, 1])
    assert call_fwd(lib, t) == E["ATTN_E_LAYOUT"]
    t = dense()
    t["dk"] = desc([2, 77, 2, 128], stride=[77 * 2 * 128, 128, 77 * 128, 1])
    assert call_bwd(lib, t) == E["ATTN_E_LAYOUT"]


def test_rejects_non_finite_scale(lib):
    assert call_fwd(lib, dense(), scale=float("nan")) == E["ATTN_E_ARG"]
    assert call_fwd(lib, dense(), scale=float("inf")) == E["ATTN_E_ARG"]


def test_mask_contract(lib):
    bad = desc([2, 4, 100, 76], _lib.ATTN_U8)
    assert call_fwd(lib, dense(), mask=bad) == E["ATTN_E_SHAPE"]
    i32 = desc([2, 1, 1, 77], _lib.ATTN_I32)
    assert call_fwd(lib, dense(), mask=i32) == E["ATTN_E_DTYPE"]
    three = desc([2, 100, 77], _lib.ATTN_U8)
    assert call_fwd(lib, dense(), mask=three) == E["ATTN_E_SHAPE"]


def test_rejects_misaligned_mask(lib):
    # the kernels load mask elements one at a time: element alignment is the rule
    stop = (E["ATTN_E_DEVICE"], E["ATTN_E_CUDA"])
    for dtype, off, ok in ((_lib.ATTN_F32, 2, False), (_lib.ATTN_F32, 4, True),
                           (_lib.ATTN_BF16, 1, False), (_lib.ATTN_F16, 1, False),
                           (_lib.ATTN_BF16, 2, True), (_lib.ATTN_U8, 1, True)):
        mask = desc([2, 1, 1, 77], dtype, data=FAKE + off)
        rc = call_fwd(lib, dense(), mask=mask)
        assert (rc in stop) if ok else rc == E["ATTN_E_LAYOUT"], (dtype, off)
        rc = call_bwd(lib, dense(), mask=mask)
        assert (rc in stop) if ok else rc == E["ATTN_E_LAYOUT"], (dtype, off)


def test_bwd_lse_contract(lib):
    t = dense()
    t["lse"] = desc([2, 4, 100], _lib.ATTN_F32, data=0)
    assert call_bwd(lib, t) == E["ATTN_E_ARG"]
    t = dense()
    t["lse"] = desc([2, 4, 100], _lib.ATTN_F32, data=FAKE + 4)
    assert call_bwd(lib, t) == E["ATTN_E_LAYOUT"]
    t = dense()
    t["lse"] = desc([2, 4, 100], _lib.ATTN_F32, stride=[4 * 101, 101, 1])   # padded rows
    assert call_bwd(lib, t) == E["ATTN_E_LAYOUT"]


def varlen(T=1000, Hq=4, Hkv=2, D=64, n=3):
    return dict(q=desc([T, Hq, D]), k=desc([T, Hkv, D]), v=desc([T, Hkv, D]),
                out=desc([T, Hq, D]), lse=desc([Hq, T], _lib.ATTN_F32), dout=desc([T, Hq, D]),
                dq=desc([T, Hq, D]), dk=desc([T, Hkv, D]), dv=desc([T, Hkv, D])), \
        desc([n + 1], _lib.ATTN_I32)


def test_varlen_contract(lib):
    t, cu = varlen()
    t["lse"] = desc([1000, 4], _lib.ATTN_F32)
    assert call_fwd(lib, t, cu=cu, max_seqlen=512) == E["ATTN_E_SHAPE"]
    t, cu = varlen()
    cu.dtype = _lib.ATTN_F32
    assert call_fwd(lib, t, cu=cu, max_seqlen=512) == E["ATTN_E_DTYPE"]
    t, cu = varlen()
    mask = desc([1, 1, 1, 512], _lib.ATTN_U8)
    assert call_fwd(lib, t, mask=mask, cu=cu, max_seqlen=512) == E["ATTN_E_UNSUPPORTED"]
    t, cu = varlen()
    t["k"] = desc([999, 2, 64]); t["v"] = desc([999, 2, 64])
    assert call_fwd(lib, t, cu=cu, max_seqlen=512) == E["ATTN_E_SHAPE"]
    t, cu = varlen()
    cu.data = FAKE + 2                     # int32 offsets must be 4-byte aligned
    assert call_fwd(lib, t, cu=cu, max_seqlen=512) == E["ATTN_E_LAYOUT"]
    assert call_bwd(lib, t, cu=cu, max_seqlen=512) == E["ATTN_E_LAYOUT"]


def test_host_pointers_rejected(lib):
    t = dense()
    t["q"] = desc([2, 100, 4, 128], device=-1)
    rc = call_fwd(lib, t)
    assert rc in (E["ATTN_E_DEVICE"], E["ATTN_E_CUDA"])


def test_workspace_size_and_checks(lib):
    t = dense(B=2, Sq=100, Hq=4, D=128)
    n = lib.attn_bwd_workspace_bytes(R(t["q"]), R(t["k"]), 0)
    acc = -(-2 * 100 * 4 * 128 * 4 // 256) * 256
    vec = -(-2 * 100 * 4 * 4 // 256) * 256
    assert n == acc + 2 * vec
    nd = lib.attn_bwd_workspace_bytes(R(t["q"]), R(t["k"]), _lib.ATTN_DETERMINISTIC)
    assert nd == 2 * vec
    assert call_bwd(lib, t, ws_bytes=n - 1) == E["ATTN_E_WORKSPACE"]
    assert call_bwd(lib, t, ws=0, ws_bytes=n) == E["ATTN_E_WORKSPACE"]
    assert call_bwd(lib, t, ws=FAKE + 16, ws_bytes=n) == E["ATTN_E_WORKSPACE"]
    assert lib.attn_bwd_workspace_bytes(R(dense(D=96)["q"]), R(t["k"]), 0) == 0


def test_selftest_wait_timeout_rejects_bad_budget(lib):
    # checked before the device is touched
    assert lib.attn_selftest_wait_timeout(0, None) == E["ATTN_E_ARG"]
    assert lib.attn_selftest_wait_timeout(1000001, None) == E["ATTN_E_ARG"]


# ---------------------------------------------------------------- fp8 forward

def fp8_dense(B=2, Sq=300, Sk=200, Hq=4, Hkv=2, D=128):
    E4 = _lib.ATTN_E4M3
    return dict(q=desc([B, Sq, Hq, D], E4), k=desc([B, Sk, Hkv, D], E4),
                v=desc([B, Sk, Hkv, D], E4), out=desc([B, Sq, Hq, D]),
                lse=desc([B, Hq, Sq], _lib.ATTN_F32))


def call_fwd_fp8(lib, t, descales=(0.01, 0.02, 0.03), scale=0.1, ws=FAKE, ws_bytes=1 << 40):
    return lib.attn_fwd_fp8(R(t["q"]), R(t["k"]), R(t["v"]), *descales, 0, scale, R(t["out"]),
                            R(t["lse"]), ctypes.c_void_p(ws), ws_bytes, 0, None)


def test_fp8_forward_contract(lib):
    stop = (E["ATTN_E_DEVICE"], E["ATTN_E_CUDA"])
    assert call_fwd_fp8(lib, fp8_dense()) in stop                    # valid: stops at the device
    t = fp8_dense()
    t["k"] = desc([2, 200, 2, 128])                                  # bf16 k
    assert call_fwd_fp8(lib, t) == E["ATTN_E_DTYPE"]
    t = fp8_dense(D=64)
    assert call_fwd_fp8(lib, t) == E["ATTN_E_UNSUPPORTED"]
    t = fp8_dense()
    t["out"] = desc([2, 300, 4, 128], _lib.ATTN_F32)
    assert call_fwd_fp8(lib, t) == E["ATTN_E_DTYPE"]
    t = fp8_dense()
    t["lse"] = desc([2, 300, 4], _lib.ATTN_F32)                      # transposed lse
    assert call_fwd_fp8(lib, t) == E["ATTN_E_SHAPE"]
    t = fp8_dense(Hq=3)
    assert call_fwd_fp8(lib, t) == E["ATTN_E_SHAPE"]                 # 3 % 2 != 0
    t = fp8_dense()
    t["q"] = desc([2, 300, 4, 128], _lib.ATTN_E4M3, stride=[300 * 4 * 136, 4 * 136, 136, 1])
    assert call_fwd_fp8(lib, t) == E["ATTN_E_LAYOUT"]                # 136-byte rows
    for bad in ((0.0, 0.02, 0.03), (0.01, -1.0, 0.03), (0.01, 0.02, float("nan"))):
        assert call_fwd_fp8(lib, fp8_dense(), descales=bad) == E["ATTN_E_ARG"]
    n = lib.attn_fwd_fp8_workspace_bytes(R(fp8_dense()["k"]))
    assert n == -(-2 * 2 * 128 * 208 // 256) * 256                  # keys padded to 208
    assert call_fwd_fp8(lib, fp8_dense(), ws_bytes=n - 1) == E["ATTN_E_WORKSPACE"]
    assert call_fwd_fp8(lib, fp8_dense(), ws=FAKE + 16, ws_bytes=n) == E["ATTN_E_WORKSPACE"]


# ---------------------------------------------------------------- score recompute

def call_score(lib, t, score, l1, cu=None, max_seqlen=0, ws=FAKE, ws_bytes=1 << 40, flags=0):
    return lib.attn_score_recompute(R(t["q"]), R(t["k"]), R(t["lse"]), R(cu), max_seqlen, 0, 0.1,
                                    R(score), R(l1), ctypes.c_void_p(ws), ws_bytes, flags, None)


def test_score_recompute_contract(lib):
    """The score recompute takes attn_fwd's q, k and lse (PFCCLab PR #9,
    section 3) and writes fp32 [B,Sq,Sk] scores and [B,Sq] L1 norms; every
    malformed call is rejected before a launch."""
    t = dense()
    sc, l1 = desc([2, 100, 77], _lib.ATTN_F32), desc([2, 100], _lib.ATTN_F32)
    stop = (E["ATTN_E_DEVICE"], E["ATTN_E_CUDA"])
    assert call_score(lib, t, sc, l1) in stop                      # valid: stops at the device
    assert call_score(lib, t, sc, l1, flags=1) == E["ATTN_E_ARG"]
    assert call_score(lib, t, desc([2, 100, 77]), l1) == E["ATTN_E_DTYPE"]         # bf16 score
    assert call_score(lib, t, desc([2, 77, 100], _lib.ATTN_F32), l1) == E["ATTN_E_SHAPE"]
    assert call_score(lib, t, sc, desc([100, 2], _lib.ATTN_F32)) == E["ATTN_E_SHAPE"]
    t2 = dense()
    t2["lse"] = desc([2, 100, 4], _lib.ATTN_F32)                     # transposed lse
    assert call_score(lib, t2, sc, l1) == E["ATTN_E_SHAPE"]
    assert call_score(lib, dense(D=96), sc, l1) == E["ATTN_E_UNSUPPORTED"]
    strided = desc([2, 100, 77], _lib.ATTN_F32, stride=[100 * 80, 80, 1])
    assert call_score(lib, t, strided, l1) == E["ATTN_E_LAYOUT"]
    n = lib.attn_score_workspace_bytes(R(t["q"]), R(t["k"]), None, 0)
    assert n == -(-1 * 200 * 4 // 256) * 256                        # one key tile x 200 rows
    assert call_score(lib, t, sc, l1, ws_bytes=n - 1) == E["ATTN_E_WORKSPACE"]
    assert call_score(lib, t, sc, l1, ws=FAKE + 16, ws_bytes=n) == E["ATTN_E_WORKSPACE"]
    # varlen: score [T, max_seqlen], l1 [T]
    T = 300
    tv = dict(q=desc([T, 4, 64]), k=desc([T, 2, 64]), lse=desc([4, T], _lib.ATTN_F32))
    cu = desc([4], _lib.ATTN_I32)
    assert call_score(lib, tv, desc([T, 130], _lib.ATTN_F32), desc([T], _lib.ATTN_F32), cu=cu,
                      max_seqlen=130) in stop
    assert call_score(lib, tv, desc([T, 129], _lib.ATTN_F32), desc([T], _lib.ATTN_F32), cu=cu,
                      max_seqlen=130) == E["ATTN_E_SHAPE"]
    assert lib.attn_score_workspace_bytes(R(tv["q"]), R(tv["k"]), R(cu), 130) == \
        -(-2 * T * 4 // 256) * 256                                  # two key tiles


def test_poisoned_staging_variant_builds_and_exports_the_abi():
    """The race-check debug library (ATTN_POISON_SMEM) compiles for sm_103a
    from the same sources and exports the same C ABI."""
    path = build.build(variant="poison")
    assert path == build.POISON_LIB and os.path.exists(path)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True).stdout
    for name in declared_functions():
        assert re.search(r"\bT %s\b" % name, out), name
    with pytest.raises(ValueError):
        build.build(variant="nonexistent")


def test_checked_variant_builds_and_exports_the_abi_and_the_stall_hook():
    """The bounds-check / stall-injection debug library (ATTN_DEBUG_CHECKS)
    compiles from the same sources, exports the same C ABI plus
    attn_debug_inject_stall, which the product library does not export;
    the hook only sets a host-side value and validates its arguments."""
    path = build.build(variant="checked")
    assert path == build.CHECKED_LIB and os.path.exists(path)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True).stdout
    for name in declared_functions():
        assert re.search(r"\bT %s\b" % name, out), name
    assert re.search(r"\bT attn_debug_inject_stall\b", out)
    prod = subprocess.run(["nm", "-D", "--defined-only", build.build()], capture_output=True,
                          text=True).stdout
    assert not re.search(r"\battn_debug_inject_stall\b", prod)
    dbg = ctypes.CDLL(path)
    fn = dbg.attn_debug_inject_stall
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_int]
    assert fn(7, 0) == E["ATTN_E_ARG"]
    assert fn(1, -1) == E["ATTN_E_ARG"]
    assert fn(2, 70000) == E["ATTN_E_ARG"]
    assert fn(2, 3) == 0
    assert fn(0, 0) == 0


def test_use_library_swaps_and_restores(lib):
    """Calls inside `use_library` go through the named build; the previous
    library comes back afterwards, also when the block raises."""
    path = build.build(variant="poison")
    before = _lib.load()
    with _lib.use_library(path) as dbg:
        assert _lib.load() is dbg and dbg is not before
        assert dbg.attn_version() == before.attn_version()
    assert _lib.load() is before
    with pytest.raises(RuntimeError):
        with _lib.use_library(path):
            raise RuntimeError("inside")
    assert _lib.load() is before
    with pytest.raises(RuntimeError, match="not built"):
        with _lib.use_library(os.path.join(build.LIB_DIR, "missing.so")):
            pass
    assert _lib.load() is before


def sparse(B=2, S=100, Skv=300, H=64, D=576, K=128, sink=True, length=True):
    return dict(q=desc([B, S, H, D]), kv=desc([B, Skv, D]), out=desc([B, S, H, 512]),
                dout=desc([B, S, H, 512]), lse=desc([B, S, H], _lib.ATTN_F32),
                sink=desc([H], _lib.ATTN_F32) if sink else None,
                idx=desc([B, S, K], _lib.ATTN_I32),
                len=desc([B, S], _lib.ATTN_I32) if length else None,
                dq=desc([B, S, H, D]), dkv=desc([B, Skv, D]),
                dsink=desc([H], _lib.ATTN_F32) if sink else None)


def call_sparse(lib, t, scale=0.04, ws=FAKE, ws_bytes=1 << 40, flags=0):
    return lib.attn_sparse_bwd(R(t["q"]), R(t["kv"]), R(t["out"]), R(t["dout"]), R(t["lse"]),
                               R(t["sink"]), R(t["idx"]), R(t["len"]), scale, R(t["dq"]),
                               R(t["dkv"]), R(t["dsink"]), ctypes.c_void_p(ws), ws_bytes, flags,
                               None)


def test_sparse_bwd_contract(lib):
    """NVIDIA/cudnn-frontend PR #429: every companion tensor of the DSA
    backward is checked against q before launch (a transposed dout or lse, a
    mis-shaped index tensor, a wrong dtype, a strided out-parameter or an
    unsupported head dim fails instead of running)."""
    stop = (E["ATTN_E_DEVICE"], E["ATTN_E_CUDA"])
    assert call_sparse(lib, sparse()) in stop                          # valid: stops at the device
    assert call_sparse(lib, sparse(D=512, sink=False, length=False)) in stop
    assert call_sparse(lib, sparse(K=0)) in stop
    assert call_sparse(lib, sparse(), flags=1) == E["ATTN_E_ARG"]
    assert call_sparse(lib, sparse(), scale=float("nan")) == E["ATTN_E_ARG"]
    assert call_sparse(lib, sparse(H=32)) == E["ATTN_E_UNSUPPORTED"]
    assert call_sparse(lib, sparse(D=128)) == E["ATTN_E_UNSUPPORTED"]

    def bad(key, value, code):
        t = sparse()
        t[key] = value
        assert call_sparse(lib, t) == E[code], (key, code)

    bad("dout", desc([2, 100, 512, 64]), "ATTN_E_SHAPE")               # transposed dout
    bad("lse", desc([2, 64, 100], _lib.ATTN_F32), "ATTN_E_SHAPE")      # transposed lse
    bad("lse", desc([2, 100, 64]), "ATTN_E_DTYPE")                     # bf16 lse
    bad("kv", desc([2, 300, 512]), "ATTN_E_SHAPE")
    bad("kv", desc([1, 300, 576]), "ATTN_E_SHAPE")
    bad("out", desc([2, 100, 64, 512], _lib.ATTN_F16), "ATTN_E_DTYPE")
    bad("idx", desc([2, 99, 128], _lib.ATTN_I32), "ATTN_E_SHAPE")
    bad("idx", desc([2, 100, 128], _lib.ATTN_F32), "ATTN_E_DTYPE")
    bad("idx", desc([2, 100, 128], _lib.ATTN_I32, stride=[100 * 256, 256, 1]), "ATTN_E_LAYOUT")
    bad("len", desc([2, 101], _lib.ATTN_I32), "ATTN_E_SHAPE")
    bad("sink", desc([32], _lib.ATTN_F32), "ATTN_E_SHAPE")
    bad("sink", None, "ATTN_E_ARG")                                    # d_sink without a sink
    bad("dsink", None, "ATTN_E_ARG")                                   # a sink without d_sink
    bad("dq", desc([2, 100, 64, 576], stride=[100 * 64 * 640, 64 * 640, 640, 1]), "ATTN_E_LAYOUT")
    bad("dkv", desc([2, 300, 576], _lib.ATTN_F16), "ATTN_E_DTYPE")
    bad("q", desc([2, 100, 64, 576], _lib.ATTN_F32), "ATTN_E_DTYPE")
    bad("idx", None, "ATTN_E_ARG")
    t = sparse()
    n = lib.attn_sparse_bwd_workspace_bytes(R(t["q"]), R(t["kv"]), 1)
    vec = -(-2 * 100 * 64 * 4 // 256) * 256
    assert n == -(-2 * 300 * 576 * 4 // 256) * 256 + 2 * vec
    assert lib.attn_sparse_bwd_workspace_bytes(R(t["q"]), R(t["kv"]), 0) == n - vec
    assert call_sparse(lib, t, ws_bytes=n - 1) == E["ATTN_E_WORKSPACE"]
    assert call_sparse(lib, t, ws=FAKE + 16, ws_bytes=n) == E["ATTN_E_WORKSPACE"]
