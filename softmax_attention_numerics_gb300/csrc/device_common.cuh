// Device helpers shared by the attention kernels: sequence bounds, mask and
// predicate evaluation, shared-memory swizzle, and thin PTX wrappers.
#pragma once

#include <math.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy-rescale threshold and forward exponent clamp, in log2 units of the
// scaled logits (FlyDSL PR #1033, Root cause: the threshold of 8).
constexpr float kLazyTau = 8.0f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Hardware base-2 exponential (MUFU); -inf -> +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void set_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Bounds of batch / sequence b.  For varlen, a malformed cu_seqlens entry
// (decreasing, past T, or longer than max_seqlen) flags ATTN_E_SEQLENS and
// the sequence is skipped.
struct SeqInfo {
    int row0;
    int len_q;
    int len_k;
    bool ok;
};

__device__ __forceinline__ SeqInfo seq_info(const Problem& p, int b) {
    SeqInfo s;
    if (!p.varlen) {
        s.row0 = 0;
        s.len_q = p.Sq;
        s.len_k = p.Sk;
        s.ok = true;
        return s;
    }
    const int a = __ldg(p.cu + b);
    const int e = __ldg(p.cu + b + 1);
    s.ok = (a >= 0) && (e >= a) && (e <= p.T) && (e - a <= p.Sq);
    s.row0 = s.ok ? a : 0;
    s.len_q = s.ok ? e - a : 0;
    s.len_k = s.len_q;
    if (!s.ok && threadIdx.x == 0) set_error(p.err, DEV_E_SEQLENS);
    return s;
}

// Mask contribution in log2 units for (b, h, i, j): 0 / -inf for a bool
// mask, value * log2(e) for an additive one.  Caller guarantees i < Sq and
// j < Sk (the mask is dense-only).
__device__ __forceinline__ float mask_log2(const Problem& p, int b, int h, int i, int j) {
    const int64_t off = b * p.m_b + h * p.m_h + static_cast<int64_t>(i) * p.m_q +
                        static_cast<int64_t>(j) * p.m_k;
    if (p.mask_kind == MASK_BOOL) {
        return static_cast<const uint8_t*>(p.mask)[off] ? 0.0f : -INFINITY;
    } else if (p.mask_kind == MASK_F32) {
        return static_cast<const float*>(p.mask)[off] * kLog2e;
    } else {
        return __bfloat162float(static_cast<const bf16*>(p.mask)[off]) * kLog2e;
    }
}

// Scaled logit in log2 units with every predicate applied: keys past the
// sequence (the partial last key tile), query rows past the sequence,
// causal j > i, and the user's mask.  Hidden -> -inf.
__device__ __forceinline__ float logit_log2(const Problem& p, float acc, int b, int h, int i,
                                            int j, int len_q, int len_k) {
    const bool vis = (j < len_k) && (i < len_q) && (!p.causal || j <= i);
    if (!vis) return -INFINITY;
    float x = acc * p.scale_log2;
    if (p.mask_kind != MASK_NONE) x += mask_log2(p, b, h, i, j);
    return x;
}

// ---------------------------------------------------------------- cp.async

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool pred) {
    const int sz = pred ? 16 : 0;   // 0 bytes read -> 16 zero bytes written
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Element offset of 16-byte chunk c of row r in a [rows][D] bf16 tile whose
// chunks are XOR-swizzled by (r mod 8) (conflict-free ldmatrix).
template <int D>
__device__ __forceinline__ int swz(int r, int c) {
    return r * D + ((c ^ (r & 7)) << 3);
}

// Copy rows [0, R) of a bf16 [*, D] matrix (row stride `rs` elements) into a
// swizzled shared tile; rows >= rows_valid are zero-filled (never read).
template <int R, int D, int NT>
__device__ __forceinline__ void load_tile(bf16* s, const bf16* g, int64_t rs, int rows_valid,
                                          const bf16* safe, int tid) {
    constexpr int CH = D / 8;
#pragma unroll
    for (int idx = tid; idx < R * CH; idx += NT) {
        const int r = idx / CH, c = idx % CH;
        const bool ok = r < rows_valid;
        const bf16* src = ok ? g + static_cast<int64_t>(r) * rs + c * 8 : safe;
        cp_async_16(smem_u32(s + swz<D>(r, c)), src, ok);
    }
}

// ---------------------------------------------------------------- mma.sync

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_round(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

}  // namespace attn
