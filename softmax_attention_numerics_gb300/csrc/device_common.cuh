// Device helpers shared by the attention kernels: sequence bounds, mask and
// predicate evaluation, exp2 / log2 and 16-bit packing.
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
    } else if (p.mask_kind == MASK_F16) {
        return __half2float(static_cast<const __half*>(p.mask)[off]) * kLog2e;
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

// Two floats -> one 32-bit word of two 16-bit elements (lo in the low half),
// round to nearest even: bf16, or fp16 when F16.
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (F16) {
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    } else {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    }
    return r;
}

// The two 16-bit elements of a packed word as floats (lo, hi).
template <bool F16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (F16) {
        const __half2 h = *reinterpret_cast<const __half2*>(&w);
        return __half22float2(h);
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
}

}  // namespace attn
