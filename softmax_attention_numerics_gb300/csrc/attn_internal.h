// Internal problem description shared by the host entry points and the
// kernels.  Not part of the public ABI (include/attn_gb300.h is).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

// 16-bit element storage.  The pointers below are typed bf16 for both
// element types; `f16` says how the bits are read (bf16 or IEEE fp16).
typedef __nv_bfloat16 bf16;

enum MaskKind { MASK_NONE = 0, MASK_BOOL = 1, MASK_F32 = 2, MASK_BF16 = 3, MASK_F16 = 4 };

// Every stride is in elements.  Row addressing for a (batch b, head h, row i
// of that batch/sequence) is  ptr + b * x_b + (row0(b) + i) * x_s + h * x_h,
// where row0(b) = cu[b] for varlen (and x_b = 0) or 0 for dense.
struct Problem {
    const bf16* q;
    const bf16* k;
    const bf16* v;
    const bf16* o;      // forward output, read by the backward
    const bf16* dout;
    bf16* out;
    float* lse;
    bf16* dq;
    bf16* dk;
    bf16* dv;
    float* dq_acc;      // workspace: fp32 [rows, Hq, D]
    float* delta;       // workspace: fp32, indexed like lse
    float* lse2;        // workspace: lse * log2(e), indexed like lse

    int64_t q_b, q_s, q_h;
    int64_t k_b, k_s, k_h;
    int64_t v_b, v_s, v_h;
    int64_t o_b, o_s, o_h;
    int64_t do_b, do_s, do_h;
    int64_t out_b, out_s, out_h;   // out and dq (contiguous like q)
    int64_t dk_b, dk_s, dk_h;      // dk and dv (contiguous like k)
    int64_t lse_b, lse_h;          // lse / delta / lse2: b*lse_b + h*lse_h + row0 + i
    int64_t acc_b;                 // dq_acc row of (b, i): b*acc_b + row0 + i

    int B;          // batches (dense) or sequences (varlen)
    int Hq, Hkv, G; // G = Hq / Hkv
    int Sq, Sk;     // dense lengths; varlen: max_seqlen for both
    int D;
    int f16;        // 1: q, k, v, out, dout, dq, dk, dv hold fp16; 0: bf16
    int varlen;
    const int* cu;  // varlen: int32 [B + 1]
    int T;          // varlen: total rows of q/k/v

    const void* mask;
    int mask_kind;
    int64_t m_b, m_h, m_q, m_k;

    int causal;
    float scale;
    float scale_log2;   // scale * log2(e)
    int lazy;           // 1: lazy rescale with threshold 8 (log2 units)
    int* err;           // device error word
    int debug_stall;    // debug builds: (kernel << 16 | iteration) whose wait runs out; -1 none

    // score recompute: score [rows, sc_w] fp32 (rows = B*Sq dense, T varlen),
    // l1 [rows], l1_part [key tiles][l1_rows] workspace
    float* score;
    float* l1;
    float* l1_part;
    int64_t sc_w;
    int64_t l1_rows;
};

// Error codes written to the device error word (match include/attn_gb300.h).
constexpr int DEV_E_TIMEOUT = -8;
constexpr int DEV_E_SEQLENS = -9;
constexpr int DEV_E_INTERNAL = -11;

// Debug builds: the stall point set by attn_debug_inject_stall (-1: none).
int debug_stall_point();

// TMA tensor map over a 16-bit (bf16, or fp16 when f16) [B, S, H, D] view
// (dims innermost first: D, H, S, B; strides in elements), box 64 x 1 x 128 x 1,
// 128-byte swizzle.  Rows past S read as zero and are clipped on store.
bool make_tile_map(CUtensorMap* m, const void* base, int64_t D, int64_t H, int64_t S, int64_t B,
                   int64_t sh, int64_t ss, int64_t sb, bool f16);

// TMA tensor map over a 16-bit [B, S, H, D] view with box 64 x 64 x 1 x 1
// (64 columns of 64 heads of one token), 128-byte swizzle; H >= 64.
bool make_heads_map(CUtensorMap* m, const void* base, int64_t D, int64_t H, int64_t S, int64_t B,
                    int64_t sh, int64_t ss, int64_t sb, bool f16);

// TMA tensor map over the fp32 dQ workspace [R, H, D] (dims D, H, R), box
// 32 x 1 x 128, 128-byte swizzle; the target of bulk reduce-adds.
bool make_f32_reduce_map(CUtensorMap* m, void* base, int64_t D, int64_t H, int64_t R);

// fp8 forward: E4M3 q [B,Sq,Hq,D], k [B,Sk,Hkv,D] and V transposed into the
// workspace as vt [B,Hkv,D,Sk_pad] (Sk_pad = Sk rounded up to 16), one
// descale factor per tensor; D = 128; out bf16 and lse fp32 contiguous.
struct Fp8Problem {
    const uint8_t* q;
    const uint8_t* k;
    const uint8_t* v;
    uint8_t* vt;
    int64_t q_b, q_s, q_h;      // elements (= bytes)
    int64_t k_b, k_s, k_h;
    int64_t v_b, v_s, v_h;
    int64_t vt_b, vt_h;         // vt: b * vt_b + hk * vt_h + d * Sk_pad + key
    bf16* out;
    float* lse;
    int64_t out_b, out_s, out_h;
    int64_t lse_b, lse_h;
    int B, Hq, Hkv, G, Sq, Sk, Sk_pad;
    int causal;
    int lazy;
    float scale_log2;           // scale * descale_q * descale_k * log2(e)
    float out_scale;            // descale_v
    int* err;
    int debug_stall;            // as in Problem
};

// TMA tensor map over a 4-D uint8 view (dims innermost first, strides in
// bytes), box {128, box1, box2, 1}, 128-byte swizzle.
bool make_u8_map(CUtensorMap* m, const void* base, const int64_t dims[4], const int64_t strides[3],
                 int box1, int box2);

// Sparse top-k (DSA) backward: q [B,S,H,Dqk], kv [B,Skv,Dqk] (one row set
// shared by the H query heads; values are its first Dv = 512 columns), out /
// dout [B,S,H,Dv], lse [B,S,H] fp32 (natural log, the sink included),
// topk_idxs int32 [B,S,K], optional topk_length int32 [B,S], optional sink
// fp32 [H].  H = 64, Dqk = 512 or 576.  Strides in elements.
struct SparseProblem {
    const bf16* q;
    const bf16* kv;
    const bf16* out;
    const bf16* dout;
    const float* lse;        // contiguous [B, S, H]
    const float* sink;       // [H] or null
    const int* idx;
    const int* len;          // [B, S] or null
    bf16* dq;                // contiguous like q
    bf16* dkv;               // contiguous like kv
    float* dsink;            // [H] (when sink)
    float* dkv_acc;          // workspace: fp32 [B * Skv, Dqk]
    float* delta;            // workspace: fp32 [B * S, H]
    float* dsink_part;       // workspace: fp32 [B * S, H] (when sink)
    int64_t q_b, q_s, q_h;
    int64_t kv_b, kv_s;
    int64_t o_b, o_s, o_h;
    int64_t do_b, do_s, do_h;
    int64_t idx_b, idx_s;    // topk_idxs: b * idx_b + i * idx_s + e
    int64_t len_b, len_s;    // topk_length: b * len_b + i * len_s
    int B, S, Skv, H, Dqk, Dv, K;
    int f16;
    float scale;
    float scale_log2;        // scale * log2(e)
    int* err;
    int debug_stall;
};

// Launchers (each enqueues on `stream`, returns cudaGetLastError()).
cudaError_t launch_fwd(const Problem& p, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const Problem& p, cudaStream_t stream);
cudaError_t launch_bwd_main(const Problem& p, bool with_dq_atomics, cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(const Problem& p, cudaStream_t stream);
cudaError_t launch_bwd_dq_deterministic(const Problem& p, cudaStream_t stream);
cudaError_t launch_zero_trailing_fwd(const Problem& p, cudaStream_t stream);
cudaError_t launch_score_recompute(const Problem& p, cudaStream_t stream);
// Sparse backward stages: Delta (and the sink terms), the main kernel, the
// dkv conversion, the ordered d_sink sum.
cudaError_t launch_sparse_prep(const SparseProblem& p, cudaStream_t stream);
cudaError_t launch_sparse_bwd_main(const SparseProblem& p, cudaStream_t stream);
cudaError_t launch_sparse_dkv_convert(const SparseProblem& p, cudaStream_t stream);
cudaError_t launch_sparse_dsink(const SparseProblem& p, cudaStream_t stream);
int score_key_tiles(int64_t width);
cudaError_t launch_zero_trailing_bwd(const Problem& p, cudaStream_t stream);
cudaError_t launch_fp8_transpose_v(const Fp8Problem& p, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const Fp8Problem& p, cudaStream_t stream);
// One CTA whose thread 0 waits, bounded by budget_ns, on an mbarrier that no
// one arrives on, and then reports DEV_E_TIMEOUT through `err`.
cudaError_t launch_wait_timeout_probe(int* err, uint64_t budget_ns, cudaStream_t stream);

}  // namespace attn
