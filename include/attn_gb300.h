/*
 * attn_gb300.h - C ABI of the fused scaled-dot-product attention library
 * (forward and backward) for NVIDIA GB300 (sm_103a).
 *
 * The operation (the formula every source page assumes; see "Sources" below):
 *
 *   s_ij  = scale * q_i . k_j + mask_ij            (mask: additive, or a bool
 *                                                    mask with False = -inf;
 *                                                    causal hides j > i)
 *   out_i = sum_j softmax_j(s_i)_j v_j
 *   lse_i = log sum_j exp(s_ij)                      (natural log, fp32)
 *
 *   backward, given dO = d(loss)/d(out):
 *   Delta_i = sum_d dO_id out_id,  P = softmax(s),  dP = dO V^T,
 *   dS = P o (dP - Delta),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 *
 * Sources (the web pages this library follows):
 *   - flash-dmattn PR #122 "Fix NaN/Inf values in dV gradients", Problem and
 *     Root Cause: the causal B=1,H=1,S=256,D=64 bf16 call, and the rule that
 *     gradient accumulators must be zero-initialised (never empty_like).
 *   - ROCm/FlyDSL PR #1033 "Fix NaN from the lazy rescale on a wide score
 *     range", Root cause / The fix: the online softmax must take
 *     m_new = max(m_row, m_tile) before it rescales.
 *   - NVIDIA/cudnn-frontend PR #429 "Fix stream-ordering and input-validation
 *     holes in the SM100 DSA backward interface": every allocation and
 *     zero-fill goes on the launch stream; the dtype gate must match the
 *     kernel; companion tensors are checked against the shape contract; all
 *     inputs on one device; strided out-parameters are rejected.
 *   - PFCCLab/cudnn-frontend PR #9 "DSA: fix dK SMEM handoff race ...",
 *     sections 1-4: barrier-protected staging before a bulk store, rows the
 *     scheduler never visits are written (0, not -inf), the exp2 exponent is
 *     clamped, unsupported head_dim is rejected.
 *   - OpenWAM PR #64, Summary / Fix: the last partial key tile must be
 *     predicated in the backward too, or a row whose lse is below -88.7
 *     evaluates exp(0 - lse) = inf there.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *   Tensors are described by attn_tensor_t: a device pointer, an element type,
 *   a rank, a shape and strides counted in ELEMENTS.  The library never
 *   allocates and never frees; the caller owns every buffer.  All work
 *   (zero-fills included) is enqueued on the caller's `stream`; nothing runs
 *   on the legacy default stream, and the calls do not synchronise.
 *
 *   Layouts
 *     dense  : q, out, dout [B, Sq, Hq, D]; k, v [B, Sk, Hkv, D];
 *              lse [B, Hq, Sq] fp32; mask broadcastable to [B, Hq, Sq, Sk].
 *     varlen : q, out, dout [T, Hq, D]; k, v [T, Hkv, D]; lse [Hq, T];
 *              cu_seqlens int32 [nseq + 1] on the device, cu[0] = 0,
 *              non-decreasing, cu[nseq] <= T.  Sequence s owns rows
 *              [cu[s], cu[s+1]) of q, k and v (so Sq = Sk per sequence).
 *              Rows >= cu[nseq] belong to no sequence; the library writes
 *              them as out = 0, lse = 0, dq = dk = dv = 0.
 *   Inputs q, k, v, dout, out (as a backward input): bf16 or fp16 (all the
 *   same type; it also sets the type of out, dq, dk, dv), last-dim stride 1,
 *   every other stride a multiple of 8 elements (16 bytes), base 16-byte
 *   aligned.  Outputs out, lse, dq, dk, dv: contiguous in the layouts above,
 *   base 16-byte aligned (lse keeps that contract as a backward input).  A
 *   mask's base must be aligned to its element size, cu_seqlens to 4 bytes.
 *   Head dim D must be 64 or 128; Hq must be a multiple of Hkv (GQA).
 *   Causal masking is top-left aligned: key j is hidden from query i when
 *   j > i.  A query row with no visible key gets out = 0, lse = 0 and a zero
 *   dq row; keys that no query sees get zero dk and dv.
 *
 *   Inputs must be finite.  Values in rows outside a sequence (varlen) may be
 *   read by a partial tile and are multiplied by exact zeros.
 *
 *   Errors: every entry point returns ATTN_OK (0) or a negative ATTN_E_*
 *   code.  A validation failure launches nothing.  Faults found on the device
 *   (a malformed cu_seqlens, a bounded wait that ran out) are recorded in a
 *   per-device error word and the affected tiles are skipped; read and clear
 *   it with attn_get_error().
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st* attn_stream_t;

/* Element types. */
enum {
    ATTN_BF16 = 1,
    ATTN_F16 = 2,   /* IEEE half: computed like bf16 (fp32 accumulation) */
    ATTN_F32 = 3,
    ATTN_I32 = 4,
    ATTN_U8 = 5,    /* bool mask: nonzero = visible, 0 = hidden */
    ATTN_E4M3 = 6   /* fp8 E4M3 (finite-only, max 448): attn_fwd_fp8 inputs */
};

/* Return codes. */
enum {
    ATTN_OK = 0,
    ATTN_E_DTYPE = -1,        /* element type not supported for this argument */
    ATTN_E_SHAPE = -2,        /* shape breaks the contract derived from q      */
    ATTN_E_LAYOUT = -3,       /* stride / alignment / contiguity violation     */
    ATTN_E_DEVICE = -4,       /* tensors on different devices, or host memory  */
    ATTN_E_UNSUPPORTED = -5,  /* head dim, mask+varlen, ... not implemented    */
    ATTN_E_WORKSPACE = -6,    /* workspace missing, too small or misaligned    */
    ATTN_E_CUDA = -7,         /* a CUDA runtime call failed                    */
    ATTN_E_TIMEOUT = -8,      /* device: a bounded wait gave up                */
    ATTN_E_SEQLENS = -9,      /* device: cu_seqlens malformed / over max_seqlen*/
    ATTN_E_ARG = -10,         /* null pointer or non-finite scale              */
    ATTN_E_INTERNAL = -11,    /* device: an internal invariant failed          */
    ATTN_E_TOO_LARGE = -12    /* attn_bwd_noalloc: needs more scratch than the
                                 library's built-in array holds               */
};

/* Flags (bitwise OR). */
enum {
    ATTN_DETERMINISTIC = 1u,  /* backward: dQ by a separate kernel, no atomics;
                                 dq, dk, dv are bitwise reproducible */
    ATTN_EAGER_RESCALE = 2u   /* forward: rescale the running output on every
                                 new row max (disables the lazy threshold) */
};

typedef struct {
    void* data;          /* device pointer */
    int32_t dtype;       /* ATTN_BF16, ATTN_F16, ATTN_F32, ATTN_I32, ATTN_U8, ATTN_E4M3 */
    int32_t ndim;        /* 1 .. 4 */
    int64_t shape[4];
    int64_t stride[4];   /* in elements; 0 = broadcast (masks only) */
    int32_t device;      /* CUDA device ordinal, or -1 for host memory */
} attn_tensor_t;

/*
 * attn_fwd - forward pass: out and lse.
 *
 * Defined by the formula above.  Passages it follows: the online softmax
 * always takes m_new = max(m_row, m_tile) (ROCm/FlyDSL PR #1033, The fix);
 * the last partial key tile is predicated (OpenWAM PR #64, Root cause);
 * the exponent is clamped (PFCCLab/cudnn-frontend PR #9, section 3); varlen
 * rows outside every sequence are written as out = 0, lse = 0 (PFCCLab PR #9,
 * section 2); all work on the caller's stream (NVIDIA/cudnn-frontend PR #429,
 * first fix).
 *
 *   q, k, v     bf16 or fp16 inputs, all three the same type (dense
 *               [B,S,H,D] or varlen [T,H,D]); any other type or a mix gives
 *               ATTN_E_DTYPE before anything is launched.
 *   mask        NULL, or a dense-only mask broadcastable to [B,Hq,Sq,Sk]
 *               (rank 4, stride 0 on broadcast axes): ATTN_U8 (bool,
 *               0 = hidden), ATTN_F32, ATTN_BF16 or ATTN_F16 (additive,
 *               -inf = hidden).
 *               The mask is added after scaling.
 *   cu_seqlens  NULL for dense, else int32 [nseq+1] on the device (varlen).
 *   max_seqlen  varlen only: an upper bound on every sequence length (a
 *               longer sequence is skipped and flagged ATTN_E_SEQLENS; every
 *               sequence is checked, also when max_seqlen is 0).
 *   causal      nonzero = causal (top-left).
 *   scale       finite softmax scale (callers usually pass 1/sqrt(D)).
 *   out         q's element type, same shape as q, contiguous; fully written.
 *   lse         fp32 [B,Hq,Sq] (dense) or [Hq,T] (varlen), contiguous; fully
 *               written, natural log.
 *   flags       0 or ATTN_EAGER_RESCALE.
 *   stream      every launch and zero-fill is enqueued here.
 */
int attn_fwd(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
             const attn_tensor_t* mask, const attn_tensor_t* cu_seqlens, int32_t max_seqlen,
             int causal, float scale, attn_tensor_t* out, attn_tensor_t* lse,
             uint32_t flags, attn_stream_t stream);

/*
 * attn_fwd_fp8 - forward pass on fp8 inputs: out (bf16) and lse.
 *
 * Follows FlyDSL PR #1033 ("The fp8 helper, second commit"): the logits come
 * from fp8 operands and the probabilities enter the P.V product as fp8; the
 * result is still softmax(scale * q k^T) v of the real-valued inputs.
 *
 *   q, k, v     ATTN_E4M3 codes, dense [B,Sq,Hq,D] / [B,Sk,Hkv,D], D = 128;
 *               last-dim stride 1, other strides multiples of 16 elements,
 *               16-byte aligned bases.  Real value = decoded code * descale.
 *   descale_q, descale_k, descale_v   finite, > 0 (one per tensor).
 *   causal      nonzero = causal (top-left).  No mask, no varlen.
 *   scale       finite softmax scale applied to the real-valued q . k.
 *   out         ATTN_BF16 [B,Sq,Hq,D], contiguous; fully written.
 *   lse         fp32 [B,Hq,Sq], contiguous; natural log; fully written.
 *   workspace   device buffer of attn_fwd_fp8_workspace_bytes(k) bytes,
 *               256-byte aligned (holds V transposed to [B,Hkv,D,Sk']).
 *   flags       0 or ATTN_EAGER_RESCALE.
 */
int attn_fwd_fp8(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
                 float descale_q, float descale_k, float descale_v, int causal, float scale,
                 attn_tensor_t* out, attn_tensor_t* lse, void* workspace,
                 size_t workspace_bytes, uint32_t flags, attn_stream_t stream);

/* attn_fwd_fp8_workspace_bytes - workspace size attn_fwd_fp8 needs for k's
 * shape (0 if k is malformed). */
size_t attn_fwd_fp8_workspace_bytes(const attn_tensor_t* k);

/*
 * attn_bwd_workspace_bytes - size of the scratch buffer attn_bwd needs for
 * this q / k / flags combination (fp32 dQ accumulator and the per-row
 * Delta and log2-domain lse vectors).  Returns 0 if q or k is malformed.
 * The caller allocates it, on its own stream: NVIDIA/cudnn-frontend PR #429
 * (first fix) moves every scratch allocation and zero-fill onto the launch
 * stream, and flash-dmattn PR #122 (Root Cause 1) requires the accumulator to
 * start at zero, which attn_bwd does itself on `stream`.
 */
size_t attn_bwd_workspace_bytes(const attn_tensor_t* q, const attn_tensor_t* k, uint32_t flags);

/*
 * attn_bwd - backward pass: dq, dk, dv.
 *
 * Defined by the backward formulas above.  Passages it follows: the
 * probabilities are recomputed with the forward's predicates, the last
 * partial key tile included (OpenWAM PR #64, Root cause / Fix); the dK / dV
 * staging tile is handed to the bulk store behind a fence and a barrier
 * (PFCCLab/cudnn-frontend PR #9, section 1); accumulators start at zero
 * (flash-dmattn PR #122, Root Cause 1); the deterministic dQ path is
 * bitwise reproducible and the atomic one stays within the fp32
 * reassociation bound (PFCCLab PR #9, How it was verified); inputs are
 * validated against the shape and dtype contract before any launch
 * (NVIDIA/cudnn-frontend PR #429, the input-validation fixes).
 *
 *   q, k, v, out, dout, lse   as produced / consumed by attn_fwd with the
 *               same mask, cu_seqlens, max_seqlen, causal and scale.
 *   dq, dk, dv  q's element type, shapes of q, k, v, contiguous; fully written (the
 *               caller may pass uninitialised memory).
 *   workspace   device buffer of at least attn_bwd_workspace_bytes() bytes,
 *               256-byte aligned; contents on entry are ignored (it is
 *               zero-filled on `stream`) and are undefined on return.
 *   flags       0 or ATTN_DETERMINISTIC.
 */
int attn_bwd(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
             const attn_tensor_t* out, const attn_tensor_t* dout, const attn_tensor_t* lse,
             const attn_tensor_t* mask, const attn_tensor_t* cu_seqlens, int32_t max_seqlen,
             int causal, float scale, attn_tensor_t* dq, attn_tensor_t* dk, attn_tensor_t* dv,
             void* workspace, size_t workspace_bytes, uint32_t flags, attn_stream_t stream);

/*
 * attn_bwd_noalloc - attn_bwd for callers that cannot allocate device memory
 * when they run the backward (for example a plugin inside a framework that
 * owns all device memory and gives it no allocator, or a real-time caller
 * whose device-memory budget is fixed at start-up).  The source pages have no
 * counterpart: this is a convenience of this library.
 *
 * Same arguments as attn_bwd minus the workspace: the scratch is a 32 MiB
 * array compiled into the library, which every GPU that loads the library
 * keeps until the process exits.  Problems whose attn_bwd_workspace_bytes()
 * exceeds 32 MiB (about 64 K (query row, head) pairs at D = 128) are rejected
 * with ATTN_E_TOO_LARGE.  Nothing is allocated or freed by the call.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and may load the library's device code
 * there; this happens before the arguments are checked, so make the first
 * call of any kind, valid or not, before any stream capture.  The address is
 * kept for the life of the process: after cudaDeviceReset() on a device,
 * this entry point must not be used on that device again.
 * All calls on one device share the array: calls whose work overlaps on the
 * GPU (unordered streams) race on it; order them.  The part that must start
 * at zero is zero-filled on `stream` by every call.
 */
int attn_bwd_noalloc(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
                     const attn_tensor_t* out, const attn_tensor_t* dout, const attn_tensor_t* lse,
                     const attn_tensor_t* mask, const attn_tensor_t* cu_seqlens, int32_t max_seqlen,
                     int causal, float scale, attn_tensor_t* dq, attn_tensor_t* dk,
                     attn_tensor_t* dv, uint32_t flags, attn_stream_t stream);

/*
 * attn_score_recompute - attention targets recomputed from the forward's lse
 * and summed over the query heads, with each row's L1 norm.
 *
 * Follows PFCCLab/cudnn-frontend PR #9, section 3 (the dense score recompute
 * behind a sparse-attention indexer's training targets) and section 2 (rows
 * no tile visits are written as 0, not -inf):
 *
 *   score_ij = sum_h exp2(min(log2(e) (scale q_hi . k_j - lse_hi), 120))
 *   l1_i     = sum_j score_ij          (the consumer's target: score / l1)
 *
 * The clamp bounds each term by 2^120 so that the sum over heads stays
 * finite when an lse is far too small; with the forward's own lse it never
 * fires and l1_i is the number of heads.  Hidden pairs (causal j > i) add 0.
 *
 *   q, k        as for attn_fwd (bf16 or fp16, D = 64 or 128, GQA allowed);
 *               no mask.
 *   lse         fp32, as attn_fwd wrote it: [B,Hq,Sq] or [Hq,T].
 *   cu_seqlens, max_seqlen, causal, scale   as for attn_fwd.
 *   score       fp32, contiguous: dense [B,Sq,Sk]; varlen [T,max_seqlen], row
 *               cu[s] + i holding sequence s's keys in columns 0..len-1 and 0
 *               past them; rows >= cu[nseq] are 0.  Fully written.
 *   l1          fp32, contiguous: dense [B,Sq]; varlen [T].  Fully written.
 *   workspace   attn_score_workspace_bytes() bytes, 256-byte aligned (per
 *               key-tile partial sums, added in a fixed order so that both
 *               outputs are bit-reproducible).
 *   flags       0.
 */
int attn_score_recompute(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* lse,
                         const attn_tensor_t* cu_seqlens, int32_t max_seqlen, int causal,
                         float scale, attn_tensor_t* score, attn_tensor_t* l1, void* workspace,
                         size_t workspace_bytes, uint32_t flags, attn_stream_t stream);

/* attn_score_workspace_bytes - workspace attn_score_recompute needs (0 if q or
 * k is malformed). */
size_t attn_score_workspace_bytes(const attn_tensor_t* q, const attn_tensor_t* k,
                                  const attn_tensor_t* cu_seqlens, int32_t max_seqlen);

/*
 * attn_sparse_bwd - backward of sparse top-k attention with an attention sink
 * (the DSA backward).  NVIDIA/cudnn-frontend PR #429 fixes the interface
 * (inputs q, kv, out, dout, lse, attn_sink, topk_idxs, optional topk_length;
 * outputs dq, dkv, d_sink; head dim 512, or 576 in the MLA form whose values
 * are the first 512 columns of the kv rows), the shape contract checked
 * against q before launch, the zero-fills on the launch stream and a real
 * fp16 path.  The page prints no formula; the library computes, for token i
 * of batch b and its listed kv rows k_e (v_e = k_e[:512]):
 *
 *   P_he = exp(scale q_h . k_e - lse_h),   Delta_h = dout_h . out_h,
 *   dS_he = P_he (dout_h . v_e - Delta_h),
 *   dq_h = scale sum_e dS_he k_e,
 *   dkv[b, idx_e] += scale sum_h dS_he q_h  (+ sum_h P_he dout_h on the
 *                                             first 512 columns),
 *   d_sink[h] = - sum over all tokens of exp(attn_sink[h] - lse_h) Delta_h.
 *
 *   q            [B, S, H, Dqk] bf16 or fp16, H = 64, Dqk = 512 or 576
 *   kv           [B, S_kv, Dqk] q's type: one row set shared by the heads
 *   out, dout    [B, S, H, 512] q's type (out: the forward's output)
 *   lse          [B, S, H] fp32, contiguous: log of each (token, head)'s
 *                softmax normaliser, exp(attn_sink[h]) included (natural log)
 *   attn_sink    [H] fp32 contiguous, or NULL (no sink)
 *   topk_idxs    [B, S, K] int32 contiguous, K >= 0: kv rows of each token.
 *                Entry e takes part when e < topk_length[b, i] and
 *                0 <= idx < S_kv; other entries (e.g. -1 padding) are
 *                ignored.  Repeated rows count once per entry.
 *   topk_length  [B, S] int32 contiguous, or NULL (all K entries)
 *   scale        finite
 *   dq, dkv      q's / kv's shape and type, contiguous; written (not
 *                accumulated into).  A token with no valid entry gets dq = 0.
 *   d_sink       [H] fp32, written; given exactly when attn_sink is
 *   workspace    attn_sparse_bwd_workspace_bytes(q, kv, attn_sink != NULL)
 *                bytes, 256-byte aligned (fp32 dkv accumulator, Delta and the
 *                sink terms)
 *   flags        0
 * dq and d_sink are bitwise reproducible; dkv is the 16-bit rounding of fp32
 * sums whose order varies from run to run.  Returns ATTN_E_UNSUPPORTED for
 * H != 64 or Dqk not in {512, 576}, ATTN_E_SHAPE / ATTN_E_DTYPE /
 * ATTN_E_LAYOUT / ATTN_E_DEVICE for any tensor off the contract, ATTN_E_ARG
 * for a missing tensor, a non-finite scale, nonzero flags or a sink without
 * d_sink (or the reverse).
 */
int attn_sparse_bwd(const attn_tensor_t* q, const attn_tensor_t* kv, const attn_tensor_t* out,
                    const attn_tensor_t* dout, const attn_tensor_t* lse,
                    const attn_tensor_t* attn_sink, const attn_tensor_t* topk_idxs,
                    const attn_tensor_t* topk_length, float scale, attn_tensor_t* dq,
                    attn_tensor_t* dkv, attn_tensor_t* d_sink, void* workspace,
                    size_t workspace_bytes, uint32_t flags, attn_stream_t stream);

/* attn_sparse_bwd_workspace_bytes - workspace attn_sparse_bwd needs (0 if q
 * or kv break the contract); with_sink: nonzero when attn_sink is given. */
size_t attn_sparse_bwd_workspace_bytes(const attn_tensor_t* q, const attn_tensor_t* kv,
                                       int with_sink);

/*
 * attn_get_error - synchronises `stream`, then returns and clears the error
 * word of the current device: ATTN_OK, ATTN_E_SEQLENS, ATTN_E_TIMEOUT or
 * ATTN_E_INTERNAL
 * (ATTN_E_CUDA if the synchronisation itself failed).  Device-side faults are
 * reported rather than hidden, following NVIDIA/cudnn-frontend PR #429
 * (a clear error instead of silently wrong gradients) and PFCCLab PR #9
 * (bounded waits instead of a hang).
 */
int attn_get_error(attn_stream_t stream);

/* attn_strerror - static, human-readable text for a return code (the error
 * texts NVIDIA/cudnn-frontend PR #429 asks for: say which contract failed). */
const char* attn_strerror(int code);

/* attn_last_cuda_error - the CUDA runtime error behind the last ATTN_E_CUDA
 * returned to this thread ("" if none): which step failed, the error name and
 * its text.  The string is owned by the library (thread-local storage). */
const char* attn_last_cuda_error(void);

/* attn_version - library version as major * 10000 + minor * 100 + patch. */
int attn_version(void);

/*
 * attn_selftest_wait_timeout - exercises the failure path of the bounded
 * device waits on the current device: one thread waits on a device barrier
 * that nothing will ever complete, gives up after `budget_us` microseconds
 * (1 .. 1,000,000) of global time and sets the error word, so that a
 * following attn_get_error(stream) returns ATTN_E_TIMEOUT.  The same wait
 * loop bounds every wait in the attention kernels (there with a 2 s budget).
 * Nothing hangs and the CUDA context stays usable.  Returns ATTN_OK once the
 * probe is launched on `stream`, ATTN_E_ARG for a budget out of range.
 */
int attn_selftest_wait_timeout(uint32_t budget_us, attn_stream_t stream);

/*
 * Debug builds (not part of this ABI).  The build script makes two debug
 * variants of the library from the same sources.  In the poisoned-staging
 * build every writer of a backward staging tile first stores NaN into it,
 * so a consumer that reads the tile too early yields NaN gradients.  The
 * checked build adds per-tile bounds checks that record ATTN_E_INTERNAL and
 * skip the access instead of trapping, and exports one more function,
 * int attn_debug_inject_stall(int kernel, int iteration): from then on the
 * MMA issuer of block (0, 0, 0) of `kernel` (1 forward, 2 backward main,
 * 3 deterministic dQ, 4 fp8 forward, 5 score recompute, 6 sparse backward, whose
 * loop runs over work items) lets its wait at loop iteration
 * `iteration` (0 .. 65535) run out after 200 us, so that the kernel unwinds
 * and reports ATTN_E_TIMEOUT; kernel <= 0 turns it off; ATTN_E_ARG for
 * arguments out of range.
 */

/*
 * Profiling hooks (used by the benchmark; no effect on results).
 *
 * attn_profile_events - from now on, record the CUDA events `before` and
 * `after` (cudaEvent_t handles created by the caller, or NULL to stop) on the
 * launch stream immediately around the kernel of `stage`.  Process-wide
 * setting; not thread-safe against concurrent attn_fwd / attn_bwd calls.
 * Returns ATTN_E_ARG for an unknown stage.
 */
enum {
    ATTN_STAGE_FWD = 0,            /* forward kernel                        */
    ATTN_STAGE_BWD_PREPROCESS = 1, /* Delta = rowsum(dO o out), lse2         */
    ATTN_STAGE_BWD_MAIN = 2,       /* dK, dV (and atomic dQ partials)        */
    ATTN_STAGE_BWD_DQ = 3,         /* dQ convert, or the deterministic dQ    */
    ATTN_STAGE_SCORE = 4,          /* score recompute (then its L1 reduce)   */
    ATTN_STAGE_SPARSE = 5,         /* sparse top-k backward main kernel      */
    ATTN_STAGE_COUNT = 6
};
int attn_profile_events(int stage, void* before, void* after);

/* attn_launch_count - number of kernels this library has launched in this
 * process (all devices), for launch accounting. */
unsigned long long attn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
