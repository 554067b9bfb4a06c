// Attention forward for sm_103a: TMA + tcgen05 (UMMA) + TMEM, warp-specialised.
//
// One CTA = two 128-row query tiles (256 rows) of one (batch/sequence, q head).
//   warps 0-3   softmax for query tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for query tile 1
//   warp  8     TMA producer: Q tiles once, then K_j, V_j through a ring
//   warp  9     TMEM allocator and single-thread UMMA issuer
// TMEM (512 columns): S0 | S1 (128 fp32 columns each; the 16-bit P of a tile,
// bf16 or fp16 like the inputs, is written over the first 64 columns of its S)
// | O0 | O1 (D columns each).
//
// Per key tile j the issuer runs, for t = 0, 1:
//     O_t += P_t(j) V_j      (P from TMEM, V from shared memory)
//     S_t  = Q_t K_{j+1}^T   (after O_t's MMA has completed: P_t(j) and
//                             S_t(j+1) share TMEM columns)
// so the softmax of one query tile overlaps the MMAs of the other.
//
// Softmax (one thread per row, exp2 domain): x = s*scale*log2e (+ mask, with
// the predicates for the partial last key tile, causal pairs and rows past
// the sequence), m_tile = max_j x, and ALWAYS m_new = max(m_ref, m_tile)
// (FlyDSL PR #1033, The fix).  The lazy rule keeps the old reference max
// while m_tile - m_ref <= 8 and otherwise rescales O_t and l by
// exp2(m_ref - m_new) in TMEM; rows of the same warp that did not ask for a
// rescale use a factor of exactly 1.  p = exp2(min(x - m_ref, 8)): the clamp
// never fires on correct statistics (PFCCLab/cudnn-frontend PR #9, section 3).
// Epilogue: out = O/lr (lr = sum of the 16-bit-rounded p that entered the MMA),
// lse = (m_ref + log2 l) ln 2 (l = sum of the exact p); l = 0 gives out = 0,
// lse = 0.  Rows past the sequence are never stored (varlen neighbours).
#include "sm100_ptx.cuh"

namespace attn {
namespace {

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// max(a, b, c) in one instruction (the three-input form of sm_100).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

using namespace sm100;

constexpr int kFwdThreads = 320;
constexpr int kTile = 128;

template <int D>
struct FwdLayout {
    static constexpr int kBlocks = D / 64;                  // 128-byte column blocks
    static constexpr int kTileBytes = kTile * D * 2;        // one 128-row bf16 tile
    static constexpr int kStages = (D == 128) ? 4 : 6;      // K/V ring depth
    static constexpr int kQ = 0;                            // Q0, Q1
    static constexpr int kKV = 2 * kTileBytes;
    // D = 64: O gets 16 more columns from a 128-row block of ones appended to
    // V in the P V product, so O's column 64 is the sum of the rounded p (the
    // softmax then does not add them up itself).  TMEM has room for it there.
    static constexpr bool kOnesCol = (D == 64);
    static constexpr int kOnes = kKV + kStages * kTileBytes;   // one 128 x 64 swizzled atom of ones
    static constexpr int kBar = kOnes + (kOnesCol ? 16384 : 0);
    // barrier slots (8 bytes each)
    static constexpr int kBarQ = 0;
    static constexpr int kBarKVFull = 1;
    static constexpr int kBarKVEmpty = kBarKVFull + kStages;
    static constexpr int kBarSFull = kBarKVEmpty + kStages;   // [2]
    static constexpr int kBarPFull = kBarSFull + 2;           // [2]
    static constexpr int kBarPVDone = kBarPFull + 2;          // [2]
    static constexpr int kBarDrain = kBarPVDone + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;         // tmem base, abort flag
    static constexpr int kBytes = kMisc + 16 + 1024;          // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    static constexpr int kNO = kOnesCol ? D + 16 : D;         // N of the P V product
    static constexpr int kOStride = kOnesCol ? D + 32 : D;    // O columns, 32-aligned
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + kOStride;
    static_assert(kColO1 + kOStride <= kTmemCols, "TMEM columns");
};

struct FwdMaps {
    CUtensorMap q, k, v;
};

template <int D, bool F16>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_sm100_kernel(const Problem p, const __grid_constant__ FwdMaps maps) {
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::kBar + 8u * i; };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int m0 = (gridDim.x - 1 - blockIdx.x) * 2 * kTile;   // heaviest (causal) CTAs first
    const SeqInfo si = seq_info(p, b);
    if (!si.ok || m0 >= si.len_q) return;
    const int hk = h / p.G;

    // Key tiles per query tile (causal: up to the diagonal); 0 for an empty tile.
    int n_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int r0 = m0 + t * kTile;
        int kend = si.len_k;
        if (p.causal) kend = min(kend, r0 + kTile);
        n_t[t] = (r0 < si.len_q) ? (kend + kTile - 1) / kTile : 0;
    }
    const int n_all = max(n_t[0], n_t[1]);

    if constexpr (L::kOnesCol) {
        // the block of ones (bf16 0x3f80 or fp16 0x3c00 in every element)
        const uint32_t one2 = F16 ? 0x3c003c00u : 0x3f803f80u;
        uint4* ones = reinterpret_cast<uint4*>(smem + L::kOnes);
        for (int k = tid; k < 16384 / 16; k += kFwdThreads) ones[k] = make_uint4(one2, one2, one2, one2);
        fence_proxy_async_smem();              // generic stores -> tensor core reads
    }
    if (tid == 0) {
        for (int i = 0; i < L::kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == L::kBarPFull || i == L::kBarPFull + 1) cnt = kTile;
            mbar_init(bar(i), cnt);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const int row_base = si.row0;      // sequence start in the packed row dimension
    const int bcoord = p.varlen ? 0 : b;

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(&maps.v);
            mbar_arrive_expect_tx(bar(L::kBarQ), 2 * L::kTileBytes);
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int c = 0; c < L::kBlocks; ++c)
                    tma_load_4d(sbase + L::kQ + t * L::kTileBytes + c * 16384, &maps.q, 64 * c, h,
                                row_base + m0 + t * kTile, bcoord, bar(L::kBarQ));
            int issued = 0;
            for (int j = 0; j < n_all && !*abort_flag; ++j) {
                for (int which = 0; which < 2; ++which) {
                    const int li = 2 * j + which;
                    const int s = li % L::kStages, r = li / L::kStages;
                    if (!mbar_wait(bar(L::kBarKVEmpty + s), (r & 1) ^ 1, abort_flag)) break;
                    // every key tile starts inside the sequence (debug builds check it)
                    if (!dbg_check(j * kTile < si.len_k && s < L::kStages, p.err)) break;
                    mbar_arrive_expect_tx(bar(L::kBarKVFull + s), L::kTileBytes);
                    const CUtensorMap* m = which ? &maps.v : &maps.k;
#pragma unroll
                    for (int c = 0; c < L::kBlocks; ++c)
                        tma_load_4d(sbase + L::kKV + s * L::kTileBytes + c * 16384, m, 64 * c, hk,
                                    row_base + j * kTile, bcoord, bar(L::kBarKVFull + s));
                    issued = li + 1;
                }
            }
            if (*abort_flag) {
                // Let the copies in flight (the Q tiles too) land before the CTA exits.
                volatile int no_abort = 0;
                mbar_wait(bar(L::kBarQ), 0, &no_abort, kDrainBudgetNs);
                for (int li = max(0, issued - L::kStages); li < issued; ++li) {
                    const int s = li % L::kStages, r = li / L::kStages;
                    mbar_wait(bar(L::kBarKVFull + s), r & 1, &no_abort, kDrainBudgetNs);
                }
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16kind(128, 128, 0, 0, F16);
            constexpr uint32_t idesc_pv = idesc_f16kind(128, L::kNO, 0, 1, F16);
            const uint32_t colS[2] = {L::kColS0, L::kColS1};
            const uint32_t colO[2] = {L::kColO0, L::kColO1};
            auto kv_stage = [&](int li) { return li % L::kStages; };
            auto kv_par = [&](int li) { return (uint32_t)((li / L::kStages) & 1); };
            // TMEM columns of every accumulator stay inside the allocation
            dbg_check(L::kColS1 + kTile <= L::kTmemCols && L::kColO1 + D <= L::kTmemCols, p.err);
            auto issue_qk = [&](int t, int j) {
                const int s = kv_stage(2 * j);
                const uint64_t qd = smem_desc(sbase + L::kQ + t * L::kTileBytes, 16, 1024, kSwizzle128B);
                const uint64_t kd = smem_desc(sbase + L::kKV + s * L::kTileBytes, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(tmem + colS[t], desc_add(qd, off), desc_add(kd, off), idesc_qk, kk > 0);
                }
            };
            auto issue_pv = [&](int t, int j) {
                const int s = kv_stage(2 * j + 1);
                const uint32_t va = sbase + L::kKV + s * L::kTileBytes;
                // MN-major V: with the ones block, its 64-column atom at LBO after V's
                const uint32_t lbo = L::kOnesCol ? static_cast<uint32_t>(L::kOnes - (L::kKV + s * L::kTileBytes))
                                                 : 16384u;
                const uint64_t vd = smem_desc(va, lbo, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    mma_ts(tmem + colO[t], tmem + colS[t] + kk * 8, desc_add(vd, kk * 2048), idesc_pv,
                           (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = mbar_wait(bar(L::kBarQ), 0, abort_flag);
            if (ok && n_all > 0) {
                ok = mbar_wait(bar(L::kBarKVFull + kv_stage(0)), kv_par(0), abort_flag);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t) {
                        if (n_t[t] > 0) {
                            issue_qk(t, 0);
                            mma_commit(bar(L::kBarSFull + t));
                        }
                    }
                    mma_commit(bar(L::kBarKVEmpty + kv_stage(0)));
                }
            }
            for (int j = 0; ok && j < n_all; ++j) {
                if (!(ok = dbg_stall(p.debug_stall, kStallFwd, j, bar(L::kBarDrain), abort_flag))) break;
                const int lv = 2 * j + 1, lk = 2 * j + 2;
                if (!(ok = mbar_wait(bar(L::kBarKVFull + kv_stage(lv)), kv_par(lv), abort_flag)))
                    break;
                const bool next = j + 1 < n_all;
                if (next && !(ok = mbar_wait(bar(L::kBarKVFull + kv_stage(lk)), kv_par(lk),
                                             abort_flag)))
                    break;
                for (int t = 0; t < 2; ++t) {
                    if (j < n_t[t]) {
                        if (!(ok = mbar_wait(bar(L::kBarPFull + t), j & 1, abort_flag))) break;
                        tc_fence_after();
                        issue_pv(t, j);
                        mma_commit(bar(L::kBarPVDone + t));
                    }
                    if (t == 1) mma_commit(bar(L::kBarKVEmpty + kv_stage(lv)));
                    if (j + 1 < n_t[t]) {
                        // P_t(j) and S_t(j+1) share TMEM columns: O_t's MMA must be done.
                        if (!(ok = mbar_wait(bar(L::kBarPVDone + t), j & 1, abort_flag))) break;
                        tc_fence_after();
                        issue_qk(t, j + 1);
                        mma_commit(bar(L::kBarSFull + t));
                    }
                }
                if (ok && next) mma_commit(bar(L::kBarKVEmpty + kv_stage(lk)));
            }
            if (!ok) {
                mma_commit(bar(L::kBarDrain));
                volatile int no_abort = 0;
                mbar_wait(bar(L::kBarDrain), 0, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax WGs
        const int t = warp >> 2;                    // query tile of this warpgroup
        const int wq = warp & 3;                    // TMEM lane quarter
        const int r_local = wq * 32 + lane;
        const int i = m0 + t * kTile + r_local;     // query row in the sequence
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + (t ? L::kColS1 : L::kColS0);
        const uint32_t tO = tmem + lane_off + (t ? L::kColO1 : L::kColO0);
        const int n_mine = n_t[t];
        const int r0_tile = m0 + t * kTile;
        float m_ref = -INFINITY;
        float2 l2 = make_float2(0.f, 0.f);    // sum of the exact probabilities (-> lse)
        float2 lr2 = make_float2(0.f, 0.f);   // sum of the bf16-rounded ones fed to P V (-> out)
        bool ok = true;

        for (int j = 0; j < n_mine; ++j) {
            ok = mbar_wait(bar(L::kBarSFull + t), j & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // The whole row of S comes to registers with one TMEM load; P is
            // then written over S columns [0, 64).  With a user mask the
            // logits are first rewritten in TMEM chunk by chunk (the mask
            // loads would otherwise hold too many registers).
            const int n0 = j * kTile;
            const bool has_mask = p.mask_kind != MASK_NONE;
            const bool pred = (n0 + kTile > si.len_k) || (p.causal && n0 + kTile - 1 > r0_tile);
            float x[kTile];
            float mt = -INFINITY;
            if (has_mask) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tS + 32 * c, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = __float_as_uint(logit_log2(p, __uint_as_float(v[e]), b, h, i,
                                                          n0 + 32 * c + e, si.len_q, si.len_k));
                    tmem_st32(tS + 32 * c, v);
                }
                tmem_wait_st();
                tmem_ld128(tS, reinterpret_cast<uint32_t*>(x));
#pragma unroll
                for (int c = 0; c < kTile; ++c) mt = fmaxf(mt, x[c]);
            } else if (pred) {
                tmem_ld128(tS, reinterpret_cast<uint32_t*>(x));
                const int jmax = p.causal ? min(si.len_k, i + 1) : si.len_k;   // keys < jmax visible
                const bool row_in = i < si.len_q;
#pragma unroll
                for (int c = 0; c < kTile; ++c) {
                    x[c] = (row_in && n0 + c < jmax) ? x[c] * p.scale_log2 : -INFINITY;
                    mt = fmaxf(mt, x[c]);
                }
            } else {
                // full tile, no mask: the max of the raw scores, scaled once
                // (x stays unscaled; P below folds the scale into one FMA).  The
                // second half of the row is still loading from TMEM while the
                // max of the first half runs.
                uint32_t* xu = reinterpret_cast<uint32_t*>(x);
                tmem_ld32x2(tS, xu, tS + 32, xu + 32);
                tmem_ld64_nowait(tS + 64, xu + 64);
                // At D = 64 with the three-input max (one instruction per pair), and
                // two chains for the half on the critical path; both measured faster
                // at D = 64 and slower at D = 128.
                float mr = -INFINITY;
                if constexpr (D == 64) {
#pragma unroll
                    for (int c = 0; c < kTile / 2; c += 2) mr = fmax3(mr, x[c], x[c + 1]);
                } else {
#pragma unroll
                    for (int c = 0; c < kTile / 2; ++c) mr = fmaxf(mr, x[c]);
                }
                tmem_wait_ld_regs64(xu + 64);
                if constexpr (D == 64) {
                    float mr1 = -INFINITY;
#pragma unroll
                    for (int c = kTile / 2; c < kTile; c += 4) {
                        mr = fmax3(mr, x[c], x[c + 1]);
                        mr1 = fmax3(mr1, x[c + 2], x[c + 3]);
                    }
                    mr = fmaxf(mr, mr1);
                } else {
#pragma unroll
                    for (int c = kTile / 2; c < kTile; ++c) mr = fmaxf(mr, x[c]);
                }
                if (p.scale_log2 > 0.f) {
                    mt = mr * p.scale_log2;
                } else {
#pragma unroll
                    for (int c = 0; c < kTile; ++c) mt = fmaxf(mt, x[c] * p.scale_log2);
                }
            }
            const bool raw = !has_mask && !pred;   // x holds unscaled scores
            // Online max: always m_new = max(m_ref, m_tile); lazy threshold 8.
            const float m_new = fmaxf(m_ref, mt);
            bool rescale;
            if (m_new == -INFINITY) {
                rescale = false;
            } else if (p.lazy && m_ref != -INFINITY && mt - m_ref <= kLazyTau) {
                rescale = false;
            } else {
                rescale = true;
            }
            float corr = 1.f;
            if (rescale) {
                corr = ex2(m_ref - m_new);          // m_ref = -inf -> 0
                l2 = fmul2(l2, make_float2(corr, corr));
                lr2 = fmul2(lr2, make_float2(corr, corr));
                // O holds data only after the first PV; a row whose m_ref was
                // -inf has O = 0 there and needs no correction.
                if (j == 0 || m_ref == -INFINITY) corr = 1.f;
                m_ref = m_new;
            }
            const float ms = (m_ref == -INFINITY) ? 0.f : m_ref;
            const float2 nms2 = make_float2(-ms, -ms);
            const float2 c2 = raw ? make_float2(p.scale_log2, p.scale_log2) : make_float2(1.f, 1.f);
            // P = exp2(min(x - m_ref, 8)).  The clamp cannot bind on a row whose tile
            // max is within 8 of m_ref (the lazy test passed) or that rescaled
            // (m_ref >= the tile max); when that holds for the whole warp with a
            // margin for rounding, the per-element min is skipped.
            auto exps = [&](auto clamp_tag) {
                constexpr bool kClamp = decltype(clamp_tag)::value;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        // x - m_ref in one packed FMA (the scale folded in when x is raw)
                        const float2 d2 = ffma2(make_float2(x[32 * c + 2 * e], x[32 * c + 2 * e + 1]), c2, nms2);
                        float2 p2;
                        p2.x = ex2(kClamp ? fminf(d2.x, kLazyTau) : d2.x);
                        p2.y = ex2(kClamp ? fminf(d2.y, kLazyTau) : d2.y);
                        l2 = fadd2(l2, p2);
                        pk[e] = pack2<F16>(p2.x, p2.y);
                        if constexpr (!L::kOnesCol) lr2 = fadd2(lr2, unpack2<F16>(pk[e]));
                    }
                    tmem_st16(tS + 16 * c, pk);
                }
            };
            if (__all_sync(0xffffffffu, mt - ms <= kLazyTau - 0.015625f))
                exps(BoolTag<false>{});
            else
                exps(BoolTag<true>{});
            // Rescale O_t in TMEM (its previous MMA has completed: the commit that
            // signalled S_t(j) was issued after it).
            if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < L::kOStride / 32; ++c) {    // the sum column too
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                    tmem_st32(tO + 32 * c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(L::kBarPFull + t));
        }

        // Epilogue.
        const bool store = ok && i < si.len_q;
        bf16* orow = p.out + b * p.out_b + static_cast<int64_t>(row_base + i) * p.out_s + h * p.out_h;
        if (ok && n_mine > 0) {
            ok = mbar_wait(bar(L::kBarPVDone + t), (n_mine - 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        if (ok) {
            // Normalise by the rounded sum: out stays an exact weighted mean of V
            // even when the lazy reference max lags (largest weight up to 2^8).
            const float l = l2.x + l2.y;
            float lr = lr2.x + lr2.y;
            if constexpr (L::kOnesCol) {
                lr = 0.f;
                if (n_mine > 0) {
                    uint32_t o[32];
                    tmem_ld32(tO + D, o);              // column D: sum of the rounded p
                    lr = __uint_as_float(o[0]);
                }
            }
            const float inv = lr > 0.f ? 1.0f / lr : 0.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (n_mine > 0) {
                    tmem_ld32(tO + 32 * c, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (store) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack2<F16>(__uint_as_float(o[2 * e]) * inv,
                                          __uint_as_float(o[2 * e + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (store)
                p.lse[b * p.lse_b + h * p.lse_h + row_base + i] =
                    l > 0.f ? (m_ref + lg2(l)) * kLn2 : 0.f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    if (tid == 0 && *abort_flag) set_error(p.err, DEV_E_TIMEOUT);
}

// ------------------------------------------------------------------ host side

template <int D, bool F16>
cudaError_t launch_fwd_sm100_d(const Problem& p, cudaStream_t stream) {
    using L = FwdLayout<D>;
    if (p.B == 0 || p.Sq == 0) return cudaSuccess;
    FwdMaps maps;
    const int64_t S = p.varlen ? p.T : p.Sq;
    const int64_t Sk = p.varlen ? p.T : p.Sk;
    const int64_t Bm = p.varlen ? 1 : p.B;
    // An empty key set still needs legal maps; point them at q.
    const bool no_keys = Sk == 0;
    if (!make_tile_map(&maps.q, p.q, D, p.Hq, S, Bm, p.q_h, p.q_s, p.q_b, F16)) return cudaErrorInvalidValue;
    if (!make_tile_map(&maps.k, no_keys ? p.q : p.k, D, no_keys ? p.Hq : p.Hkv, no_keys ? S : Sk, Bm,
                  no_keys ? p.q_h : p.k_h, no_keys ? p.q_s : p.k_s, no_keys ? p.q_b : p.k_b, F16))
        return cudaErrorInvalidValue;
    if (!make_tile_map(&maps.v, no_keys ? p.q : p.v, D, no_keys ? p.Hq : p.Hkv, no_keys ? S : Sk, Bm,
                  no_keys ? p.q_h : p.v_h, no_keys ? p.q_s : p.v_s, no_keys ? p.q_b : p.v_b, F16))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fwd_sm100_kernel<D, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sq + 2 * kTile - 1) / (2 * kTile), p.Hq, p.B);
    fwd_sm100_kernel<D, F16><<<grid, kFwdThreads, L::kBytes, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, cudaStream_t stream) {
    if (p.f16)
        return p.D == 64 ? launch_fwd_sm100_d<64, true>(p, stream) : launch_fwd_sm100_d<128, true>(p, stream);
    return p.D == 64 ? launch_fwd_sm100_d<64, false>(p, stream) : launch_fwd_sm100_d<128, false>(p, stream);
}

}  // namespace attn
