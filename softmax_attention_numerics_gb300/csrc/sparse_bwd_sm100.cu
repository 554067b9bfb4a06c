// Sparse top-k attention backward with an attention sink (the DSA backward of
// NVIDIA/cudnn-frontend PR #429: q, kv, out, dout, lse, attn_sink,
// topk_idxs, topk_length -> dq, dkv, d_sink; head dim 512, or 576 in the MLA
// form whose values are the first 512 columns of the kv rows), for sm_103a:
// cp.async gathers + TMA + tcgen05 + TMEM.
//
// For token i of batch b, the valid entries e of its index list (e below the
// token's length, 0 <= idx < S_kv) select kv rows k_e, v_e = k_e[:512]:
//     P_he  = exp(scale q_h . k_e - lse_h)           (lse includes the sink)
//     dP_he = dout_h . v_e,   Delta_h = dout_h . out_h
//     dS_he = scale P_he (dP_he - Delta_h)
//     dq_h  = sum_e dS_he k_e
//     dkv[idx_e]       += sum_h dS_he q_h,   dkv[idx_e, :512] += sum_h P_he dout_h
//     d_sink_h = - sum_tokens exp(sink_h - lse_h) Delta_h
//
// Work item = (token, 128 consecutive entries of its list).  One persistent
// CTA per SM walks the items of the tokens blockIdx.x, blockIdx.x + grid, ...
// All 64 heads of a token share the gathered rows, so the entries are the M
// of the products and the heads their N:
//   S^T  [128 e x 64 h]  = K_sel . Q^T        (A: gathered rows, B: Q block)
//   dP^T [128 e x 64 h]  = V_sel . dO^T
//   dQ^T [128 d x 64 h] += K_sel^T . dS^T     (A, B MN-major; 5 row chunks)
//   dKV  [128 e x 64 d]  = dS^T . Q[:, d] + P^T . dO[:, d]   (A from TMEM)
// Roles (256 threads, so that no register cap below 255 applies):
//   warps 0-3  one entry per thread (TMEM lane): P^T, dS^T; the dKV rows,
//              bulk-reduced (fp32 add) into the workspace row idx_e two
//              operations per half row (pieces of 32 columns, 5 + 4 or
//              4 + 4), staged in half-row slots of the gathered-rows region
//              once dQ^T no longer reads it, each group's slots reused as soon
//              as its add has read them (few large bulk operations: their
//              count, not their bytes, is the limit, and adds that start
//              early overlap the dKV MMAs); dq
//   warps 4-5  gather the 128 selected kv rows with 16-byte cp.async (each
//              warp instruction covers whole 128-byte row blocks) into the
//              128-byte-swizzled operand layout, one 64-column block at a
//              time, each signalled on a barrier of its own as it lands (the
//              rows stay resident for S^T, dP^T and dQ^T)
//   warp 6     TMA: the 64 x 64 blocks of Q and dO of one 64-column slice
//              together through a 3-stage ring (one wait and one release per
//              slice), in the order the MMA issuer consumes them (twice per
//              item); an L2 prefetch of the next token's blocks
//   warp 7     TMEM allocator and single-thread UMMA issuer
// TMEM: S^T at 0 (P^T packed over its first 32 columns, dS^T over the next
// 32), dP^T at 64 (after use: dKV buffer 1), dQ^T at 128 + 64 m, dKV buffer 0
// at 448.  Delta and the sink terms come from sparse_prep_kernel; d_sink is
// their ordered sum; dkv is converted from the fp32 workspace at the end.
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using namespace sm100;

constexpr int kSpH = 64;             // query heads per token
constexpr int kSpE = 128;            // index entries per work item
constexpr int kSpDv = 512;           // value columns
constexpr int kSpThreads = 256;
constexpr int kRing = 3;             // ring of (Q block, dO block) pairs, 16 KB a stage

template <int NB>   // 64-column blocks of the kv rows: 8 (512) or 9 (576)
struct SpLayout {
    static constexpr int kNBV = kSpDv / 64;
    static constexpr int kNM = (NB + 1) / 2;                // dQ^T chunks of 128 columns
    static constexpr int kKV = 0;                           // NB x [128 entries][64 cols] bf16
    // dKV staging over the same region during the dKV phase: 128 rows of half
    // a kv row in fp32 (NB x 128 bytes) + 16 bytes of padding (bank spread)
    static constexpr int kStRow = NB * 128 + 16;
    // the staged pieces of a half row go out in two groups: pieces [0, kH1) and
    // [kH1, NB) (5 + 4 at NB = 9, 4 + 4 at NB = 8)
    static constexpr int kH1 = (NB + 1) / 2;
    __device__ static constexpr int gfirst(int q) { return q < kH1 ? 0 : kH1; }
    __device__ static constexpr bool glast(int q) { return q == kH1 - 1 || q == NB - 1; }
    static constexpr int kRingOff = 128 * kStRow;           // kRing x {Q, dO} x [64 heads][64 cols] bf16
    static constexpr int kDS = kRingOff + kRing * 16384;    // dS^T [128 entries][64 heads] bf16
    static constexpr int kBar = kDS + 16384;
    static constexpr int kBarKV = 0;                        // [NB] a block of the gathered rows landed (64)
    static constexpr int kBarRFull = NB, kBarREmpty = NB + kRing;
    static constexpr int kBarSdp = NB + 2 * kRing;          // S^T and dP^T complete
    static constexpr int kBarPds = kBarSdp + 1;             // P^T, dS^T written (128)
    static constexpr int kBarKVFree = kBarPds + 1;          // gathered rows no longer read
    static constexpr int kBarDkvFull = kBarKVFree + 1;      // 2
    static constexpr int kBarDkvFree = kBarDkvFull + 2;     // 2 (128)
    static constexpr int kBarItemDone = kBarDkvFree + 2;    // every dKV chunk read out (128)
    static constexpr int kBarDQFull = kBarItemDone + 1;
    static constexpr int kBarDQRead = kBarDQFull + 1;       // dQ^T read out (128)
    static constexpr int kBarStageFree = kBarDQRead + 1;    // staging read by the bulk adds (128)
    static constexpr int kBarDrain = kBarStageFree + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16 + 1024;        // + alignment slack
    static constexpr uint32_t kColS = 0, kColDP = 64, kColDQ = 128, kColKV0 = 448;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kColDQ + 64 * kNM <= kColKV0, "TMEM columns");
    static_assert(kBytes <= 232448, "shared memory");
    static_assert(kRingOff % 1024 == 0 && kRingOff >= NB * 16384, "ring placement");
};

struct SparseMaps {
    CUtensorMap q, dout;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most n of this thread's cp.async groups are pending.
__device__ __forceinline__ void cp_async_wait(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        case 7: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 8;" ::: "memory"); break;
    }
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
// fp32 add of `bytes` from shared memory into global memory (bulk group).
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                     dst),
                 "r"(src), "r"(bytes)
                 : "memory");
}
// Prefetch a 4-D tiled box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_4d(const void* tmap, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(tmap),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
__device__ __forceinline__ void bulk_wait_read_0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until at most N of this thread's bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

struct TokenInfo {
    int b, i, nlen, nch;
};

// Token t = b * S + i: its number of listed entries (clamped to [0, K]) and
// of work items (at least one, so that its dq row is written).
__device__ __forceinline__ TokenInfo token_info(const SparseProblem& p, int t) {
    TokenInfo r;
    r.b = t / p.S;
    r.i = t - r.b * p.S;
    int n = p.K;
    if (p.len) {
        const int l = __ldg(p.len + r.b * p.len_b + r.i * p.len_s);
        n = l < 0 ? 0 : (l < p.K ? l : p.K);
    }
    r.nlen = n;
    r.nch = n > 0 ? (n + kSpE - 1) / kSpE : 1;
    return r;
}

// kv row of entry e of the token, or -1 when the entry takes no part.
__device__ __forceinline__ int entry_row(const SparseProblem& p, const TokenInfo& ti, int e) {
    if (e >= ti.nlen) return -1;
    const int r = __ldg(p.idx + ti.b * p.idx_b + ti.i * p.idx_s + e);
    return (r >= 0 && r < p.Skv) ? r : -1;
}

template <int NB, bool F16>
__global__ void __launch_bounds__(kSpThreads, 1)
    sparse_bwd_sm100_kernel(const SparseProblem p, const __grid_constant__ SparseMaps maps) {
    using L = SpLayout<NB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::kBar + 8u * i; };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.B * p.S;

    if (tid == 0) {
        for (int i = 0; i < L::kNumBars; ++i) {
            const bool by128 = i == L::kBarPds || i == L::kBarDkvFree || i == L::kBarDkvFree + 1 ||
                               i == L::kBarItemDone || i == L::kBarDQRead || i == L::kBarStageFree;
            mbar_init(bar(i), i < L::kBarKV + NB ? 64 : (by128 ? 128 : 1));
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 7) {
        tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 4 || warp == 5) {
        // ------------------------------------------------------------ row gather
        // Thread g copies 16-byte chunk (g & 7) of rows (g >> 3) + 8 k, k < 16:
        // every warp instruction moves four whole 128-byte row blocks.
        const int g = tid - 128, j = g & 7, rs = g >> 3;
        int n = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < T; t += gridDim.x) {
            const TokenInfo ti = token_info(p, t);
            for (int c = 0; c < ti.nch; ++c, ++n) {
                // the previous item's MMAs have read the rows and its dKV
                // staging over the same region has been read by the bulk adds
                if (n > 0 && !(ok = mbar_wait(bar(L::kBarStageFree), (n - 1) & 1, abort_flag))) break;
                const uint8_t* src[kSpE / 8];
#pragma unroll
                for (int k = 0; k < kSpE / 8; ++k) {
                    const int row = entry_row(p, ti, c * kSpE + 8 * k + rs);
                    src[k] = reinterpret_cast<const uint8_t*>(
                                 p.kv + ti.b * p.kv_b + static_cast<int64_t>(row < 0 ? 0 : row) * p.kv_s) +
                             16 * j;
                }
                const uint32_t dst = sbase + L::kKV + rs * 128 + ((j ^ rs) << 4);   // (8k + rs) & 7 = rs
                // one copy group per 64-column block, each block signalled as it
                // lands, so that the S^T / dP^T MMAs start on the first blocks
                // while the later ones are still being copied
#pragma unroll
                for (int blk = 0; blk < NB; ++blk) {
#pragma unroll
                    for (int k = 0; k < kSpE / 8; ++k)
                        cp_async16(dst + blk * 16384 + k * 1024, src[k] + blk * 128);
                    cp_async_commit();
                    if (blk > 0) {
                        cp_async_wait(1);                    // this thread's part of block blk - 1
                        fence_proxy_async_smem();            // generic-proxy writes -> UMMA reads
                        mbar_arrive(bar(L::kBarKV + blk - 1));
                    }
                }
                cp_async_wait(0);
                fence_proxy_async_smem();
                mbar_arrive(bar(L::kBarKV + NB - 1));
            }
        }
        cp_async_wait(0);
    } else if (warp == 6) {
        // ------------------------------------------------------------ TMA: Q / dO blocks
        if (lane == 0) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.dout);
            int r = 0;
            bool ok = true;
            auto load = [&](int blk, const TokenInfo& ti) {       // Q block (and dO block) blk
                const int s = r % kRing;
                if (!(ok = mbar_wait(bar(L::kBarREmpty + s), ((r / kRing) & 1) ^ 1, abort_flag))) return;
                const bool with_do = blk < L::kNBV;
                mbar_arrive_expect_tx(bar(L::kBarRFull + s), with_do ? 16384 : 8192);
                const uint32_t d = sbase + L::kRingOff + s * 16384;
                tma_load_4d(d, &maps.q, 64 * blk, 0, ti.i, ti.b, bar(L::kBarRFull + s));
                if (with_do) tma_load_4d(d + 8192, &maps.dout, 64 * blk, 0, ti.i, ti.b, bar(L::kBarRFull + s));
                ++r;
            };
            for (int t = blockIdx.x; ok && t < T; t += gridDim.x) {
                const TokenInfo ti = token_info(p, t);
                if (t + static_cast<int>(gridDim.x) < T) {
                    const int tn = t + gridDim.x, bn = tn / p.S, in = tn - bn * p.S;
                    for (int blk = 0; blk < NB; ++blk) {
                        tma_prefetch_l2_4d(&maps.q, 64 * blk, 0, in, bn);
                        if (blk < L::kNBV) tma_prefetch_l2_4d(&maps.dout, 64 * blk, 0, in, bn);
                    }
                }
                for (int c = 0; ok && c < ti.nch; ++c)
                    for (int pass = 0; ok && pass < 2; ++pass)       // S^T / dP^T, then dKV
                        for (int blk = 0; ok && blk < NB; ++blk) load(blk, ti);
            }
            if (*abort_flag) {
                volatile int no_abort = 0;
                for (int k = max(0, r - kRing); k < r; ++k)
                    mbar_wait(bar(L::kBarRFull + k % kRing), (k / kRing) & 1, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else if (warp == 7) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_f16kind(128, 64, 0, 0, F16);     // S^T, dP^T
            constexpr uint32_t id_dq = idesc_f16kind(128, 64, 1, 1, F16);    // dQ^T (A, B MN-major)
            constexpr uint32_t id_kv = idesc_f16kind(128, 64, 0, 1, F16);    // dKV (B MN-major)
            const uint64_t ds_mn = smem_desc(sbase + L::kDS, 8192, 1024, kSwizzle128B);
            int n = 0, r = 0, g = 0, tk = 0;
            bool ok = true;
            // next ring stage: wait for it, return its shared address (Q block,
            // then the dO block 8 KB later)
            auto ring_next = [&](uint32_t* addr) -> int {
                const int s = r % kRing;
                if (!(ok = mbar_wait(bar(L::kBarRFull + s), (r / kRing) & 1, abort_flag))) return s;
                tc_fence_after();
                *addr = sbase + L::kRingOff + s * 16384;
                ++r;
                return s;
            };
            for (int t = blockIdx.x; ok && t < T; t += gridDim.x, ++tk) {
                const TokenInfo ti = token_info(p, t);
                for (int c = 0; ok && c < ti.nch; ++c, ++n) {
                    if (!(ok = dbg_stall(p.debug_stall, kStallSparse, n, bar(L::kBarDrain), abort_flag)))
                        break;
                    // TMEM columns 0-127 and dKV buffer 0 are free once the
                    // previous item's dKV chunks have all been read out.
                    if (n > 0 && !(ok = mbar_wait(bar(L::kBarItemDone), (n - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    // S^T and dP^T over the 64-column blocks of the gathered rows, each
                    // once it has landed
                    for (int blk = 0; ok && blk < NB; ++blk) {
                        if (!(ok = mbar_wait(bar(L::kBarKV + blk), n & 1, abort_flag))) break;
                        const uint64_t a = smem_desc(sbase + L::kKV + blk * 16384, 16, 1024, kSwizzle128B);
                        uint32_t ra;
                        const int s = ring_next(&ra);
                        if (!ok) break;
                        const uint64_t bq = smem_desc(ra, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(ra + 8192, 16, 1024, kSwizzle128B);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tmem + L::kColS, desc_add(a, 32 * kk), desc_add(bq, 32 * kk), id_s,
                                   (blk | kk) != 0);
                        if (blk < L::kNBV) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss(tmem + L::kColDP, desc_add(a, 32 * kk), desc_add(bd, 32 * kk), id_s,
                                       (blk | kk) != 0);
                        }
                        mma_commit(bar(L::kBarREmpty + s));
                    }
                    if (!ok) break;
                    mma_commit(bar(L::kBarSdp));
                    // dQ^T += K_sel^T dS^T once P^T / dS^T are written (and, on a
                    // token's first item, once the previous token's dQ^T is read out)
                    if (!(ok = mbar_wait(bar(L::kBarPds), n & 1, abort_flag))) break;
                    if (c == 0 && tk > 0 && !(ok = mbar_wait(bar(L::kBarDQRead), (tk - 1) & 1, abort_flag)))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int m = 0; m < L::kNM; ++m) {
                        // rows 128m .. 128m + 127 of K_sel^T: blocks 2m and 2m + 1 (for an odd
                        // block count the second half of the last chunk reads the next
                        // region and lands in TMEM lanes that are never read)
                        const uint64_t a = smem_desc(sbase + L::kKV + 2 * m * 16384, 16384, 1024, kSwizzle128B);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tmem + L::kColDQ + 64 * m, desc_add(a, 2048 * kk), desc_add(ds_mn, 2048 * kk),
                                   id_dq, (c | kk) != 0);
                    }
                    mma_commit(bar(L::kBarKVFree));
                    if (c == ti.nch - 1) mma_commit(bar(L::kBarDQFull));
                    // dKV chunk j (columns 64j .. 64j + 63) = dS^T Q[:, j] + P^T dO[:, j]
                    for (int j = 0; ok && j < NB; ++j, ++g) {
                        const int buf = g & 1, u = g >> 1;
                        if (u >= 1 && !(ok = mbar_wait(bar(L::kBarDkvFree + buf), (u - 1) & 1, abort_flag)))
                            break;
                        tc_fence_after();
                        const uint32_t dkv = tmem + (buf ? L::kColDP : L::kColKV0);
                        uint32_t ra;
                        const int s = ring_next(&ra);
                        if (!ok) break;
                        const uint64_t bq = smem_desc(ra, 8192, 1024, kSwizzle128B);        // MN-major
                        const uint64_t bd = smem_desc(ra + 8192, 8192, 1024, kSwizzle128B);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ts(dkv, tmem + L::kColS + 32 + 8 * kk, desc_add(bq, 2048 * kk), id_kv, kk > 0);
                        if (j < L::kNBV) {
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ts(dkv, tmem + L::kColS + 8 * kk, desc_add(bd, 2048 * kk), id_kv, 1);
                        }
                        mma_commit(bar(L::kBarREmpty + s));
                        mma_commit(bar(L::kBarDkvFull + buf));
                    }
                }
            }
            if (!ok) {
                mma_commit(bar(L::kBarDrain));
                volatile int no_abort = 0;
                mbar_wait(bar(L::kBarDrain), 0, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ entries (warps 0-3)
        const int key = warp * 32 + lane;                    // TMEM lane = entry of the item
        const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float c2 = p.scale_log2;
        int n = 0, g = 0, tk = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < T; t += gridDim.x, ++tk) {
            const TokenInfo ti = token_info(p, t);
            // the token's 64 lse and Delta values: the same address in every
            // lane (L1 broadcasts); no block-level barrier, so that a warp that
            // unwinds early cannot leave the others waiting
            const float4* lse_t = reinterpret_cast<const float4*>(p.lse + static_cast<int64_t>(t) * kSpH);
            const float4* delta_t = reinterpret_cast<const float4*>(p.delta + static_cast<int64_t>(t) * kSpH);
            for (int c = 0; ok && c < ti.nch; ++c, ++n) {
                const int row = entry_row(p, ti, c * kSpE + key);
                const bool valid = row >= 0;
                ok = mbar_wait(bar(L::kBarSdp), n & 1, abort_flag);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // P^T over columns 0-31 (all of S^T is in registers first)
                float P[kSpH];
                {
                    uint32_t x[kSpH];
                    tmem_ld32x2(tl + L::kColS, x, tl + L::kColS + 32, x + 32);
#pragma unroll
                    for (int h4 = 0; h4 < kSpH / 4; ++h4) {
                        const float4 l = __ldg(lse_t + h4);
                        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int h = 4 * h4 + u;
                            P[h] = valid ? ex2(fminf(fmaf(__uint_as_float(x[h]), c2, -lv[u] * kLog2e), 0.f))
                                         : 0.f;
                        }
                    }
                    uint32_t pk[32];
#pragma unroll
                    for (int h = 0; h < 32; ++h) pk[h] = pack2<F16>(P[2 * h], P[2 * h + 1]);
                    tmem_st32(tl + L::kColS, pk);
                }
                // dS^T = scale P^T (dP^T - Delta) over columns 32-63, and into
                // shared memory as the B operand of dQ^T (128-byte swizzle)
                const uint32_t ds_row = sbase + L::kDS + key * 128;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t y[32];
                    tmem_ld32(tl + L::kColDP + 32 * half, y);
                    uint32_t dk[16];
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 dl = __ldg(delta_t + 8 * half + e4);
                        const int h = 32 * half + 4 * e4;
                        dk[2 * e4] = pack2<F16>(P[h] * (__uint_as_float(y[4 * e4]) - dl.x) * p.scale,
                                                P[h + 1] * (__uint_as_float(y[4 * e4 + 1]) - dl.y) * p.scale);
                        dk[2 * e4 + 1] = pack2<F16>(P[h + 2] * (__uint_as_float(y[4 * e4 + 2]) - dl.z) * p.scale,
                                                    P[h + 3] * (__uint_as_float(y[4 * e4 + 3]) - dl.w) * p.scale);
                    }
                    tmem_st16(tl + L::kColS + 32 + 16 * half, dk);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int chunk = 4 * half + q4;
                        sts128(ds_row + ((chunk ^ (key & 7)) << 4), dk[4 * q4], dk[4 * q4 + 1],
                               dk[4 * q4 + 2], dk[4 * q4 + 3]);
                    }
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar(L::kBarPds));
                // dKV chunks: read out and stage the row in 32-column pieces; a
                // bulk fp32 add of each half row (NB pieces) into dkv_acc[row]
                float* acc_row = p.dkv_acc + (static_cast<int64_t>(ti.b) * p.Skv + (valid ? row : 0)) * p.Dqk;
                const uint32_t st_row = sbase + L::kKV + key * L::kStRow;
                for (int j = 0; j < NB; ++j, ++g) {
                    const int buf = g & 1, u = g >> 1;
                    ok = mbar_wait(bar(L::kBarDkvFull + buf), u & 1, abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col = buf ? L::kColDP : L::kColKV0;
                    uint32_t x[64];
                    tmem_ld32x2(tl + col, x, tl + col + 32, x + 32);
                    tc_fence_before();
                    mbar_arrive(bar(L::kBarDkvFree + buf));
                    if (j == 0) {
                        // dQ^T's MMAs have read the gathered rows: the region is staging now
                        ok = mbar_wait(bar(L::kBarKVFree), n & 1, abort_flag);
                        if (!__all_sync(0xffffffffu, ok)) {
                            ok = false;
                            break;
                        }
                    }
                    if (valid) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const int pc = 2 * j + half, q = pc % NB;
                            // the group that read this slot in the first half row is done
                            if (pc >= NB && L::gfirst(q) == q) bulk_wait_read<1>();
#pragma unroll
                            for (int q4 = 0; q4 < 8; ++q4)
                                sts128(st_row + 128 * q + 16 * q4, x[32 * half + 4 * q4],
                                       x[32 * half + 4 * q4 + 1], x[32 * half + 4 * q4 + 2],
                                       x[32 * half + 4 * q4 + 3]);
                            if (L::glast(q)) {
                                // a group of pieces (32 columns each) complete: add them
                                const int q0 = L::gfirst(q), p0 = pc - (q - q0);
                                fence_proxy_async_smem();
                                bulk_reduce_add_f32(acc_row + p0 * 32, st_row + 128 * q0, (q - q0 + 1) * 128);
                                bulk_commit();
                            }
                        }
                    }
                }
                if (ok) {
                    bulk_wait_read_0();
                    mbar_arrive(bar(L::kBarStageFree));
                }
                if (!ok) break;
                mbar_arrive(bar(L::kBarItemDone));
            }
            if (!ok) break;
            // dq of the token: dQ^T lane = column d, TMEM column = head
            ok = mbar_wait(bar(L::kBarDQFull), tk & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint16_t* dq = reinterpret_cast<uint16_t*>(p.dq) + static_cast<int64_t>(t) * kSpH * p.Dqk;
#pragma unroll 1
            for (int m = 0; m < L::kNM; ++m) {
                uint32_t x[kSpH];
                tmem_ld32x2(tl + L::kColDQ + 64 * m, x, tl + L::kColDQ + 64 * m + 32, x + 32);
                const int d = 128 * m + key;
                if (d < p.Dqk) {
#pragma unroll
                    for (int h = 0; h < kSpH; ++h) {
                        const float v = __uint_as_float(x[h]);
                        dq[h * p.Dqk + d] = static_cast<uint16_t>(pack2<F16>(v, 0.f) & 0xffffu);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(L::kBarDQRead));
        }
        bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 7) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    if (tid == 0 && *abort_flag) set_error(p.err, DEV_E_TIMEOUT);
}

// Delta[t, h] = dout . out over the value columns, and the sink terms
// -exp(sink_h - lse) Delta (one warp per head, lanes over columns, a fixed
// summation order).
template <bool F16>
__global__ void __launch_bounds__(256) sparse_prep_kernel(const SparseProblem p) {
    const int t = blockIdx.x;
    const int b = t / p.S, i = t - b * p.S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int h = warp; h < p.H; h += 8) {
        const bf16* o = p.out + b * p.o_b + i * p.o_s + h * p.o_h;
        const bf16* d = p.dout + b * p.do_b + i * p.do_s + h * p.do_h;
        float acc = 0.f;
        for (int c = lane * 8; c < p.Dv; c += 256) {
            const uint4 ov = *reinterpret_cast<const uint4*>(o + c);
            const uint4 dv = *reinterpret_cast<const uint4*>(d + c);
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
            const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 a = unpack2<F16>(ow[k]);
                const float2 e = unpack2<F16>(dw[k]);
                acc = fmaf(a.x, e.x, acc);
                acc = fmaf(a.y, e.y, acc);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            const int64_t th = static_cast<int64_t>(t) * p.H + h;
            p.delta[th] = acc;
            if (p.sink) p.dsink_part[th] = -ex2((p.sink[h] - p.lse[th]) * kLog2e) * acc;
        }
    }
}

// d_sink[h] = sum over tokens of the sink terms, in a fixed order.
__global__ void __launch_bounds__(256) sparse_dsink_kernel(const SparseProblem p) {
    __shared__ float red[256];
    const int h = blockIdx.x;
    const int64_t T = static_cast<int64_t>(p.B) * p.S;
    float s = 0.f;
    for (int64_t t = threadIdx.x; t < T; t += 256) s += p.dsink_part[t * p.H + h];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) p.dsink[h] = red[0];
}

// dkv (16-bit) from the fp32 workspace, 8 elements per thread.
template <bool F16>
__global__ void __launch_bounds__(256) sparse_dkv_convert_kernel(const SparseProblem p, int64_t n8) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n8; x += stride) {
        const float4 a = reinterpret_cast<const float4*>(p.dkv_acc)[2 * x];
        const float4 c = reinterpret_cast<const float4*>(p.dkv_acc)[2 * x + 1];
        uint4 o;
        o.x = pack2<F16>(a.x, a.y);
        o.y = pack2<F16>(a.z, a.w);
        o.z = pack2<F16>(c.x, c.y);
        o.w = pack2<F16>(c.z, c.w);
        reinterpret_cast<uint4*>(p.dkv)[x] = o;
    }
}

int sm_count() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 1;
}

template <int NB, bool F16>
cudaError_t launch_main(const SparseProblem& p, cudaStream_t stream) {
    using L = SpLayout<NB>;
    const int64_t T = static_cast<int64_t>(p.B) * p.S;
    if (T == 0) return cudaSuccess;
    SparseMaps maps;
    if (!make_heads_map(&maps.q, p.q, p.Dqk, p.H, p.S, p.B, p.q_h, p.q_s, p.q_b, F16) ||
        !make_heads_map(&maps.dout, p.dout, p.Dv, p.H, p.S, p.B, p.do_h, p.do_s, p.do_b, F16))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(sparse_bwd_sm100_kernel<NB, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(T < sm_count() ? T : sm_count());
    sparse_bwd_sm100_kernel<NB, F16><<<grid, kSpThreads, L::kBytes, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_prep(const SparseProblem& p, cudaStream_t stream) {
    const int64_t T = static_cast<int64_t>(p.B) * p.S;
    if (T == 0) return cudaSuccess;
    if (p.f16)
        sparse_prep_kernel<true><<<static_cast<unsigned>(T), 256, 0, stream>>>(p);
    else
        sparse_prep_kernel<false><<<static_cast<unsigned>(T), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_sparse_bwd_main(const SparseProblem& p, cudaStream_t stream) {
    if (p.Dqk == 576)
        return p.f16 ? launch_main<9, true>(p, stream) : launch_main<9, false>(p, stream);
    return p.f16 ? launch_main<8, true>(p, stream) : launch_main<8, false>(p, stream);
}

cudaError_t launch_sparse_dkv_convert(const SparseProblem& p, cudaStream_t stream) {
    const int64_t n8 = static_cast<int64_t>(p.B) * p.Skv * p.Dqk / 8;
    if (n8 == 0) return cudaSuccess;
    const int64_t want = (n8 + 255) / 256;
    const int64_t cap = 8ll * sm_count();
    const int grid = static_cast<int>(want < cap ? want : cap);
    if (p.f16)
        sparse_dkv_convert_kernel<true><<<grid, 256, 0, stream>>>(p, n8);
    else
        sparse_dkv_convert_kernel<false><<<grid, 256, 0, stream>>>(p, n8);
    return cudaGetLastError();
}

cudaError_t launch_sparse_dsink(const SparseProblem& p, cudaStream_t stream) {
    if (!p.sink || p.H == 0) return cudaSuccess;
    sparse_dsink_kernel<<<p.H, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
