// Attention backward (main kernel) for sm_103a: TMA + tcgen05 + TMEM.
//
// One CTA = 128 keys (one K/V tile) of one (batch/sequence, kv head).  It
// walks every q head of the GQA group and every 128-row query tile that can
// see its keys (causal: tiles at or below the diagonal):
//     S^T  = K Q_i^T            (TMEM, 128 x 128 fp32)
//     dP^T = V dO_i^T           (TMEM)
//     P^T  = exp2(min(S^T*scale*log2e + mask - lse2, 0)), with the forward's
//            predicates: partial last key tile, query rows past the
//            sequence, causal pairs, the mask (OpenWAM PR #64: an unmasked
//            partial key tile turns exp(0 - lse) into inf once lse < -88.7).
//            The clamp at 0 holds because P <= 1 (PFCCLab/cudnn-frontend PR #9,
//            section 3).  Hidden entries are 0 by selection.
//     dS^T = P^T o (dP^T - Delta)
//     dV  += P^T dO_i, dK += dS^T Q_i       (TMEM accumulators, no atomics)
//     dQ_i = dS K  -> fp32 bulk tensor reductions into the dQ workspace
// Warps: 0-7 compute (thread = key row = TMEM lane; warps 0-3 take the
// 32-query chunks 0 and 1, warps 4-7 chunks 2 and 3, two chunks at once), then
// read their half of dQ_i out of TMEM (thread = query row) and stage it in
// shared memory; 8 = TMA producer (+ lse2 / Delta vectors); 9 = TMEM allocator
// and UMMA issuer; 10 = issues the dQ reductions and waits for them to read
// the staging, so no compute warp ever blocks on the L2.
// TMEM: dV | dK (D columns each) | S^T | dP^T (128 each).  Chunk c of S^T
// (columns 32c .. 32c+31) is overwritten by its own packed 16-bit (bf16 or fp16,
// the inputs' type) P^T (first 16 columns) and dS^T (last 16) once read, so
// chunks never wait on each other;
// dQ_i = dS K then takes dP^T's columns as one N = D accumulator.
// dV / dK MMAs for chunks 0 and 2 run while chunks 1 and 3 are computed.
// D = 64 (TMEM has 128 spare columns, and the N = 64 dV / dK / dQ products
// hold the tensor pipe for twice their math time): dQ_i has columns of its
// own, dP^T(i+1) is issued once every compute warp has loaded its last dP^T
// chunk, S^T(i+1) once the dV / dK MMAs have read P^T / dS^T, dQ_i after
// them, and the compute warps read dQ_i out after tile i+1's P / dS into an
// fp32 staging tile of its own (dS double-buffered), so dQ_i is off the
// serial chain.
//
// Epilogue (PFCCLab/cudnn-frontend PR #9, section 1): every thread writes its
// dK / dV row into a shared staging tile, fences its own writes for the async
// proxy, the warpgroup meets at a named barrier, ONE thread issues the bulk
// tensor store and only that thread waits on its bulk group, and the group
// meets again before the tile could be reused.  A partial key tile of a
// packed varlen sequence is stored with predicated plain stores instead, so
// the neighbouring sequence's rows are never touched.
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using namespace sm100;

constexpr int kT = 128;
constexpr int kBwdThreads = 352;
constexpr int kWarpProducer = 8, kWarpMma = 9, kWarpReduce = 10;

template <int D>
struct BwdLayout {
    static constexpr int kBlocks = D / 64;
    static constexpr int kTileBytes = kT * D * 2;
    static constexpr int kK = 0;
    static constexpr int kV = kTileBytes;
    static constexpr int kQ = 2 * kTileBytes;           // 2 stages
    static constexpr int kDO = 4 * kTileBytes;          // 2 stages
    // D = 64 (kDefer): the dV/dK/dQ products have N = 64 and run at half rate,
    // so dQ_i leaves the chain: S^T/dP^T of the next tile are issued ahead of
    // it, dQ has TMEM columns of its own, dS is double-buffered, and dQ_i is
    // read out after the next tile's P/dS into an fp32 staging tile of its own.
    static constexpr bool kDefer = (D == 64);
    static constexpr int kDS = 6 * kTileBytes;          // dS as [128 keys][128 q] bf16 ([2] if kDefer)
    static constexpr int kDSBytes = kT * kT * 2;
    static constexpr int kDQS = kDS + (kDefer ? 2 : 1) * kDSBytes;   // kDefer: fp32 dQ staging
    static constexpr int kVec = kDQS + (kDefer ? kT * D * 4 : 0);    // lse2[2][128], delta[2][128]
    static constexpr int kBar = kVec + 4 * kT * 4;
    static constexpr int kBarKV = 0;
    static constexpr int kBarQFull = 1;    // [2]
    static constexpr int kBarQEmpty = 3;   // [2]: dV/dK MMAs done + dQ reduction read the stage
                                           // (kDefer: the MMAs alone)
    static constexpr int kBarSdp = 5;      // S^T and dP^T done
    static constexpr int kBarP = 6;        // [2]: P^T, dS^T of chunks {0, 2} / {1, 3} written
    static constexpr int kBarDQFull = 8;
    static constexpr int kBarDQRead = 9;   // both dQ halves read out of TMEM
    static constexpr int kBarDQStaged = 10;
    static constexpr int kBarAcc = 11;
    static constexpr int kBarDrain = 12;
    static constexpr int kBarDP = 13;      // dP^T done (split schedule; S^T alone on kBarSdp)
    static constexpr int kBarAccRead = 14; // kDefer: the tile's dV/dK MMAs have read P^T / dS^T
    static constexpr int kBarDQSFree = 15; // kDefer: the reduction has read the dQ staging tile
    static constexpr int kBarDPRead = 16;  // kDefer: every compute warp has loaded all its dP^T
    static constexpr int kNumBars = 17;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColDV = 0, kColDK = D, kColS = 2 * D, kColDP = 2 * D + 128;
    static constexpr uint32_t kColDQ = kDefer ? 2 * D + 256 : kColDP;   // dQ: own columns or dP^T's
    static_assert(kColDQ + D <= kTmemCols && kColDP + 128 <= kTmemCols, "TMEM columns");
    static_assert(kBytes <= 232448, "shared memory per CTA");
};

struct BwdMaps {
    CUtensorMap k, v, q, dout, dk, dv, dq_acc;
};

// Debug build (ATTN_POISON_SMEM): fill 16 staging bytes with NaN (all-ones is
// NaN in fp32, bf16 and fp16) right before the real data, so that a consumer
// that reads the tile before the writes land yields non-finite output.
__device__ __forceinline__ void poison16(const void* p) {
#ifdef ATTN_POISON_SMEM
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(smem_u32(p)), "r"(0xffffffffu)
                 : "memory");
#else
    (void)p;
#endif
}

// Write one 32-column chunk of a row into a TMA-layout staging tile
// ([blocks][128 rows][128 B], 16-byte chunks XOR-swizzled by row mod 8).
__device__ __forceinline__ void stage_row_chunk(uint8_t* tile, int row, int col0,
                                                const uint32_t* pk16) {
    const int blk = col0 >> 6;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const int ch = ((col0 & 63) >> 3) + v;
        uint4* dst = reinterpret_cast<uint4*>(tile + blk * 16384 + row * 128 + ((ch ^ (row & 7)) << 4));
        poison16(dst);
        *dst = make_uint4(pk16[4 * v], pk16[4 * v + 1], pk16[4 * v + 2], pk16[4 * v + 3]);
    }
}

// kSplit: S^T and dP^T complete on separate barriers, so that the P^T half of
// the first chunks runs while dP^T is still on the tensor pipe (used at
// D = 128, where it measured 1.5 % faster; at D = 64 it measured 1.3 % slower).
// kMask: a user mask is present (its path is compiled only into that variant).
template <int D, bool F16, bool kMask, bool kSplit>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_sm100_kernel(const Problem p, const __grid_constant__ BwdMaps maps, int with_dq) {
    using L = BwdLayout<D>;
    static_assert(!(L::kDefer && kSplit), "the deferred dQ schedule has one S^T/dP^T barrier");
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::kBar + 8u * i; };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
    float* vec = reinterpret_cast<float*>(smem + L::kVec);   // -lse2[s][128] at s*256, -delta at +128

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, hk = blockIdx.y;
    const int n0 = blockIdx.x * kT;
    const SeqInfo si = seq_info(p, b);
    if (!si.ok || n0 >= si.len_k) return;
    if ((sbase & 1023u) != 0) {            // swizzle atoms need 1 KiB alignment
        if (tid == 0) set_error(p.err, DEV_E_INTERNAL);
        return;
    }

    const int mt_first = p.causal ? n0 / kT : 0;
    const int mt_count = (si.len_q + kT - 1) / kT;
    const int per_head = max(mt_count - mt_first, 0);
    const int n_iter = per_head * p.G;
    const int row_base = si.row0;
    const int bcoord = p.varlen ? 0 : b;

    if (tid == 0) {
        for (int i = 0; i < L::kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == L::kBarQFull || i == L::kBarQFull + 1) cnt = 33;
            // q_empty: the MMAs' commit + the reduction issuer once the stage was read
            if (i == L::kBarQEmpty || i == L::kBarQEmpty + 1) cnt = L::kDefer ? 1 : 2;
            if (i == L::kBarP || i == L::kBarP + 1) cnt = 256;
            if (i == L::kBarDQRead || i == L::kBarDQStaged || i == L::kBarDPRead) cnt = 256;
            mbar_init(bar(i), cnt);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    // Each CTA starts its walk at a different (head, query tile): CTAs that run
    // at the same time then reduce into different dQ rows instead of all
    // hammering the same L2 lines.
    const int rot = n_iter > 0 ? static_cast<int>(blockIdx.x % n_iter) : 0;
    // Byte offset of fp32 dQ staging block `blk` (32 columns): inside query/dO
    // stage `s`, or (kDefer) in the staging tile of its own.
    auto dq_stage_off = [&](int blk, int s) {
        if constexpr (L::kDefer) return L::kDQS + blk * 16384;
        return ((blk & 1) ? L::kDO : L::kQ) + s * L::kTileBytes + (blk >> 1) * 16384;
    };
    auto iter_tile = [&](int it, int* h, int* m0) {
        int itr = it + rot;
        if (itr >= n_iter) itr -= n_iter;
        const int gi = itr / per_head;
        *m0 = (mt_first + itr % per_head) * kT;
        *h = hk * p.G + gi;
    };

    if (warp == kWarpProducer) {
        // ------------------------------------------------------------ producer (whole warp)
        bool ok = true;
        if (lane == 0) {
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(&maps.q);
            mbar_arrive_expect_tx(bar(L::kBarKV), 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kBlocks; ++c) {
                tma_load_4d(sbase + L::kK + c * 16384, &maps.k, 64 * c, hk, row_base + n0, bcoord,
                            bar(L::kBarKV));
                tma_load_4d(sbase + L::kV + c * 16384, &maps.v, 64 * c, hk, row_base + n0, bcoord,
                            bar(L::kBarKV));
            }
        }
        int issued = 0;
        for (int it = 0; it < n_iter; ++it) {
            const int s = it & 1, r = it >> 1;
            int h, m0;
            iter_tile(it, &h, &m0);
            // this tile's -lse2 / -Delta to registers before the wait for the
            // stage, so that their latency overlaps it
            float nlv[4], ndv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = m0 + 4 * lane + e;
                const int64_t li = b * p.lse_b + h * p.lse_h + row_base + i;
                const bool in = i < si.len_q;
                nlv[e] = in ? -p.lse2[li] : 0.f;     // both stored negated
                ndv[e] = in ? -p.delta[li] : 0.f;
            }
            ok = mbar_wait(bar(L::kBarQEmpty + s), (r & 1) ^ 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            // every query tile starts inside the sequence, every head inside the group
            if (lane == 0 && dbg_check(m0 < si.len_q && h >= hk * p.G && h < (hk + 1) * p.G, p.err)) {
                mbar_arrive_expect_tx(bar(L::kBarQFull + s), 2 * L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kBlocks; ++c) {
                    tma_load_4d(sbase + L::kQ + s * L::kTileBytes + c * 16384, &maps.q, 64 * c, h,
                                row_base + m0, bcoord, bar(L::kBarQFull + s));
                    tma_load_4d(sbase + L::kDO + s * L::kTileBytes + c * 16384, &maps.dout, 64 * c,
                                h, row_base + m0, bcoord, bar(L::kBarQFull + s));
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                vec[s * 256 + 4 * lane + e] = nlv[e];
                vec[s * 256 + 128 + 4 * lane + e] = ndv[e];
            }
            mbar_arrive(bar(L::kBarQFull + s));
            issued = it + 1;
        }
        if (*abort_flag && lane == 0) {
            volatile int no_abort = 0;
            mbar_wait(bar(L::kBarKV), 0, &no_abort, kDrainBudgetNs);
            for (int it = max(0, issued - 2); it < issued; ++it)
                mbar_wait(bar(L::kBarQFull + (it & 1)), (it >> 1) & 1, &no_abort, kDrainBudgetNs);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t id_sdp = idesc_f16kind(128, 128, 0, 0, F16);    // S^T, dP^T
            constexpr uint32_t id_acc = idesc_f16kind(128, D, 0, 1, F16);      // dV, dK (B MN-major)
            constexpr uint32_t id_dq = idesc_f16kind(128, D, 1, 1, F16);       // dQ (A, B MN-major)
            const uint32_t tS = tmem + L::kColS, tDP = tmem + L::kColDP;
            const uint32_t tDV = tmem + L::kColDV, tDK = tmem + L::kColDK;
            const uint64_t k_k = smem_desc(sbase + L::kK, 16, 1024, kSwizzle128B);
            const uint64_t v_k = smem_desc(sbase + L::kV, 16, 1024, kSwizzle128B);
            const uint64_t k_mn = smem_desc(sbase + L::kK, 16384, 1024, kSwizzle128B);
            const uint64_t ds_mn0 = smem_desc(sbase + L::kDS, 16384, 1024, kSwizzle128B);
            bool ok = mbar_wait(bar(L::kBarKV), 0, abort_flag);
            dbg_check(L::kColDP + 128 <= L::kTmemCols && L::kColDK + D <= L::kColS, p.err);
            for (int it = 0; ok && it < n_iter; ++it) {
                const int s = it & 1, r = it >> 1;
                if (!(ok = dbg_stall(p.debug_stall, kStallBwd, it, bar(L::kBarDrain), abort_flag))) break;
                const uint32_t qa = sbase + L::kQ + s * L::kTileBytes;
                const uint32_t da = sbase + L::kDO + s * L::kTileBytes;
                const uint64_t q_mn = smem_desc(qa, 16384, 1024, kSwizzle128B);  // MN-major
                const uint64_t do_mn = smem_desc(da, 16384, 1024, kSwizzle128B);
                // S^T = K Q^T and dP^T = V dO^T of the tile in stage `sn` (K-major Q / dO)
                auto issue_s = [&](int sn) {
                    const uint64_t q_k = smem_desc(sbase + L::kQ + sn * L::kTileBytes, 16, 1024, kSwizzle128B);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_ss(tS, desc_add(k_k, off), desc_add(q_k, off), id_sdp, kk > 0);
                    }
                };
                auto issue_dp = [&](int sn) {
                    const uint64_t do_k = smem_desc(sbase + L::kDO + sn * L::kTileBytes, 16, 1024, kSwizzle128B);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_ss(tDP, desc_add(v_k, off), desc_add(do_k, off), id_sdp, kk > 0);
                    }
                };
                if (!L::kDefer || it == 0) {
                    if (!(ok = mbar_wait(bar(L::kBarQFull + s), r & 1, abort_flag))) break;
                    // S^T / dP^T columns are free once the previous dQ has been read out
                    // (its commit covered every earlier MMA, including dV and dK).
                    if (it > 0 && !(ok = mbar_wait(bar(L::kBarDQRead), (it - 1) & 1, abort_flag))) break;
                    tc_fence_after();
                    issue_s(s);
                    if constexpr (kSplit) mma_commit(bar(L::kBarSdp));
                    issue_dp(s);
                    mma_commit(bar(kSplit ? L::kBarDP : L::kBarSdp));
                }
                // dV += P^T dO, dK += dS^T Q as the chunks arrive: phase 0 covers
                // chunks 0 and 2, phase 1 chunks 1 and 3 (16 queries = 8 packed
                // columns per step; P^T at 32c, dS^T at 32c + 16).
#pragma unroll
                for (int ph = 0; ph < 2; ++ph) {
                    if (L::kDefer && ph == 1 && it + 1 < n_iter) {
                        // the next tile's dP^T while this tile's second chunks are
                        // worked on, once every compute warp has loaded its dP^T
                        const int s1 = (it + 1) & 1;
                        if (!(ok = mbar_wait(bar(L::kBarDPRead), it & 1, abort_flag))) break;
                        if (!(ok = mbar_wait(bar(L::kBarQFull + s1), ((it + 1) >> 1) & 1, abort_flag))) break;
                        tc_fence_after();
                        issue_dp(s1);
                    }
                    if (!(ok = mbar_wait(bar(L::kBarP + ph), it & 1, abort_flag))) break;
                    tc_fence_after();
#pragma unroll
                    for (int cq = 0; cq < 2; ++cq) {
                        const int c = ph + 2 * cq;
#pragma unroll
                        for (int kq = 0; kq < 2; ++kq) {
                            const int kk = 2 * c + kq;
                            const uint32_t acc = (it > 0 || ph > 0 || cq > 0 || kq > 0) ? 1u : 0u;
                            mma_ts(tDV, tS + 32 * c + 8 * kq, desc_add(do_mn, kk * 2048), id_acc, acc);
                            mma_ts(tDK, tS + 32 * c + 16 + 8 * kq, desc_add(q_mn, kk * 2048), id_acc, acc);
                        }
                    }
                }
                if (!ok) break;
                mma_commit(bar(L::kBarQEmpty + s));
                {
                    if (L::kDefer && it + 1 < n_iter) {
                        // the next tile's S^T once the dV/dK MMAs have read P^T / dS^T
                        // out of the S^T columns (its dP^T is already issued)
                        mma_commit(bar(L::kBarAccRead));
                        if (!(ok = mbar_wait(bar(L::kBarAccRead), it & 1, abort_flag))) break;
                        tc_fence_after();
                        issue_s((it + 1) & 1);
                        mma_commit(bar(L::kBarSdp));
                    }
                }
                if (with_dq) {
                    // dQ's columns: dP^T's (every compute warp has read them) or
                    // (kDefer) its own, once the previous dQ has been read out
                    if (L::kDefer && it > 0 &&
                        !(ok = mbar_wait(bar(L::kBarDQRead), (it - 1) & 1, abort_flag)))
                        break;
                    tc_fence_after();
                    const uint64_t ds_mn = desc_add(ds_mn0, L::kDefer ? (it & 1) * L::kDSBytes : 0);
#pragma unroll
                    for (int kk = 0; kk < kT / 16; ++kk)
                        mma_ss(tmem + L::kColDQ, desc_add(ds_mn, kk * 2048), desc_add(k_mn, kk * 2048), id_dq,
                               kk > 0);
                }
                mma_commit(bar(L::kBarDQFull));
            }
            mma_commit(bar(L::kBarAcc));
            if (!ok) {
                mma_commit(bar(L::kBarDrain));
                volatile int no_abort = 0;
                mbar_wait(bar(L::kBarDrain), 0, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else if (warp == kWarpReduce) {
        // ------------------------------------------------------------ dQ reduction issuer
        // Reduce each staged dQ_i into the fp32 workspace with bulk tensor
        // reductions; the stage (kDefer: the staging tile) is released once
        // they have read it.
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; ok && it < n_iter; ++it) {
                const int s = it & 1;
                if (!(ok = mbar_wait(bar(L::kBarDQStaged), it & 1, abort_flag))) break;
                if (with_dq) {
                    int h, m0;
                    iter_tile(it, &h, &m0);
                    const int acc_row = static_cast<int>(b * p.acc_b) + row_base + m0;
#pragma unroll
                    for (int blk = 0; blk < D / 32; ++blk)
                        tma_reduce_add_3d(&maps.dq_acc, sbase + dq_stage_off(blk, s), 32 * blk, h,
                                          acc_row);
                    bulk_commit();
                    bulk_wait_read_all();          // only the committing thread may wait
                }
                mbar_arrive(bar(L::kDefer ? L::kBarDQSFree : L::kBarQEmpty + s));
            }
        }
        __syncwarp();
        named_bar_sync(3, 160);    // warps 4-7 may reuse query stage 0 for the dK epilogue
    } else {
        // ------------------------------------------------------------ compute (warps 0-7)
        const int wq = warp & 3;                    // TMEM lane quarter
        const int hq = warp >> 2;                   // query half (P^T / dS^T), d half (dQ)
        const int r = wq * 32 + lane;               // key row = TMEM lane (dQ: query row)
        const int j = n0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + L::kColS;
        const uint32_t tDP = tmem + lane_off + L::kColDP;
        uint8_t* ds_tile = smem + L::kDS;
        bool ok = true;
        // dQ_i: this warp's D/2 columns for its 32 query rows, out of TMEM,
        // then staged as fp32 in tile i's query/dO stage (every MMA that read
        // the stage has completed once dq_full fires) or, with kDefer, in the
        // staging tile of its own once the reduction has read dQ_{i-1} there.
        auto read_out_dq = [&](int i) {
            if (ok) {
                ok = mbar_wait(bar(L::kBarDQFull), i & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (!ok) return;
            tc_fence_after();
            uint32_t dq[D / 2];
            if (with_dq) {
                const uint32_t src = tmem + lane_off + L::kColDQ + hq * (D / 2);
                if constexpr (D == 128) {
                    tmem_ld32x2(src, dq, src + 32, dq + 32);
                } else {
                    tmem_ld32(src, dq);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(L::kBarDQRead));
            if (L::kDefer && with_dq && i > 0) {
                ok = mbar_wait(bar(L::kBarDQSFree), (i - 1) & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) return;
            }
#pragma unroll
            for (int bb = 0; bb < D / 64; ++bb) {
                if (with_dq) {
                    // fp32 staging: 32-column blocks of [128 rows][128 B], 16-byte
                    // chunks swizzled; even blocks in the query stage, odd in the dO stage.
                    const int off = dq_stage_off(hq * (D / 64) + bb, i & 1) + r * 128;
                    // the fp32 staging row lies inside tile i's query / dO stage or
                    // the staging tile
                    constexpr int lo = L::kDefer ? L::kDQS : L::kQ;
                    constexpr int hi = L::kDefer ? L::kVec : L::kDS;
                    if (!dbg_check(off >= lo && off + 128 <= hi, p.err)) continue;
                    uint8_t* base = smem + off;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        poison16(base + ((k ^ (r & 7)) << 4));
                        *reinterpret_cast<uint4*>(base + ((k ^ (r & 7)) << 4)) =
                            make_uint4(dq[32 * bb + 4 * k], dq[32 * bb + 4 * k + 1],
                                       dq[32 * bb + 4 * k + 2], dq[32 * bb + 4 * k + 3]);
                    }
                }
            }
            if (with_dq) fence_proxy_async_smem();   // each writer: its stores -> async proxy
            mbar_arrive(bar(L::kBarDQStaged));
        };
        for (int it = 0; it < n_iter; ++it) {
            const int s = it & 1;
            int h, m0;
            iter_tile(it, &h, &m0);
            const float* lse2 = vec + s * 256;
            const bool pred = (n0 + kT > si.len_k) || (m0 + kT > si.len_q) ||
                              (p.causal && n0 + kT - 1 > m0) || kMask;
            // After a wait gives up, `ok` stays false: the warp skips the work
            // but still meets every named barrier, so none is left short.
            if (ok) {
                // q_full[s] also publishes the producer's lse2 / Delta vectors.
                ok = mbar_wait(bar(L::kBarQFull + s), (it >> 1) & 1, abort_flag) &&
                     mbar_wait(bar(L::kBarSdp), it & 1, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
            }
            if (ok) {
                tc_fence_after();
                if constexpr (kMask) {
                    // With a user mask, rewrite this warp's chunks of S^T in TMEM as
                    // finished logits first (mask loads in the main loop would spill).
#pragma unroll 1
                    for (int cc = 0; cc < 2; ++cc) {
                        const int c = 2 * hq + cc;
                        uint32_t v[32];
                        tmem_ld32(tS + 32 * c, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(logit_log2(p, __uint_as_float(v[e]), b, h,
                                                              m0 + 32 * c + e, j, si.len_q, si.len_k));
                        tmem_st32(tS + 32 * c, v);
                    }
                    tmem_wait_st();
                }
                bool dp_ready = !kSplit;
#pragma unroll 1
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * hq + cc;
                    uint32_t sv[32], dv[32];
                    if constexpr (kSplit) {
                        tmem_ld32(tS + 32 * c, sv);
                    } else {
                        tmem_ld32x2(tS + 32 * c, sv, tDP + 32 * c, dv);
                        if (L::kDefer && cc == 1) {
                            // this warp's last dP^T chunk is in registers: the next
                            // tile's dP^T may overwrite the columns
                            tc_fence_before();
                            mbar_arrive(bar(L::kBarDPRead));
                        }
                    }
                    // -lse2 / -Delta of this chunk's query rows, four at a time, one
                    // group ahead of use (16-byte shared loads, every lane the same
                    // address): loading all 32 up front costs 64 live registers.
                    const uint32_t va = smem_u32(lse2 + 32 * c);
                    uint32_t pk[16], dk[16];
                    // Phase A: P^T = exp2(min(x - lse2, 0)), kept in sv as fp32 and
                    // packed into pk; hidden entries are exactly 0.
                    if (!kSplit && !pred && !kMask) {
                        // one pass: P^T and dS^T together (dP^T is already loaded)
                        const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
                        float4 lv = lds128(va), dl = lds128(va + 512), lvn, dln;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            if ((e & 3) == 0 && e + 4 < 32) {
                                lvn = lds128(va + 4 * e + 16);
                                dln = lds128(va + 512 + 4 * e + 16);
                            }
                            const float2 l2 = (e & 2) ? make_float2(lv.z, lv.w) : make_float2(lv.x, lv.y);
                            const float2 nd2 = (e & 2) ? make_float2(dl.z, dl.w) : make_float2(dl.x, dl.y);
                            const float2 x2 = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                    c2, l2);
                            const float p0 = ex2(fminf(x2.x, 0.f));
                            const float p1 = ex2(fminf(x2.y, 0.f));
                            const float2 d2 = fadd2(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                                    nd2);
                            const float2 ds2 = fmul2(make_float2(p0, p1), d2);
                            pk[e >> 1] = pack2<F16>(p0, p1);
                            dk[e >> 1] = pack2<F16>(ds2.x, ds2.y);
                            if ((e & 3) == 2) {
                                lv = lvn;
                                dl = dln;
                            }
                        }
                    } else if (!pred && !kMask) {
                        const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
                        float4 lv = lds128(va), lvn;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            if ((e & 3) == 0 && e + 4 < 32) lvn = lds128(va + 4 * e + 16);
                            const float2 l2 = (e & 2) ? make_float2(lv.z, lv.w) : make_float2(lv.x, lv.y);
                            // packed pair: x - lse2 = s*c + (-lse2)
                            const float2 x2 = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                    c2, l2);
                            const float p0 = ex2(fminf(x2.x, 0.f));
                            const float p1 = ex2(fminf(x2.y, 0.f));
                            sv[e] = __float_as_uint(p0);
                            sv[e + 1] = __float_as_uint(p1);
                            pk[e >> 1] = pack2<F16>(p0, p1);
                            if ((e & 3) == 2) lv = lvn;
                        }
                    } else if (!kMask) {
                        // keys past the sequence, query rows past it, causal pairs
                        const int qlo = p.causal ? j - m0 : -1;          // visible: q >= qlo
                        const int qhi = (j < si.len_k) ? si.len_q - m0 : 0;  // visible: q < qhi
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float pr[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int q = 32 * c + e + u;
                                const bool vis = q >= qlo && q < qhi;
                                const float x = __uint_as_float(sv[e + u]) * p.scale_log2;
                                const float pv = ex2(fminf(x + lds32(va + 4 * (e + u)), 0.f));
                                pr[u] = vis ? pv : 0.f;
                                sv[e + u] = __float_as_uint(pr[u]);
                            }
                            pk[e >> 1] = pack2<F16>(pr[0], pr[1]);
                        }
                    } else {
                        // mask: S^T already holds the finished log2-domain logits
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float pr[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const float x = __uint_as_float(sv[e + u]);
                                const bool vis = x != -INFINITY;
                                const float pv = ex2(fminf(x + lds32(va + 4 * (e + u)), 0.f));
                                pr[u] = vis ? pv : 0.f;
                                sv[e + u] = __float_as_uint(pr[u]);
                            }
                            pk[e >> 1] = pack2<F16>(pr[0], pr[1]);
                        }
                    }
                    if constexpr (kSplit) {
                        if (!dp_ready) {
                            // dP^T of this iteration (the first chunk waits for both)
                            bool okd = mbar_wait(bar(L::kBarDP), it & 1, abort_flag);
                            if (!__all_sync(0xffffffffu, okd)) {
                                ok = false;
                                break;
                            }
                            dp_ready = true;
                            tc_fence_after();
                        }
                        tmem_ld32(tDP + 32 * c, dv);
                    }
                    // Phase B: dS^T = P^T o (dP^T - Delta); hidden entries stay exactly 0.
                    if (!kSplit && !pred && !kMask) {
                        // done in the one-pass loop above
                    } else if (!pred && !kMask) {
                        float4 dl = lds128(va + 512), dln;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            if ((e & 3) == 0 && e + 4 < 32) dln = lds128(va + 512 + 4 * e + 16);
                            const float2 nd2 = (e & 2) ? make_float2(dl.z, dl.w) : make_float2(dl.x, dl.y);
                            const float2 d2 = fadd2(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                                    nd2);
                            const float2 ds2 = fmul2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), d2);
                            dk[e >> 1] = pack2<F16>(ds2.x, ds2.y);
                            if ((e & 3) == 2) dl = dln;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float ds[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const float pr = __uint_as_float(sv[e + u]);
                                const float nd = lds32(va + 512 + 4 * (e + u));
                                ds[u] = pr != 0.f ? pr * (__uint_as_float(dv[e + u]) + nd) : 0.f;
                            }
                            dk[e >> 1] = pack2<F16>(ds[0], ds[1]);
                        }
                    }
                    tmem_st16(tS + 32 * c, pk);
                    tmem_st16(tS + 32 * c + 16, dk);
                    if (with_dq) stage_row_chunk(ds_tile + (L::kDefer ? (it & 1) * L::kDSBytes : 0), r, 32 * c, dk);
                    tmem_wait_st();
                    fence_proxy_async_smem();      // dS in shared memory -> the dQ MMA
                    tc_fence_before();
                    mbar_arrive(bar(L::kBarP + cc));
                }
            }
            // dQ of this tile (kDefer: of the previous one, after this tile's P/dS)
            if (!L::kDefer || it > 0) read_out_dq(L::kDefer ? it - 1 : it);
        }
        if (L::kDefer && n_iter > 0) read_out_dq(n_iter - 1);
        // Epilogue: warps 0-3 store dV (staging tile = the dS buffer), warps 4-7
        // dK (staging tile = query stage 0, free once the reduction issuer has
        // seen its last reduction read it).  Both need every MMA done.
        const int nb = hq ? 2 : 1;                   // named barrier of this warpgroup
        if (hq) named_bar_sync(3, 160);
        if (ok) {
            ok = mbar_wait(bar(L::kBarAcc), 0, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        {
            if (ok) tc_fence_after();
            uint8_t* tile = hq ? smem + L::kQ : ds_tile;
            const uint32_t tile_addr = sbase + (hq ? L::kQ : L::kDS);
            const uint32_t col = hq ? L::kColDK : L::kColDV;
            const float mul = hq ? p.scale : 1.f;    // dK = scale * dS^T Q
            const bool tma_path = !p.varlen || n0 + kT <= si.len_k;
            bf16* grow = (hq ? p.dk : p.dv) + b * p.dk_b + static_cast<int64_t>(row_base + j) * p.dk_s +
                         hk * p.dk_h;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (ok && n_iter > 0) {
                    tmem_ld32(tmem + lane_off + col + 32 * c, o);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    pk[e] = pack2<F16>(__uint_as_float(o[2 * e]) * mul,
                                      __uint_as_float(o[2 * e + 1]) * mul);
                if (!ok) {
                } else if (tma_path) {
                    if (dbg_check(r < kT && 32 * c < D, p.err)) stage_row_chunk(tile, r, 32 * c, pk);
                } else if (j < si.len_k) {
                    uint4* dst = reinterpret_cast<uint4*>(grow + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (tma_path) {
                if (ok) fence_proxy_async_smem();   // each writer: its stores -> async proxy
                named_bar_sync(nb, 128);            // all 128 rows are in the staging tile
                if (ok && r == 0) {
#pragma unroll
                    for (int c = 0; c < L::kBlocks; ++c)
                        tma_store_4d(hq ? &maps.dk : &maps.dv, tile_addr + c * 16384, 64 * c, hk,
                                     row_base + n0, bcoord);
                    bulk_commit();
                    bulk_wait_read_all();   // only the committing thread may wait
                }
                named_bar_sync(nb, 128);    // staging tile no longer read
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    if (tid == 0 && *abort_flag) set_error(p.err, DEV_E_TIMEOUT);
}

// ------------------------------------------------------------------ host side

template <int D, bool F16, bool kMask, bool kSplit>
cudaError_t launch_bwd_sm100_v(const Problem& p, bool with_dq, cudaStream_t stream) {
    using L = BwdLayout<D>;
    if (p.B == 0 || p.Sk == 0) return cudaSuccess;
    const int64_t Sq = p.varlen ? p.T : p.Sq;
    const int64_t Sk = p.varlen ? p.T : p.Sk;
    const int64_t Bm = p.varlen ? 1 : p.B;
    // With no queries the maps are never read; keep them legal by pointing at k.
    const bool no_q = Sq == 0;
    BwdMaps maps;
    bool ok = make_tile_map(&maps.k, p.k, D, p.Hkv, Sk, Bm, p.k_h, p.k_s, p.k_b, F16) &&
              make_tile_map(&maps.v, p.v, D, p.Hkv, Sk, Bm, p.v_h, p.v_s, p.v_b, F16) &&
              make_tile_map(&maps.q, no_q ? p.k : p.q, D, no_q ? p.Hkv : p.Hq, no_q ? Sk : Sq, Bm,
                       no_q ? p.k_h : p.q_h, no_q ? p.k_s : p.q_s, no_q ? p.k_b : p.q_b, F16) &&
              make_tile_map(&maps.dout, no_q ? p.k : p.dout, D, no_q ? p.Hkv : p.Hq, no_q ? Sk : Sq, Bm,
                       no_q ? p.k_h : p.do_h, no_q ? p.k_s : p.do_s, no_q ? p.k_b : p.do_b, F16) &&
              make_tile_map(&maps.dk, p.dk, D, p.Hkv, Sk, Bm, p.dk_h, p.dk_s, p.dk_b, F16) &&
              make_tile_map(&maps.dv, p.dv, D, p.Hkv, Sk, Bm, p.dk_h, p.dk_s, p.dk_b, F16);
    if (with_dq) {
        const int64_t rows = p.varlen ? p.T : static_cast<int64_t>(p.B) * p.Sq;
        ok = ok && make_f32_reduce_map(&maps.dq_acc, p.dq_acc, D, p.Hq, rows);
    } else {
        maps.dq_acc = maps.k;   // never read without dQ
    }
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_sm100_kernel<D, F16, kMask, kSplit>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sk + kT - 1) / kT, p.Hkv, p.B);
    bwd_sm100_kernel<D, F16, kMask, kSplit><<<grid, kBwdThreads, L::kBytes, stream>>>(
        p, maps, with_dq ? 1 : 0);
    return cudaGetLastError();
}

template <int D, bool F16, bool kMask>
cudaError_t launch_bwd_sm100_d(const Problem& p, bool with_dq, cudaStream_t stream) {
    return launch_bwd_sm100_v<D, F16, kMask, D == 128>(p, with_dq, stream);
}

}  // namespace

cudaError_t launch_bwd_main(const Problem& p, bool with_dq_atomics, cudaStream_t stream) {
    const bool m = p.mask_kind != MASK_NONE;
    const bool w = with_dq_atomics;
    if (p.f16) {
        if (m) return p.D == 64 ? launch_bwd_sm100_d<64, true, true>(p, w, stream)
                                : launch_bwd_sm100_d<128, true, true>(p, w, stream);
        return p.D == 64 ? launch_bwd_sm100_d<64, true, false>(p, w, stream)
                         : launch_bwd_sm100_d<128, true, false>(p, w, stream);
    }
    if (m) return p.D == 64 ? launch_bwd_sm100_d<64, false, true>(p, w, stream)
                            : launch_bwd_sm100_d<128, false, true>(p, w, stream);
    return p.D == 64 ? launch_bwd_sm100_d<64, false, false>(p, w, stream)
                     : launch_bwd_sm100_d<128, false, false>(p, w, stream);
}

}  // namespace attn
