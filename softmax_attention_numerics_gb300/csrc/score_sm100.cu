// Attention targets recomputed from the forward's lse and summed over the
// query heads, for sm_103a: TMA + tcgen05 + TMEM (PFCCLab/cudnn-frontend PR #9,
// sections 2 and 3: the dense score recompute that feeds a sparse-attention
// indexer's training targets).
//
//     score_ij = sum_h exp2(min(s_hij * scale * log2 e - lse_hi * log2 e, 120))
//     l1_i     = sum_j score_ij
//
// The clamp at 120 bounds every term by 2^120, so a sum over 64 heads stays
// finite (2^120 * 64 < FLT_MAX) even when an lse is far too small (section 3);
// with the forward's own lse it never fires.  Hidden pairs (causal j > i,
// keys past the sequence) contribute exactly 0.
//
// One CTA = a 128 x 128 (query, key) tile of one batch / sequence; it loops
// over the query heads:
//   warp 8   TMA producer: Q_h tiles through a 4-stage ring, the K tile of
//            each kv head through a 2-stage one (q heads of a GQA group share it)
//   warp 9   TMEM allocator and single-thread UMMA issuer: S_h = Q_h K^T into
//            TMEM buffer h & 1
//   warps 0-3 / 4-7  key columns 0-63 / 64-127 of every head: thread = query
//            row = TMEM lane, its 64 terms accumulated in registers; one
//            TMEM load per head, and both warpgroups release the buffer
// Each thread stores its row's 64 sums from registers (rows past the sequence
// are never written).  Each CTA writes its rows' partial L1 norm for this key
// tile; l1_reduce_kernel adds the partials of a row in key-tile order, so both
// outputs are bit-reproducible.
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using namespace sm100;

constexpr int kScThreads = 320;
constexpr int kSt = 128;                 // query and key tile
constexpr float kScoreClamp = 120.0f;    // log2 units

template <int D>
struct ScLayout {
    static constexpr int kBlocks = D / 64;
    static constexpr int kTileBytes = kSt * D * 2;
    static constexpr int kQStages = 4;                   // a Q_h tile per head: keep loads ahead
    static constexpr int kQ = 0;
    static constexpr int kK = kQStages * kTileBytes;     // 2 stages
    static constexpr int kHalf = kK + 2 * kTileBytes;    // fp32 [128]: odd half-row sums
    static constexpr int kBar = kHalf + kSt * 4;
    static constexpr int kBarQFull = 0, kBarQEmpty = kQStages, kBarKFull = 2 * kQStages;
    static constexpr int kBarKEmpty = kBarKFull + 2, kBarSFull = kBarKEmpty + 2;
    static constexpr int kBarSFree = kBarSFull + 2, kBarDrain = kBarSFree + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16 + 1024;     // + alignment slack
    static_assert(kBytes <= 232448, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 256;
};

struct ScoreMaps {
    CUtensorMap q, k;
};

// Zeros for rows [m0, m0 + 128) x columns [n0, n0 + 128) of the score (a tile
// with no visible pair); warp w writes rows 16w .. 16w + 15, lane l columns
// 4l .. 4l + 3.
__device__ __forceinline__ void store_zero_tile(const Problem& p, int b, int row_base, int m0, int n0,
                                                int len_q, int warp, int lane) {
    const int64_t W = p.sc_w;
    const int64_t rb = p.varlen ? row_base : static_cast<int64_t>(b) * p.Sq;
    for (int rr = 0; rr < 16; ++rr) {
        const int row = warp * 16 + rr;
        if (m0 + row >= len_q) break;
        float* dst = p.score + (rb + m0 + row) * W;
        const int c0 = n0 + 4 * lane;
        if (c0 + 3 < W && (W & 3) == 0) {
            *reinterpret_cast<float4*>(dst + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c0 + u < W) dst[c0 + u] = 0.f;
        }
    }
}

template <int D, bool F16>
__global__ void __launch_bounds__(kScThreads, 1)
    score_sm100_kernel(const Problem p, const __grid_constant__ ScoreMaps maps) {
    using L = ScLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::kBar + 8u * i; };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
    float* half_sum = reinterpret_cast<float*>(smem + L::kHalf);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z;
    const int m0 = blockIdx.y * kSt, n0 = blockIdx.x * kSt;
    const SeqInfo si = seq_info(p, b);
    if (!si.ok || m0 >= si.len_q) return;                 // rows of another sequence
    const int row_base = si.row0;
    const int bcoord = p.varlen ? 0 : b;
    const int nrow = min(kSt, si.len_q - m0);
    const int64_t part_row = p.varlen ? row_base + m0 : static_cast<int64_t>(b) * p.Sq + m0;
    float* part = p.l1_part + static_cast<int64_t>(blockIdx.x) * p.l1_rows + part_row;

    // A tile with no visible pair (keys past the sequence, or wholly above
    // the causal diagonal) is written as zeros.
    if (n0 >= si.len_k || (p.causal && n0 > m0 + kSt - 1)) {
        if (warp < 8) store_zero_tile(p, b, row_base, m0, n0, si.len_q, warp, lane);
        for (int r = tid; r < nrow; r += kScThreads) part[r] = 0.f;
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < L::kNumBars; ++i)
            mbar_init(bar(i), (i == L::kBarSFree || i == L::kBarSFree + 1) ? 256 : 1);
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
    const int H = p.Hq, G = p.G;

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.k);
            int q_issued = 0, k_issued = 0;
            for (int h = 0; h < H && !*abort_flag; ++h) {
                if (h % G == 0) {
                    const int kv = h / G, ks = kv & 1;
                    if (!mbar_wait(bar(L::kBarKEmpty + ks), ((kv >> 1) & 1) ^ 1, abort_flag)) break;
                    if (!dbg_check(kv < p.Hkv, p.err)) break;
                    mbar_arrive_expect_tx(bar(L::kBarKFull + ks), L::kTileBytes);
#pragma unroll
                    for (int c = 0; c < L::kBlocks; ++c)
                        tma_load_4d(sbase + L::kK + ks * L::kTileBytes + c * 16384, &maps.k, 64 * c, kv,
                                    row_base + n0, bcoord, bar(L::kBarKFull + ks));
                    k_issued = kv + 1;
                }
                const int s = h % L::kQStages, qr = h / L::kQStages;
                if (!mbar_wait(bar(L::kBarQEmpty + s), (qr & 1) ^ 1, abort_flag)) break;
                mbar_arrive_expect_tx(bar(L::kBarQFull + s), L::kTileBytes);
#pragma unroll
                for (int c = 0; c < L::kBlocks; ++c)
                    tma_load_4d(sbase + L::kQ + s * L::kTileBytes + c * 16384, &maps.q, 64 * c, h,
                                row_base + m0, bcoord, bar(L::kBarQFull + s));
                q_issued = h + 1;
            }
            if (*abort_flag) {
                // Let the copies in flight land before the CTA exits.
                volatile int no_abort = 0;
                for (int h = max(0, q_issued - L::kQStages); h < q_issued; ++h)
                    mbar_wait(bar(L::kBarQFull + h % L::kQStages), (h / L::kQStages) & 1, &no_abort,
                              kDrainBudgetNs);
                for (int kv = max(0, k_issued - 2); kv < k_issued; ++kv)
                    mbar_wait(bar(L::kBarKFull + (kv & 1)), (kv >> 1) & 1, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16kind(128, 128, 0, 0, F16);
            bool ok = true;
            for (int h = 0; ok && h < H; ++h) {
                if (!(ok = dbg_stall(p.debug_stall, kStallScore, h, bar(L::kBarDrain), abort_flag))) break;
                const int s = h % L::kQStages, kv = h / G, ks = kv & 1, buf = h & 1;
                if (!(ok = mbar_wait(bar(L::kBarQFull + s), (h / L::kQStages) & 1, abort_flag))) break;
                if (!(ok = mbar_wait(bar(L::kBarKFull + ks), (kv >> 1) & 1, abort_flag))) break;
                // buffer `buf` is free once both warpgroups have read head h - 2
                if (h >= 2 && !(ok = mbar_wait(bar(L::kBarSFree + buf), ((h >> 1) - 1) & 1, abort_flag)))
                    break;
                tc_fence_after();
                const uint64_t qd = smem_desc(sbase + L::kQ + s * L::kTileBytes, 16, 1024, kSwizzle128B);
                const uint64_t kd = smem_desc(sbase + L::kK + ks * L::kTileBytes, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(tmem + 128 * buf, desc_add(qd, off), desc_add(kd, off), idesc, kk > 0);
                }
                mma_commit(bar(L::kBarSFull + buf));
                mma_commit(bar(L::kBarQEmpty + s));                  // Q_h consumed
                if (h % G == G - 1 || h == H - 1) mma_commit(bar(L::kBarKEmpty + ks));
            }
            if (!ok) {
                mma_commit(bar(L::kBarDrain));
                volatile int no_abort = 0;
                mbar_wait(bar(L::kBarDrain), 0, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ head sums (warps 0-7)
        const int wg = warp >> 2, wq = warp & 3;
        const int row = wq * 32 + lane;
        const int i = m0 + row;                              // query row in the sequence
        const bool row_in = i < si.len_q;
        const int c0 = 64 * wg;                              // this warpgroup's key columns
        const uint32_t tS = tmem + (static_cast<uint32_t>(wq * 32) << 16) + c0;
        const int jmax = p.causal ? min(si.len_k, i + 1) : si.len_k;   // keys < jmax visible
        const bool full = n0 + c0 + 64 <= jmax;              // every key of the half visible
        const float c = p.scale_log2;
        // rows past the sequence read the last row's lse (a valid address) and
        // discard it, so the load needs no predicate
        const int64_t lse_row = b * p.lse_b + row_base + min(i, si.len_q - 1);
        float acc[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) acc[e] = 0.f;
        bool ok = true;
        // The next head's lse is loaded one head ahead and only converted when
        // it is used: arithmetic on the value right after its load would wait
        // for the load there, every head.
        float lse_next = p.lse[lse_row];
        for (int h = 0; h < H; ++h) {
            const float lse_h = lse_next;
            if (h + 1 < H) lse_next = p.lse[lse_row + (h + 1) * p.lse_h];
            const int buf = h & 1;
            ok = mbar_wait(bar(L::kBarSFull + buf), (h >> 1) & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[64];
            tmem_ld32x2(tS + 128 * buf, v, tS + 128 * buf + 32, v + 32);
            tc_fence_before();
            mbar_arrive(bar(L::kBarSFree + buf));            // the values are in registers
            const float nl = row_in ? -lse_h * kLog2e : 0.f;  // -lse2 of (row, h)
            if (full && row_in) {
                // packed pairs: one FMA and one add per two terms
                const float2 c2 = make_float2(c, c), nl2 = make_float2(nl, nl);
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 x2 = ffma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), c2, nl2);
                    const float2 t2 = make_float2(ex2(fminf(x2.x, kScoreClamp)), ex2(fminf(x2.y, kScoreClamp)));
                    const float2 a2 = fadd2(make_float2(acc[e], acc[e + 1]), t2);
                    acc[e] = a2.x;
                    acc[e + 1] = a2.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    const bool vis = row_in && n0 + c0 + e < jmax;
                    const float t = ex2(fminf(fmaf(__uint_as_float(v[e]), c, nl), kScoreClamp));
                    acc[e] += vis ? t : 0.f;
                }
            }
        }
        // Each thread stores its row's 64 sums directly (full 16-byte vectors
        // where the row stride allows); warpgroup 1 leaves its half-row sum in
        // shared memory and warpgroup 0 adds it to its own: the row's partial
        // L1 norm for this key tile, in a fixed order.
        float hs = 0.f;
#pragma unroll
        for (int e = 0; e < 64; e += 4) hs += (acc[e] + acc[e + 1]) + (acc[e + 2] + acc[e + 3]);
        if (wg == 1) half_sum[row] = hs;
        if (ok && row_in) {
            const int64_t W = p.sc_w;
            const int64_t rb = p.varlen ? row_base : static_cast<int64_t>(b) * p.Sq;
            float* dst = p.score + (rb + i) * W + n0 + c0;
            if (n0 + c0 + 63 < W && (W & 3) == 0) {
#pragma unroll
                for (int e = 0; e < 64; e += 4)
                    *reinterpret_cast<float4*>(dst + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    if (n0 + c0 + e < W) dst[e] = acc[e];
            }
        }
        named_bar_sync(1, 256);
        if (wg == 0 && ok && row_in) part[row] = hs + half_sum[row];
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
    if (tid == 0 && *abort_flag) set_error(p.err, DEV_E_TIMEOUT);
}

// l1[r] = sum over key tiles t, in order, of part[t][r]; rows past cu[-1]
// (varlen) are 0, as are their score rows.
__global__ void __launch_bounds__(256) l1_reduce_kernel(const Problem p, int n_tiles) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t r_end = p.l1_rows;
    if (p.varlen) {
        int e = __ldg(p.cu + p.B);
        r_end = (e < 0) ? 0 : (e > p.T ? p.T : e);
    }
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < p.l1_rows;
         r += stride) {
        float s = 0.f;
        if (r < r_end)
            for (int t = 0; t < n_tiles; ++t) s += p.l1_part[static_cast<int64_t>(t) * p.l1_rows + r];
        p.l1[r] = s;
    }
    if (p.varlen) {   // unvisited rows of the score: 0, not whatever the buffer held
        const int64_t n = (p.T - r_end) * p.sc_w;
        float* base = p.score + r_end * p.sc_w;
        for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n; x += stride)
            base[x] = 0.f;
    }
}

template <int D, bool F16>
cudaError_t launch_score_d(const Problem& p, cudaStream_t stream) {
    using L = ScLayout<D>;
    const int64_t rows = p.varlen ? p.T : p.Sq;
    const int64_t keys = p.varlen ? p.T : p.Sk;
    const int64_t Bm = p.varlen ? 1 : p.B;
    const int n_tiles = static_cast<int>((p.sc_w + kSt - 1) / kSt);
    if (p.B > 0 && p.Sq > 0 && p.sc_w > 0 && keys > 0) {
        ScoreMaps maps;
        if (!make_tile_map(&maps.q, p.q, D, p.Hq, rows, Bm, p.q_h, p.q_s, p.q_b, F16) ||
            !make_tile_map(&maps.k, p.k, D, p.Hkv, keys, Bm, p.k_h, p.k_s, p.k_b, F16))
            return cudaErrorInvalidValue;
        cudaError_t e = cudaFuncSetAttribute(score_sm100_kernel<D, F16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) return e;
        dim3 grid(n_tiles, (p.Sq + kSt - 1) / kSt, p.B);
        score_sm100_kernel<D, F16><<<grid, kScThreads, L::kBytes, stream>>>(p, maps);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.l1_rows > 0) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t want = (p.l1_rows + 255) / 256;
        const int grid = static_cast<int>(want < 4 * sms ? (want > 0 ? want : 1) : 4 * sms);
        l1_reduce_kernel<<<grid, 256, 0, stream>>>(p, p.sc_w > 0 ? n_tiles : 0);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace

int score_key_tiles(int64_t width) { return static_cast<int>((width + kSt - 1) / kSt); }

cudaError_t launch_score_recompute(const Problem& p, cudaStream_t stream) {
    if (p.f16)
        return p.D == 64 ? launch_score_d<64, true>(p, stream) : launch_score_d<128, true>(p, stream);
    return p.D == 64 ? launch_score_d<64, false>(p, stream) : launch_score_d<128, false>(p, stream);
}

}  // namespace attn
