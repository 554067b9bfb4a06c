// Deterministic dQ of the attention backward for sm_103a (TMA + tcgen05 + TMEM).
//
// One CTA = 128 query rows of one (batch/sequence, q head).  It walks the key
// tiles of its kv head in a fixed order and accumulates dQ in TMEM, so no
// atomics are involved and dq is bitwise reproducible (the ordering argument
// of PFCCLab/cudnn-frontend PR #9, How it was verified).  Per key tile j:
//     S_j  = Q K_j^T,  dP_j = dO V_j^T                 (TMEM, fp32)
//     P    = exp2(min(S*scale*log2e + mask - lse2, 0))  with the predicates of
//            the other passes (partial last key tile, query rows past the
//            sequence, causal pairs, the mask: OpenWAM PR #64)
//     dS   = P o (dP - Delta)  -> bf16, written over S_j in TMEM
//     dQ  += dS K_j                                     (TMEM A operand)
// Warps: 0-7 compute (thread = query row = TMEM lane; its lse2 and Delta live
// in registers; warps 0-3 take keys 0-63 of the tile, warps 4-7 keys 64-127,
// each half writing its packed dS over the first 32 of its own 64 S columns),
// 8 = TMA producer (Q, dO once; K_j, V_j through a ring), 9 = TMEM allocator
// and UMMA issuer.  TMEM: S0 | S1 (double buffer) | dP | dQ.  S_{j+1} is
// computed while the warps work on tile j.
#include "sm100_ptx.cuh"

namespace attn {
namespace {

using namespace sm100;

constexpr int kDqThreads = 320;
constexpr int kT = 128;

template <int D>
struct DqLayout {
    static constexpr int kBlocks = D / 64;
    static constexpr int kTileBytes = kT * D * 2;
    // K/V ring.  At iteration j the issuer needs K_j (until dQ_j), K_{j+1} and
    // V_{j+1} resident at once (dP_{j+1} is issued before dQ_j), plus a slot
    // being filled: at least four slots.  With five, K_{j+2} goes into the
    // slot V_{j-1} left (free early) instead of K_j's, so its load is not
    // held until dQ_j completes.
    static constexpr int kStages = (D == 128) ? 5 : 6;
    static constexpr int kQ = 0;
    static constexpr int kDO = kTileBytes;
    static constexpr int kKV = 2 * kTileBytes;
    static constexpr int kBar = kKV + kStages * kTileBytes;
    static constexpr int kBarQ = 0;
    static constexpr int kBarKVFull = 1;
    static constexpr int kBarKVEmpty = kBarKVFull + kStages;
    static constexpr int kBarSFull = kBarKVEmpty + kStages;   // [2]
    static constexpr int kBarDPFull = kBarSFull + 2;
    static constexpr int kBarDSReady = kBarDPFull + 1;
    static constexpr int kBarDQDone = kBarDSReady + 1;        // [2]: dQ_j read S buffer j&1
    static constexpr int kBarFinal = kBarDQDone + 2;
    static constexpr int kBarDrain = kBarFinal + 1;
    static constexpr int kBarDPRead = kBarDrain + 1;          // dP_j in registers (256)
    static constexpr int kNumBars = kBarDPRead + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16;
    static_assert(kBytes <= 232448, "shared memory");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColDP = 256, kColDQ = 384;
};

struct DqMaps {
    CUtensorMap q, dout, k, v;
};

template <int D, bool F16>
__global__ void __launch_bounds__(kDqThreads, 1)
    bwd_dq_sm100_kernel(const Problem p, const __grid_constant__ DqMaps maps) {
    using L = DqLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::kBar + 8u * i; };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int m0 = (gridDim.x - 1 - blockIdx.x) * kT;      // heaviest (causal) CTAs first
    const SeqInfo si = seq_info(p, b);
    if (!si.ok || m0 >= si.len_q) return;
    if ((sbase & 1023u) != 0) {
        if (tid == 0) set_error(p.err, DEV_E_INTERNAL);
        return;
    }
    const int hk = h / p.G;
    int kend = si.len_k;
    if (p.causal) kend = min(kend, m0 + kT);
    const int n = (kend + kT - 1) / kT;
    const int row_base = si.row0;
    const int bcoord = p.varlen ? 0 : b;

    if (tid == 0) {
        for (int i = 0; i < L::kNumBars; ++i)
            mbar_init(bar(i), (i == L::kBarDSReady || i == L::kBarDPRead) ? 2 * kT : 1);
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

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            mbar_arrive_expect_tx(bar(L::kBarQ), 2 * L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kBlocks; ++c) {
                tma_load_4d(sbase + L::kQ + c * 16384, &maps.q, 64 * c, h, row_base + m0, bcoord,
                            bar(L::kBarQ));
                tma_load_4d(sbase + L::kDO + c * 16384, &maps.dout, 64 * c, h, row_base + m0, bcoord,
                            bar(L::kBarQ));
            }
            int issued = 0;
            for (int j = 0; j < n && !*abort_flag; ++j) {
                for (int which = 0; which < 2; ++which) {
                    const int li = 2 * j + which;
                    const int s = li % L::kStages, r = li / L::kStages;
                    if (!mbar_wait(bar(L::kBarKVEmpty + s), (r & 1) ^ 1, abort_flag)) break;
                    mbar_arrive_expect_tx(bar(L::kBarKVFull + s), L::kTileBytes);
                    const CUtensorMap* m = which ? &maps.v : &maps.k;
#pragma unroll
                    for (int c = 0; c < L::kBlocks; ++c)
                        tma_load_4d(sbase + L::kKV + s * L::kTileBytes + c * 16384, m, 64 * c, hk,
                                    row_base + j * kT, bcoord, bar(L::kBarKVFull + s));
                    issued = li + 1;
                }
            }
            if (*abort_flag) {
                volatile int no_abort = 0;
                mbar_wait(bar(L::kBarQ), 0, &no_abort, kDrainBudgetNs);
                for (int li = max(0, issued - L::kStages); li < issued; ++li)
                    mbar_wait(bar(L::kBarKVFull + li % L::kStages), (li / L::kStages) & 1, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_f16kind(128, 128, 0, 0, F16);    // S, dP (K-major)
            constexpr uint32_t id_dq = idesc_f16kind(128, D, 0, 1, F16);     // dQ += dS K (B MN-major)
            const uint64_t q_k = smem_desc(sbase + L::kQ, 16, 1024, kSwizzle128B);
            const uint64_t do_k = smem_desc(sbase + L::kDO, 16, 1024, kSwizzle128B);
            auto stage = [&](int li) { return li % L::kStages; };
            auto par = [&](int li) { return (uint32_t)((li / L::kStages) & 1); };
            auto issue_s = [&](int j) {
                const uint64_t kd = smem_desc(sbase + L::kKV + stage(2 * j) * L::kTileBytes, 16, 1024,
                                              kSwizzle128B);
                const uint32_t dst = tmem + ((j & 1) ? L::kColS1 : L::kColS0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(dst, desc_add(q_k, off), desc_add(kd, off), id_s, kk > 0);
                }
            };
            auto issue_dp = [&](int j) {
                const uint64_t vd = smem_desc(sbase + L::kKV + stage(2 * j + 1) * L::kTileBytes, 16,
                                              1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_ss(tmem + L::kColDP, desc_add(do_k, off), desc_add(vd, off), id_s, kk > 0);
                }
            };
            bool ok = mbar_wait(bar(L::kBarQ), 0, abort_flag);
            if (ok && n > 0) {
                ok = mbar_wait(bar(L::kBarKVFull + stage(0)), par(0), abort_flag) &&
                     mbar_wait(bar(L::kBarKVFull + stage(1)), par(1), abort_flag);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                    mma_commit(bar(L::kBarSFull + 0));
                    issue_dp(0);
                    mma_commit(bar(L::kBarDPFull));
                    mma_commit(bar(L::kBarKVEmpty + stage(1)));     // V_0 consumed
                }
            }
            for (int j = 0; ok && j < n; ++j) {
                if (!(ok = dbg_stall(p.debug_stall, kStallDq, j, bar(L::kBarDrain), abort_flag))) break;
                const bool next = j + 1 < n;
                if (next) {
                    // S_{j+1} goes into the buffer dQ_{j-1} read dS_{j-1} from.
                    if (!(ok = mbar_wait(bar(L::kBarKVFull + stage(2 * j + 2)), par(2 * j + 2),
                                         abort_flag)))
                        break;
                    if (j >= 1 &&
                        !(ok = mbar_wait(bar(L::kBarDQDone + ((j + 1) & 1)), ((j - 1) >> 1) & 1,
                                         abort_flag)))
                        break;
                    tc_fence_after();
                    issue_s(j + 1);
                    mma_commit(bar(L::kBarSFull + ((j + 1) & 1)));
                    // dP_{j+1} as soon as the compute warps hold dP_j in registers
                    // (it runs while they work on tile j, ahead of dQ_j)
                    if (!(ok = mbar_wait(bar(L::kBarDPRead), j & 1, abort_flag))) break;
                    if (!(ok = mbar_wait(bar(L::kBarKVFull + stage(2 * j + 3)), par(2 * j + 3),
                                         abort_flag)))
                        break;
                    tc_fence_after();
                    issue_dp(j + 1);
                    mma_commit(bar(L::kBarDPFull));
                    mma_commit(bar(L::kBarKVEmpty + stage(2 * j + 3)));   // V_{j+1} consumed
                }
                // dS_j written by the compute warps.
                if (!(ok = mbar_wait(bar(L::kBarDSReady), j & 1, abort_flag))) break;
                tc_fence_after();
                {
                    const uint64_t kmn = smem_desc(sbase + L::kKV + stage(2 * j) * L::kTileBytes,
                                                   16384, 1024, kSwizzle128B);
                    const uint32_t a = tmem + ((j & 1) ? L::kColS1 : L::kColS0);
#pragma unroll
                    for (int kk = 0; kk < kT / 16; ++kk)    // dS of keys 16kk..: see dS_col
                        mma_ts(tmem + L::kColDQ, a + 8 * kk + (kk >= 4 ? 32 : 0), desc_add(kmn, kk * 2048),
                               id_dq, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(L::kBarDQDone + (j & 1)));
                mma_commit(bar(L::kBarKVEmpty + stage(2 * j)));     // K_j consumed
            }
            mma_commit(bar(L::kBarFinal));
            if (!ok) {
                mma_commit(bar(L::kBarDrain));
                volatile int no_abort = 0;
                mbar_wait(bar(L::kBarDrain), 0, &no_abort, kDrainBudgetNs);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ dS rows
        const int wq = warp & 3;                      // TMEM lane quarter
        const int hq = warp >> 2;                     // key half of the tile (dQ: d half)
        const int r = wq * 32 + lane;
        const int i = m0 + r;                         // query row in the sequence
        const bool row_in = i < si.len_q;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const int64_t li = b * p.lse_b + h * p.lse_h + row_base + i;
        const float nl = row_in ? -p.lse2[li] : 0.f;   // -lse2 of this row
        const float dl = row_in ? p.delta[li] : 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            ok = mbar_wait(bar(L::kBarSFull + (j & 1)), (j >> 1) & 1, abort_flag) &&
                 mbar_wait(bar(L::kBarDPFull), j & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t tS = tmem + lane_off + ((j & 1) ? L::kColS1 : L::kColS0);
            const uint32_t tDP = tmem + lane_off + L::kColDP;
            const int n0 = j * kT;
            const bool has_mask = p.mask_kind != MASK_NONE;
            const bool pred = (n0 + kT > si.len_k) || (m0 + kT > si.len_q) ||
                              (p.causal && n0 + kT - 1 > m0);
            if (has_mask) {
                // logits rewritten in TMEM chunk by chunk (mask loads would spill)
#pragma unroll 1
                for (int c = 2 * hq; c < 2 * hq + 2; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tS + 32 * c, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        v[e] = __float_as_uint(logit_log2(p, __uint_as_float(v[e]), b, h, i,
                                                          n0 + 32 * c + e, si.len_q, si.len_k));
                    tmem_st32(tS + 32 * c, v);
                }
                tmem_wait_st();
            }
            const int jmax = p.causal ? min(si.len_k, i + 1) : si.len_k;   // keys < jmax visible
            // this warp's half of dP_j to registers first, so that dP_{j+1} can
            // start on the tensor cores while the tile is worked on
            uint32_t dph[64];
            tmem_ld32x2(tDP + 64 * hq, dph, tDP + 64 * hq + 32, dph + 32);
            tc_fence_before();
            mbar_arrive(bar(L::kBarDPRead));
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int c = 2 * hq + cc;
                uint32_t sv[32];
                const uint32_t* dv = dph + 32 * cc;
                tmem_ld32(tS + 32 * c, sv);
                uint32_t pk[16];
                if (!pred && !has_mask) {
                    const float2 c2 = make_float2(p.scale_log2, p.scale_log2);
                    const float2 nl2 = make_float2(nl, nl);
                    const float2 nd2 = make_float2(-dl, -dl);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 x2 = ffma2(make_float2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])),
                                                c2, nl2);
                        const float p0 = ex2(fminf(x2.x, 0.f));
                        const float p1 = ex2(fminf(x2.y, 0.f));
                        const float2 d2 = fadd2(make_float2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                                nd2);
                        const float2 ds2 = fmul2(make_float2(p0, p1), d2);
                        pk[e >> 1] = pack2<F16>(ds2.x, ds2.y);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float ds[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int key = n0 + 32 * c + e + u;
                            float x;
                            bool vis;
                            if (has_mask) {
                                x = __uint_as_float(sv[e + u]);
                                vis = x != -INFINITY;
                            } else {
                                x = __uint_as_float(sv[e + u]) * p.scale_log2;
                                vis = row_in && key < jmax;
                            }
                            const float pv = ex2(fminf(x + nl, 0.f));
                            ds[u] = vis ? pv * (__uint_as_float(dv[e + u]) - dl) : 0.f;
                        }
                        pk[e >> 1] = pack2<F16>(ds[0], ds[1]);
                    }
                }
                // dS of chunk c over S columns this thread has already read:
                // 16c (chunks 0, 1) and 32 + 16c (chunks 2, 3).
                tmem_st16(tS + 16 * c + (c >= 2 ? 32 : 0), pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(L::kBarDSReady));
        }
        // Epilogue: dq = bf16(dQ * scale); rows past the sequence are not written.
        if (ok) {
            ok = mbar_wait(bar(L::kBarFinal), 0, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            tc_fence_after();
            bf16* grow = p.dq + b * p.out_b + static_cast<int64_t>(row_base + i) * p.out_s + h * p.out_h;
#pragma unroll 1
            for (int c = hq * (D / 64); c < (hq + 1) * (D / 64); ++c) {
                uint32_t o[32];
                if (n > 0) {
                    tmem_ld32(tmem + lane_off + L::kColDQ + 32 * c, o);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (row_in) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack2<F16>(__uint_as_float(o[2 * e]) * p.scale,
                                          __uint_as_float(o[2 * e + 1]) * p.scale);
                    uint4* dst = reinterpret_cast<uint4*>(grow + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
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

template <int D, bool F16>
cudaError_t launch_dq_sm100_d(const Problem& p, cudaStream_t stream) {
    using L = DqLayout<D>;
    if (p.B == 0 || p.Sq == 0) return cudaSuccess;
    const int64_t Sq = p.varlen ? p.T : p.Sq;
    const int64_t Sk = p.varlen ? p.T : p.Sk;
    const int64_t Bm = p.varlen ? 1 : p.B;
    const bool no_keys = Sk == 0;    // maps must stay legal; they are never read then
    DqMaps maps;
    const bool ok =
        make_tile_map(&maps.q, p.q, D, p.Hq, Sq, Bm, p.q_h, p.q_s, p.q_b, F16) &&
        make_tile_map(&maps.dout, p.dout, D, p.Hq, Sq, Bm, p.do_h, p.do_s, p.do_b, F16) &&
        make_tile_map(&maps.k, no_keys ? p.q : p.k, D, no_keys ? p.Hq : p.Hkv, no_keys ? Sq : Sk, Bm,
                      no_keys ? p.q_h : p.k_h, no_keys ? p.q_s : p.k_s, no_keys ? p.q_b : p.k_b, F16) &&
        make_tile_map(&maps.v, no_keys ? p.q : p.v, D, no_keys ? p.Hq : p.Hkv, no_keys ? Sq : Sk, Bm,
                      no_keys ? p.q_h : p.v_h, no_keys ? p.q_s : p.v_s, no_keys ? p.q_b : p.v_b, F16);
    if (!ok) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_sm100_kernel<D, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sq + kT - 1) / kT, p.Hq, p.B);
    bwd_dq_sm100_kernel<D, F16><<<grid, kDqThreads, L::kBytes, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_deterministic(const Problem& p, cudaStream_t stream) {
    if (p.f16)
        return p.D == 64 ? launch_dq_sm100_d<64, true>(p, stream) : launch_dq_sm100_d<128, true>(p, stream);
    return p.D == 64 ? launch_dq_sm100_d<64, false>(p, stream) : launch_dq_sm100_d<128, false>(p, stream);
}

}  // namespace attn
