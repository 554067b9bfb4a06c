// Attention forward on fp8 (E4M3) inputs for sm_103a: TMA + tcgen05 + TMEM.
//
// Inputs: q [B,Sq,Hq,D], k [B,Sk,Hkv,D] as E4M3 codes, and V transposed by
// transpose_v_kernel into the caller's workspace as vt [B,Hkv,D,Sk_pad] (keys
// contiguous; Sk_pad = Sk rounded up to 16, padding keys 0), one descale
// factor per tensor, D = 128.  Both MMAs are tcgen05 kind::f8f6f4 with E4M3 A
// and B, fp32 accumulate, B K-major in shared memory:
//     S_t  = Q_t K_j^T          A = Q tile [128 rows][128 bytes], B = K tile
//     O_t += P^_t(j) V_j        A = P^ in TMEM [128 lanes][32 columns of 4 keys], B = V^T tile
// The softmax is the 16-bit kernel's (FlyDSL PR #1033, "The fix": always
// m_new = max(m_ref, m_tile), lazy threshold 8): x = s * scale * dq * dk *
// log2 e, p = exp2(min(x - m_ref, 8)), P^ = E4M3(p) written over the first
// 32 columns of S_t for the P V product.  The fp8 helper of the same PR instead
// rebases the running max down to a lower tile max with a bounded factor;
// that keeps the top P of a tile exact in E4M3 but leaves earlier terms
// under-weighted, which a V = ones check cannot see, so it is not used here.
// out = O * dv / sum(P^) (bf16; the rounded sum keeps out an exact weighted
// mean of V), lse = (m_ref + log2 sum(p)) ln 2.
//
// One CTA = two 128-row query tiles of one (b, q head):
//   warps 0-3 softmax tile 0, 4-7 tile 1, 8 TMA producer, 9 TMEM + MMA issuer.
// TMEM: S0 | S1 | O0 | O1 (128 fp32 columns each; P^_t over S_t's first 32).
// Shared: Q0 Q1 (16 KB each) | K / V^T ring (16 KB stages) | barriers.  Every
// tile is one 128-byte-wide swizzle-128 block.
#include "sm100_ptx.cuh"

namespace attn {
namespace {

template <bool B>
struct F8Tag {
    static constexpr bool value = B;
};

using namespace sm100;

constexpr int kF8Threads = 320;
constexpr int kF8Tile = 128;


struct Fp8Maps {
    CUtensorMap q, k, vt;
};

struct Fp8Layout {
    static constexpr int kTileBytes = kF8Tile * 128;      // 128 rows x 128 bytes
    static constexpr int kStages = 6;
    static constexpr int kQ = 0;
    static constexpr int kKV = 2 * kTileBytes;
    static constexpr int kBar = kKV + kStages * kTileBytes;
    static constexpr int kBarQ = 0;
    static constexpr int kBarKVFull = 1;
    static constexpr int kBarKVEmpty = kBarKVFull + kStages;
    static constexpr int kBarSFull = kBarKVEmpty + kStages;   // [2]
    static constexpr int kBarPFull = kBarSFull + 2;           // [2]
    static constexpr int kBarPVDone = kBarPFull + 2;          // [2]
    static constexpr int kBarDrain = kBarPVDone + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kMisc = kBar + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16 + 1024;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 384;
};

// kind::f8f6f4, fp32 accumulate, A and B E4M3 (format code 0), both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// A with P^ in TMEM (the TS form): [128 lanes][8 columns] = 32 E4M3 of K per row.
__device__ __forceinline__ void mma_ts_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 8 consecutive TMEM columns from registers.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// Two fp32 -> two E4M3 (round to nearest even, saturating to +-448), lo in the low byte.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// acc.x += the low E4M3 of v, acc.y += the high one: both widen exactly to f16
// and the mixed-precision add of sm_100 takes the f16 operand as it is (one
// fp32 rounding per add, the same sums as converting to fp32 first).
__device__ __forceinline__ float2 add_e4m3x2(float2 acc, uint16_t v) {
    asm("{\n\t.reg .b16 lo, hi;\n\t.reg .b32 h2;\n\t"
        "cvt.rn.f16x2.e4m3x2 h2, %2;\n\t"
        "mov.b32 {lo, hi}, h2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\t"
        "add.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(acc.x), "+f"(acc.y) : "h"(v));
    return acc;
}

__global__ void __launch_bounds__(kF8Threads, 1)
    fwd_fp8_sm100_kernel(const Fp8Problem p, const __grid_constant__ Fp8Maps maps) {
    using L = Fp8Layout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + L::kBar + 8u * i; };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int m0 = (gridDim.x - 1 - blockIdx.x) * 2 * kF8Tile;
    if (m0 >= p.Sq) return;
    const int hk = h / p.G;

    int n_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int r0 = m0 + t * kF8Tile;
        int kend = p.Sk;
        if (p.causal) kend = min(kend, r0 + kF8Tile);
        n_t[t] = (r0 < p.Sq) ? (kend + kF8Tile - 1) / kF8Tile : 0;
    }
    const int n_all = max(n_t[0], n_t[1]);

    if (tid == 0) {
        for (int i = 0; i < L::kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == L::kBarPFull || i == L::kBarPFull + 1) cnt = kF8Tile;
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

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&maps.q);
            tma_prefetch_desc(&maps.k);
            tma_prefetch_desc(&maps.vt);
            mbar_arrive_expect_tx(bar(L::kBarQ), 2 * L::kTileBytes);
#pragma unroll
            for (int t = 0; t < 2; ++t)
                tma_load_4d(sbase + L::kQ + t * L::kTileBytes, &maps.q, 0, h, m0 + t * kF8Tile, b,
                            bar(L::kBarQ));
            int issued = 0;
            for (int j = 0; j < n_all && !*abort_flag; ++j) {
                for (int which = 0; which < 2; ++which) {
                    const int li = 2 * j + which;
                    const int s = li % L::kStages, r = li / L::kStages;
                    if (!mbar_wait(bar(L::kBarKVEmpty + s), (r & 1) ^ 1, abort_flag)) break;
                    if (!dbg_check(j * kF8Tile < p.Sk && s < L::kStages, p.err)) break;
                    mbar_arrive_expect_tx(bar(L::kBarKVFull + s), L::kTileBytes);
                    const uint32_t dst = sbase + L::kKV + s * L::kTileBytes;
                    if (which == 0)   // K_j: keys j*128.., all D bytes
                        tma_load_4d(dst, &maps.k, 0, hk, j * kF8Tile, b, bar(L::kBarKVFull + s));
                    else              // V^T_j: all D rows, keys j*128..
                        tma_load_4d(dst, &maps.vt, j * kF8Tile, 0, hk, b, bar(L::kBarKVFull + s));
                    issued = li + 1;
                }
            }
            if (*abort_flag) {
                // Let every copy in flight (the Q tiles too) land before the CTA exits.
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
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3(128, 128);
            const uint32_t colS[2] = {L::kColS0, L::kColS1};
            const uint32_t colO[2] = {L::kColO0, L::kColO1};
            auto kv_stage = [&](int li) { return li % L::kStages; };
            auto kv_par = [&](int li) { return (uint32_t)((li / L::kStages) & 1); };
            auto issue_qk = [&](int t, int j) {
                const uint64_t qd = smem_desc(sbase + L::kQ + t * L::kTileBytes, 16, 1024, kSwizzle128B);
                const uint64_t kd = smem_desc(sbase + L::kKV + kv_stage(2 * j) * L::kTileBytes, 16,
                                              1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)      // 32 E4M3 (32 bytes) of D per MMA
                    mma_ss_f8(tmem + colS[t], desc_add(qd, kk * 32), desc_add(kd, kk * 32), idesc, kk > 0);
            };
            auto issue_pv = [&](int t, int j) {
                const uint64_t vd = smem_desc(sbase + L::kKV + kv_stage(2 * j + 1) * L::kTileBytes, 16,
                                              1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)      // 32 keys (8 TMEM columns of P^) per MMA
                    mma_ts_f8(tmem + colO[t], tmem + colS[t] + 8 * kk, desc_add(vd, kk * 32), idesc,
                              (j > 0 || kk > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(bar(L::kBarQ), 0, abort_flag);
            if (ok && n_all > 0) {
                ok = mbar_wait(bar(L::kBarKVFull + kv_stage(0)), kv_par(0), abort_flag);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t)
                        if (n_t[t] > 0) {
                            issue_qk(t, 0);
                            mma_commit(bar(L::kBarSFull + t));
                        }
                    mma_commit(bar(L::kBarKVEmpty + kv_stage(0)));
                }
            }
            for (int j = 0; ok && j < n_all; ++j) {
                if (!(ok = dbg_stall(p.debug_stall, kStallFp8, j, bar(L::kBarDrain), abort_flag))) break;
                const int lv = 2 * j + 1, lk = 2 * j + 2;
                if (!(ok = mbar_wait(bar(L::kBarKVFull + kv_stage(lv)), kv_par(lv), abort_flag))) break;
                const bool next = j + 1 < n_all;
                if (next && !(ok = mbar_wait(bar(L::kBarKVFull + kv_stage(lk)), kv_par(lk), abort_flag)))
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
                        // S_t(j+1) overwrites P^_t(j), and its softmax rescales O_t: PV_t(j) first.
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
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2;
        const int wq = warp & 3;
        const int r_local = wq * 32 + lane;
        const int i = m0 + t * kF8Tile + r_local;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off + (t ? L::kColS1 : L::kColS0);
        const uint32_t tO = tmem + lane_off + (t ? L::kColO1 : L::kColO0);
        const int r0_tile = m0 + t * kF8Tile;
        const int n_mine = n_t[t];
        float m_ref = -INFINITY;
        float2 l2 = make_float2(0.f, 0.f), lr2 = make_float2(0.f, 0.f);
        bool ok = true;

        for (int j = 0; j < n_mine; ++j) {
            ok = mbar_wait(bar(L::kBarSFull + t), j & 1, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int n0 = j * kF8Tile;
            // keys past the sequence or causal pairs in this tile: predicated path
            const bool pred = (n0 + kF8Tile > p.Sk) || (p.causal && n0 + kF8Tile - 1 > r0_tile);
            float x[kF8Tile];
            float mt = -INFINITY;
            uint32_t* xu = reinterpret_cast<uint32_t*>(x);
            if (pred) {
                tmem_ld128(tS, xu);
                const int jmax = p.causal ? min(p.Sk, i + 1) : p.Sk;
                const bool row_in = i < p.Sq;
#pragma unroll
                for (int c = 0; c < kF8Tile; ++c) {
                    x[c] = (row_in && n0 + c < jmax) ? x[c] * p.scale_log2 : -INFINITY;
                    mt = fmaxf(mt, x[c]);
                }
            } else {
                // full tile: the max of the raw scores, scaled once (x stays
                // unscaled; P folds the scale into one FMA).  The row loaded in two
                // halves with the first half's max under the second load, as in the
                // 16-bit kernel, spills here.
                tmem_ld128(tS, xu);
                float mr = -INFINITY;
#pragma unroll
                for (int c = 0; c < kF8Tile; ++c) mr = fmaxf(mr, x[c]);
                if (p.scale_log2 > 0.f) {
                    mt = mr * p.scale_log2;
                } else {
#pragma unroll
                    for (int c = 0; c < kF8Tile; ++c) mt = fmaxf(mt, x[c] * p.scale_log2);
                }
            }
            const float m_new = fmaxf(m_ref, mt);
            bool rescale = true;
            if (m_new == -INFINITY || (p.lazy && m_ref != -INFINITY && mt - m_ref <= 8.f)) rescale = false;
            float corr = 1.f;
            if (rescale) {
                corr = ex2(m_ref - m_new);
                l2 = fmul2(l2, make_float2(corr, corr));
                lr2 = fmul2(lr2, make_float2(corr, corr));
                if (j == 0 || m_ref == -INFINITY) corr = 1.f;
                m_ref = m_new;
            }
            const float ms = (m_ref == -INFINITY) ? 0.f : m_ref;
            const float2 nms2 = make_float2(-ms, -ms);
            const float2 c2 = pred ? make_float2(1.f, 1.f) : make_float2(p.scale_log2, p.scale_log2);
            // P^ row: 128 E4M3, four keys per TMEM column, over S_t's columns [0, 32).
            // p = exp2(min(x - m_ref, 8)); x - m_ref <= m_tile - m_ref up to the
            // rounding of the scaled maximum, so when every row of the warp has
            // m_tile - m_ref <= 8 - 1/64 the per-element min is skipped.
            auto exps = [&](auto clamp_tag) {
                constexpr bool kClamp = decltype(clamp_tag)::value;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int k0 = 32 * c + 4 * e;
                        const float2 d01 = ffma2(make_float2(x[k0], x[k0 + 1]), c2, nms2);
                        const float2 d23 = ffma2(make_float2(x[k0 + 2], x[k0 + 3]), c2, nms2);
                        const float2 p01 = make_float2(ex2(kClamp ? fminf(d01.x, 8.f) : d01.x),
                                                       ex2(kClamp ? fminf(d01.y, 8.f) : d01.y));
                        const float2 p23 = make_float2(ex2(kClamp ? fminf(d23.x, 8.f) : d23.x),
                                                       ex2(kClamp ? fminf(d23.y, 8.f) : d23.y));
                        l2 = fadd2(fadd2(l2, p01), p23);
                        const uint16_t lo = pack_e4m3x2(p01.x, p01.y), hi = pack_e4m3x2(p23.x, p23.y);
                        lr2 = add_e4m3x2(add_e4m3x2(lr2, lo), hi);
                        w[e] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
                    }
                    tmem_st8(tS + 8 * c, w);
                }
            };
            if (__all_sync(0xffffffffu, mt - ms <= 8.f - 0.015625f))
                exps(F8Tag<false>{});
            else
                exps(F8Tag<true>{});
            if (__any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                    tmem_st32(tO + 32 * c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(L::kBarPFull + t));
        }

        const bool store = ok && i < p.Sq;
        bf16* orow = p.out + b * p.out_b + static_cast<int64_t>(i) * p.out_s + h * p.out_h;
        if (ok && n_mine > 0) {
            ok = mbar_wait(bar(L::kBarPVDone + t), (n_mine - 1) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
        }
        if (ok) {
            const float l = l2.x + l2.y, lr = lr2.x + lr2.y;
            const float inv = lr > 0.f ? p.out_scale / lr : 0.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
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
                        pk[e] = pack2<false>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (store) p.lse[b * p.lse_b + h * p.lse_h + i] = l > 0.f ? (m_ref + lg2(l)) * kLn2 : 0.f;
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

// V [B,Sk,Hkv,D] (E4M3) -> vt [B,Hkv,D,Sk_pad]: 64 keys x 64 d bytes per block
// through shared memory; keys past Sk in the padding are written as 0.
__global__ void __launch_bounds__(256) transpose_v_kernel(const uint8_t* __restrict__ v, int64_t v_b,
                                                          int64_t v_s, int64_t v_h, uint8_t* __restrict__ vt,
                                                          int Sk, int Sk_pad, int Hkv, int D) {
    __shared__ uint8_t tile[64][65];
    const int s0 = blockIdx.x * 64, d0 = blockIdx.y * 64;
    const int bh = blockIdx.z, b = bh / Hkv, hk = bh % Hkv;
    for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
        const int ls = e / 64, ld = e % 64;
        const int s = s0 + ls, d = d0 + ld;
        tile[ls][ld] = (s < Sk && d < D) ? v[b * v_b + s * v_s + hk * v_h + d] : uint8_t(0);
    }
    __syncthreads();
    uint8_t* base = vt + (static_cast<int64_t>(b) * Hkv + hk) * D * Sk_pad;
    for (int e = threadIdx.x; e < 64 * 64; e += blockDim.x) {
        const int ld = e / 64, ls = e % 64;
        const int s = s0 + ls, d = d0 + ld;
        if (s < Sk_pad && d < D) base[static_cast<int64_t>(d) * Sk_pad + s] = tile[ls][ld];
    }
}

}  // namespace

cudaError_t launch_fp8_transpose_v(const Fp8Problem& p, cudaStream_t stream) {
    if (p.B == 0 || p.Sk == 0) return cudaSuccess;
    dim3 grid((p.Sk_pad + 63) / 64, 2, p.B * p.Hkv);
    transpose_v_kernel<<<grid, 256, 0, stream>>>(p.v, p.v_b, p.v_s, p.v_h, p.vt, p.Sk, p.Sk_pad,
                                                 p.Hkv, 128);
    return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const Fp8Problem& p, cudaStream_t stream) {
    using L = Fp8Layout;
    if (p.B == 0 || p.Sq == 0) return cudaSuccess;
    Fp8Maps maps;
    const int64_t qd[4] = {128, p.Hq, p.Sq, p.B};
    const int64_t qs[3] = {p.q_h, p.q_s, p.q_b};
    if (!make_u8_map(&maps.q, p.q, qd, qs, 1, 128)) return cudaErrorInvalidValue;
    if (p.Sk == 0) {
        maps.k = maps.q;      // no key tile is ever loaded
        maps.vt = maps.q;
    } else {
        const int64_t kd[4] = {128, p.Hkv, p.Sk, p.B};
        const int64_t ks[3] = {p.k_h, p.k_s, p.k_b};
        const int64_t vd[4] = {p.Sk_pad, 128, p.Hkv, p.B};
        const int64_t vs[3] = {p.Sk_pad, p.vt_h, p.vt_b};
        if (!make_u8_map(&maps.k, p.k, kd, ks, 1, 128) || !make_u8_map(&maps.vt, p.vt, vd, vs, 128, 1))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(fwd_fp8_sm100_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sq + 2 * kF8Tile - 1) / (2 * kF8Tile), p.Hq, p.B);
    fwd_fp8_sm100_kernel<<<grid, kF8Threads, L::kBytes, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace attn
