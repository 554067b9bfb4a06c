// Attention backward on the warp-level mma.sync tensor path.
//
// bwd_main: one CTA = 128 keys of one (batch/sequence, kv head); 8 warps own
// 16 keys each.  The CTA walks every q head of the GQA group and every
// 64-row query tile that can see its keys (causal: only tiles at or below
// the diagonal), recomputing
//     S^T = K Q^T,  P^T = exp2(min(S^T*scale*log2e + mask - lse2, 0))
// with the same predicates as the forward (partial last key tile, query
// rows past the sequence, causal, mask: OpenWAM PR #64, Summary), then
//     dP^T = V dO^T,  dS^T = P^T o (dP^T - Delta),
//     dV += P^T dO,  dK += dS^T Q          (registers, no atomics)
// and, on the atomic path, dQ_part = dS K added into an fp32 workspace.
// The exponent clamp at 0 holds because P <= 1 exactly (PFCCLab/cudnn-
// frontend PR #9, section 3).  Hidden entries give P = dS = 0 by selection,
// never by multiplying possibly non-finite values by zero.
//
// bwd_dq: the deterministic dQ path, one CTA = 128 query rows of one q head
// walking the key tiles in a fixed order (no atomics).
#include "device_common.cuh"

namespace attn {
namespace {

constexpr int kThreads = 256;

// ------------------------------------------------------------------ main

constexpr int kMainBN = 128;   // keys per CTA
constexpr int kMainBM = 64;    // query rows per inner tile

template <int D>
struct MainSmem {
    static constexpr int K = 0;
    static constexpr int V = K + kMainBN * D;
    static constexpr int Q = V + kMainBN * D;          // 2 stages
    static constexpr int DO = Q + 2 * kMainBM * D;     // 2 stages
    static constexpr int DS = DO + 2 * kMainBM * D;    // [128 keys][64 q]
    static constexpr int END_BF16 = DS + kMainBN * kMainBM;
    static constexpr size_t bytes = END_BF16 * sizeof(bf16) + 4 * kMainBM * sizeof(float);
};

template <int D>
__global__ void __launch_bounds__(kThreads) bwd_main_kernel(const Problem p, int with_dq) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    bf16* sb = reinterpret_cast<bf16*>(smem_raw);
    bf16* sK = sb + MainSmem<D>::K;
    bf16* sV = sb + MainSmem<D>::V;
    bf16* sQ = sb + MainSmem<D>::Q;
    bf16* sDO = sb + MainSmem<D>::DO;
    bf16* sDS = sb + MainSmem<D>::DS;
    float* sL = reinterpret_cast<float*>(sb + MainSmem<D>::END_BF16);   // [2][64] lse2
    float* sDel = sL + 2 * kMainBM;                                      // [2][64] Delta

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int b = blockIdx.z, hk = blockIdx.y;
    const int n0 = blockIdx.x * kMainBN;
    const SeqInfo si = seq_info(p, b);
    if (!si.ok || n0 >= si.len_k) return;

    const bf16* kg = p.k + b * p.k_b + static_cast<int64_t>(si.row0 + n0) * p.k_s + hk * p.k_h;
    const bf16* vg = p.v + b * p.v_b + static_cast<int64_t>(si.row0 + n0) * p.v_s + hk * p.v_h;
    load_tile<kMainBN, D, kThreads>(sK, kg, p.k_s, si.len_k - n0, p.k, tid);
    load_tile<kMainBN, D, kThreads>(sV, vg, p.v_s, si.len_k - n0, p.v, tid);

    const int mt_first = p.causal ? n0 / kMainBM : 0;
    const int mt_count = (si.len_q + kMainBM - 1) / kMainBM;
    const int per_head = max(mt_count - mt_first, 0);
    const int n_iter = per_head * p.G;

    // Issue the loads of iteration `it` into stage `st`.
    auto issue = [&](int it, int st) {
        const int gi = it / per_head;
        const int m0 = (mt_first + it % per_head) * kMainBM;
        const int h = hk * p.G + gi;
        const bf16* qg = p.q + b * p.q_b + static_cast<int64_t>(si.row0 + m0) * p.q_s + h * p.q_h;
        const bf16* dg =
            p.dout + b * p.do_b + static_cast<int64_t>(si.row0 + m0) * p.do_s + h * p.do_h;
        load_tile<kMainBM, D, kThreads>(sQ + st * kMainBM * D, qg, p.q_s, si.len_q - m0, p.q, tid);
        load_tile<kMainBM, D, kThreads>(sDO + st * kMainBM * D, dg, p.do_s, si.len_q - m0, p.dout,
                                        tid);
        if (tid < kMainBM) {
            const int i = m0 + tid;
            const int64_t li = b * p.lse_b + h * p.lse_h + si.row0 + i;
            sL[st * kMainBM + tid] = i < si.len_q ? p.lse2[li] : 0.f;
            sDel[st * kMainBM + tid] = i < si.len_q ? p.delta[li] : 0.f;
        }
    };

    if (n_iter > 0) issue(0, 0);
    cp_async_commit();

    float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) dk[n][e] = dv[n][e] = 0.f;
    }
    const int jrow[2] = {n0 + warp * 16 + g, n0 + warp * 16 + g + 8};   // this thread's keys

    for (int it = 0; it < n_iter; ++it) {
        const int st = it & 1;
        if (it + 1 < n_iter) issue(it + 1, st ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();

        const int gi = it / per_head;
        const int m0 = (mt_first + it % per_head) * kMainBM;
        const int h = hk * p.G + gi;
        const bf16* cQ = sQ + st * kMainBM * D;
        const bf16* cDO = sDO + st * kMainBM * D;
        const float* cL = sL + st * kMainBM;
        const float* cDel = sDel + st * kMainBM;

        // S^T (16 keys x 64 q) and dP^T.
        float sT[kMainBM / 8][4], dpT[kMainBM / 8][4];
#pragma unroll
        for (int n = 0; n < kMainBM / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sT[n][e] = dpT[n][e] = 0.f;
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t ka[4], va[4];
            {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = 2 * kk + (lane >> 4);
                ldsm_x4(smem_u32(sK + swz<D>(r, c)), ka[0], ka[1], ka[2], ka[3]);
                ldsm_x4(smem_u32(sV + swz<D>(r, c)), va[0], va[1], va[2], va[3]);
            }
#pragma unroll
            for (int np = 0; np < kMainBM / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = 2 * kk + ((lane >> 3) & 1);
                ldsm_x4(smem_u32(cQ + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(sT[2 * np], ka[0], ka[1], ka[2], ka[3], b0, b1);
                mma16816(sT[2 * np + 1], ka[0], ka[1], ka[2], ka[3], b2, b3);
                ldsm_x4(smem_u32(cDO + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(dpT[2 * np], va[0], va[1], va[2], va[3], b0, b1);
                mma16816(dpT[2 * np + 1], va[0], va[1], va[2], va[3], b2, b3);
            }
        }

        // P^T and dS^T, packed as A fragments (rows = keys, k = query rows).
        uint32_t pa[kMainBM / 16][4], da[kMainBM / 16][4];
#pragma unroll
        for (int n = 0; n < kMainBM / 8; ++n) {
            float pv[4], dsv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int ql = 8 * n + 2 * t4 + (e & 1);
                const int i = m0 + ql;
                const int j = jrow[e >> 1];
                const float x = logit_log2(p, sT[n][e], b, h, i, j, si.len_q, si.len_k);
                float pr = 0.f, ds = 0.f;
                if (x != -INFINITY) {
                    pr = ex2(fminf(x - cL[ql], 0.f));
                    ds = pr * (dpT[n][e] - cDel[ql]);
                }
                pv[e] = pr;
                dsv[e] = ds;
            }
            pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(pv[0], pv[1]);
            pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(pv[2], pv[3]);
            da[n >> 1][(n & 1) * 2 + 0] = pack_bf16(dsv[0], dsv[1]);
            da[n >> 1][(n & 1) * 2 + 1] = pack_bf16(dsv[2], dsv[3]);
            if (with_dq) {
                // dS^T rows (keys) -> shared [128 keys][64 q], swizzled chunks of 8 q.
                const int r0 = warp * 16 + g;
                *reinterpret_cast<uint32_t*>(sDS + r0 * kMainBM + ((n ^ (r0 & 7)) << 3) + 2 * t4) =
                    da[n >> 1][(n & 1) * 2 + 0];
                const int r1 = r0 + 8;
                *reinterpret_cast<uint32_t*>(sDS + r1 * kMainBM + ((n ^ (r1 & 7)) << 3) + 2 * t4) =
                    da[n >> 1][(n & 1) * 2 + 1];
            }
        }

        // dV += P^T dO ; dK += dS^T Q.
#pragma unroll
        for (int kk = 0; kk < kMainBM / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = 2 * np + (lane >> 4);
                ldsm_x4_t(smem_u32(cDO + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(dv[2 * np], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                mma16816(dv[2 * np + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
                ldsm_x4_t(smem_u32(cQ + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(dk[2 * np], da[kk][0], da[kk][1], da[kk][2], da[kk][3], b0, b1);
                mma16816(dk[2 * np + 1], da[kk][0], da[kk][1], da[kk][2], da[kk][3], b2, b3);
            }
        }

        if (with_dq) {
            __syncthreads();   // every warp's dS^T rows are in shared memory
            // dQ_part (64 q x D) = dS (64 x 128 keys) K (128 x D).
            // Warp w: q rows 16*(w%4); D=128: d columns 64*(w/4), all keys;
            // D=64: all d columns, keys 64*(w/4) .. +63.
            const int q0 = (warp & 3) * 16;
            const int d0 = (D == 128) ? (warp >> 2) * 64 : 0;
            const int kb0 = (D == 128) ? 0 : (warp >> 2) * 64;
            constexpr int KSTEPS = (D == 128) ? kMainBN / 16 : kMainBN / 32;
            float dq[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                const int kb = kb0 + ks * 16;
                uint32_t a0, a1, a2, a3;
                {
                    const int r = kb + (lane & 7) + (lane >> 4) * 8;
                    const int c = (q0 >> 3) + ((lane >> 3) & 1);
                    ldsm_x4_t(smem_u32(sDS + r * kMainBM + ((c ^ (r & 7)) << 3)), a0, a1, a2, a3);
                }
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b0, b1, b2, b3;
                    const int r = kb + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int c = (d0 >> 3) + 2 * np + (lane >> 4);
                    ldsm_x4_t(smem_u32(sK + swz<D>(r, c)), b0, b1, b2, b3);
                    mma16816(dq[2 * np], a0, a1, a2, a3, b0, b1);
                    mma16816(dq[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const int i = m0 + q0 + g + rr * 8;
                if (i >= si.len_q) continue;
                float* dst = p.dq_acc + (b * p.acc_b + si.row0 + i) * static_cast<int64_t>(p.Hq) * D +
                             static_cast<int64_t>(h) * D + d0;
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    atomicAdd(dst + 8 * n + 2 * t4, dq[n][2 * rr]);
                    atomicAdd(dst + 8 * n + 2 * t4 + 1, dq[n][2 * rr + 1]);
                }
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // Epilogue: dK *= scale; rows past the sequence are not written.
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int j = jrow[r];
        if (j >= si.len_k) continue;
        bf16* dkg = p.dk + b * p.dk_b + static_cast<int64_t>(si.row0 + j) * p.dk_s + hk * p.dk_h;
        bf16* dvg = p.dv + b * p.dk_b + static_cast<int64_t>(si.row0 + j) * p.dk_s + hk * p.dk_h;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            *reinterpret_cast<uint32_t*>(dkg + 8 * n + 2 * t4) =
                pack_bf16(dk[n][2 * r] * p.scale, dk[n][2 * r + 1] * p.scale);
            *reinterpret_cast<uint32_t*>(dvg + 8 * n + 2 * t4) =
                pack_bf16(dv[n][2 * r], dv[n][2 * r + 1]);
        }
    }
}

// ------------------------------------------------------------------ deterministic dQ

constexpr int kDqBM = 128;
constexpr int kDqBN = 64;

template <int D>
__global__ void __launch_bounds__(kThreads) bwd_dq_kernel(const Problem p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
    bf16* sDO = sQ + kDqBM * D;
    bf16* sK = sDO + kDqBM * D;     // 2 stages
    bf16* sV = sK + 2 * kDqBN * D;  // 2 stages

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int b = blockIdx.z, h = blockIdx.y;
    const int m0 = blockIdx.x * kDqBM;
    const SeqInfo si = seq_info(p, b);
    if (!si.ok || m0 >= si.len_q) return;
    const int hk = h / p.G;

    const bf16* qg = p.q + b * p.q_b + static_cast<int64_t>(si.row0 + m0) * p.q_s + h * p.q_h;
    const bf16* dg = p.dout + b * p.do_b + static_cast<int64_t>(si.row0 + m0) * p.do_s + h * p.do_h;
    const bf16* kg = p.k + b * p.k_b + static_cast<int64_t>(si.row0) * p.k_s + hk * p.k_h;
    const bf16* vg = p.v + b * p.v_b + static_cast<int64_t>(si.row0) * p.v_s + hk * p.v_h;

    int n_end = si.len_k;
    if (p.causal) n_end = min(n_end, m0 + kDqBM);
    const int n_tiles = (n_end + kDqBN - 1) / kDqBN;

    load_tile<kDqBM, D, kThreads>(sQ, qg, p.q_s, si.len_q - m0, p.q, tid);
    load_tile<kDqBM, D, kThreads>(sDO, dg, p.do_s, si.len_q - m0, p.dout, tid);
    if (n_tiles > 0) {
        load_tile<kDqBN, D, kThreads>(sK, kg, p.k_s, si.len_k, p.k, tid);
        load_tile<kDqBN, D, kThreads>(sV, vg, p.v_s, si.len_k, p.v, tid);
    }
    cp_async_commit();

    const int row_i[2] = {m0 + warp * 16 + g, m0 + warp * 16 + g + 8};
    float lse2[2], del[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int i = row_i[r];
        const int64_t li = b * p.lse_b + h * p.lse_h + si.row0 + i;
        lse2[r] = i < si.len_q ? p.lse2[li] : 0.f;
        del[r] = i < si.len_q ? p.delta[li] : 0.f;
    }

    float dq[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;
    uint32_t qf[D / 16][4], df[D / 16][4];

    for (int t = 0; t < n_tiles; ++t) {
        const int st = t & 1;
        if (t + 1 < n_tiles) {
            const int nn = (t + 1) * kDqBN;
            load_tile<kDqBN, D, kThreads>(sK + (st ^ 1) * kDqBN * D, kg + nn * p.k_s, p.k_s,
                                          si.len_k - nn, p.k, tid);
            load_tile<kDqBN, D, kThreads>(sV + (st ^ 1) * kDqBN * D, vg + nn * p.v_s, p.v_s,
                                          si.len_k - nn, p.v, tid);
        }
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = 2 * kk + (lane >> 4);
                ldsm_x4(smem_u32(sQ + swz<D>(r, c)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
                ldsm_x4(smem_u32(sDO + swz<D>(r, c)), df[kk][0], df[kk][1], df[kk][2], df[kk][3]);
            }
        }
        const bf16* cK = sK + st * kDqBN * D;
        const bf16* cV = sV + st * kDqBN * D;

        float s[kDqBN / 8][4], dp[kDqBN / 8][4];
#pragma unroll
        for (int n = 0; n < kDqBN / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = dp[n][e] = 0.f;
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < kDqBN / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = 2 * kk + ((lane >> 3) & 1);
                ldsm_x4(smem_u32(cK + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(s[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
                mma16816(s[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
                ldsm_x4(smem_u32(cV + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(dp[2 * np], df[kk][0], df[kk][1], df[kk][2], df[kk][3], b0, b1);
                mma16816(dp[2 * np + 1], df[kk][0], df[kk][1], df[kk][2], df[kk][3], b2, b3);
            }
        }
        const int n0 = t * kDqBN;
        uint32_t da[kDqBN / 16][4];
#pragma unroll
        for (int n = 0; n < kDqBN / 8; ++n) {
            float dsv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = n0 + 8 * n + 2 * t4 + (e & 1);
                const int r = e >> 1;
                const float x = logit_log2(p, s[n][e], b, h, row_i[r], j, si.len_q, si.len_k);
                float ds = 0.f;
                if (x != -INFINITY) {
                    const float pr = ex2(fminf(x - lse2[r], 0.f));
                    ds = pr * (dp[n][e] - del[r]);
                }
                dsv[e] = ds;
            }
            da[n >> 1][(n & 1) * 2 + 0] = pack_bf16(dsv[0], dsv[1]);
            da[n >> 1][(n & 1) * 2 + 1] = pack_bf16(dsv[2], dsv[3]);
        }
#pragma unroll
        for (int kk = 0; kk < kDqBN / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = 2 * np + (lane >> 4);
                ldsm_x4_t(smem_u32(cK + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(dq[2 * np], da[kk][0], da[kk][1], da[kk][2], da[kk][3], b0, b1);
                mma16816(dq[2 * np + 1], da[kk][0], da[kk][1], da[kk][2], da[kk][3], b2, b3);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int i = row_i[r];
        if (i >= si.len_q) continue;
        bf16* og = p.dq + b * p.out_b + static_cast<int64_t>(si.row0 + i) * p.out_s + h * p.out_h;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            *reinterpret_cast<uint32_t*>(og + 8 * n + 2 * t4) =
                pack_bf16(dq[n][2 * r] * p.scale, dq[n][2 * r + 1] * p.scale);
        }
    }
}

template <int D>
cudaError_t launch_main_d(const Problem& p, bool with_dq, cudaStream_t stream) {
    const size_t smem = MainSmem<D>::bytes;
    cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sk + kMainBN - 1) / kMainBN, p.Hkv, p.B);
    if (grid.x == 0 || p.B == 0) return cudaSuccess;
    bwd_main_kernel<D><<<grid, kThreads, smem, stream>>>(p, with_dq ? 1 : 0);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_dq_d(const Problem& p, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(2 * kDqBM + 4 * kDqBN) * D * sizeof(bf16);
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sq + kDqBM - 1) / kDqBM, p.Hq, p.B);
    if (grid.x == 0 || p.B == 0) return cudaSuccess;
    bwd_dq_kernel<D><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main(const Problem& p, bool with_dq_atomics, cudaStream_t stream) {
    return p.D == 64 ? launch_main_d<64>(p, with_dq_atomics, stream)
                     : launch_main_d<128>(p, with_dq_atomics, stream);
}

cudaError_t launch_bwd_dq_deterministic(const Problem& p, cudaStream_t stream) {
    return p.D == 64 ? launch_dq_d<64>(p, stream) : launch_dq_d<128>(p, stream);
}

}  // namespace attn
