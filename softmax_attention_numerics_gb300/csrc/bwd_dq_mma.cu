// Deterministic dQ of the attention backward, on the warp-level mma.sync
// tensor path (m16n8k16 bf16).
//
// bwd_dq: one CTA = 128 query rows of one q head; 8 warps own 16 rows each
// and walk the key tiles (64 keys, double-buffered by cp.async) in a fixed
// order, recomputing
//     S = Q K^T,  P = exp2(min(S*scale*log2e + mask - lse2, 0)),
//     dP = dO V^T,  dS = P o (dP - Delta),  dQ += dS K
// with the same predicates as the other passes (partial last key tile,
// query rows past the sequence, causal pairs, the mask: OpenWAM PR #64).
// No atomics: dq is bitwise reproducible (the ordering argument of
// PFCCLab/cudnn-frontend PR #9, How it was verified).  Hidden entries give
// dS = 0 by selection.
#include "device_common.cuh"

namespace attn {
namespace {

constexpr int kThreads = 256;

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

cudaError_t launch_bwd_dq_deterministic(const Problem& p, cudaStream_t stream) {
    return p.D == 64 ? launch_dq_d<64>(p, stream) : launch_dq_d<128>(p, stream);
}

}  // namespace attn
