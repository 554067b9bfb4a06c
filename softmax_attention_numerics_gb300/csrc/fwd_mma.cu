// Attention forward on the warp-level mma.sync tensor path (m16n8k16 bf16).
//
// One CTA = 128 query rows of one (batch/sequence, q head); 8 warps own 16
// rows each.  K/V tiles of 64 keys are double-buffered through cp.async.
// Online softmax in exp2: per row the running reference max m_ref, the
// running sum l and the unnormalised output O (registers).  Each new tile
// takes m_new = max(m_ref, m_tile) (FlyDSL PR #1033, "The fix"); with the
// lazy rule the rescale is skipped while m_tile - m_ref <= 8 and the
// exponent is clamped at 8, which never fires on correct statistics
// (PFCCLab/cudnn-frontend PR #9, section 3: bound the exp2 argument).
#include "device_common.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;
constexpr int kBN = 64;
constexpr int kThreads = 256;

template <int D>
__global__ void __launch_bounds__(kThreads) fwd_mma_kernel(const Problem p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
    bf16* sK = sQ + kBM * D;
    bf16* sV = sK + 2 * kBN * D;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int b = blockIdx.z, h = blockIdx.y;
    const int m0 = blockIdx.x * kBM;
    const SeqInfo si = seq_info(p, b);
    if (!si.ok || m0 >= si.len_q) return;
    const int hk = h / p.G;

    const bf16* qg = p.q + b * p.q_b + static_cast<int64_t>(si.row0 + m0) * p.q_s + h * p.q_h;
    const bf16* kg = p.k + b * p.k_b + static_cast<int64_t>(si.row0) * p.k_s + hk * p.k_h;
    const bf16* vg = p.v + b * p.v_b + static_cast<int64_t>(si.row0) * p.v_s + hk * p.v_h;

    int n_end = si.len_k;
    if (p.causal) n_end = min(n_end, m0 + kBM);
    const int n_tiles = (n_end + kBN - 1) / kBN;

    load_tile<kBM, D, kThreads>(sQ, qg, p.q_s, si.len_q - m0, p.q, tid);
    if (n_tiles > 0) {
        load_tile<kBN, D, kThreads>(sK, kg, p.k_s, si.len_k, p.k, tid);
        load_tile<kBN, D, kThreads>(sV, vg, p.v_s, si.len_k, p.v, tid);
    }
    cp_async_commit();

    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_ref[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};     // sum of the exact probabilities (-> lse)
    float lr[2] = {0.f, 0.f};    // sum of the bf16-rounded ones fed to P V (-> out)
    uint32_t qf[D / 16][4];
    const int row_i[2] = {m0 + warp * 16 + g, m0 + warp * 16 + g + 8};

    for (int t = 0; t < n_tiles; ++t) {
        const int st = t & 1;
        if (t + 1 < n_tiles) {
            const int nn = (t + 1) * kBN;
            load_tile<kBN, D, kThreads>(sK + (st ^ 1) * kBN * D, kg + nn * p.k_s, p.k_s,
                                        si.len_k - nn, p.k, tid);
            load_tile<kBN, D, kThreads>(sV + (st ^ 1) * kBN * D, vg + nn * p.v_s, p.v_s,
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
            }
        }
        const bf16* cK = sK + st * kBN * D;
        const bf16* cV = sV + st * kBN * D;

        // S = Q K^T for this warp's 16 rows x 64 keys.
        float s[kBN / 8][4];
#pragma unroll
        for (int n = 0; n < kBN / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < kBN / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                const int c = 2 * kk + ((lane >> 3) & 1);
                ldsm_x4(smem_u32(cK + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(s[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
                mma16816(s[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
            }
        }

        // Predicates, then the online-softmax update.
        const int n0 = t * kBN;
        float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < kBN / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = n0 + 8 * n + 2 * t4 + (e & 1);
                const float x = logit_log2(p, s[n][e], b, h, row_i[e >> 1], j, si.len_q, si.len_k);
                s[n][e] = x;
                mt[e >> 1] = fmaxf(mt[e >> 1], x);
            }
        }
        float msafe[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 1));
            mt[r] = fmaxf(mt[r], __shfl_xor_sync(0xffffffffu, mt[r], 2));
            const float m_new = fmaxf(m_ref[r], mt[r]);
            bool rescale;
            if (m_new == -INFINITY) {
                rescale = false;                  // nothing visible in this row yet
            } else if (p.lazy && m_ref[r] != -INFINITY && mt[r] - m_ref[r] <= kLazyTau) {
                rescale = false;                  // lazy: keep the old reference max
            } else {
                rescale = true;
            }
            if (rescale) {
                const float corr = ex2(m_ref[r] - m_new);   // m_ref = -inf -> 0
                l[r] *= corr;
                lr[r] *= corr;
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    o[n][2 * r] *= corr;
                    o[n][2 * r + 1] *= corr;
                }
                m_ref[r] = m_new;
            }
            msafe[r] = (m_ref[r] == -INFINITY) ? 0.f : m_ref[r];
        }

        uint32_t pf[kBN / 16][4];
#pragma unroll
        for (int n = 0; n < kBN / 8; ++n) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pv[e] = ex2(fminf(s[n][e] - msafe[e >> 1], kLazyTau));
                l[e >> 1] += pv[e];
                lr[e >> 1] += bf16_round(pv[e]);
            }
            pf[n >> 1][(n & 1) * 2 + 0] = pack_bf16(pv[0], pv[1]);
            pf[n >> 1][(n & 1) * 2 + 1] = pack_bf16(pv[2], pv[3]);
        }

        // O += P V.
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int c = 2 * np + (lane >> 4);
                ldsm_x4_t(smem_u32(cV + swz<D>(r, c)), b0, b1, b2, b3);
                mma16816(o[2 * np], pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3], b0, b1);
                mma16816(o[2 * np + 1], pf[kk][0], pf[kk][1], pf[kk][2], pf[kk][3], b2, b3);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // Epilogue: out = O / lr, lse = (m_ref + log2 l) ln 2; a row with l = 0
    // (no visible key) gets out = 0 and lse = 0.
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
        l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
        lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 1);
        lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int i = row_i[r];
        if (i >= si.len_q) continue;
        // Normalising by the sum of the rounded weights keeps out an exact
        // weighted mean of V even when the lazy reference max lags the true
        // one (then the largest weight is up to 2^8 and not exact in bf16).
        const float inv = lr[r] > 0.f ? 1.0f / lr[r] : 0.f;
        bf16* og = p.out + b * p.out_b + static_cast<int64_t>(si.row0 + i) * p.out_s + h * p.out_h;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            *reinterpret_cast<uint32_t*>(og + 8 * n + 2 * t4) =
                pack_bf16(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
        }
        if (t4 == 0) {
            const float lse = l[r] > 0.f ? (m_ref[r] + lg2(l[r])) * kLn2 : 0.f;
            p.lse[b * p.lse_b + h * p.lse_h + si.row0 + i] = lse;
        }
    }
}

template <int D>
cudaError_t launch_fwd_d(const Problem& p, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(kBM + 4 * kBN) * D * sizeof(bf16);
    cudaError_t e = cudaFuncSetAttribute(fwd_mma_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.Sq + kBM - 1) / kBM, p.Hq, p.B);
    if (grid.x == 0 || p.B == 0) return cudaSuccess;
    fwd_mma_kernel<D><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const Problem& p, cudaStream_t stream) {
    return p.D == 64 ? launch_fwd_d<64>(p, stream) : launch_fwd_d<128>(p, stream);
}

}  // namespace attn
