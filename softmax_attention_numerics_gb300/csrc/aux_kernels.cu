// Memory-bound helper kernels of the backward and the varlen tails:
//   bwd_preprocess  Delta = rowsum(dO o O) in fp32 and lse2 = lse * log2(e)
//   dq_convert      dq = bf16 / fp16 (dq_acc * scale)
//   zero_trailing   rows >= cu[nseq] of a packed varlen buffer: out = 0 and
//                   lse = 0 (forward), dq = dk = dv = 0 (backward); also
//                   checks every sequence's bounds against T and max_seqlen.  Rows that no
//                   tile visits must still be written (PFCCLab/cudnn-frontend
//                   PR #9, section 2; flash-dmattn PR #122, Root Cause 1).
// All are grid-stride loops sized to a multiple of the SM count.
#include "device_common.cuh"
#include "sm100_ptx.cuh"

namespace attn {
namespace {

// D/8 threads per (row, head), 8 elements (16 bytes) of O and of dO per
// thread: every load is a full 16-byte vector and a warp covers 32*8/D rows,
// so the reduction is log2(D/8) shuffles within each row's lane group.
template <int D, bool F16>
__global__ void __launch_bounds__(256) preprocess_kernel(const Problem p, int64_t rows) {
    constexpr int kTpr = D / 8;                       // threads per (row, head)
    constexpr int kGpw = 32 / kTpr;                   // (row, head) groups per warp
    const int sub = threadIdx.x & (kTpr - 1);         // position within the row
    const int gw = (threadIdx.x & 31) / kTpr;         // group within the warp
    const int64_t groups = static_cast<int64_t>(gridDim.x) * (blockDim.x / kTpr);
    const int64_t total = rows * p.Hq;
    // The loop bound is the warp's first group, so all 32 lanes run the same
    // iterations and meet every shuffle; groups past the end idle.
    for (int64_t w0 = ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * kGpw;
         w0 < total; w0 += groups) {
        const int64_t w = w0 + gw;
        const bool active = w < total;
        int b = 0, h = 0;
        int64_t i = 0;
        float acc = 0.f;
        if (active) {
            h = static_cast<int>(w % p.Hq);
            const int64_t r = w / p.Hq;
            if (p.varlen) {
                i = r;
            } else {
                b = static_cast<int>(r / p.Sq);
                i = r - static_cast<int64_t>(b) * p.Sq;
            }
            const uint4 ov = *reinterpret_cast<const uint4*>(p.o + b * p.o_b + i * p.o_s +
                                                             h * p.o_h + sub * 8);
            const uint4 dv = *reinterpret_cast<const uint4*>(p.dout + b * p.do_b + i * p.do_s +
                                                             h * p.do_h + sub * 8);
            const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a = unpack2<F16>(ow[e]);
                const float2 c = unpack2<F16>(dw[e]);
                acc = fmaf(a.x, c.x, acc);
                acc = fmaf(a.y, c.y, acc);
            }
        }
#pragma unroll
        for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (active && sub == 0) {
            const int64_t li = b * p.lse_b + h * p.lse_h + i;
            p.delta[li] = acc;
            p.lse2[li] = p.lse[li] * kLog2e;
        }
    }
}

// dq = 16-bit(acc * scale), 4 elements per thread-iteration.
template <bool F16>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         bf16* __restrict__ dq, int64_t n4,
                                                         float scale) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride) {
        const float4 a = reinterpret_cast<const float4*>(acc)[i];
        uint2 o;
        o.x = pack2<F16>(a.x * scale, a.y * scale);
        o.y = pack2<F16>(a.z * scale, a.w * scale);
        reinterpret_cast<uint2*>(dq)[i] = o;
    }
}

__device__ __forceinline__ int64_t trailing_start(const Problem& p) {
    int e = __ldg(p.cu + p.B);
    if (e < 0) e = 0;
    if (e > p.T) e = p.T;
    return e;
}

// Zero rows [cu[B], T) of a contiguous [T, H, D] 16-bit buffer (8 elems per op).
__device__ __forceinline__ void zero_rows_bf16(bf16* base, int64_t r0, int64_t T, int H, int D) {
    const int64_t per_row = static_cast<int64_t>(H) * D / 8;
    const int64_t n = (T - r0) * per_row;
    uint4* dst = reinterpret_cast<uint4*>(base + r0 * H * D);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride)
        dst[i] = make_uint4(0u, 0u, 0u, 0u);
}

// Every sequence's bounds, checked once per varlen call: the attention
// kernels check only the sequences their blocks visit, and with max_seqlen = 0
// no attention block runs at all.
__device__ __forceinline__ void check_seqlens(const Problem& p) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; b < p.B;
         b += stride) {
        const int a = __ldg(p.cu + b), e = __ldg(p.cu + b + 1);
        if (!(a >= 0 && e >= a && e <= p.T && e - a <= p.Sq)) set_error(p.err, DEV_E_SEQLENS);
    }
}

__global__ void zero_trailing_fwd_kernel(const Problem p) {
    check_seqlens(p);
    const int64_t r0 = trailing_start(p);
    zero_rows_bf16(p.out, r0, p.T, p.Hq, p.D);
    const int64_t n = (p.T - r0) * p.Hq;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const int64_t h = i / (p.T - r0);
        const int64_t r = r0 + i % (p.T - r0);
        p.lse[h * p.lse_h + r] = 0.f;
    }
}

__global__ void zero_trailing_bwd_kernel(const Problem p) {
    check_seqlens(p);
    const int64_t r0 = trailing_start(p);
    zero_rows_bf16(p.dq, r0, p.T, p.Hq, p.D);
    zero_rows_bf16(p.dk, r0, p.T, p.Hkv, p.D);
    zero_rows_bf16(p.dv, r0, p.T, p.Hkv, p.D);
}

// The bounded-wait path of the tcgen05 kernels, on its own: a wait that
// nothing will satisfy gives up after budget_ns of global time and the error
// word reports a timeout.  The barrier expects one arrival that never comes.
__global__ void wait_timeout_probe_kernel(int* err, uint64_t budget_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        sm100::mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        sm100::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int* flag = &abort_flag;
        if (!sm100::mbar_wait(smem_u32(&bar), 0, flag, budget_ns)) set_error(err, DEV_E_TIMEOUT);
    }
}

int grid_for(int64_t work, int threads) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const Problem& p, cudaStream_t stream) {
    const int64_t rows = p.varlen ? p.T : static_cast<int64_t>(p.B) * p.Sq;
    if (rows == 0) return cudaSuccess;
    const int blocks = grid_for(rows * p.Hq * (p.D / 8), 256);
    if (p.f16) {
        if (p.D == 64)
            preprocess_kernel<64, true><<<blocks, 256, 0, stream>>>(p, rows);
        else
            preprocess_kernel<128, true><<<blocks, 256, 0, stream>>>(p, rows);
    } else {
        if (p.D == 64)
            preprocess_kernel<64, false><<<blocks, 256, 0, stream>>>(p, rows);
        else
            preprocess_kernel<128, false><<<blocks, 256, 0, stream>>>(p, rows);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(const Problem& p, cudaStream_t stream) {
    const int64_t rows = p.varlen ? p.T : static_cast<int64_t>(p.B) * p.Sq;
    const int64_t n4 = rows * p.Hq * p.D / 4;
    if (n4 == 0) return cudaSuccess;
    if (p.f16)
        dq_convert_kernel<true><<<grid_for(n4, 256), 256, 0, stream>>>(p.dq_acc, p.dq, n4, p.scale);
    else
        dq_convert_kernel<false><<<grid_for(n4, 256), 256, 0, stream>>>(p.dq_acc, p.dq, n4, p.scale);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(int* err, uint64_t budget_ns, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(err, budget_ns);
    return cudaGetLastError();
}

cudaError_t launch_zero_trailing_fwd(const Problem& p, cudaStream_t stream) {
    if (!p.varlen || (p.T == 0 && p.B == 0)) return cudaSuccess;
    zero_trailing_fwd_kernel<<<grid_for(static_cast<int64_t>(p.T) * p.Hq * p.D / 8, 256), 256, 0,
                               stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_zero_trailing_bwd(const Problem& p, cudaStream_t stream) {
    if (!p.varlen || (p.T == 0 && p.B == 0)) return cudaSuccess;
    zero_trailing_bwd_kernel<<<grid_for(static_cast<int64_t>(p.T) * p.Hq * p.D / 8, 256), 256,
                               0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace attn
