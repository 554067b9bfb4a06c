// Host side of the C ABI declared in include/attn_gb300.h: argument
// validation (before any launch), problem set-up and the launch sequence on
// the caller's stream.
//
// The checks follow NVIDIA/cudnn-frontend PR #429 ("Fix stream-ordering and
// input-validation holes ..."): every companion tensor is checked against
// the shape contract derived from q (a transposed dout or lse must fail, not
// run), all tensors sit on one device, the dtype gate matches what the
// kernels compute (bf16 or fp16, templated on the element type and never
// reinterpreted: q, k, v, out, dout, dq, dk, dv must all have q's type), and
// out-parameters must be contiguous.  Unsupported head dims are rejected
// before launch (PFCCLab/cudnn-frontend PR #9, section 4).
#include <atomic>
#include <math.h>
#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "../../include/attn_gb300.h"
#include "attn_internal.h"

namespace attn {
namespace {

// Device error word (one per device that loads the library).
__device__ int g_attn_error = 0;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices] = {nullptr};
std::mutex g_err_mu;

int* error_word(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_attn_error) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(ptr);
    }
    return g_err_ptr[dev];
}

std::atomic<unsigned long long> g_launches{0};
std::atomic<int> g_debug_stall{-1};
thread_local char g_cuda_detail[256] = "";

int cuda_fail(cudaError_t e, const char* what) {
    snprintf(g_cuda_detail, sizeof(g_cuda_detail), "%s: %s (%s)", what, cudaGetErrorName(e),
             cudaGetErrorString(e));
    return ATTN_E_CUDA;
}
cudaEvent_t g_prof[ATTN_STAGE_COUNT][2] = {};

// Launch one stage: optional profiling events around it, launch accounting.
template <class F>
int run_stage(int stage, cudaStream_t st, F&& launch) {
    cudaEvent_t a = stage >= 0 ? g_prof[stage][0] : nullptr;
    cudaEvent_t b = stage >= 0 ? g_prof[stage][1] : nullptr;
    cudaError_t e;
    if (a && (e = cudaEventRecord(a, st)) != cudaSuccess) return cuda_fail(e, "event record");
    e = launch();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (b && (e = cudaEventRecord(b, st)) != cudaSuccess) return cuda_fail(e, "event record");
    return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 16-bit input of element type `dtype`: rank r, last stride 1, other strides
// multiples of 8 elements (for dims longer than 1), 16-byte aligned base.
int check_input(const attn_tensor_t* t, int rank, int dtype) {
    if (!t) return ATTN_E_ARG;
    if (t->dtype != dtype) return ATTN_E_DTYPE;
    if (t->ndim != rank) return ATTN_E_SHAPE;
    int64_t n = 1;
    for (int i = 0; i < rank; ++i) {
        if (t->shape[i] < 0) return ATTN_E_SHAPE;
        n *= t->shape[i];
    }
    if (n > 0 && !t->data) return ATTN_E_ARG;
    if (t->stride[rank - 1] != 1) return ATTN_E_LAYOUT;
    for (int i = 0; i < rank - 1; ++i)
        if (t->shape[i] > 1 && (t->stride[i] <= 0 || (t->stride[i] % 8) != 0)) return ATTN_E_LAYOUT;
    if (!aligned16(t->data)) return ATTN_E_LAYOUT;
    return ATTN_OK;
}

bool is_contiguous(const attn_tensor_t* t) {
    for (int i = 0; i < t->ndim; ++i)
        if (t->shape[i] == 0) return true;   // no elements: any strides describe it
    int64_t s = 1;
    for (int i = t->ndim - 1; i >= 0; --i) {
        if (t->shape[i] != 1 && t->stride[i] != s) return false;
        s *= t->shape[i];
    }
    return true;
}

bool same_shape(const attn_tensor_t* t, const int64_t* shape, int rank) {
    if (t->ndim != rank) return false;
    for (int i = 0; i < rank; ++i)
        if (t->shape[i] != shape[i]) return false;
    return true;
}

int check_output(const attn_tensor_t* t, int dtype, const int64_t* shape, int rank) {
    if (!t) return ATTN_E_ARG;
    if (t->dtype != dtype) return ATTN_E_DTYPE;
    if (!same_shape(t, shape, rank)) return ATTN_E_SHAPE;
    int64_t n = 1;
    for (int i = 0; i < rank; ++i) n *= shape[i];
    if (n > 0 && !t->data) return ATTN_E_ARG;
    if (!is_contiguous(t)) return ATTN_E_LAYOUT;
    if (n > 0 && !aligned16(t->data)) return ATTN_E_LAYOUT;
    return ATTN_OK;
}

int check_device(const attn_tensor_t* t, int dev) {
    if (!t) return ATTN_OK;
    if (t->device < 0) return ATTN_E_DEVICE;
    if (t->device != dev) return ATTN_E_DEVICE;
    return ATTN_OK;
}

#define ATTN_TRY(x)                       \
    do {                                  \
        const int _rc = (x);              \
        if (_rc != ATTN_OK) return _rc;   \
    } while (0)

// Shape contract derived from q and k; fills the shape-related fields of p.
struct Shapes {
    int varlen;
    int elt;        // ATTN_BF16 or ATTN_F16: the element type of q and every 16-bit tensor
    int64_t B, Sq, Sk, Hq, Hkv, D, T, nseq;
    int64_t q_shape[4], k_shape[4], lse_shape[3];
    int rank, lse_rank;
};

int derive_shapes(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
                  const attn_tensor_t* cu, int32_t max_seqlen, Shapes* s) {
    s->varlen = cu != nullptr;
    s->rank = s->varlen ? 3 : 4;
    if (!q || !k || !v) return ATTN_E_ARG;
    // bf16 or fp16, the same for q, k, v (and for out, dout, dq, dk, dv).
    if (q->dtype != ATTN_BF16 && q->dtype != ATTN_F16) return ATTN_E_DTYPE;
    s->elt = q->dtype;
    if (q->ndim == s->rank && q->shape[s->rank - 1] != 64 && q->shape[s->rank - 1] != 128)
        return ATTN_E_UNSUPPORTED;
    ATTN_TRY(check_input(q, s->rank, s->elt));
    ATTN_TRY(check_input(k, s->rank, s->elt));
    ATTN_TRY(check_input(v, s->rank, s->elt));
    if (s->varlen) {
        s->T = q->shape[0];
        s->Hq = q->shape[1];
        s->D = q->shape[2];
        s->Hkv = k->shape[1];
        if (k->shape[0] != s->T || k->shape[2] != s->D) return ATTN_E_SHAPE;
        if (!same_shape(v, k->shape, 3)) return ATTN_E_SHAPE;
        if (cu->dtype != ATTN_I32) return ATTN_E_DTYPE;
        if (cu->ndim != 1 || cu->shape[0] < 1) return ATTN_E_SHAPE;
        if (cu->stride[0] != 1 && cu->shape[0] > 1) return ATTN_E_LAYOUT;
        if (!cu->data) return ATTN_E_ARG;
        if ((reinterpret_cast<uintptr_t>(cu->data) & 3u) != 0) return ATTN_E_LAYOUT;
        if (max_seqlen < 0) return ATTN_E_ARG;
        s->nseq = cu->shape[0] - 1;
        s->B = s->nseq;
        s->Sq = s->Sk = max_seqlen;
        const int64_t qs[3] = {s->T, s->Hq, s->D};
        const int64_t ks[3] = {s->T, s->Hkv, s->D};
        for (int i = 0; i < 3; ++i) {
            s->q_shape[i] = qs[i];
            s->k_shape[i] = ks[i];
        }
        s->lse_rank = 2;
        s->lse_shape[0] = s->Hq;
        s->lse_shape[1] = s->T;
    } else {
        s->B = q->shape[0];
        s->Sq = q->shape[1];
        s->Hq = q->shape[2];
        s->D = q->shape[3];
        s->Sk = k->shape[1];
        s->Hkv = k->shape[2];
        s->T = 0;
        if (k->shape[0] != s->B || k->shape[3] != s->D) return ATTN_E_SHAPE;
        if (!same_shape(v, k->shape, 4)) return ATTN_E_SHAPE;
        for (int i = 0; i < 4; ++i) {
            s->q_shape[i] = q->shape[i];
            s->k_shape[i] = k->shape[i];
        }
        s->lse_rank = 3;
        s->lse_shape[0] = s->B;
        s->lse_shape[1] = s->Hq;
        s->lse_shape[2] = s->Sq;
    }
    if (s->D != 64 && s->D != 128) return ATTN_E_UNSUPPORTED;
    if (s->Hkv <= 0 || s->Hq <= 0 || s->Hq % s->Hkv != 0) return ATTN_E_SHAPE;
    if (s->Sq > INT32_MAX / 2 || s->Sk > INT32_MAX / 2 || s->T > INT32_MAX / 2 ||
        s->B > 65535 || s->Hq > 65535)
        return ATTN_E_UNSUPPORTED;
    return ATTN_OK;
}

void strides_in(const attn_tensor_t* t, int varlen, int64_t* xb, int64_t* xs, int64_t* xh) {
    if (varlen) {
        *xb = 0;
        *xs = t->stride[0];
        *xh = t->stride[1];
    } else {
        *xb = t->stride[0];
        *xs = t->stride[1];
        *xh = t->stride[2];
    }
}

int fill_common(Problem* p, const Shapes& s, const attn_tensor_t* q, const attn_tensor_t* k,
                const attn_tensor_t* v, const attn_tensor_t* mask, const attn_tensor_t* cu,
                int causal, float scale, uint32_t flags) {
    *p = Problem();
    p->q = static_cast<const bf16*>(q->data);
    p->k = static_cast<const bf16*>(k->data);
    p->v = static_cast<const bf16*>(v->data);
    strides_in(q, s.varlen, &p->q_b, &p->q_s, &p->q_h);
    strides_in(k, s.varlen, &p->k_b, &p->k_s, &p->k_h);
    strides_in(v, s.varlen, &p->v_b, &p->v_s, &p->v_h);
    p->B = static_cast<int>(s.B);
    p->Hq = static_cast<int>(s.Hq);
    p->Hkv = static_cast<int>(s.Hkv);
    p->G = static_cast<int>(s.Hq / s.Hkv);
    p->Sq = static_cast<int>(s.Sq);
    p->Sk = static_cast<int>(s.Sk);
    p->D = static_cast<int>(s.D);
    p->f16 = s.elt == ATTN_F16 ? 1 : 0;
    p->varlen = s.varlen;
    p->cu = s.varlen ? static_cast<const int*>(cu->data) : nullptr;
    p->T = static_cast<int>(s.T);
    if (s.varlen) {
        p->out_b = 0;
        p->out_s = s.Hq * s.D;
        p->out_h = s.D;
        p->dk_b = 0;
        p->dk_s = s.Hkv * s.D;
        p->dk_h = s.D;
        p->lse_b = 0;
        p->lse_h = s.T;
        p->acc_b = 0;
    } else {
        p->out_b = s.Sq * s.Hq * s.D;
        p->out_s = s.Hq * s.D;
        p->out_h = s.D;
        p->dk_b = s.Sk * s.Hkv * s.D;
        p->dk_s = s.Hkv * s.D;
        p->dk_h = s.D;
        p->lse_b = s.Hq * s.Sq;
        p->lse_h = s.Sq;
        p->acc_b = s.Sq;
    }
    p->mask_kind = MASK_NONE;
    if (mask) {
        if (s.varlen) return ATTN_E_UNSUPPORTED;
        if (!mask->data) return ATTN_E_ARG;
        if (mask->ndim != 4) return ATTN_E_SHAPE;
        const int64_t full[4] = {s.B, s.Hq, s.Sq, s.Sk};
        int64_t st[4];
        for (int i = 0; i < 4; ++i) {
            if (mask->shape[i] != full[i] && mask->shape[i] != 1) return ATTN_E_SHAPE;
            st[i] = mask->shape[i] == 1 ? 0 : mask->stride[i];
            if (st[i] < 0) return ATTN_E_LAYOUT;
        }
        if (mask->dtype == ATTN_U8)
            p->mask_kind = MASK_BOOL;
        else if (mask->dtype == ATTN_F32)
            p->mask_kind = MASK_F32;
        else if (mask->dtype == ATTN_BF16)
            p->mask_kind = MASK_BF16;
        else if (mask->dtype == ATTN_F16)
            p->mask_kind = MASK_F16;
        else
            return ATTN_E_DTYPE;
        // the kernels load mask elements one by one: element alignment suffices
        const uintptr_t esz = mask->dtype == ATTN_U8 ? 1 : (mask->dtype == ATTN_F32 ? 4 : 2);
        if ((reinterpret_cast<uintptr_t>(mask->data) & (esz - 1)) != 0) return ATTN_E_LAYOUT;
        p->mask = mask->data;
        p->m_b = st[0];
        p->m_h = st[1];
        p->m_q = st[2];
        p->m_k = st[3];
    }
    if (!isfinite(scale)) return ATTN_E_ARG;
    p->causal = causal ? 1 : 0;
    p->scale = scale;
    p->scale_log2 = scale * 1.4426950408889634f;
    p->lazy = (flags & ATTN_EAGER_RESCALE) ? 0 : 1;
    p->debug_stall = debug_stall_point();
    return ATTN_OK;
}

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return ATTN_E_CUDA;
    return ATTN_OK;
}

// Device checks and the error word; runs after every host-only check.
int bind_device(Problem* p, std::initializer_list<const attn_tensor_t*> ts) {
    int dev;
    ATTN_TRY(current_device(&dev));
    for (const attn_tensor_t* t : ts) ATTN_TRY(check_device(t, dev));
    p->err = error_word(dev);
    return p->err ? ATTN_OK : ATTN_E_CUDA;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t acc, delta, lse2, total;
};

WsLayout ws_layout(const Shapes& s, uint32_t flags) {
    const int64_t rows = s.varlen ? s.T : s.B * s.Sq;
    WsLayout w;
    const size_t acc_bytes =
        (flags & ATTN_DETERMINISTIC) ? 0 : round256(static_cast<size_t>(rows * s.Hq * s.D) * 4);
    const size_t vec_bytes = round256(static_cast<size_t>(rows * s.Hq) * 4);
    w.acc = 0;
    w.delta = acc_bytes;
    w.lse2 = w.delta + vec_bytes;
    w.total = w.lse2 + vec_bytes;
    return w;
}


}  // namespace

int debug_stall_point() { return g_debug_stall.load(std::memory_order_relaxed); }

}  // namespace attn

using namespace attn;

extern "C" int attn_fwd(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
                        const attn_tensor_t* mask, const attn_tensor_t* cu_seqlens,
                        int32_t max_seqlen, int causal, float scale, attn_tensor_t* out,
                        attn_tensor_t* lse, uint32_t flags, attn_stream_t stream) {
    Shapes s;
    ATTN_TRY(derive_shapes(q, k, v, cu_seqlens, max_seqlen, &s));
    ATTN_TRY(check_output(out, s.elt, s.q_shape, s.rank));
    ATTN_TRY(check_output(lse, ATTN_F32, s.lse_shape, s.lse_rank));
    Problem p;
    ATTN_TRY(fill_common(&p, s, q, k, v, mask, cu_seqlens, causal, scale, flags));
    ATTN_TRY(bind_device(&p, {q, k, v, mask, cu_seqlens, out, lse}));
    p.out = static_cast<bf16*>(out->data);
    p.lse = static_cast<float*>(lse->data);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (s.varlen) ATTN_TRY(run_stage(-1, st, [&] { return launch_zero_trailing_fwd(p, st); }));
    return run_stage(ATTN_STAGE_FWD, st, [&] { return launch_fwd(p, st); });
}

namespace attn {
namespace {

// E4M3 input of the fp8 forward: rank 4, last stride 1, other strides multiples
// of 16 elements (bytes) for dims longer than 1, 16-byte aligned base.
int check_fp8_input(const attn_tensor_t* t) {
    if (!t) return ATTN_E_ARG;
    if (t->dtype != ATTN_E4M3) return ATTN_E_DTYPE;
    if (t->ndim != 4) return ATTN_E_SHAPE;
    int64_t n = 1;
    for (int i = 0; i < 4; ++i) {
        if (t->shape[i] < 0) return ATTN_E_SHAPE;
        n *= t->shape[i];
    }
    if (n > 0 && !t->data) return ATTN_E_ARG;
    if (t->stride[3] != 1) return ATTN_E_LAYOUT;
    for (int i = 0; i < 3; ++i)
        if (t->shape[i] > 1 && (t->stride[i] <= 0 || (t->stride[i] % 16) != 0)) return ATTN_E_LAYOUT;
    if (!aligned16(t->data)) return ATTN_E_LAYOUT;
    return ATTN_OK;
}

int64_t fp8_keys_padded(int64_t Sk) { return (Sk + 15) / 16 * 16; }

size_t fp8_workspace(const attn_tensor_t* k) {
    if (!k || k->ndim != 4 || k->shape[3] != 128) return 0;
    for (int i = 0; i < 4; ++i)
        if (k->shape[i] < 0) return 0;
    return round256(static_cast<size_t>(k->shape[0] * k->shape[2] * 128 * fp8_keys_padded(k->shape[1])));
}

}  // namespace
}  // namespace attn

extern "C" size_t attn_fwd_fp8_workspace_bytes(const attn_tensor_t* k) { return fp8_workspace(k); }

extern "C" int attn_fwd_fp8(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
                            float descale_q, float descale_k, float descale_v, int causal,
                            float scale, attn_tensor_t* out, attn_tensor_t* lse, void* workspace,
                            size_t workspace_bytes, uint32_t flags, attn_stream_t stream) {
    if (!q || !k || !v) return ATTN_E_ARG;
    if (q->dtype != ATTN_E4M3 || k->dtype != ATTN_E4M3 || v->dtype != ATTN_E4M3) return ATTN_E_DTYPE;
    if (q->ndim == 4 && q->shape[3] != 128) return ATTN_E_UNSUPPORTED;
    ATTN_TRY(check_fp8_input(q));
    ATTN_TRY(check_fp8_input(k));
    ATTN_TRY(check_fp8_input(v));
    const int64_t B = q->shape[0], Sq = q->shape[1], Hq = q->shape[2], D = q->shape[3];
    const int64_t Sk = k->shape[1], Hkv = k->shape[2];
    if (k->shape[0] != B || k->shape[3] != D || !same_shape(v, k->shape, 4)) return ATTN_E_SHAPE;
    if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return ATTN_E_SHAPE;
    if (Sq > INT32_MAX / 2 || Sk > INT32_MAX / 2 || B > 65535 || Hq > 65535) return ATTN_E_UNSUPPORTED;
    const int64_t qshape[4] = {B, Sq, Hq, D};
    const int64_t lshape[3] = {B, Hq, Sq};
    ATTN_TRY(check_output(out, ATTN_BF16, qshape, 4));
    ATTN_TRY(check_output(lse, ATTN_F32, lshape, 3));
    if (!isfinite(scale) || !isfinite(descale_q) || !isfinite(descale_k) || !isfinite(descale_v) ||
        !(descale_q > 0.f) || !(descale_k > 0.f) || !(descale_v > 0.f))
        return ATTN_E_ARG;
    const size_t need = fp8_workspace(k);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return ATTN_E_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_E_WORKSPACE;
    }
    Fp8Problem p = {};
    p.q = static_cast<const uint8_t*>(q->data);
    p.k = static_cast<const uint8_t*>(k->data);
    p.v = static_cast<const uint8_t*>(v->data);
    p.vt = static_cast<uint8_t*>(workspace);
    p.q_b = q->stride[0]; p.q_s = q->stride[1]; p.q_h = q->stride[2];
    p.k_b = k->stride[0]; p.k_s = k->stride[1]; p.k_h = k->stride[2];
    p.v_b = v->stride[0]; p.v_s = v->stride[1]; p.v_h = v->stride[2];
    p.Sk_pad = static_cast<int>(fp8_keys_padded(Sk));
    p.vt_h = static_cast<int64_t>(128) * p.Sk_pad;
    p.vt_b = p.vt_h * Hkv;
    p.out = static_cast<bf16*>(out->data);
    p.lse = static_cast<float*>(lse->data);
    p.out_b = Sq * Hq * D; p.out_s = Hq * D; p.out_h = D;
    p.lse_b = Hq * Sq; p.lse_h = Sq;
    p.B = static_cast<int>(B); p.Hq = static_cast<int>(Hq); p.Hkv = static_cast<int>(Hkv);
    p.G = static_cast<int>(Hq / Hkv);
    p.Sq = static_cast<int>(Sq); p.Sk = static_cast<int>(Sk);
    p.causal = causal ? 1 : 0;
    p.lazy = (flags & ATTN_EAGER_RESCALE) ? 0 : 1;
    p.scale_log2 = scale * descale_q * descale_k * 1.4426950408889634f;
    p.out_scale = descale_v;
    p.debug_stall = debug_stall_point();
    int dev;
    ATTN_TRY(current_device(&dev));
    for (const attn_tensor_t* t : {q, k, v, static_cast<const attn_tensor_t*>(out),
                                   static_cast<const attn_tensor_t*>(lse)})
        ATTN_TRY(check_device(t, dev));
    p.err = error_word(dev);
    if (!p.err) return ATTN_E_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    ATTN_TRY(run_stage(-1, st, [&] { return launch_fp8_transpose_v(p, st); }));
    return run_stage(ATTN_STAGE_FWD, st, [&] { return launch_fwd_fp8(p, st); });
}

extern "C" size_t attn_bwd_workspace_bytes(const attn_tensor_t* q, const attn_tensor_t* k,
                                           uint32_t flags) {
    if (!q || !k) return 0;
    Shapes s;
    s.varlen = q->ndim == 3;
    if (s.varlen) {
        s.T = q->shape[0];
        s.Hq = q->shape[1];
        s.D = q->shape[2];
        s.B = 0;
        s.Sq = 0;
    } else if (q->ndim == 4) {
        s.B = q->shape[0];
        s.Sq = q->shape[1];
        s.Hq = q->shape[2];
        s.D = q->shape[3];
        s.T = 0;
    } else {
        return 0;
    }
    if (s.D != 64 && s.D != 128) return 0;
    return ws_layout(s, flags).total;
}

extern "C" int attn_bwd(const attn_tensor_t* q, const attn_tensor_t* k, const attn_tensor_t* v,
                        const attn_tensor_t* out, const attn_tensor_t* dout,
                        const attn_tensor_t* lse, const attn_tensor_t* mask,
                        const attn_tensor_t* cu_seqlens, int32_t max_seqlen, int causal,
                        float scale, attn_tensor_t* dq, attn_tensor_t* dk, attn_tensor_t* dv,
                        void* workspace, size_t workspace_bytes, uint32_t flags,
                        attn_stream_t stream) {
    Shapes s;
    ATTN_TRY(derive_shapes(q, k, v, cu_seqlens, max_seqlen, &s));
    if (!out || !dout || !lse) return ATTN_E_ARG;
    ATTN_TRY(check_input(out, s.rank, s.elt));
    ATTN_TRY(check_input(dout, s.rank, s.elt));
    if (!same_shape(out, s.q_shape, s.rank) || !same_shape(dout, s.q_shape, s.rank))
        return ATTN_E_SHAPE;
    // lse is read back in the layout attn_fwd wrote it: the same contract as its output
    ATTN_TRY(check_output(lse, ATTN_F32, s.lse_shape, s.lse_rank));
    ATTN_TRY(check_output(dq, s.elt, s.q_shape, s.rank));
    ATTN_TRY(check_output(dk, s.elt, s.k_shape, s.rank));
    ATTN_TRY(check_output(dv, s.elt, s.k_shape, s.rank));
    const WsLayout w = ws_layout(s, flags);
    if (w.total > 0) {
        if (!workspace) return ATTN_E_WORKSPACE;
        if (workspace_bytes < w.total) return ATTN_E_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_E_WORKSPACE;
    }
    Problem p;
    ATTN_TRY(fill_common(&p, s, q, k, v, mask, cu_seqlens, causal, scale, flags));
    ATTN_TRY(bind_device(&p, {q, k, v, out, dout, lse, mask, cu_seqlens, dq, dk, dv}));
    p.o = static_cast<const bf16*>(out->data);
    strides_in(out, s.varlen, &p.o_b, &p.o_s, &p.o_h);
    p.dout = static_cast<const bf16*>(dout->data);
    strides_in(dout, s.varlen, &p.do_b, &p.do_s, &p.do_h);
    p.lse = static_cast<float*>(lse->data);
    p.dq = static_cast<bf16*>(dq->data);
    p.dk = static_cast<bf16*>(dk->data);
    p.dv = static_cast<bf16*>(dv->data);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool det = (flags & ATTN_DETERMINISTIC) != 0;
    p.dq_acc = det ? nullptr : reinterpret_cast<float*>(ws + w.acc);
    p.delta = reinterpret_cast<float*>(ws + w.delta);
    p.lse2 = reinterpret_cast<float*>(ws + w.lse2);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!det && w.delta > 0) {
        const cudaError_t e = cudaMemsetAsync(ws + w.acc, 0, w.delta, st);
        if (e != cudaSuccess) return cuda_fail(e, "workspace zero-fill");
    }
    ATTN_TRY(run_stage(ATTN_STAGE_BWD_PREPROCESS, st, [&] { return launch_bwd_preprocess(p, st); }));
    if (s.varlen) ATTN_TRY(run_stage(-1, st, [&] { return launch_zero_trailing_bwd(p, st); }));
    ATTN_TRY(run_stage(ATTN_STAGE_BWD_MAIN, st, [&] { return launch_bwd_main(p, !det, st); }));
    if (det)
        return run_stage(ATTN_STAGE_BWD_DQ, st, [&] { return launch_bwd_dq_deterministic(p, st); });
    return run_stage(ATTN_STAGE_BWD_DQ, st, [&] { return launch_bwd_dq_convert(p, st); });
}

// ------------------------------------------------------------------ score recompute

namespace attn {
namespace {

// Rows and width of the score output and the L1-partial workspace size.
void score_dims(const Shapes& s, int64_t* rows, int64_t* width) {
    *rows = s.varlen ? s.T : s.B * s.Sq;
    *width = s.varlen ? s.Sq : s.Sk;
}

size_t score_workspace(const Shapes& s) {
    int64_t rows, width;
    score_dims(s, &rows, &width);
    return round256(static_cast<size_t>(score_key_tiles(width)) * static_cast<size_t>(rows) * 4);
}

}  // namespace
}  // namespace attn

extern "C" size_t attn_score_workspace_bytes(const attn_tensor_t* q, const attn_tensor_t* k,
                                             const attn_tensor_t* cu_seqlens, int32_t max_seqlen) {
    Shapes s;
    if (!q || !k) return 0;
    if (derive_shapes(q, k, k, cu_seqlens, max_seqlen, &s) != ATTN_OK) return 0;
    return score_workspace(s);
}

extern "C" int attn_score_recompute(const attn_tensor_t* q, const attn_tensor_t* k,
                                    const attn_tensor_t* lse, const attn_tensor_t* cu_seqlens,
                                    int32_t max_seqlen, int causal, float scale,
                                    attn_tensor_t* score, attn_tensor_t* l1, void* workspace,
                                    size_t workspace_bytes, uint32_t flags,
                                    attn_stream_t stream) {
    if (flags != 0) return ATTN_E_ARG;
    Shapes s;
    ATTN_TRY(derive_shapes(q, k, k, cu_seqlens, max_seqlen, &s));
    // lse is read in the layout attn_fwd wrote it
    ATTN_TRY(check_output(lse, ATTN_F32, s.lse_shape, s.lse_rank));
    int64_t rows, width;
    score_dims(s, &rows, &width);
    const int64_t sshape_d[3] = {s.B, s.Sq, s.Sk};
    const int64_t sshape_v[2] = {s.T, s.Sq};
    ATTN_TRY(check_output(score, ATTN_F32, s.varlen ? sshape_v : sshape_d, s.varlen ? 2 : 3));
    const int64_t lshape_d[2] = {s.B, s.Sq};
    const int64_t lshape_v[1] = {s.T};
    ATTN_TRY(check_output(l1, ATTN_F32, s.varlen ? lshape_v : lshape_d, s.varlen ? 1 : 2));
    const size_t need = score_workspace(s);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return ATTN_E_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_E_WORKSPACE;
    }
    Problem p;
    ATTN_TRY(fill_common(&p, s, q, k, k, nullptr, cu_seqlens, causal, scale, 0));
    ATTN_TRY(bind_device(&p, {q, k, lse, cu_seqlens, score, l1}));
    p.lse = static_cast<float*>(lse->data);
    p.score = static_cast<float*>(score->data);
    p.l1 = static_cast<float*>(l1->data);
    p.l1_part = static_cast<float*>(workspace);
    p.sc_w = width;
    p.l1_rows = rows;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return run_stage(ATTN_STAGE_SCORE, st, [&] { return launch_score_recompute(p, st); });
}

namespace attn {
namespace {

// Sparse top-k backward: the shape contract, every tensor against q
// (NVIDIA/cudnn-frontend PR #429: a transposed dout or lse, a mis-shaped
// index tensor or an unsupported head dim must fail before launch).
struct SparseShapes {
    int elt;
    int64_t B, S, H, D, Skv, K;
};

int sparse_shapes(const attn_tensor_t* q, const attn_tensor_t* kv, SparseShapes* s) {
    if (!q || !kv) return ATTN_E_ARG;
    if (q->dtype != ATTN_BF16 && q->dtype != ATTN_F16) return ATTN_E_DTYPE;
    s->elt = q->dtype;
    ATTN_TRY(check_input(q, 4, s->elt));
    s->B = q->shape[0];
    s->S = q->shape[1];
    s->H = q->shape[2];
    s->D = q->shape[3];
    if (s->H != 64 || (s->D != 512 && s->D != 576)) return ATTN_E_UNSUPPORTED;
    ATTN_TRY(check_input(kv, 3, s->elt));
    if (kv->shape[0] != s->B || kv->shape[2] != s->D) return ATTN_E_SHAPE;
    s->Skv = kv->shape[1];
    if (s->B * s->S > INT32_MAX / 2 || s->Skv > INT32_MAX / 2) return ATTN_E_SHAPE;
    return ATTN_OK;
}

struct SparseWs {
    size_t acc, delta, sink, total;
};

SparseWs sparse_ws(const SparseShapes& s, bool with_sink) {
    SparseWs w;
    const size_t vec = round256(static_cast<size_t>(s.B * s.S * s.H) * 4);
    w.acc = 0;
    w.delta = round256(static_cast<size_t>(s.B * s.Skv * s.D) * 4);
    w.sink = w.delta + vec;
    w.total = w.sink + (with_sink ? vec : 0);
    return w;
}

// int32 index tensor: the given shape, contiguous, 4-byte aligned.
int check_index(const attn_tensor_t* t, const int64_t* shape, int rank) {
    if (!t) return ATTN_E_ARG;
    if (t->dtype != ATTN_I32) return ATTN_E_DTYPE;
    if (!same_shape(t, shape, rank)) return ATTN_E_SHAPE;
    int64_t n = 1;
    for (int i = 0; i < rank; ++i) n *= shape[i];
    if (n > 0 && !t->data) return ATTN_E_ARG;
    if (!is_contiguous(t)) return ATTN_E_LAYOUT;
    if ((reinterpret_cast<uintptr_t>(t->data) & 3u) != 0) return ATTN_E_LAYOUT;
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" size_t attn_sparse_bwd_workspace_bytes(const attn_tensor_t* q, const attn_tensor_t* kv,
                                                  int with_sink) {
    attn::SparseShapes s;
    if (attn::sparse_shapes(q, kv, &s) != ATTN_OK) return 0;
    return attn::sparse_ws(s, with_sink != 0).total;
}

extern "C" int attn_sparse_bwd(const attn_tensor_t* q, const attn_tensor_t* kv,
                               const attn_tensor_t* out, const attn_tensor_t* dout,
                               const attn_tensor_t* lse, const attn_tensor_t* attn_sink,
                               const attn_tensor_t* topk_idxs, const attn_tensor_t* topk_length,
                               float scale, attn_tensor_t* dq, attn_tensor_t* dkv,
                               attn_tensor_t* d_sink, void* workspace, size_t workspace_bytes,
                               uint32_t flags, attn_stream_t stream) {
    using namespace attn;
    if (flags != 0) return ATTN_E_ARG;
    if (!isfinite(scale)) return ATTN_E_ARG;
    SparseShapes s;
    ATTN_TRY(sparse_shapes(q, kv, &s));
    const int64_t oshape[4] = {s.B, s.S, s.H, 512};
    ATTN_TRY(check_input(out, 4, s.elt));
    ATTN_TRY(check_input(dout, 4, s.elt));
    if (!same_shape(out, oshape, 4) || !same_shape(dout, oshape, 4)) return ATTN_E_SHAPE;
    const int64_t lshape[3] = {s.B, s.S, s.H};
    ATTN_TRY(check_output(lse, ATTN_F32, lshape, 3));
    if (!topk_idxs) return ATTN_E_ARG;
    if (topk_idxs->ndim != 3) return ATTN_E_SHAPE;
    s.K = topk_idxs->shape[2];
    const int64_t ishape[3] = {s.B, s.S, s.K};
    ATTN_TRY(check_index(topk_idxs, ishape, 3));
    const int64_t nshape[2] = {s.B, s.S};
    if (topk_length) ATTN_TRY(check_index(topk_length, nshape, 2));
    const int64_t hshape[1] = {s.H};
    if ((attn_sink == nullptr) != (d_sink == nullptr)) return ATTN_E_ARG;
    if (attn_sink) {
        ATTN_TRY(check_output(attn_sink, ATTN_F32, hshape, 1));
        ATTN_TRY(check_output(d_sink, ATTN_F32, hshape, 1));
    }
    ATTN_TRY(check_output(dq, s.elt, q->shape, 4));
    ATTN_TRY(check_output(dkv, s.elt, kv->shape, 3));
    const SparseWs w = sparse_ws(s, attn_sink != nullptr);
    if (!workspace || workspace_bytes < w.total) return ATTN_E_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_E_WORKSPACE;
    int dev;
    ATTN_TRY(current_device(&dev));
    for (const attn_tensor_t* t : {q, kv, out, dout, lse, attn_sink, topk_idxs, topk_length,
                                   static_cast<const attn_tensor_t*>(dq),
                                   static_cast<const attn_tensor_t*>(dkv),
                                   static_cast<const attn_tensor_t*>(d_sink)})
        ATTN_TRY(check_device(t, dev));
    SparseProblem p{};
    p.err = error_word(dev);
    if (!p.err) return ATTN_E_CUDA;
    p.q = static_cast<const bf16*>(q->data);
    p.kv = static_cast<const bf16*>(kv->data);
    p.out = static_cast<const bf16*>(out->data);
    p.dout = static_cast<const bf16*>(dout->data);
    p.lse = static_cast<const float*>(lse->data);
    p.sink = attn_sink ? static_cast<const float*>(attn_sink->data) : nullptr;
    p.idx = static_cast<const int*>(topk_idxs->data);
    p.len = topk_length ? static_cast<const int*>(topk_length->data) : nullptr;
    p.dq = static_cast<bf16*>(dq->data);
    p.dkv = static_cast<bf16*>(dkv->data);
    p.dsink = d_sink ? static_cast<float*>(d_sink->data) : nullptr;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.dkv_acc = reinterpret_cast<float*>(ws + w.acc);
    p.delta = reinterpret_cast<float*>(ws + w.delta);
    p.dsink_part = attn_sink ? reinterpret_cast<float*>(ws + w.sink) : nullptr;
    p.q_b = q->stride[0], p.q_s = q->stride[1], p.q_h = q->stride[2];
    p.kv_b = kv->stride[0], p.kv_s = kv->stride[1];
    p.o_b = out->stride[0], p.o_s = out->stride[1], p.o_h = out->stride[2];
    p.do_b = dout->stride[0], p.do_s = dout->stride[1], p.do_h = dout->stride[2];
    p.idx_b = s.S * s.K, p.idx_s = s.K;
    p.len_b = s.S, p.len_s = 1;
    p.B = static_cast<int>(s.B), p.S = static_cast<int>(s.S), p.Skv = static_cast<int>(s.Skv);
    p.H = static_cast<int>(s.H), p.Dqk = static_cast<int>(s.D), p.Dv = 512;
    p.K = static_cast<int>(s.K);
    p.f16 = s.elt == ATTN_F16;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.debug_stall = debug_stall_point();
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    const size_t acc_bytes = static_cast<size_t>(s.B * s.Skv * s.D) * 4;
    if (acc_bytes > 0 && (e = cudaMemsetAsync(p.dkv_acc, 0, acc_bytes, st)) != cudaSuccess)
        return cuda_fail(e, "dkv workspace zero-fill");
    ATTN_TRY(run_stage(-1, st, [&] { return launch_sparse_prep(p, st); }));
    if (s.Skv > 0) {
        ATTN_TRY(run_stage(ATTN_STAGE_SPARSE, st, [&] { return launch_sparse_bwd_main(p, st); }));
    } else {
        // no kv row exists, so no entry takes part: dq is zero
        const size_t dq_bytes = static_cast<size_t>(s.B * s.S * s.H * s.D) * 2;
        if (dq_bytes > 0 && (e = cudaMemsetAsync(p.dq, 0, dq_bytes, st)) != cudaSuccess)
            return cuda_fail(e, "dq zero-fill");
    }
    ATTN_TRY(run_stage(-1, st, [&] { return launch_sparse_dkv_convert(p, st); }));
    if (attn_sink) ATTN_TRY(run_stage(-1, st, [&] { return launch_sparse_dsink(p, st); }));
    return ATTN_OK;
}

extern "C" int attn_get_error(attn_stream_t stream) {
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_E_CUDA;
    int* ptr = error_word(dev);
    if (!ptr) return ATTN_E_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_E_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_E_CUDA;
    const int zero = 0;
    if (cudaMemcpy(ptr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return ATTN_E_CUDA;
    return v;
}

extern "C" const char* attn_strerror(int code) {
    switch (code) {
        case ATTN_OK: return "ok";
        case ATTN_E_DTYPE: return "unsupported or mismatched element type (bf16 or fp16 inputs, all alike; fp32 lse)";
        case ATTN_E_SHAPE: return "shape does not match the contract derived from q";
        case ATTN_E_LAYOUT: return "stride, alignment or contiguity violation";
        case ATTN_E_DEVICE: return "tensors are not all on the current CUDA device";
        case ATTN_E_UNSUPPORTED: return "unsupported configuration (head dim must be 64 or 128)";
        case ATTN_E_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case ATTN_E_CUDA: return "a CUDA runtime call failed";
        case ATTN_E_TIMEOUT: return "a bounded device wait gave up";
        case ATTN_E_SEQLENS: return "cu_seqlens malformed or a sequence exceeds max_seqlen";
        case ATTN_E_ARG: return "null pointer, non-finite scale or descale, or descale <= 0";
        case ATTN_E_INTERNAL: return "an internal invariant failed on the device";
        case ATTN_E_TOO_LARGE:
            return "problem needs more scratch than attn_bwd_noalloc's built-in 32 MiB array";
        default: return "unknown error code";
    }
}

extern "C" int attn_version(void) { return 100; }

extern "C" int attn_selftest_wait_timeout(uint32_t budget_us, attn_stream_t stream) {
    if (budget_us == 0 || budget_us > 1000000u) return ATTN_E_ARG;
    int dev;
    ATTN_TRY(current_device(&dev));
    int* err = error_word(dev);
    if (!err) return ATTN_E_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return run_stage(-1, st, [&] {
        return launch_wait_timeout_probe(err, static_cast<uint64_t>(budget_us) * 1000ull, st);
    });
}

extern "C" int attn_profile_events(int stage, void* before, void* after) {
    if (stage < 0 || stage >= ATTN_STAGE_COUNT) return ATTN_E_ARG;
    g_prof[stage][0] = static_cast<cudaEvent_t>(before);
    g_prof[stage][1] = static_cast<cudaEvent_t>(after);
    return ATTN_OK;
}

extern "C" const char* attn_last_cuda_error(void) { return g_cuda_detail; }

extern "C" unsigned long long attn_launch_count(void) {
    return g_launches.load(std::memory_order_relaxed);
}

#ifdef ATTN_DEBUG_CHECKS
// Debug builds only: from now on, the MMA issuer of block (0, 0, 0) of
// `kernel` (1 forward, 2 backward main, 3 deterministic dQ, 4 fp8 forward,
// 5 score recompute) lets its wait at iteration `iteration` run out; kernel <= 0 clears it.
extern "C" int attn_debug_inject_stall(int kernel, int iteration) {
    if (kernel <= 0) {
        g_debug_stall.store(-1);
        return ATTN_OK;
    }
    if (kernel > 6 || iteration < 0 || iteration > 0xffff) return ATTN_E_ARG;
    g_debug_stall.store((kernel << 16) | iteration);
    return ATTN_OK;
}
#endif
