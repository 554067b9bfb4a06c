// attn_bwd_noalloc: the backward pass for callers that cannot hand the
// library a workspace.
//
// attn_bwd needs a scratch buffer (the fp32 dQ accumulator and two per-row
// vectors) that the caller allocates.  Some callers cannot allocate device
// memory at the moment they run the backward: a plugin living inside a host
// framework that owns all device memory and exposes no allocator to it, or a
// real-time / embedded caller whose device-memory budget is fixed when the
// process starts.  For them this entry point uses a scratch array that is
// part of the library image itself: a file-scope __device__ array that the
// CUDA runtime places in device memory when the module is loaded on a GPU,
// so nothing is allocated at call time.
//
// Costs and limits, stated for the user:
//   * every GPU that loads the library holds kNoallocScratchBytes of device
//     memory for the scratch until the process exits;
//   * problems whose workspace (attn_bwd_workspace_bytes) is larger than that
//     are rejected with ATTN_E_TOO_LARGE before anything is launched;
//   * the first call on a device looks up the array's device address (and,
//     if nothing else has yet, makes the runtime load the library's device
//     code on that device); make that first call before any stream capture;
//   * all calls on a device share the one array: two calls whose work
//     overlaps on the GPU (different streams, no ordering between them) race
//     on it and give wrong gradients.  Order such calls on one stream, or
//     with events;
//   * the array keeps whatever the previous call left in it; the part that
//     must start at zero (the dQ accumulator) is zero-filled on `stream` by
//     every call, and the rest is fully overwritten before it is read.
#include <mutex>

#include "../../include/attn_gb300.h"
#include "attn_internal.h"

namespace attn {
namespace {

// 32 MiB: at D = 128 the workspace is 520 bytes per (query row, head), so
// this covers about 64 K (row, head) pairs, e.g. B*S*Hq = 4 * 1024 * 16.
constexpr size_t kNoallocScratchBytes = size_t(32) << 20;

// In host code this name is only a stand-in for the device array: its host
// address must never reach a kernel.  The device address comes from
// cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_dev_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

int scratch_for_device(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return ATTN_E_DEVICE;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_dev_ptr[dev]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) return ATTN_E_CUDA;
        g_scratch_dev_ptr[dev] = ptr;
    }
    *out = g_scratch_dev_ptr[dev];
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" int attn_bwd_noalloc(const attn_tensor_t* q, const attn_tensor_t* k,
                                const attn_tensor_t* v, const attn_tensor_t* out,
                                const attn_tensor_t* dout, const attn_tensor_t* lse,
                                const attn_tensor_t* mask, const attn_tensor_t* cu_seqlens,
                                int32_t max_seqlen, int causal, float scale, attn_tensor_t* dq,
                                attn_tensor_t* dk, attn_tensor_t* dv, uint32_t flags,
                                attn_stream_t stream) {
    if (!q || !k) return ATTN_E_ARG;
    const size_t need = attn_bwd_workspace_bytes(q, k, flags);
    if (need > attn::kNoallocScratchBytes) return ATTN_E_TOO_LARGE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_E_CUDA;
    void* scratch = nullptr;
    const int rc = attn::scratch_for_device(dev, &scratch);
    if (rc != ATTN_OK) return rc;
    return attn_bwd(q, k, v, out, dout, lse, mask, cu_seqlens, max_seqlen, causal, scale, dq, dk,
                    dv, scratch, attn::kNoallocScratchBytes, flags, stream);
}
