// Host-side construction of TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry-point query so the library needs no
// link-time dependency on libcuda).
#include "attn_internal.h"

namespace attn {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

}  // namespace

bool make_tile_map(CUtensorMap* m, const void* base, int64_t D, int64_t H, int64_t S, int64_t B,
                   int64_t sh, int64_t ss, int64_t sb, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)(sh * 2), (cuuint64_t)(ss * 2), (cuuint64_t)(sb * 2)};
    // Strides of size-1 dims are never used; keep them legal (16-byte multiples).
    if (H == 1) strides[0] = (cuuint64_t)(D * 2);
    if (B == 1) strides[2] = strides[1] * (cuuint64_t)(S > 0 ? S : 1);
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_heads_map(CUtensorMap* m, const void* base, int64_t D, int64_t H, int64_t S, int64_t B,
                    int64_t sh, int64_t ss, int64_t sb, bool f16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(S > 0 ? S : 1),
                          (cuuint64_t)(B > 0 ? B : 1)};
    cuuint64_t strides[3] = {(cuuint64_t)(sh * 2), (cuuint64_t)(ss * 2), (cuuint64_t)(sb * 2)};
    // Strides of size-1 dims are never used; keep them legal (16-byte multiples).
    if (dims[2] == 1) strides[1] = strides[0] * dims[1];
    if (dims[3] == 1) strides[2] = strides[1] * dims[2];
    cuuint32_t box[4] = {64, 64, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_f32_reduce_map(CUtensorMap* m, void* base, int64_t D, int64_t H, int64_t R) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(R > 0 ? R : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)(D * 4), (cuuint64_t)(H * D * 4)};
    cuuint32_t box[3] = {32, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_u8_map(CUtensorMap* m, const void* base, const int64_t dims[4], const int64_t strides[3],
                 int box1, int box2) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t d[4], st[3];
    for (int i = 0; i < 4; ++i) d[i] = (cuuint64_t)(dims[i] > 0 ? dims[i] : 1);
    for (int i = 0; i < 3; ++i) st[i] = (cuuint64_t)strides[i];
    // Strides of size-1 dims are never used; keep them legal (16-byte multiples).
    if (d[1] == 1) st[0] = d[0];
    if (d[2] == 1) st[1] = st[0] * d[1];
    if (d[3] == 1) st[2] = st[1] * d[2];
    cuuint32_t box[4] = {128, (cuuint32_t)box1, (cuuint32_t)box2, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), d, st, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace attn
