// tmap.cu -- host helpers of the tensor-core path: TMA tensor-map encoding
// (through the driver entry point, so the library does not link libcuda) and
// the SM count.
#include <cudaTypedefs.h>

#include "gdn_internal.h"

namespace gdn {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return (PFN_cuTensorMapEncodeTiled_v12000)p;
    }();
    return fn;
}

// [B, T, H, D] bf16 -> 4D map (D, H, T, B); box 64 x 1 x 64 x 1, 128B swizzle.
bool tmap_bthd(CUtensorMap* m, const void* ptr, int B, int T, int H, int D) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, cols] bf16 row-major -> 2D map; box 64 x 64, 128B swizzle.
bool tmap_rows(CUtensorMap* m, const void* ptr, int64_t rows, int cols) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t str[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int n = [] {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        return v > 0 ? v : 148;
    }();
    return n;
}

// [rows, cols] bf16 row-major seen as 3D (8, rows, cols/8): a box (8, R, n) lands in
// shared memory as the no-swizzle MN-major operand layout [n][R][8] (core matrices
// of 8 rows x 16 bytes).  Box rows R = box_rows, n = box_groups.
bool tmap_core8_rows(CUtensorMap* m, const void* ptr, int64_t rows, int cols, int box_rows,
                     int box_groups) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {8, (cuuint64_t)rows, (cuuint64_t)(cols / 8)};
    cuuint64_t str[2] = {(cuuint64_t)cols * 2, 16};
    cuuint32_t box[3] = {8, (cuuint32_t)box_rows, (cuuint32_t)box_groups};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B, T, H, D] bf16 seen as 5D (8, T, D/8, H, B): a box (8, 64, n, 1, 1) lands as
// the operand layout [n][64 tokens][8] for one (b, h).
bool tmap_core8_bthd(CUtensorMap* m, const void* ptr, int B, int T, int H, int D, int box_groups) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[5] = {8, (cuuint64_t)T, (cuuint64_t)(D / 8), (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t str[4] = {(cuuint64_t)H * D * 2, 16, (cuuint64_t)D * 2, (cuuint64_t)T * H * D * 2};
    cuuint32_t box[5] = {8, 64, (cuuint32_t)box_groups, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(ptr), dims, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_available() { return encode_fn() != nullptr; }

}  // namespace gdn
