// TMA tensor maps (cuTensorMapEncodeTiled, reached through the runtime's
// driver entry-point lookup so the library needs no link-time libcuda).
#include <cuda.h>

#include "common.cuh"

namespace kvc {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

bool encode3d(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int cols, int64_t ld, int rows,
              int H, uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)ld * esize, (cuuint64_t)rows * ld * esize};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool tc_maps_available() { return encode_fn() != nullptr; }

// [H][rows][d] bf16 as a 3-D tensor (d, rows, H): boxes of [128 rows][64
// elements] (128 bytes) with 128-byte swizzle; rows past a head's end read 0.
bool make_map(CUtensorMap* m, const void* base, int d, int rows, int H) {
    return encode3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, d, d, rows, H, 64, 128);
}

// The same with boxes of [256 rows][64 elements]: the 256-query operand
// blocks of the key-score pass.
bool make_map_rows256(CUtensorMap* m, const void* base, int d, int rows, int H) {
    return encode3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, d, d, rows, H, 64, 256);
}

// [H][rows][ld] fp32 (first `cols` columns addressed) as a 3-D tensor: boxes
// of [32 rows][32 columns] (128 bytes) with 128-byte swizzle; reads past the
// addressed columns or rows return 0.
bool make_map_f32(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H) {
    return encode3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, cols, ld, rows, H, 32, 32);
}

// [H][rows][ld] bf16 (first `cols` columns addressed) as a 3-D tensor: boxes
// of [64 rows][64 columns] (128 bytes) with 128-byte swizzle, the MN-major
// operand layout of the Gram products; reads past the addressed columns or
// rows return 0.
bool make_map_bf16(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H) {
    return encode3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, ld, rows, H, 64, 64);
}

// The same bf16 layout with boxes of [32 rows][64 columns]: the store boxes
// of a warp's 32 rows.
bool make_map_bf16_rows32(CUtensorMap* m, const void* base, int cols, int64_t ld, int rows, int H) {
    return encode3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, ld, rows, H, 64, 32);
}

}  // namespace kvc
