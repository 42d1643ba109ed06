// Host: TMA tensor maps. The driver's cuTensorMapEncodeTiled is fetched once
// per process through the runtime, so the library does not link libcuda.
#include <mutex>

#include "tc_helpers.cuh"

namespace sparsp {
namespace {

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

}  // namespace

bool make_tmap_bf16_rows(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_rows) {
  EncodeTiled enc = encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16_raster(CUtensorMap* map, const void* base, const Dims& s) {
  EncodeTiled enc = encoder();
  if (enc == nullptr) return false;
  // [B, T, Y, X, H, d] with B and T merged: (column, head, x, y, frame)
  const uint64_t d = (uint64_t)s.d, H = (uint64_t)s.H;
  const cuuint64_t dims[5] = {d, H, (uint64_t)s.X, (uint64_t)s.Y, (uint64_t)s.B * s.T};
  const cuuint64_t strides[4] = {d * 2, H * d * 2, (uint64_t)s.X * H * d * 2, (uint64_t)s.Y * s.X * H * d * 2};
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)s.tc, (cuuint32_t)s.tb, (cuuint32_t)s.ta};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace sparsp
