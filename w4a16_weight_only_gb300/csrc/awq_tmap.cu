// Host helper: encode 2D TMA tensor maps through the driver entry point obtained from the
// runtime (no link-time dependency on libcuda, so the library loads without a driver).
#include <mutex>

#include "awq_internal.cuh"

namespace awq {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                  const void* base, uint64_t dim0, uint64_t dim1, uint32_t box0, uint32_t box1,
                  CUtensorMapSwizzle swizzle, const char** why) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {dim0 * elem_bytes};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled rejected a tensor map";
    return false;
  }
  return true;
}

bool make_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                  const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2, uint32_t box0,
                  uint32_t box1, CUtensorMapSwizzle swizzle, const char** why) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    *why = "cuTensorMapEncodeTiled unavailable";
    return false;
  }
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {dim0 * elem_bytes, dim0 * dim1 * elem_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled rejected a 3D tensor map";
    return false;
  }
  return true;
}

}  // namespace awq
