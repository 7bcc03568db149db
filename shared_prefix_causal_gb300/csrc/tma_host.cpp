// Tensor-map encoding through the driver entry point (looked up once through
// the runtime, so the library needs no link-time dependency on libcuda).
#include "tma_host.h"

#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace spc {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

}  // namespace

int encode_bf16_3d(CUtensorMap *map, const void *base, int inner, int mid, int outer, int box_inner, int box_mid,
                   int box_outer) {
  EncodeFn fn = encoder();
  if (!fn) return SP_ERR_CUDA;
  const cuuint64_t dims[3] = {cuuint64_t(inner), cuuint64_t(mid), cuuint64_t(outer)};
  const cuuint64_t strides[2] = {cuuint64_t(inner) * 2, cuuint64_t(inner) * mid * 2};
  const cuuint32_t box[3] = {cuuint32_t(box_inner), cuuint32_t(box_mid), cuuint32_t(box_outer)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SP_OK : SP_ERR_CUDA;
}

int encode_bf16_2d(CUtensorMap *map, const void *base, int cols, int rows, int box_cols, int box_rows) {
  EncodeFn fn = encoder();
  if (!fn) return SP_ERR_CUDA;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SP_OK : SP_ERR_CUDA;
}

}  // namespace spc
