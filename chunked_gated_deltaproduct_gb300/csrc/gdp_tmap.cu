// gdp_tmap.cu -- host-side TMA tensor-map encoding shared by the kernels' launchers.
//
// The encoder (cuTensorMapEncodeTiled) is a driver function; it is fetched once through the
// runtime's driver entry point so that the library links against the runtime only.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "gdp_internal.cuh"

namespace gdp {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

cudaError_t encode(CUtensorMap *m, CUtensorMapDataType type, cuuint32_t rank, void *base, const cuuint64_t *dims,
                   const cuuint64_t *strides, const cuuint32_t *box,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, type, rank, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t tmap_state(void *map, float *base, int64_t rows, int d) {
  memset(map, 0, sizeof(CUtensorMap));
  if (!base || rows <= 0) return cudaSuccess;  // unused: left zeroed
  const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d * sizeof(float)};
  const cuuint32_t box[2] = {32, 32};
  return encode(static_cast<CUtensorMap *>(map), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box);
}

cudaError_t tmap_rows_16(void *map, const void *base, int64_t rows, int H, int K, int64_t stride_t, int64_t stride_h,
                         int box_rows, int f16) {
  memset(map, 0, sizeof(CUtensorMap));
  if (!base || rows <= 0) return cudaSuccess;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)stride_h * 2u, (cuuint64_t)stride_t * 2u};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  return encode(static_cast<CUtensorMap *>(map),
                f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                dims, strides, box);
}

cudaError_t tmap_out_rows(void *map, void *base, int64_t T, int H, int V, int box_rows, int f16) {
  memset(map, 0, sizeof(CUtensorMap));
  if (!base || T <= 0) return cudaSuccess;
  const cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)V * 2u, (cuuint64_t)H * V * 2u};
  const cuuint32_t box[3] = {(cuuint32_t)V, 1, (cuuint32_t)box_rows};
  return encode(static_cast<CUtensorMap *>(map),
                f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box,
                CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace gdp
