// tma.cu -- host side of the TMA helpers: tensor-map encoding through the
// driver entry point (resolved once; no link-time dependency on libcuda).
#include <mutex>

#include "tma.cuh"

namespace csa {
namespace tma {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
}  // namespace

cudaError_t encode_rows128(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  return encode_rows(map, base, 128, rows, box_rows);
}

cudaError_t encode_rows(CUtensorMap* map, const void* base, uint32_t row_elems, uint64_t rows,
                        uint32_t box_rows) {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &fn, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return cudaErrorNotSupported;
  if (rows == 0) rows = 1;
  const cuuint64_t dims[2] = {row_elems, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_elems * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tma
}  // namespace csa
