// static_scratch.cu -- csa_indexer_topk_static: the Lightning-Indexer top-k
// call with its scratch in a fixed device array owned by the library, for
// callers that cannot allocate device memory when they make the call (a
// decode step running inside a device-memory budget reserved up front, where
// the device allocator may synchronise the device; a host runtime with no
// device allocator of its own).  Nothing here allocates: the array is a
// file-scope __device__ object, and its address is looked up once per device.
#include <mutex>

#include "csa.h"
#include "kernels.h"

namespace csa {
namespace {

// One per device (module-scope device variables are instantiated on every
// device the library runs on).  256-byte aligned: the workspace carve keeps
// every region 256-byte aligned relative to the base.
__device__ __align__(256) uint8_t g_indexer_scratch[CSA_INDEXER_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device; looked up on first use.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CSA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_indexer_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return CSA_ERR_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return CSA_OK;
}

}  // namespace
}  // namespace csa

extern "C" CSA_API int csa_indexer_topk_static(
    const void* q_idx, const float* q_scale, const float* w, const void* k_idx, int64_t k_bstride,
    const float* k_scale, int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
    const int32_t* n_cmp, int B, int T, int H_I, int d_I, int N_cap, int m, int k,
    int32_t* topk_idx, float* topk_score, int32_t* err_word, void* stream) {
  // sizes past the array's capacity are refused before any CUDA call
  if (B > 0 && T > 0 && N_cap > 0 && N_cap <= csa::kMaxNcap && (int64_t)B * T <= (1 << 30) &&
      csa_indexer_topk_workspace(B, T, N_cap, k) > CSA_INDEXER_STATIC_SCRATCH_BYTES)
    return CSA_ERR_WORKSPACE;
  if (B == 0 || T == 0) {
    return csa_indexer_topk(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride, idx_dtype,
                            q_pos, n_cmp, B, T, H_I, d_I, N_cap, m, k, topk_idx, topk_score,
                            nullptr, 0, err_word, stream);
  }
  void* ws = nullptr;
  const int st = csa::scratch_address(&ws);
  if (st != CSA_OK) return st;
  return csa_indexer_topk(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride, idx_dtype,
                          q_pos, n_cmp, B, T, H_I, d_I, N_cap, m, k, topk_idx, topk_score, ws,
                          CSA_INDEXER_STATIC_SCRATCH_BYTES, err_word, stream);
}
