// static_scratch.cu -- csa_indexer_topk_static: the Lightning-Indexer top-k
// call with its scratch in a fixed device array owned by the library, for
// callers that cannot allocate device memory when they make the call (a
// decode step running inside a device-memory budget reserved up front, where
// the device allocator may synchronise the device; a host runtime with no
// device allocator of its own).  Nothing here allocates: the array is a
// file-scope __device__ object, and its address is looked up once per device
// context.
#include <cuda.h>

#include <mutex>

#include "csa.h"
#include "kernels.h"

namespace csa {
namespace {

// One per device (module-scope device variables are instantiated on every
// device the library runs on).  256-byte aligned: the workspace carve keeps
// every region 256-byte aligned relative to the base.
__device__ __align__(256) uint8_t g_indexer_scratch[CSA_INDEXER_STATIC_SCRATCH_BYTES];

// The array's address is cached per device together with the id of the
// context it was looked up in: a device reset (cudaDeviceReset) destroys the
// primary context, the module is loaded again into the new one and the array
// may move, so a changed context id repeats the lookup.
constexpr int kMaxDevices = 64;
struct Slot {
  void* addr = nullptr;
  unsigned long long ctx_id = 0;
};
std::mutex g_mu;
Slot g_slot[kMaxDevices];

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);
typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long*);
PFN_ctxGetCurrent g_ctx_current = nullptr;
PFN_ctxGetId g_ctx_id = nullptr;
std::once_flag g_once;

// Id of the calling thread's current context (the device's primary context
// once the runtime has initialised it); 0 if it cannot be read.
unsigned long long current_context_id() {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuCtxGetCurrent", &fn, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_ctxGetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPoint("cuCtxGetId", &fn, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_ctxGetId>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx ||
      g_ctx_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array on the current device (cudaGetSymbolAddress
// with that device current; looked up on first use and again after a reset).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CSA_ERR_CUDA;
  }
  // (before the runtime's first call on this thread there may be no current
  // context yet: id 0, so the lookup runs, and the id is read after it)
  std::lock_guard<std::mutex> lock(g_mu);
  Slot& s = g_slot[dev];
  const unsigned long long id = current_context_id();
  if (!s.addr || id == 0 || id != s.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_indexer_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return CSA_ERR_CUDA;
    }
    s.addr = p;
    s.ctx_id = current_context_id();  // the lookup made the context current if it was not
  }
  *out = s.addr;
  return CSA_OK;
}

}  // namespace
}  // namespace csa

extern "C" CSA_API int csa_indexer_topk_static(
    const void* q_idx, const float* q_scale, const float* w, const void* k_idx, int64_t k_bstride,
    const float* k_scale, int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
    const int32_t* n_cmp, int B, int T, int H_I, int d_I, int N_cap, int m, int k,
    int32_t* topk_idx, float* topk_score, int32_t* err_word, void* stream) {
  // the same argument checks (and statuses) as csa_indexer_topk, then the
  // capacity; all of them before any CUDA call
  const int c = csa::indexer_topk_arg_status(q_idx, q_scale, w, k_idx, k_bstride, k_scale,
                                             ks_bstride, idx_dtype, q_pos, n_cmp, B, T, H_I, d_I,
                                             N_cap, m, k, topk_idx, topk_score);
  if (c >= 0) return c;
  if (csa_indexer_topk_workspace(B, T, N_cap, k) > CSA_INDEXER_STATIC_SCRATCH_BYTES)
    return CSA_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = csa::scratch_address(&ws);
  if (st != CSA_OK) return st;
  return csa_indexer_topk(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride, idx_dtype,
                          q_pos, n_cmp, B, T, H_I, d_I, N_cap, m, k, topk_idx, topk_score, ws,
                          CSA_INDEXER_STATIC_SCRATCH_BYTES, err_word, stream);
}
