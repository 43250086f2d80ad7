// selftest.cu -- csa_selftest_bounded_wait: drives the bounded mbarrier wait
// that every pipelined kernel of the library uses (tc::mbar_wait with an
// iteration limit, then CSA_EW_TIMEOUT into the caller's error word) on a
// barrier that nobody completes, so that the give-up path can be checked on a
// real GPU without faulting or hanging it: one thread, no bulk copy, no MMA
// and no tensor memory in flight, and the wait's limit set by the caller.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace csa {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(int arrive, uint32_t limit,
                                                                   int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  tc::fence_mbar_init();
  // with `arrive` the one expected arrival completes phase 0 and the wait
  // returns at once; without it nothing ever arrives
  if (arrive) tc::mbar_arrive(&bar);
  if (!tc::mbar_wait(&bar, 0, limit)) flag_error(err, CSA_EW_TIMEOUT);
}

}  // namespace
}  // namespace csa

extern "C" CSA_API int csa_selftest_bounded_wait(int arrive, uint32_t limit, int32_t* err_word,
                                                 void* stream) {
  if (!err_word || (reinterpret_cast<uintptr_t>(err_word) & 3u) != 0) return CSA_ERR_INVALID_ARG;
  if (limit == 0 || limit > (1u << 20)) return CSA_ERR_INVALID_ARG;
  csa::bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      arrive != 0, limit, err_word);
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
