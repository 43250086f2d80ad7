// Feed probes: the read rates the attention and indexer kernels are measured
// against.  Neither computes anything of the method; `bench.py --probe` times
// them.
//
// csa_probe_stream_read: every CTA streams an equal contiguous share of a
//   buffer with 16-byte loads, `in_flight` of them per thread before any is
//   used (the indexer scorer's situation: keys read once).
// csa_probe_row_gather: every CTA gathers `stages` stages of 64 rows of 512
//   bytes (a K row and a V row of 256 bytes) at the row indices it is given,
//   with 16-byte cp.async copies into a ring of `ring` stages of shared
//   memory, a block barrier per stage; the rows are summed as they are
//   consumed (the sparse attention's loader situation without the tensor
//   cores).  The ring depth sets the shared memory and so the CTAs per SM.
#include "common.cuh"
#include "kernels.h"

namespace csa {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kGatherThreads = 256;
constexpr int kGatherRowBytes = 512;
constexpr int kGatherStageBytes = 64 * kGatherRowBytes;  // 32 KB

template <int K>
__global__ void __launch_bounds__(kProbeThreads)
    stream_read_kernel(const uint4* __restrict__ src, int64_t per, float* sink) {
  const int64_t base = (int64_t)blockIdx.x * per;
  uint32_t acc = 0u;
  for (int64_t i = threadIdx.x; i < per; i += (int64_t)K * kProbeThreads) {
    uint4 v[K];
#pragma unroll
    for (int u = 0; u < K; ++u) {
      const int64_t j = i + (int64_t)u * kProbeThreads;
      v[u] = j < per ? __ldg(src + base + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < K; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  if (acc == 0x9E3779B9u) sink[0] = 1.f;  // keeps the loads; practically never stored
}

template <int RING>
__global__ void __launch_bounds__(kGatherThreads)
    row_gather_kernel(const uint4* __restrict__ table, int64_t n_rows,
                      const int32_t* __restrict__ idx, int stages, float* sink) {
  extern __shared__ __align__(16) uint4 ring[];  // [RING][64 rows][32 chunks]
  const int t = threadIdx.x;
  const int32_t* my = idx + (int64_t)blockIdx.x * stages * 64;
  uint32_t acc = 0u;
  auto issue = [&](int s) {
    if (s < stages) {
      for (int c = t; c < 64 * 32; c += kGatherThreads) {
        const int r = c >> 5, ch = c & 31;
        int64_t row = __ldg(my + s * 64 + r);
        row = row < 0 ? 0 : (row >= n_rows ? n_rows - 1 : row);  // every read stays in the table
        cp_async16(smem_u32(&ring[(s % RING) * 2048 + c]), table + (int64_t)row * 32 + ch, 16);
      }
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int s = 0; s < RING; ++s) issue(s);
  for (int s = 0; s < stages; ++s) {
    cp_async_wait<RING - 1>();
    __syncthreads();  // every thread's copies of stage s have landed
    for (int c = t; c < 2048; c += kGatherThreads) acc ^= ring[(s % RING) * 2048 + c].x;
    __syncthreads();  // stage s's slot is free again
    issue(s + RING);
  }
  cp_async_wait<0>();
  if (acc == 0x9E3779B9u) sink[0] = 1.f;
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" {

CSA_API int csa_probe_stream_read(const void* src, int64_t bytes, int ctas_per_sm, int in_flight,
                                  float* sink, void* stream) {
  if (!src || !sink || bytes <= 0 || ctas_per_sm < 1 || ctas_per_sm > 4 ||
      (in_flight != 1 && in_flight != 4 && in_flight != 8) ||
      (reinterpret_cast<uintptr_t>(src) & 15))
    return CSA_ERR_INVALID_ARG;
  const int grid = kNumSMs * ctas_per_sm;
  const int64_t per = bytes / 16 / grid;  // 16-byte vectors per CTA (the remainder is not read)
  if (per < 1) return CSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint4* s = static_cast<const uint4*>(src);
  if (in_flight == 1) stream_read_kernel<1><<<grid, kProbeThreads, 0, st>>>(s, per, sink);
  else if (in_flight == 4) stream_read_kernel<4><<<grid, kProbeThreads, 0, st>>>(s, per, sink);
  else stream_read_kernel<8><<<grid, kProbeThreads, 0, st>>>(s, per, sink);
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

CSA_API int csa_probe_row_gather(const void* table, int64_t n_rows, const int32_t* idx, int n_ctas,
                                 int stages, int ring, float* sink, void* stream) {
  if (!table || !idx || !sink || n_rows <= 0 || n_ctas <= 0 || stages <= 0 ||
      (ring != 2 && ring != 4 && ring != 6) || (reinterpret_cast<uintptr_t>(table) & 15))
    return CSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint4* tb = static_cast<const uint4*>(table);
  const int smem = ring * kGatherStageBytes;
  cudaError_t e;
  if (ring == 2) {
    e = ensure_smem_attr((const void*)row_gather_kernel<2>, smem);
    if (e == cudaSuccess)
      row_gather_kernel<2><<<n_ctas, kGatherThreads, smem, st>>>(tb, n_rows, idx, stages, sink);
  } else if (ring == 4) {
    e = ensure_smem_attr((const void*)row_gather_kernel<4>, smem);
    if (e == cudaSuccess)
      row_gather_kernel<4><<<n_ctas, kGatherThreads, smem, st>>>(tb, n_rows, idx, stages, sink);
  } else {
    e = ensure_smem_attr((const void*)row_gather_kernel<6>, smem);
    if (e == cudaSuccess)
      row_gather_kernel<6><<<n_ctas, kGatherThreads, smem, st>>>(tb, n_rows, idx, stages, sink);
  }
  if (e != cudaSuccess) return CSA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

}  // extern "C"
