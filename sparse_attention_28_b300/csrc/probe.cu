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
//   cores).  The CTA's row indices are first staged in shared memory (one
//   coalesced read), so that no copy waits on an index load, as in the
//   attention, whose loaders look their rows up stages ahead.  The ring depth
//   sets the shared memory and so the CTAs per SM.  Mode 1 moves the same
//   rows with TMA `tile::gather4` (four 128-byte row pieces per instruction,
//   128-byte swizzled, issued by 16 lanes of one warp) into the attention's
//   layout (K and V halves as four 8 KB regions per stage), with a full and
//   an empty mbarrier per ring slot.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.cuh"

namespace csa {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kGatherRowBytes = 512;
constexpr int kGatherStageBytes = 64 * kGatherRowBytes;  // 32 KB
constexpr int kMaxGatherStages = 64;                     // the index list: at most 16 KB

// The CTA's stages * 64 row indices into shared memory, each clamped into the
// table; ends with a block barrier.
__device__ __forceinline__ void stage_indices(int32_t* dst, const int32_t* __restrict__ src,
                                              int n, int64_t n_rows) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int64_t row = __ldg(src + i);
    dst[i] = (int32_t)(row < 0 ? 0 : (row >= n_rows ? n_rows - 1 : row));  // reads stay in the table
  }
  __syncthreads();
}

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

template <int RING, int NT>
__global__ void __launch_bounds__(NT)
    row_gather_kernel(const uint4* __restrict__ table, int64_t n_rows,
                      const int32_t* __restrict__ idx, int stages, float* sink) {
  extern __shared__ __align__(16) uint4 ring[];  // [RING][64 rows][32 chunks], then the indices
  int32_t* rows = reinterpret_cast<int32_t*>(ring + RING * 2048);
  const int t = threadIdx.x;
  stage_indices(rows, idx + (int64_t)blockIdx.x * stages * 64, stages * 64, n_rows);
  uint32_t acc = 0u;
  auto issue = [&](int s) {
    if (s < stages) {
      for (int c = t; c < 64 * 32; c += NT) {
        const int r = c >> 5, ch = c & 31;
        const int64_t row = rows[s * 64 + r];
        cp_async16(smem_u32(&ring[(s % RING) * 2048 + c]), table + row * 32 + ch, 16);
      }
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int s = 0; s < RING; ++s) issue(s);
  for (int s = 0; s < stages; ++s) {
    cp_async_wait<RING - 1>();
    __syncthreads();  // every thread's copies of stage s have landed
    for (int c = t; c < 2048; c += NT) acc ^= ring[(s % RING) * 2048 + c].x;
    __syncthreads();  // stage s's slot is free again
    issue(s + RING);
  }
  cp_async_wait<0>();
  if (acc == 0x9E3779B9u) sink[0] = 1.f;
}

template <int RING, int IW>
__global__ void __launch_bounds__(32 * IW + 128 + (IW == 1 ? 96 : 0))
    row_gather4_kernel(const __grid_constant__ CUtensorMap map, int64_t n_rows,
                       const int32_t* __restrict__ idx, int stages, float* sink) {
  static_assert(IW == 1 || IW == 4 || IW == 8, "one, four or eight issuing warps");
  // threads: IW issuing warps and four consumer warps (seven with one issuer)
  constexpr int kThreadsG = 32 * IW + 128 + (IW == 1 ? 96 : 0);
  extern __shared__ uint8_t g4_raw[];
  __shared__ __align__(8) uint64_t full[RING], empty[RING];
  uint8_t* base = g4_raw + ((1024 - (smem_u32(g4_raw) & 1023)) & 1023);
  int32_t* rows = reinterpret_cast<int32_t*>(base + RING * kGatherStageBytes);
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  stage_indices(rows, idx + (int64_t)blockIdx.x * stages * 64, stages * 64, n_rows);
  constexpr uint32_t kLimit = 1u << 22;
  constexpr int kConsumers = kThreadsG - 32 * IW;
  if (t == 0) {
    for (int d = 0; d < RING; ++d) {
      tc::mbar_init(&full[d], IW);                  // one expect_tx arrival per issuing warp
      tc::mbar_init(&empty[d], kConsumers / 32);    // one arrival per consumer warp
    }
    tc::fence_mbar_init();
  }
  __syncthreads();
  bool ok = true;
  uint32_t acc = 0u;
  if (warp < IW) {
    for (int s = 0; s < stages; ++s) {
      const int d = s % RING;
      if (s >= RING) ok &= tc::mbar_wait(&empty[d], ((s / RING) - 1) & 1, kLimit);
      if (lane == 0) tma::expect_tx(&full[d], kGatherStageBytes / IW);
      __syncwarp();
      const uint32_t st = smem_u32(base + d * kGatherStageBytes);
      if constexpr (IW == 1) {
        // lane l < 16: the four pieces of rows 4l .. 4l + 3
        int r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = lane < 16 ? rows[s * 64 + 4 * lane + q] : 0;
        if (lane < 16) {
#pragma unroll
          for (int h = 0; h < 4; ++h)  // K 0-63, K 64-127, V 0-63, V 64-127
            tma::gather4(st + lane * 512 + h * 8192, &map, 64 * h, r[0], r[1], r[2], r[3],
                         &full[d]);
        }
      } else {
        // the stage's 64 instructions i = (group g, piece h) = (i / 4, i % 4):
        // lane l < 64 / IW of warp w issues i = w * 64 / IW + l
        if (lane < 64 / IW) {
          const int i = warp * (64 / IW) + lane, g = i >> 2, h = i & 3;
          const int* rg = rows + s * 64 + 4 * g;
          tma::gather4(st + g * 512 + h * 8192, &map, 64 * h, rg[0], rg[1], rg[2], rg[3],
                       &full[d]);
        }
      }
    }
  } else {
    for (int s = 0; s < stages; ++s) {
      const int d = s % RING;
      ok &= tc::mbar_wait(&full[d], (s / RING) & 1, kLimit);
      const uint4* v = reinterpret_cast<const uint4*>(base + d * kGatherStageBytes);
      for (int c = t - 32 * IW; c < 2048; c += kConsumers) acc ^= v[c].x;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[d]);
    }
  }
  if (!ok) sink[0] = 2.f;  // a wait gave up
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
                                 int stages, int ring, int mode, float* sink, void* stream) {
  if (!table || !idx || !sink || n_rows <= 0 || n_rows >= (int64_t)1 << 31 || n_ctas <= 0 ||
      stages <= 0 || stages > kMaxGatherStages || (ring != 2 && ring != 4 && ring != 6) ||
      mode < 0 || mode > 4 ||
      (reinterpret_cast<uintptr_t>(table) & 15))
    return CSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint4* tb = static_cast<const uint4*>(table);
  cudaError_t e;
  if (mode == 0 || mode == 2) {  // cp.async
    const int smem = ring * kGatherStageBytes + stages * 64 * 4;  // + the index list
    auto run = [&](auto kern, int nt) {
      e = ensure_smem_attr((const void*)kern, smem);
      if (e == cudaSuccess) kern<<<n_ctas, nt, smem, st>>>(tb, n_rows, idx, stages, sink);
    };
    if (mode == 0) {
      if (ring == 2) run(row_gather_kernel<2, 256>, 256);
      else if (ring == 4) run(row_gather_kernel<4, 256>, 256);
      else run(row_gather_kernel<6, 256>, 256);
    } else {
      if (ring == 2) run(row_gather_kernel<2, 512>, 512);
      else if (ring == 4) run(row_gather_kernel<4, 512>, 512);
      else run(row_gather_kernel<6, 512>, 512);
    }
  } else {
    // rows of 256 bf16 (a K row and a V row), boxes of 64 columns x 1 row
    CUtensorMap map;
    e = tma::encode_rows(&map, table, 256, (uint64_t)n_rows, 1);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    // + room to align the ring to 1024, + the index list
    const int smem = ring * kGatherStageBytes + 1024 + stages * 64 * 4;
    auto run = [&](auto kern, int nt) {
      e = ensure_smem_attr((const void*)kern, smem);
      if (e == cudaSuccess) kern<<<n_ctas, nt, smem, st>>>(map, n_rows, idx, stages, sink);
    };
    if (mode == 1) {
      if (ring == 2) run(row_gather4_kernel<2, 1>, 256);
      else if (ring == 4) run(row_gather4_kernel<4, 1>, 256);
      else run(row_gather4_kernel<6, 1>, 256);
    } else if (mode == 3) {
      if (ring == 2) run(row_gather4_kernel<2, 4>, 256);
      else if (ring == 4) run(row_gather4_kernel<4, 4>, 256);
      else run(row_gather4_kernel<6, 4>, 256);
    } else {
      if (ring == 2) run(row_gather4_kernel<2, 8>, 384);
      else if (ring == 4) run(row_gather4_kernel<4, 8>, 384);
      else run(row_gather4_kernel<6, 8>, 384);
    }
  }
  if (e != cudaSuccess) return CSA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

}  // extern "C"
