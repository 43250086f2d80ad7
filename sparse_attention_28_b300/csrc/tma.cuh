// tma.cuh -- Tensor Memory Accelerator helpers: host-side tensor-map encoding
// (through the driver entry point, no link-time libcuda dependency) and the
// device-side bulk tensor copies used by libcsa.so.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace csa {
namespace tma {

// 2-D bf16 tensor map over `rows` rows of 128 elements (256-byte rows), box of
// 64 columns x box_rows rows, 128-byte swizzle (the SW128 shared layout),
// out-of-range rows read as zeros.
cudaError_t encode_rows128(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);
// The same over rows of row_elems bf16 (a multiple of 64; 16-byte aligned rows).
cudaError_t encode_rows(CUtensorMap* map, const void* base, uint32_t row_elems, uint64_t rows,
                        uint32_t box_rows);

__device__ __forceinline__ void expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// box {64 cols, box_rows rows} at (col, row) -> shared dst (1024-aligned)
__device__ __forceinline__ void load_box(uint32_t dst, const CUtensorMap* map, int col, int row,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(map), "r"(col), "r"(row), "r"(smem_u32(bar))
      : "memory");
}

// contiguous bytes (a multiple of 16, both addresses 16-byte aligned)
// global -> shared, completion through the mbarrier's transaction count
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// four rows (each 64 columns from col) -> four consecutive 128-byte rows at dst
__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap* map, int col, int r0,
                                        int r1, int r2, int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(dst),
      "l"(map), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace tma
}  // namespace csa
