// out_proj.cu -- grouped output projection after the MQA core attention.
//
// Method: hyper.ai DeepSeek-V4 page, Method, CSA paragraph (the core attention
// "operates in a Multi-Query Attention manner ... followed by a grouped
// output projection").  Reading: the H heads of a query's output are split
// into G groups of H/G consecutive heads; group g's K = (H/G) * D values are
// projected by its own matrix W_g (d_g rows of K, bf16):
//     y[q][g*d_g + r] = sum_{j < K} W[g][r][j] * o[q][g*K + j]
// fp32 accumulation, bf16 output (nearest even).
//
// One tcgen05 product per (128 output channels, group, tile of up to 256
// queries): M = 128 rows of W_g, N = the queries, K in 64-wide slabs.  When
// that leaves SMs idle (decode: few queries), the K slabs are split over a
// cluster of ks CTAs; each writes its fp32 partial to its shared memory and,
// after a cluster barrier, CTA s sums rows [s*128/ks, (s+1)*128/ks) of all
// ks partials through distributed shared memory.
//   warp 0     TMA: each slab's W rows (128 x 128 B) and query rows (N x 128 B)
//              into a four-stage ring, 128-byte swizzled
//   warp 1     one thread issues 4 tcgen05.mma (M128 N K16) per slab into one
//              TMEM accumulator
//   warps 2-5  epilogue: each lane one output channel (TMEM lane), 32 queries
//              per tcgen05.ld; a warp writes 32 consecutive channels (64 B)
//              of a query at a time
// Every wait is bounded (error word on timeout).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.cuh"

namespace csa {

namespace {

constexpr int kPM = 128;      // output channels per CTA
constexpr int kPMaxN = 256;   // queries per CTA
constexpr int kPStages = 4;
constexpr int kPThreads = 192;
constexpr uint32_t kPWait = 1u << 24;
constexpr int kPABytes = kPM * 128;       // 16 KB: 128 rows x 64 bf16
constexpr int kPBBytes = kPMaxN * 128;    // up to 32 KB
constexpr int kPStageBytes = kPABytes + kPBBytes;
constexpr int kPBarOff = kPStages * kPStageBytes;
constexpr int kPSmem = kPBarOff + 256 + 1024;

struct PBars {
  uint64_t full[kPStages], empty[kPStages];
  uint64_t done;
  uint32_t tmem_slot;
};

struct ProjMaps {
  CUtensorMap w, o;
};

__global__ void __launch_bounds__(kPThreads, 1)
    out_proj_kernel(OutProjArgs a, int n_tile, int ks, int slabs_per,
                    const __grid_constant__ ProjMaps maps) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ uint8_t psm_raw[];
  uint8_t* sm = psm_raw + ((1024 - (smem_u32(psm_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(sm);
  PBars* bars = reinterpret_cast<PBars*>(sm + kPBarOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kspl = blockIdx.x % ks;  // this CTA's share of the K slabs
  const int m0 = (blockIdx.x / ks) * kPM, g = blockIdx.y, n0 = blockIdx.z * n_tile;
  const int K = (a.H / a.G) * a.D;
  const int s_beg = kspl * slabs_per;
  const int n_slabs = min(K / 64 - s_beg, slabs_per);  // may be <= 0 for the last split
  const int nq = min(n_tile, a.n - n0);  // queries of this tile

  if (warp == 0) {
    tc::tmem_alloc(&bars->tmem_slot, kPMaxN);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kPStages; ++s) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    tc::mbar_init(&bars->done, 1);
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;
  const uint32_t tx = (uint32_t)(kPABytes + n_tile * 128);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int i = 0; i < n_slabs; ++i) {
        const int s = i % kPStages;
        if (i >= kPStages && !tc::mbar_wait(&bars->empty[s], ((i / kPStages) - 1) & 1, kPWait)) {
          flag_error(a.err, CSA_EW_TIMEOUT);
          break;
        }
        const uint32_t st = sbase + s * kPStageBytes;
        tma::expect_tx(&bars->full[s], tx);
        tma::load_box(st, &maps.w, (s_beg + i) * 64, g * a.d_g + m0, &bars->full[s]);
        tma::load_box(st + kPABytes, &maps.o, g * K + (s_beg + i) * 64, n0, &bars->full[s]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(kPM, n_tile, false, false);
      bool ok = true;
      for (int i = 0; i < n_slabs && ok; ++i) {
        const int s = i % kPStages;
        ok = tc::mbar_wait(&bars->full[s], (i / kPStages) & 1, kPWait);
        if (!ok) {
          flag_error(a.err, CSA_EW_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
        const uint32_t st = sbase + s * kPStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = tc::desc_sw128(st + kk * 32, 16, 1024);
          const uint64_t bd = tc::desc_sw128(st + kPABytes + kk * 32, 16, 1024);
          tc::mma_ss(tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(&bars->empty[s]);
      }
      tc::mma_commit(&bars->done);  // covers every MMA issued above
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3;  // TMEM lane quarter: output channels 32 qd ..
    const uint32_t lanef = (uint32_t)(qd * 32) << 16;
    const bool ok = __all_sync(0xFFFFFFFFu, tc::mbar_wait(&bars->done, 0, kPWait));
    if (!ok) {
      if (lane == 0) flag_error(a.err, CSA_EW_TIMEOUT);
    } else {
      tc::fence_after_sync();
      const int rl = qd * 32 + lane;  // output channel within the tile
      bf16* y = a.y + (int64_t)g * a.d_g + m0 + rl;
      const int64_t ystride = (int64_t)a.G * a.d_g;
      float* part = reinterpret_cast<float*>(sm);  // [n_tile][128] (stages are done)
      for (int c0 = 0; c0 < n_tile; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lanef + c0, v);
        tc::tmem_ld_wait();
        if (n_slabs <= 0)  // a split left without slabs contributes zeros
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (c0 + j >= nq) continue;
          if (ks == 1)
            y[(int64_t)(n0 + c0 + j) * ystride] = __float2bfloat16_rn(__uint_as_float(v[j]));
          else
            part[(c0 + j) * kPM + rl] = __uint_as_float(v[j]);
        }
      }
    }
  }
  if (ks > 1) {
    // every CTA's partial is complete; CTA kspl sums its rows of all of them
    tc::cluster_sync();
    const int rs = kPM / ks;
    const int64_t ystride = (int64_t)a.G * a.d_g;
    for (int it = tid; it < nq * rs; it += kPThreads) {
      const int q = it / rs, rl = kspl * rs + it % rs;
      const uint32_t la = sbase + (uint32_t)(q * kPM + rl) * 4u;
      float acc = 0.f;
      for (int p = 0; p < ks; ++p) acc += __uint_as_float(tc::ld_cluster_u32(tc::map_shared(la, p)));
      a.y[(int64_t)(n0 + q) * ystride + (int64_t)g * a.d_g + m0 + rl] = __float2bfloat16_rn(acc);
    }
    tc::cluster_sync();  // no CTA leaves while another still reads its partial
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    // copies still in flight (after a timeout) land before TMEM and smem go
    if (lane == 0)
      for (int i = n_slabs > kPStages ? n_slabs - kPStages : 0; i < n_slabs; ++i)
        tc::mbar_wait(&bars->full[i % kPStages], (i / kPStages) & 1, kPWait);
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kPMaxN);
  }
}

}  // namespace

cudaError_t launch_out_proj(const OutProjArgs& a, cudaStream_t st) {
  if (a.n == 0) return cudaSuccess;
  cudaError_t e = ensure_smem_attr((const void*)out_proj_kernel, kPSmem);
  if (e != cudaSuccess) return e;
  const int K = (a.H / a.G) * a.D;
  const int n_slabs = K / 64;
  // queries per CTA: all of them up to 256 (a multiple of 16: the MMA's N)
  int n_tile = a.n < kPMaxN ? a.n : kPMaxN;
  n_tile = (n_tile + 15) / 16 * 16;
  // K split: the largest power of two up to 8 that keeps the CTAs within the
  // SMs, every split at least one slab
  const int64_t base = (int64_t)(a.d_g / kPM) * a.G * ((a.n + n_tile - 1) / n_tile);
  int ks = 1;
  while (ks < 8 && base * ks * 2 <= kNumSMs && ks * 2 <= n_slabs) ks *= 2;
  const int slabs_per = (n_slabs + ks - 1) / ks;
  ProjMaps maps;
  e = tma::encode_rows(&maps.w, a.W, (uint32_t)K, (uint64_t)a.G * a.d_g, kPM);
  if (e != cudaSuccess) return e;
  e = tma::encode_rows(&maps.o, a.o, (uint32_t)(a.H * a.D), (uint64_t)a.n, (uint32_t)n_tile);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.d_g / kPM * ks), (unsigned)a.G,
                     (unsigned)((a.n + n_tile - 1) / n_tile));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  set_pdl(attr[1]);
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, out_proj_kernel, a, n_tile, ks, slabs_per, maps);
}

}  // namespace csa
