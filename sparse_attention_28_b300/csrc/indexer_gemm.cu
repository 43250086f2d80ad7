// indexer_gemm.cu -- Lightning-Indexer scores for many query tokens of one
// sequence (chunked prefill) as a tensor-core GEMM.
//
// Method: hyper.ai DeepSeek-V4 page, Method (Lightning Indexer over the
// compressed entries); elamur.ai page, Summary (DeepSeek Sparse Attention
// form) -- per query token t and entry s:
//     I(t,s) = sum_h w[t][h] * ReLU(q[t][h] . k[s]).
// With many tokens sharing one sequence's keys, the dot products are one
// matrix product: keys [entries x 64] times queries^T [64 x (tokens x 4
// heads)].  One CTA owns a block of 64 tokens (256 MMA columns) and a range of
// 128-entry key tiles:
//   warp 0   TMA: the token block's queries once (256 rows x 128 bytes), then
//            key tiles (128 rows x 128 bytes) into a four-stage ring
//   warp 1   one thread issues 4 tcgen05.mma (M128 N256 K16) per tile into one
//            of two TMEM accumulators (256 columns each)
//   warps 4-11  epilogue: each lane is one entry; per token the 4 head
//            columns are combined as sum_h w_h ReLU(x_h) and the score written
//            to the token's row (32 lanes = 128 contiguous bytes per store)
// Scores of entries a token cannot see are written too; the selection reads
// only the visible ones.  Every wait is bounded (error word on timeout).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.cuh"

namespace csa {

namespace {

constexpr int kGM = 128;          // entries per tile
constexpr int kGQ = 64;           // tokens per CTA
constexpr int kGN = kGQ * 4;      // MMA columns: (token, head)
constexpr int kGStages = 4;
constexpr int kGThreads = 384;
constexpr int kGEpiWarp0 = 4;
constexpr int kGEpiWarps = 8;
constexpr uint32_t kGWait = 1u << 24;
constexpr int kGTileBytes = kGM * 128;   // 16 KB
constexpr int kGQBytes = kGN * 128;      // 32 KB
constexpr int kGQOff = 0;
constexpr int kGAOff = kGQBytes;
constexpr int kGWOff = kGAOff + kGStages * kGTileBytes;  // w [64][4] fp32
constexpr int kGBarOff = kGWOff + kGQ * 4 * 4;
// one CTA per SM (it holds all 512 TMEM columns): at least 116 KB of shared memory
constexpr int kGSmem = kGBarOff + 256 + 1024 > 116 * 1024 ? kGBarOff + 256 + 1024 : 116 * 1024;

struct GBars {
  uint64_t full[kGStages], empty[kGStages];
  uint64_t tfull[2], tempty[2];
  uint64_t qfull;
  uint32_t tmem_slot;
};

struct GemmMaps {
  CUtensorMap q, k;
};

// grid (splits, token blocks); block qb covers tokens [q0 + 64 qb, +64) of
// one sequence; scores row of token i (relative to q0) at scores + i*stride.
__global__ void __launch_bounds__(kGThreads, 1)
    indexer_gemm_kernel(IndexerArgs a, int q0, float* scores, int stride,
                        const __grid_constant__ GemmMaps maps) {
  // Until the producer's griddepcontrol.wait below the kernel reads only
  // inputs that no kernel of this library writes (positions, entry counts,
  // the chunk's queries and head weights) and sets up shared and tensor
  // memory, so that part overlaps the previous kernel (the select of the
  // previous chunk, which still reads the score workspace).
  pdl_trigger();
  extern __shared__ uint8_t gsm_raw[];
  uint8_t* sm = gsm_raw + ((1024 - (smem_u32(gsm_raw) & 1023)) & 1023);
  const uint32_t sbase = smem_u32(sm);
  GBars* bars = reinterpret_cast<GBars*>(sm + kGBarOff);
  float* wts = reinterpret_cast<float*>(sm + kGWOff);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qb = blockIdx.y;
  const int tok0 = q0 + qb * kGQ;  // first token (global query index)
  const int b = tok0 / a.T;

  // entries any token of the block can see: tiles [0, n_tiles)
  int nv_max = 0;
  bool bad = false;  // flagged after the wait (the error word may be the previous kernel's)
  for (int i = lane; i < kGQ; i += 32) {
    const int64_t t = __ldg(a.q_pos + tok0 + i);
    int64_t present = __ldg(a.n_cmp + b);
    if (blockIdx.x == 0 && (t < 0 || present < 0 || present > a.N_cap)) bad = true;
    present = present < 0 ? 0 : (present > a.N_cap ? a.N_cap : present);
    int64_t nv = t >= 0 ? (t + 1) / a.m : 0;
    nv = nv < present ? nv : present;
    nv_max = max(nv_max, (int)nv);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) nv_max = max(nv_max, __shfl_xor_sync(0xFFFFFFFFu, nv_max, o));
  const int n_tiles_all = (nv_max + kGM - 1) / kGM;
  const int per = (n_tiles_all + gridDim.x - 1) / gridDim.x;
  const int t_beg = blockIdx.x * per;
  const int t_end = min(t_beg + per, n_tiles_all);
  const int n_tiles = t_end > t_beg ? t_end - t_beg : 0;

  if (warp == 0) {
    tc::tmem_alloc(&bars->tmem_slot, 512);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kGStages; ++s) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars->tfull[i], 1);
      tc::mbar_init(&bars->tempty[i], kGEpiWarps);
    }
    tc::mbar_init(&bars->qfull, 1);
    tc::fence_mbar_init();
  }
  for (int i = tid; i < kGQ * 4; i += kGThreads) wts[i] = __ldg(a.w + (int64_t)tok0 * 4 + i);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;

  if (n_tiles > 0 && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma::expect_tx(&bars->qfull, kGQBytes);
      tma::load_box(sbase + kGQOff, &maps.q, 0, tok0 * 4, &bars->qfull);
      pdl_wait();  // the keys may be the compression's output
      const int krow0 = (int)((int64_t)b * (a.k_bstride / 64));
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kGStages;
        if (i >= kGStages && !tc::mbar_wait(&bars->empty[s], ((i / kGStages) - 1) & 1, kGWait)) {
          flag_error(a.err, CSA_EW_TIMEOUT);
          break;
        }
        tma::expect_tx(&bars->full[s], kGTileBytes);
        tma::load_box(sbase + kGAOff + s * kGTileBytes, &maps.k, 0, krow0 + (t_beg + i) * kGM,
                      &bars->full[s]);
      }
    }
    __syncwarp();
  } else if (n_tiles > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(kGM, kGN, false, false);
      bool ok = tc::mbar_wait(&bars->qfull, 0, kGWait);
      for (int i = 0; i < n_tiles && ok; ++i) {
        const int s = i % kGStages, buf = i & 1;
        ok = tc::mbar_wait(&bars->full[s], (i / kGStages) & 1, kGWait);
        if (ok && i >= 2) ok = tc::mbar_wait(&bars->tempty[buf], ((i - 2) >> 1) & 1, kGWait);
        if (!ok) {
          flag_error(a.err, CSA_EW_TIMEOUT);
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = tc::desc_sw128(sbase + kGAOff + s * kGTileBytes + kk * 32, 16, 1024);
          const uint64_t bd = tc::desc_sw128(sbase + kGQOff + kk * 32, 16, 1024);
          tc::mma_ss(tmem + buf * kGN, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bars->empty[s]);
        tc::mma_commit(&bars->tfull[buf]);
      }
    }
    __syncwarp();
  } else if (n_tiles > 0 && warp >= kGEpiWarp0 && warp < kGEpiWarp0 + kGEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int e8 = warp - kGEpiWarp0;
    const int qd = warp & 3;      // TMEM lane quarter
    const int half = e8 >> 2;     // columns [128 half, 128 half + 128): tokens 32 half ..
    const uint32_t lanef = (uint32_t)(qd * 32) << 16;
    const uint64_t keep = l2_evict_last_policy();  // read back by the select
    pdl_wait();  // the previous select has finished reading the score workspace
    for (int i = 0; i < n_tiles; ++i) {
      const int buf = i & 1;
      if (!__all_sync(0xFFFFFFFFu, tc::mbar_wait(&bars->tfull[buf], (i >> 1) & 1, kGWait))) {
        if (lane == 0) flag_error(a.err, CSA_EW_TIMEOUT);
        break;
      }
      tc::fence_after_sync();
      const int64_t e = (int64_t)(t_beg + i) * kGM + qd * 32 + lane;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lanef + buf * kGN + half * 128 + c * 32, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int tq = half * 32 + c * 8 + j;  // token within the block
          const float* wq = wts + tq * 4;
          const float sc = wq[0] * fmaxf(__uint_as_float(v[4 * j]), 0.f) +
                           wq[1] * fmaxf(__uint_as_float(v[4 * j + 1]), 0.f) +
                           wq[2] * fmaxf(__uint_as_float(v[4 * j + 2]), 0.f) +
                           wq[3] * fmaxf(__uint_as_float(v[4 * j + 3]), 0.f);
          if (e < a.N_cap) st_f32_policy(scores + (int64_t)(qb * kGQ + tq) * stride + e, sc, keep);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars->tempty[buf]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  pdl_wait();
  if (bad) flag_error(a.err, CSA_EW_BAD_POSITION);
  if (warp == 0) {
    // copies still in flight (after a timeout) land before TMEM and smem go
    if (lane == 0 && n_tiles > 0) {
      tc::mbar_wait(&bars->qfull, 0, kGWait);
      for (int i = n_tiles > kGStages ? n_tiles - kGStages : 0; i < n_tiles; ++i)
        tc::mbar_wait(&bars->full[i % kGStages], (i / kGStages) & 1, kGWait);
    }
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool indexer_gemm_applies(const IndexerArgs& a) {
  return !a.fp8 && !a.fp4 && a.T % kGQ == 0 && a.T >= kGQ && a.k_bstride % 64 == 0;
}

// Scores of queries [q0, q0 + qc) (qc a multiple of 64, whole blocks of one
// sequence) into scores[(q - q0) * stride + entry].
cudaError_t launch_indexer_gemm(const IndexerArgs& a, int q0, int qc, float* scores, int stride,
                                cudaStream_t st) {
  cudaError_t e = ensure_smem_attr((const void*)indexer_gemm_kernel, kGSmem);
  if (e != cudaSuccess) return e;
  GemmMaps maps;
  e = tma::encode_rows(&maps.q, a.q, 64, (uint64_t)a.n_query * 4, kGN);
  if (e != cudaSuccess) return e;
  const int n_seq = a.n_query / a.T;
  const uint64_t krows = (uint64_t)(n_seq - 1) * (a.k_bstride / 64) + a.N_cap;
  e = tma::encode_rows(&maps.k, a.keys, 64, krows, kGM);
  if (e != cudaSuccess) return e;
  const int n_blocks = qc / kGQ;
  int splits = (kNumSMs + n_blocks - 1) / n_blocks;
  const int max_tiles = (a.N_cap + kGM - 1) / kGM;
  splits = splits > max_tiles ? max_tiles : splits;
  splits = splits < 1 ? 1 : splits;
  return launch_pdl(indexer_gemm_kernel, dim3(splits, n_blocks), dim3(kGThreads), kGSmem, st, a, q0,
                    scores, stride, maps);
}

}  // namespace csa
