// indexer.cu -- Lightning-Indexer scores and exact top-k selection.
//
// Method: hyper.ai DeepSeek-V4 page, Method ("A Lightning Indexer then
// selects the top-k compressed KV entries"); aiboss88 DeepSeek-V4 page,
// Technical Principles (index score, then top-k sparse selection; FP8 range
// for the low-precision indexer QK path); elamur.ai page, Summary ("runs
// DeepSeek Sparse Attention"), read as
//     I(t,s) = sum_h w[t][h] * ReLU(q[t][h] . k[s]),  s < n_vis(t).
//
// Per call (queries in chunks that bound the workspace):
//   1. scores: for a few tokens per sequence (decode) a kernel with one CTA
//      per (2048-entry chunk, query) streams the compressed indexer keys once
//      (the dominant HBM traffic) and computes the 4-head scores with
//      tensor-core MMAs (entries on M, heads on N); for many tokens per
//      sequence (prefill) the scores are one tcgen05 GEMM (indexer_gemm.cu);
//      either way fp32 scores land in the workspace,
//   2. select kernel, one thread-block cluster of up to 16 CTAs per query,
//      each holding a slice of 8, 16 or 32 entries per thread of the scores
//      in shared memory (one bulk copy): three radix levels over the
//      order-preserving score keys (bits 31..20, then 19..10 and 9..0 of the
//      keys in the chosen bins) -- counts pushed into every cluster CTA with
//      remote atomics, one cluster barrier per level -- give the exact k-th
//      key k*; one more exchange of the per-CTA counts
//      of keys above k* and equal to k* gives each CTA its output offset and
//      how many ties at k* it takes (lowest indices first); each thread then
//      writes the indices of its consecutive entries in order.
// Bins, keys and the tie rule give the same set as a full sort on
// (-score, index).
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.cuh"

namespace csa {

namespace {

constexpr int kDI = 64;
constexpr int kHI = 4;
constexpr int kThreads = 256;     // score kernel
constexpr int kChunk = 2048;      // entries per score CTA
constexpr int kUnrollBf16 = 4;    // 16-entry groups in flight per warp (bf16 keys)
constexpr int kUnrollFp8 = 8;     // (E4M3 keys: half the bytes per row)
constexpr int kUnrollFp4 = 8;     // (FP4 keys)
constexpr int kQueryChunk = 256;  // queries per launch (bounds the workspace)
// from this many queries in a launch, one streaming CTA per query
// (topk_stream_kernel) instead of a cluster per query
constexpr int kStreamQueries = 128;
constexpr int kSelThreads = 1024;  // select CTA size for few queries (512 for many)
constexpr int kMaxCluster = 16;  // select CTAs per query
static_assert(kMaxNcap <= kMaxCluster * kSelThreads * 32, "select cluster");

struct WsLayout {
  float* scores;  // [QC][stride]
  int stride;     // N_cap rounded up to 32 entries (128-byte aligned rows)
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int score_stride(int n_cap) { return (n_cap + 31) & ~31; }

WsLayout carve(void* ws, int n_cap) {
  WsLayout L;
  L.stride = score_stride(n_cap);
  L.scores = reinterpret_cast<float*>(ws);
  return L;
}

__device__ __forceinline__ int64_t visible_entries(const IndexerArgs& a, int qid, int32_t* err,
                                                   bool report) {
  const int b = qid / a.T;
  const int64_t t = __ldg(a.q_pos + qid);
  int64_t present = __ldg(a.n_cmp + b);
  if (t < 0 || present < 0 || present > a.N_cap) {
    if (report) flag_error(err, CSA_EW_BAD_POSITION);
    if (t < 0) return 0;
    present = present < 0 ? 0 : a.N_cap;
  }
  const int64_t nv = (t + 1) / a.m;
  return nv < present ? nv : present;
}

// ------------------------------------------------------------------ block helpers
template <int NT>
__device__ __forceinline__ int block_excl_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < NT / 32 ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NT / 32) scratch[lane] = s;  // inclusive warp prefix
  }
  __syncthreads();
  const int before = warp > 0 ? scratch[warp - 1] : 0;
  if (total) *total = scratch[NT / 32 - 1];
  __syncthreads();
  return before + x - v;
}

// Thread t of NT holds `cnt` = the count of its bins; bins are split evenly
// and thread 0 owns the highest ones (`bins` = the thread's bins, highest
// first).  res[0] = the bin holding the need-th largest key, res[1] = the
// count in the bins above it.
template <int NT, int PER>
__device__ void bin_from_top(const int (&bins)[PER], int first_bin, int need, int* scratch,
                             int* res) {
  int local = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) local += bins[i];
  int total;
  const int before = block_excl_scan<NT>(local, scratch, &total);
  if (before < need && before + local >= need) {
    int run = before;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      if (run + bins[i] >= need) {
        res[0] = first_bin - i;
        res[1] = run;
        break;
      }
      run += bins[i];
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ scores
// Fragment mapping: 16 entries on M, heads on N (heads 4..7 zero).  The
// contraction order over the 64 dims is free, so each thread loads whole
// 16-byte vectors of a key row and the query fragments use the same
// permutation:
//   bf16 (m16n8k16): thread (g, c) holds row bytes [16c,16c+16) and
//         [64+16c, 64+16c+16); k-step s takes word s of each vector.
//   E4M3 (m16n8k32, products exact in fp32): thread (g, c) holds row bytes
//         [16c, 16c+16); k-step s takes words 2s and 2s+1.
//   FP4 (E2M1 codes, one E4M3 scale per 16 channels; m16n8k16 f16): as
//         bf16, with each byte of codes expanded to an f16 pair and
//         multiplied by its block's scale (exact: at most 6 significant
//         bits, within the f16 range), so products are exact in fp32.
// Scores of entries [e0, e1) of query qid into scores[e]: each warp takes
// 16-entry groups, kUnroll groups in flight.  FMT: 0 bf16, 1 E4M3, 2 FP4.
template <int FMT>
__device__ __forceinline__ void score_range(const IndexerArgs& a, int qid, int64_t e0, int64_t e1,
                                            float* scores, int warp, int g, int c) {
  constexpr bool FP8 = FMT == 1, FP4 = FMT == 2;
  // query fragments (heads g < 4) and head weights (heads 2c, 2c+1 for c < 2)
  uint32_t qb0[4] = {0, 0, 0, 0}, qb1[4] = {0, 0, 0, 0};
  float w0 = 0.f, w1 = 0.f;
  if (g < kHI) {
    if (FP4) {
      const uint8_t* qr = reinterpret_cast<const uint8_t*>(a.q) + ((int64_t)qid * kHI + g) * (kDI / 2);
      const uint8_t* qs = reinterpret_cast<const uint8_t*>(a.q_scale) + ((int64_t)qid * kHI + g) * (kDI / 16);
      const uint32_t v0 = __ldg(reinterpret_cast<const uint32_t*>(qr + 4 * c));
      const uint32_t v1 = __ldg(reinterpret_cast<const uint32_t*>(qr + 16 + 4 * c));
      const __half2 s0 = e4m3_half2(__ldg(qs + (c >> 1))), s1 = e4m3_half2(__ldg(qs + 2 + (c >> 1)));
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        qb0[t] = fp4x2_scaled(v0 >> (8 * t), s0);
        qb1[t] = fp4x2_scaled(v1 >> (8 * t), s1);
      }
    } else if (FP8) {
      const uint8_t* qr = reinterpret_cast<const uint8_t*>(a.q) + ((int64_t)qid * kHI + g) * kDI;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(qr + 16 * c));
      qb0[0] = v.x; qb0[1] = v.y; qb0[2] = v.z; qb0[3] = v.w;
    } else {
      const bf16* qr = reinterpret_cast<const bf16*>(a.q) + ((int64_t)qid * kHI + g) * kDI;
      const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(qr + 8 * c));
      const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(qr + 32 + 8 * c));
      qb0[0] = v0.x; qb0[1] = v0.y; qb0[2] = v0.z; qb0[3] = v0.w;
      qb1[0] = v1.x; qb1[1] = v1.y; qb1[2] = v1.z; qb1[3] = v1.w;
    }
  }
  if (c < 2) {
    w0 = __ldg(a.w + (int64_t)qid * kHI + 2 * c);
    w1 = __ldg(a.w + (int64_t)qid * kHI + 2 * c + 1);
    if (FP8) {
      w0 *= __ldg(a.q_scale + (int64_t)qid * kHI + 2 * c);
      w1 *= __ldg(a.q_scale + (int64_t)qid * kHI + 2 * c + 1);
    }
  }

  const int b = qid / a.T;
  constexpr int kUnroll = FMT == 0 ? kUnrollBf16 : FMT == 1 ? kUnrollFp8 : kUnrollFp4;
  const int n_groups = (int)((e1 - e0 + 15) / 16);
  // the keys are read once; the scores are read back by the select
  const uint64_t once = l2_evict_first_policy(), keep = l2_evict_last_policy();
  for (int gb = warp * kUnroll; gb < n_groups; gb += (kThreads / 32) * kUnroll) {
    uint4 ra[kUnroll][2], rb[kUnroll][2];  // rows g and g+8 of each group
    float ks[kUnroll];                      // E4M3: scale of the entry this thread scores
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t ea = e0 + (int64_t)(gb + u) * 16 + g, eb = ea + 8;
      if (FP4) {
        // codes (two 4-byte chunks per row) and the row's 4 block scales
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(a.keys) + (int64_t)b * (a.k_bstride / 2);
        const uint32_t* sb = reinterpret_cast<const uint32_t*>(a.k_scale) + (int64_t)b * a.ks_bstride;
        const uint4 z = make_uint4(0, 0, 0, 0);
        ra[u][0] = z;
        rb[u][0] = z;
        if (ea < e1) {
          ra[u][0].x = ldg_u32_policy(kb + ea * (kDI / 2) + 4 * c, once);
          ra[u][0].y = ldg_u32_policy(kb + ea * (kDI / 2) + 16 + 4 * c, once);
          ra[u][0].z = __ldg(sb + ea);
        }
        if (eb < e1) {
          rb[u][0].x = ldg_u32_policy(kb + eb * (kDI / 2) + 4 * c, once);
          rb[u][0].y = ldg_u32_policy(kb + eb * (kDI / 2) + 16 + 4 * c, once);
          rb[u][0].z = __ldg(sb + eb);
        }
      } else if (FP8) {
        const int64_t es = c == 1 ? eb : ea;
        ks[u] = (c < 2 && es < e1) ? __ldg(a.k_scale + (int64_t)b * a.ks_bstride + es) : 0.f;
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(a.keys) + (int64_t)b * a.k_bstride;
        ra[u][0] = ea < e1 ? ldg_u32x4_policy(kb + ea * kDI + 16 * c, once) : make_uint4(0, 0, 0, 0);
        rb[u][0] = eb < e1 ? ldg_u32x4_policy(kb + eb * kDI + 16 * c, once) : make_uint4(0, 0, 0, 0);
      } else {
        const bf16* kb = reinterpret_cast<const bf16*>(a.keys) + (int64_t)b * a.k_bstride;
        const uint4 z = make_uint4(0, 0, 0, 0);
        ra[u][0] = ea < e1 ? ldg_u32x4_policy(kb + ea * kDI + 8 * c, once) : z;
        ra[u][1] = ea < e1 ? ldg_u32x4_policy(kb + ea * kDI + 32 + 8 * c, once) : z;
        rb[u][0] = eb < e1 ? ldg_u32x4_policy(kb + eb * kDI + 8 * c, once) : z;
        rb[u][1] = eb < e1 ? ldg_u32x4_policy(kb + eb * kDI + 32 + 8 * c, once) : z;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (gb + u >= n_groups) break;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (FP4) {
        // this thread's blocks: c >> 1 (channels 8c..) and 2 + (c >> 1) (32 + 8c..)
        const int sh0 = 8 * (c >> 1), sh1 = 8 * (2 + (c >> 1));
        const __half2 sa0 = e4m3_half2(ra[u][0].z >> sh0), sa1 = e4m3_half2(ra[u][0].z >> sh1);
        const __half2 sb0 = e4m3_half2(rb[u][0].z >> sh0), sb1 = e4m3_half2(rb[u][0].z >> sh1);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t af[4] = {fp4x2_scaled(ra[u][0].x >> (8 * t), sa0),
                                  fp4x2_scaled(rb[u][0].x >> (8 * t), sb0),
                                  fp4x2_scaled(ra[u][0].y >> (8 * t), sa1),
                                  fp4x2_scaled(rb[u][0].y >> (8 * t), sb1)};
          mma_f16_16816(acc, af, qb0[t], qb1[t]);
        }
      } else if (FP8) {
        const uint32_t a0[4] = {ra[u][0].x, rb[u][0].x, ra[u][0].y, rb[u][0].y};
        const uint32_t a1[4] = {ra[u][0].z, rb[u][0].z, ra[u][0].w, rb[u][0].w};
        mma_e4m3_16832(acc, a0, qb0[0], qb0[1]);
        mma_e4m3_16832(acc, a1, qb0[2], qb0[3]);
      } else {
        const uint32_t xa0[4] = {ra[u][0].x, ra[u][0].y, ra[u][0].z, ra[u][0].w};
        const uint32_t xa1[4] = {ra[u][1].x, ra[u][1].y, ra[u][1].z, ra[u][1].w};
        const uint32_t xb0[4] = {rb[u][0].x, rb[u][0].y, rb[u][0].z, rb[u][0].w};
        const uint32_t xb1[4] = {rb[u][1].x, rb[u][1].y, rb[u][1].z, rb[u][1].w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint32_t af[4] = {xa0[s], xb0[s], xa1[s], xb1[s]};
          mma_bf16_16816(acc, af, qb0[s], qb1[s]);
        }
      }
      // epilogue: weighted ReLU over heads 2c, 2c+1, then over the 4 heads
      float sa = w0 * fmaxf(acc[0], 0.f) + w1 * fmaxf(acc[1], 0.f);
      float sb = w0 * fmaxf(acc[2], 0.f) + w1 * fmaxf(acc[3], 0.f);
      sa += __shfl_xor_sync(0xFFFFFFFFu, sa, 1);
      sb += __shfl_xor_sync(0xFFFFFFFFu, sb, 1);
      const int64_t e = e0 + (int64_t)(gb + u) * 16 + g + (c == 1 ? 8 : 0);
      float sc = c == 1 ? sb : sa;
      if (c < 2 && e < e1) {
        if (FP8) sc *= ks[u];
        st_f32_policy(scores + e, sc, keep);
      }
    }
  }
}

// One wave of CTAs; the 16-entry groups of all queries of the chunk,
// concatenated in query order, are split into equal contiguous ranges, one
// per CTA.  A CTA walks its range query by query (loading that query's
// fragments and weights), so that every CTA streams the same number of key
// bytes whatever the queries' visible counts.
// CTAs per SM (a third FP4 CTA within 85 registers spilled and was slower).
constexpr int score_ctas_per_sm(int) { return 2; }

template <int FMT>
__global__ void __launch_bounds__(kThreads, score_ctas_per_sm(FMT)) indexer_score_kernel(IndexerArgs a, int q0, int qc,
                                                                WsLayout L) {
  // the visible counts and their prefix come from inputs no kernel of this
  // library writes: computed while the previous kernel finishes
  pdl_trigger();
  __shared__ int gp[kQueryChunk + 1];  // group prefix over the chunk's queries
  __shared__ int nvs[kQueryChunk];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  {
    int nv = 0;
    if (tid < qc) {
      nv = (int)visible_entries(a, q0 + tid, nullptr, false);
      nvs[tid] = nv;
    }
    int tot;
    const int before = block_excl_scan<kThreads>((nv + 15) >> 4, reinterpret_cast<int*>(gp + 1),
                                                 &tot);
    if (tid < qc) gp[tid] = before;  // (the scan's scratch, gp[1..32], is read before this)
    __syncthreads();
    if (tid == 0) gp[qc] = tot;
    __syncthreads();
  }
  pdl_wait();
  if (tid < qc && blockIdx.x == 0) visible_entries(a, q0 + tid, a.err, true);  // flags bad input
  const int G = gp[qc];
  const int g_lo = (int)((int64_t)blockIdx.x * G / gridDim.x);
  const int g_hi = (int)((int64_t)(blockIdx.x + 1) * G / gridDim.x);
  int lq = 0;
  while (lq < qc && gp[lq + 1] <= g_lo) ++lq;
  for (; lq < qc && gp[lq] < g_hi; ++lq) {
    const int qid = q0 + lq;
    const int s_lo = max(g_lo, gp[lq]) - gp[lq], s_hi = min(g_hi, gp[lq + 1]) - gp[lq];
    if (s_hi <= s_lo) continue;
    const int64_t e0 = (int64_t)s_lo * 16;
    const int64_t e1 = min((int64_t)s_hi * 16, (int64_t)nvs[lq]);
    score_range<FMT>(a, qid, e0, e1, L.scores + (int64_t)lq * L.stride, warp, g, c);
  }
}

// ------------------------------------------------------------------ select
struct SelShared {
  uint64_t bar;
  int scratch[32];
  int res[3];
  uint32_t t1[kHistBins];     // cluster totals, key bits 31..20
  uint32_t t2[1024];          // key bits 19..10 of the keys in the chosen bin
  uint32_t t3[1024];          // key bits 9..0 under the chosen 19..10 bin
  uint32_t loc[kHistBins];    // this CTA's counts of the current level
  uint32_t above[kMaxCluster];  // per CTA of the cluster: keys above k*
  uint32_t equal[kMaxCluster];  // and equal to k*
};
constexpr int sel_smem_bytes(int threads, int per_thread) {
  return (int)((sizeof(SelShared) + 127) / 128 * 128) + threads * per_thread * 4;
}

// this CTA's counts of one level, added into `tot` of every CTA in the cluster
template <int NT>
__device__ __forceinline__ void push_level(const uint32_t* loc, uint32_t* tot, int nb, int cs) {
  for (int bin = threadIdx.x; bin < nb; bin += NT) {
    const uint32_t v = loc[bin];
    if (!v) continue;
    const uint32_t la = smem_u32(&tot[bin]);
    for (int q = 0; q < cs; ++q) tc::red_cluster_add_u32(tc::map_shared(la, q), v);
  }
}

// grid (C, queries), cluster (C, 1, 1); CTA r holds the E*1024 entries from
// r*E*1024.  Thread t owns the E consecutive entries [E t, E t + E) of the
// slice, read as 16-byte vectors in a rotated order; bit b of its masks is
// entry E t + b.
template <int NT, int E>
__global__ void __launch_bounds__(NT, 1024 / NT) topk_select_kernel(IndexerArgs a, int q0,
                                                                    WsLayout L) {
  constexpr int PER1 = kHistBins / NT;  // level-1 bins per thread
  constexpr int PER2 = 1024 / NT;       // level-2 / 3 bins per thread
  constexpr int V = E / 4;             // 16-byte vectors per thread
  constexpr int kSlice = NT * E;
  constexpr int kCopies = 8;           // bulk copies the slice is split into
  extern __shared__ __align__(128) uint8_t sel_smem[];
  SelShared* sh = reinterpret_cast<SelShared*>(sel_smem);
  pdl_trigger();
  float* sc = reinterpret_cast<float*>(sel_smem + (sizeof(SelShared) + 127) / 128 * 128);
  const int tid = threadIdx.x;
  const int cs = gridDim.x, r = blockIdx.x;
  const int lq = blockIdx.y, qid = q0 + lq;
  // positions and entry counts: inputs that no kernel of this library
  // writes, read while the scoring kernel finishes; the slice's barrier too
  const int64_t nv = visible_entries(a, qid, nullptr, false);
  if (tid == 0) {
    tc::mbar_init(&sh->bar, 1);
    tc::fence_mbar_init();
  }
  pdl_wait();
  int32_t* out = a.topk_idx + (int64_t)qid * a.k;
  float* out_s = a.topk_score ? a.topk_score + (int64_t)qid * a.k : nullptr;
  const float* scores = L.scores + (int64_t)lq * L.stride;
  const int64_t s0 = (int64_t)r * kSlice;
  const int n_slice = nv > s0 ? (int)(nv - s0 < kSlice ? nv - s0 : kSlice) : 0;

  if (nv <= a.k) {  // every visible entry is selected (the same branch in every CTA)
    for (int64_t i = s0 + tid; i < s0 + kSlice && i < a.k; i += NT) {
      out[i] = i < nv ? (int32_t)i : -1;
      if (out_s) out_s[i] = i < nv ? scores[i] : -INFINITY;
    }
    return;
  }
  // the slice's scores: one bulk copy of whole 16-byte chunks, the tail below
  const int bulk = (n_slice * 4) & ~15;
  if (tid == 0) {
    if (bulk > 0)
      tma::expect_tx(&sh->bar, (uint32_t)bulk);
    else
      tc::mbar_arrive(&sh->bar);
  }
  __syncthreads();
  if (tid < kCopies && bulk > 0) {  // a few copies in flight at once
    const int piece = ((bulk / kCopies) + 15) & ~15;
    const int b0 = tid * piece, b1 = min(bulk, b0 + piece);
    if (b1 > b0)
      tma::bulk_load(smem_u32(sc) + b0, reinterpret_cast<const uint8_t*>(scores + s0) + b0,
                     (uint32_t)(b1 - b0), &sh->bar);
  }
  for (int i = tid; i < kHistBins; i += NT) {
    sh->t1[i] = 0u;
    sh->loc[i] = 0u;
    if (i < 1024) {
      sh->t2[i] = 0u;
      sh->t3[i] = 0u;
    }
  }
  for (int i = bulk / 4 + tid; i < n_slice; i += NT) sc[i] = scores[s0 + i];
  __syncthreads();
  tc::cluster_arrive();  // the totals are zeroed before any CTA adds into them

  if (!tc::mbar_wait(&sh->bar, 0, 1u << 24) && tid == 0) flag_error(a.err, CSA_EW_TIMEOUT);

  // this thread's keys (key 0, below every score, past the slice) and the
  // entry bit of each register slot
  uint32_t kk[E];
  int bitpos[V];
#pragma unroll
  for (int q = 0; q < V; ++q) {
    const int vq = (q + tid) % V;  // rotated vector order: fewer bank conflicts
    bitpos[q] = 4 * vq;
    const float4 f = reinterpret_cast<const float4*>(sc)[tid * V + vq];
    const int e = E * tid + 4 * vq;
    kk[4 * q + 0] = e + 0 < n_slice ? score_key(f.x) : 0u;
    kk[4 * q + 1] = e + 1 < n_slice ? score_key(f.y) : 0u;
    kk[4 * q + 2] = e + 2 < n_slice ? score_key(f.z) : 0u;
    kk[4 * q + 3] = e + 3 < n_slice ? score_key(f.w) : 0u;
  }
  // (a valid key is never 0: the score_key of any finite float is positive)

  // ---- level 1: key bits 31..20
#pragma unroll
  for (int i = 0; i < E; ++i)
    if (kk[i]) atomicAdd(&sh->loc[kk[i] >> 20], 1u);
  __syncthreads();
  tc::cluster_wait();
  push_level<NT>(sh->loc, sh->t1, kHistBins, cs);
  tc::cluster_sync();
  {
    int bins[PER1];
#pragma unroll
    for (int i = 0; i < PER1; ++i) bins[i] = (int)sh->t1[kHistBins - 1 - PER1 * tid - i];
    bin_from_top<NT, PER1>(bins, kHistBins - 1 - PER1 * tid, a.k, sh->scratch, sh->res);
  }
  const uint32_t bstar = (uint32_t)sh->res[0];
  int need = a.k - sh->res[1];
  for (int i = tid; i < 1024; i += NT) sh->loc[i] = 0u;  // levels 2 and 3 use 1024 counters
  __syncthreads();

  // ---- level 2: key bits 19..10 of the B* keys
#pragma unroll
  for (int i = 0; i < E; ++i)
    if (kk[i] && (kk[i] >> 20) == bstar) atomicAdd(&sh->loc[(kk[i] >> 10) & 1023], 1u);
  __syncthreads();
  push_level<NT>(sh->loc, sh->t2, 1024, cs);
  tc::cluster_sync();
  {
    int bins[PER2];
#pragma unroll
    for (int i = 0; i < PER2; ++i) bins[i] = (int)sh->t2[1023 - PER2 * tid - i];
    bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, need, sh->scratch, sh->res);
  }
  const uint32_t p2 = (bstar << 10) | (uint32_t)sh->res[0];
  need -= sh->res[1];
  for (int i = tid; i < 1024; i += NT) sh->loc[i] = 0u;
  __syncthreads();

  // ---- level 3: key bits 9..0 under (B*, level-2 bin)
#pragma unroll
  for (int i = 0; i < E; ++i)
    if (kk[i] && (kk[i] >> 10) == p2) atomicAdd(&sh->loc[kk[i] & 1023], 1u);
  __syncthreads();
  push_level<NT>(sh->loc, sh->t3, 1024, cs);
  tc::cluster_sync();
  {
    int bins[PER2];
#pragma unroll
    for (int i = 0; i < PER2; ++i) bins[i] = (int)sh->t3[1023 - PER2 * tid - i];
    bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, need, sh->scratch, sh->res);
  }
  const uint32_t kstar = (p2 << 10) | (uint32_t)sh->res[0];
  const int need_eq = need - sh->res[1];  // entries equal to k* to take, lowest index first

  // ---- keys above / equal to k*; counts in index order by block scans
  uint32_t above_bits = 0u, eq_bits = 0u;
#pragma unroll
  for (int q = 0; q < V; ++q)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t k1 = kk[4 * q + c];
      above_bits |= (uint32_t)(k1 && k1 > kstar) << (bitpos[q] + c);
      eq_bits |= (uint32_t)(k1 && k1 == kstar) << (bitpos[q] + c);
    }
  int tot_above, tot_eq;
  const int above_before = block_excl_scan<NT>(__popc(above_bits), sh->scratch, &tot_above);
  const int eq_before = block_excl_scan<NT>(__popc(eq_bits), sh->scratch, &tot_eq);
  if (tid < cs) {
    tc::st_cluster_u32(tc::map_shared(smem_u32(&sh->above[r]), tid), (uint32_t)tot_above);
    tc::st_cluster_u32(tc::map_shared(smem_u32(&sh->equal[r]), tid), (uint32_t)tot_eq);
  }
  tc::cluster_sync();
  // ties go to the lowest indices: the lower ranks' equal keys come first
  int off = 0, eq_lower = 0;
  for (int q = 0; q < r; ++q) {
    const int take_q = min(max(need_eq - eq_lower, 0), (int)sh->equal[q]);
    off += (int)sh->above[q] + take_q;
    eq_lower += (int)sh->equal[q];
  }
  const int take_cta = min(max(need_eq - eq_lower, 0), tot_eq);
  if (r == cs - 1 && tid == 0 && off + tot_above + take_cta != a.k)
    flag_error(a.err, CSA_EW_BAD_INDEX);  // internal invariant
  // this thread's ties taken: the lowest ones, up to what the CTA takes
  int take = min(max(take_cta - eq_before, 0), __popc(eq_bits));
  uint32_t sel = above_bits;
  for (uint32_t e = eq_bits; e && take > 0; --take) {
    const uint32_t low = e & (~e + 1u);
    sel |= low;
    e ^= low;
  }
  int pos = off + above_before + min(max(take_cta, 0), eq_before);
  while (sel) {
    const int b = __ffs(sel) - 1;
    sel &= sel - 1;
    if (pos < a.k) {
      const int e = E * tid + b;
      out[pos] = (int32_t)(s0 + e);
      if (out_s) out_s[pos] = sc[e];
    }
    ++pos;
  }
}

// One CTA per query, no cluster, for calls with many queries (chunked
// prefill): the query's scores are streamed from the workspace rather than
// held in registers.  The usual case reads them once: an evenly spaced
// sample of the row gives a key bound lo (its key at the rank that
// corresponds to about (k + kList) / 2 entries of the row); one streamed
// pass lists, in index order, the entries above lo and the first k equal to
// it (per-warp segments and buckets, no block barrier per tile); when the
// list holds at least k and at most kList entries, key bits 31..20, 19..10
// and 9..0 of the listed keys give the exact k-th key k* and how many
// entries equal to it to take, and one block scan over the list writes the
// entries above k* and the lowest-index ties.  Otherwise (a skewed sample,
// k > kList / 2) the histogram passes do it: pass 1, a histogram of key bits
// 31..20 (4096 bins) and the bin B* holding the k-th key; when B* and the
// bins above it hold at most kList entries, one more streamed pass lists
// them and the selection is made from the list as above; else pass 2 keeps
// B*'s keys (at most kCand; else two more streamed passes) to find k*, and
// pass 3 walks the scores in index order once more.  Same selection as
// topk_select_kernel.
constexpr int kCand = 2048;
constexpr int kList = 4096;
constexpr int kSampleVec = 1024;  // 16-byte score vectors sampled for the list's bound
static_assert(kList >= 4 * kSampleVec, "a row longer than the list holds a whole sample");
constexpr int kStreamWarps = 16;  // warps of a select CTA (512 threads)
constexpr int kBucket = 512;      // entries a warp may take in one streamed pass
struct StreamShared {
  uint32_t hist[kHistBins];
  uint32_t lkey[kList];  // the list: keys and entry indices, in index order
  int32_t lidx[kList];
  // per-warp buckets of a streamed pass: keys [warp][kBucket], then indices;
  // the histogram passes keep threshold-bin keys (at most kCand) at the front
  uint32_t buckets[2 * kStreamWarps * kBucket];
  int wcnt[kStreamWarps];    // entries a warp took (above lo or equal to it)
  int wcnt_e[kStreamWarps];  // of those, equal to lo
  int scratch[32];
  int res[3];
  int ncand;
};
static_assert(kCand <= 2 * kStreamWarps * kBucket, "threshold-bin keys fit the buckets");

template <int NT>
__global__ void __launch_bounds__(NT, 2) topk_stream_kernel(IndexerArgs a, int q0, WsLayout L) {
  constexpr int PER1 = kHistBins / NT;
  constexpr int PER2 = 1024 / NT;
  constexpr int kE = 16;  // entries per thread per output tile
  extern __shared__ __align__(16) uint8_t stream_smem[];
  StreamShared& sh = *reinterpret_cast<StreamShared*>(stream_smem);
  uint32_t* const cand = sh.buckets;
  pdl_trigger();
  const int tid = threadIdx.x;
  const int lq = blockIdx.x, qid = q0 + lq;
  // positions and entry counts: inputs that no kernel of this library
  // writes, read while the scoring kernel finishes
  const int64_t nv = visible_entries(a, qid, nullptr, false);
  pdl_wait();
  int32_t* out = a.topk_idx + (int64_t)qid * a.k;
  float* out_s = a.topk_score ? a.topk_score + (int64_t)qid * a.k : nullptr;
  const float* scores = L.scores + (int64_t)lq * L.stride;
  if (nv <= a.k) {  // every visible entry is selected
    for (int i = tid; i < a.k; i += NT) {
      out[i] = i < nv ? (int32_t)i : -1;
      if (out_s) out_s[i] = i < nv ? scores[i] : -INFINITY;
    }
    return;
  }
  const int n = (int)nv;
  const int n4 = n >> 2;
  const float4* s4 = reinterpret_cast<const float4*>(scores);  // rows are 128-byte aligned
  // stream every visible key through f(key) (4 vectors in flight per thread)
  auto sweep = [&](auto&& f) {
    int i = tid;
    for (; i + 3 * NT < n4; i += 4 * NT) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = s4[i + u * NT];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        f(score_key(v[u].x));
        f(score_key(v[u].y));
        f(score_key(v[u].z));
        f(score_key(v[u].w));
      }
    }
    for (; i < n4; i += NT) {
      const float4 v = s4[i];
      f(score_key(v.x));
      f(score_key(v.y));
      f(score_key(v.z));
      f(score_key(v.w));
    }
    for (int e = 4 * n4 + tid; e < n; e += NT) f(score_key(scores[e]));
  };

  // ---- the exact selection among a list of entries (index order) that holds
  // every entry whose key is at or above some bound, and at least k of them
  // (so the k-th key k* is in the list): k* from key bits 31..20, 19..10 and
  // 9..0 of the listed keys, then one block scan per NT listed entries writes
  // the entries above k* and the lowest-index ties, in index order
  auto select_list = [&](int nlist) {
    for (int i = tid; i < kHistBins; i += NT) sh.hist[i] = 0u;
    __syncthreads();
    for (int c = tid; c < nlist; c += NT) atomicAdd(&sh.hist[sh.lkey[c] >> 20], 1u);
    __syncthreads();
    {
      int bins[PER1];
#pragma unroll
      for (int i = 0; i < PER1; ++i) bins[i] = (int)sh.hist[kHistBins - 1 - PER1 * tid - i];
      bin_from_top<NT, PER1>(bins, kHistBins - 1 - PER1 * tid, a.k, sh.scratch, sh.res);
    }
    const uint32_t bstar = (uint32_t)sh.res[0];
    int need = a.k - sh.res[1];
    for (int i = tid; i < 1024; i += NT) sh.hist[i] = 0u;
    __syncthreads();
    for (int c = tid; c < nlist; c += NT)
      if ((sh.lkey[c] >> 20) == bstar) atomicAdd(&sh.hist[(sh.lkey[c] >> 10) & 1023], 1u);
    __syncthreads();
    {
      int bins[PER2];
#pragma unroll
      for (int i = 0; i < PER2; ++i) bins[i] = (int)sh.hist[1023 - PER2 * tid - i];
      bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, need, sh.scratch, sh.res);
    }
    const uint32_t p2 = (bstar << 10) | (uint32_t)sh.res[0];
    need -= sh.res[1];
    for (int i = tid; i < 1024; i += NT) sh.hist[i] = 0u;
    __syncthreads();
    for (int c = tid; c < nlist; c += NT)
      if ((sh.lkey[c] >> 10) == p2) atomicAdd(&sh.hist[sh.lkey[c] & 1023], 1u);
    __syncthreads();
    {
      int bins[PER2];
#pragma unroll
      for (int i = 0; i < PER2; ++i) bins[i] = (int)sh.hist[1023 - PER2 * tid - i];
      bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, need, sh.scratch, sh.res);
    }
    const uint32_t kstar = (p2 << 10) | (uint32_t)sh.res[0];
    const int need_eq = need - sh.res[1];
    int run_above = 0, run_eq = 0;
    for (int c0 = 0; c0 < nlist; c0 += NT) {
      const int c = c0 + tid;
      const uint32_t key = c < nlist ? sh.lkey[c] : 0u;
      const int above = key > kstar ? 1 : 0, eq = (c < nlist && key == kstar) ? 1 : 0;
      int tot;
      const int before = block_excl_scan<NT>(above | (eq << 16), sh.scratch, &tot);
      const int e_rank = run_eq + (before >> 16);
      if (above || (eq && e_rank < need_eq)) {
        const int pos = run_above + (before & 0xFFFF) + min(e_rank, need_eq);
        if (pos < a.k) {
          out[pos] = sh.lidx[c];
          if (out_s) out_s[pos] = scores[sh.lidx[c]];
        }
      }
      run_above += tot & 0xFFFF;
      run_eq += tot >> 16;
    }
    if (tid == 0 && run_above + min(run_eq, need_eq) != a.k)
      flag_error(a.err, CSA_EW_BAD_INDEX);  // internal invariant
  };

  // ---- one streamed pass: the entries at or above lo, in index order, into
  // the list.  Each warp streams its own contiguous segment of the row (whole
  // 256-entry steps: lane l holds entries 4 l .. 4 l + 3 of each half, three
  // steps of loads in flight) and appends to its own bucket, in order, every
  // entry that a float compare with lo's value does not rule out (NaN scores
  // included); no barrier until the segment ends.  The exact key test comes
  // at the copy to the list: every warp counts the keys of its bucket above
  // lo and equal to it, and copies them to the list at the offsets the lower
  // warps' counts give.  Strict: the entries above lo all go in, and of
  // those equal to lo only the first k of the row (no more can be selected:
  // if k* == lo they are the lowest-index ties), so a bound that many
  // entries share still gives a short list.  Returns the list's length (at
  // most kList entries are written), or -1 when a bucket overflowed.
  constexpr int kWarps = NT / 32;
  constexpr int kStep = 256;
  constexpr int kAhead = 3;
  static_assert(kWarps == kStreamWarps, "one bucket per warp");
  auto warp_gather = [&](auto strict_tag, uint32_t lo) -> int {
    constexpr bool strict = decltype(strict_tag)::value;
    const int warp = tid >> 5, lane = tid & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    // lo's score (the inverse of score_key); !(f < lo_f) holds for every f
    // whose key is at least lo, and for NaN
    const uint32_t lo_bits = (lo & 0x80000000u) ? (lo & 0x7FFFFFFFu) : ~lo;
    const float lo_f = __uint_as_float(lo_bits);
    const int seg = (n + kWarps * kStep - 1) / (kWarps * kStep) * kStep;
    const int s_begin = min(n, warp * seg), s_end = min(n, s_begin + seg);
    uint32_t* bk = sh.buckets + warp * kBucket;
    int32_t* bi = reinterpret_cast<int32_t*>(sh.buckets + kStreamWarps * kBucket) + warp * kBucket;
    const uint64_t drop = l2_evict_first_policy();  // each score is read once here
    float4 v[kAhead][2];
    auto ld = [&](float4 (&w)[2], int base) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int e = base + 128 * j + 4 * lane;  // the row holds whole 16-byte vectors
        w[j] = e < s_end ? ld_f32x4_policy(s4 + (e >> 2), drop)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
#pragma unroll
    for (int i = 0; i < kAhead; ++i) ld(v[i], s_begin + i * kStep);
    int run = 0;
    for (int base = s_begin; base < s_end; base += kAhead * kStep) {
#pragma unroll
      for (int i = 0; i < kAhead; ++i) {
        const int b = base + i * kStep;
        if (b < s_end) {  // warp-uniform
          const float f[8] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w,
                              v[i][1].x, v[i][1].y, v[i][1].z, v[i][1].w};
          unsigned m = 0u;
#pragma unroll
          for (int c = 0; c < 8; ++c) m |= (unsigned)!(f[c] < lo_f) << c;
          if (b + kStep > s_end) {  // the segment's last step: entries past its end
            const int r0 = s_end - (b + 4 * lane), r1 = r0 - 128;
            m &= (r0 >= 4 ? 0xFu : (1u << max(r0, 0)) - 1u) |
                 ((r1 >= 4 ? 0xFu : (1u << max(r1, 0)) - 1u) << 4);
          }
          // takes before this lane, both halves at once (8 bits each)
          const int own = __popc(m & 0xFu) | (__popc(m >> 4) << 8);
          int inc = own;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += y;
          }
          const int tot = __shfl_sync(0xFFFFFFFFu, inc, 31);
          const int excl = inc - own;
          int pos0 = run + (excl & 0xFF), pos1 = run + (tot & 0xFF) + (excl >> 8);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            if ((m >> c) & 1u) {
              int& p = c < 4 ? pos0 : pos1;
              if (p < kBucket) {
                bk[p] = score_key(f[c]);
                bi[p] = b + (c < 4 ? 0 : 128) + 4 * lane + (c & 3);
              }
              ++p;
            }
          run += (tot & 0xFF) + (tot >> 8);
        }
        if (b + kAhead * kStep < s_end) ld(v[i], b + kAhead * kStep);
      }
    }
    // exact keys: above lo (at or above it when not strict), equal to it
    int cnt_a = 0, cnt_e = 0;
    if (run <= kBucket)
      for (int c0 = 0; c0 < run; c0 += 32) {
        const int c = c0 + lane;
        const uint32_t key = c < run ? bk[c] : 0u;
        const bool is_a = c < run && (strict ? key > lo : key >= lo);
        const bool is_e = c < run && strict && key == lo;
        cnt_a += __popc(__ballot_sync(0xFFFFFFFFu, is_a));
        cnt_e += __popc(__ballot_sync(0xFFFFFFFFu, is_e));
      }
    if (lane == 0) {
      sh.wcnt[warp] = run > kBucket ? -1 : cnt_a;
      sh.wcnt_e[warp] = cnt_e;
    }
    __syncthreads();
    bool over = false;
    int tot_a = 0, tot_e = 0, a_before = 0, e_before = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int ca = sh.wcnt[w], ce = sh.wcnt_e[w];
      over |= ca < 0;
      if (w < warp) {
        a_before += ca;
        e_before += ce;
      }
      tot_a += ca;
      tot_e += ce;
    }
    const int len = tot_a + min(tot_e, a.k);
    if (over) return -1;
    if (len < a.k || len > kList) return len;
    for (int c0 = 0; c0 < run; c0 += 32) {
      const int c = c0 + lane;
      const uint32_t key = c < run ? bk[c] : 0u;
      const bool is_a = c < run && (strict ? key > lo : key >= lo);
      const bool is_e = c < run && strict && key == lo;
      const unsigned be = __ballot_sync(0xFFFFFFFFu, is_e), ba = __ballot_sync(0xFFFFFFFFu, is_a);
      const int e_r = e_before + __popc(be & lt_mask);
      const int a_r = a_before + __popc(ba & lt_mask);
      int p = kList;
      if (is_a) p = a_r + min(e_r, a.k);
      else if (is_e && e_r < a.k) p = a_r + e_r;
      if (p < kList) {
        sh.lkey[p] = key;
        sh.lidx[p] = bi[c];
      }
      a_before += __popc(ba);
      e_before += __popc(be);
    }
    __syncthreads();
    return len;
  };

  // ---- the usual case: a bound from a sample.  kSampleVec evenly spaced
  // 16-byte vectors of the scores (4 * kSampleVec keys) give lo, the
  // sample's key of the rank that corresponds to (k + kList) / 2 entries of
  // the whole row; when at
  // least k entries are at or above lo and the list holds them, one streamed
  // pass lists them and the selection is made from the list.  Otherwise (a
  // skewed sample) the histogram passes below do it.  With n <= kList every
  // entry is listed.
  if (2 * a.k <= kList) {
    uint32_t lo = 1u;
    bool strict = false;
    if (n > kList) {
      constexpr int kSV = kSampleVec / NT;
      const int stride = n4 / kSampleVec;  // >= 1: n > kList >= 4 * kSampleVec
      // the sample's keys wait in the list's key array (thread t's at 4 t + ...)
      uint32_t* sk = sh.lkey;
#pragma unroll
      for (int u = 0; u < kSV; ++u) {
        const float4 f = s4[(int64_t)(tid + u * NT) * stride];
        *reinterpret_cast<uint4*>(sk + 4 * (tid + u * NT)) =
            make_uint4(score_key(f.x), score_key(f.y), score_key(f.z), score_key(f.w));
      }
      for (int i = tid; i < kHistBins; i += NT) sh.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < 4 * kSampleVec; i += NT) atomicAdd(&sh.hist[sk[i] >> 20], 1u);
      __syncthreads();
      int r = (int)((int64_t)((a.k + kList) / 2) * (4 * kSampleVec) / n);
      r = r < 1 ? 1 : r;  // < 4 * kSampleVec, since n > kList
      {
        int bins[PER1];
#pragma unroll
        for (int i = 0; i < PER1; ++i) bins[i] = (int)sh.hist[kHistBins - 1 - PER1 * tid - i];
        bin_from_top<NT, PER1>(bins, kHistBins - 1 - PER1 * tid, r, sh.scratch, sh.res);
      }
      const uint32_t b1 = (uint32_t)sh.res[0];
      r -= sh.res[1];
      for (int i = tid; i < 1024; i += NT) sh.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < 4 * kSampleVec; i += NT)
        if ((sk[i] >> 20) == b1) atomicAdd(&sh.hist[(sk[i] >> 10) & 1023], 1u);
      __syncthreads();
      {
        int bins[PER2];
#pragma unroll
        for (int i = 0; i < PER2; ++i) bins[i] = (int)sh.hist[1023 - PER2 * tid - i];
        bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, r, sh.scratch, sh.res);
      }
      const uint32_t b2 = (b1 << 10) | (uint32_t)sh.res[0];
      r -= sh.res[1];
      for (int i = tid; i < 1024; i += NT) sh.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < 4 * kSampleVec; i += NT)
        if ((sk[i] >> 10) == b2) atomicAdd(&sh.hist[sk[i] & 1023], 1u);
      __syncthreads();
      {
        int bins[PER2];
#pragma unroll
        for (int i = 0; i < PER2; ++i) bins[i] = (int)sh.hist[1023 - PER2 * tid - i];
        bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, r, sh.scratch, sh.res);
      }
      lo = (b2 << 10) | (uint32_t)sh.res[0];  // a sample key: never 0
      strict = true;
    }
    const int nlist =
        strict ? warp_gather(std::true_type{}, lo) : warp_gather(std::false_type{}, lo);
    if (nlist >= a.k && nlist <= kList) {
      select_list(nlist);
      return;
    }
  }
  // ---- pass 1: bits 31..20
  for (int i = tid; i < kHistBins; i += NT) sh.hist[i] = 0u;
  if (tid == 0) sh.ncand = 0;
  __syncthreads();
  sweep([&](uint32_t key) { atomicAdd(&sh.hist[key >> 20], 1u); });
  __syncthreads();
  {
    int bins[PER1];
#pragma unroll
    for (int i = 0; i < PER1; ++i) bins[i] = (int)sh.hist[kHistBins - 1 - PER1 * tid - i];
    bin_from_top<NT, PER1>(bins, kHistBins - 1 - PER1 * tid, a.k, sh.scratch, sh.res);
  }
  const uint32_t bstar = (uint32_t)sh.res[0];
  int need = a.k - sh.res[1];
  const bool in_smem = sh.hist[bstar] <= (uint32_t)kCand;
  const int nlist = sh.res[1] + (int)sh.hist[bstar];  // entries in B* or above it
  __syncthreads();

  if (nlist <= kList) {
    // ---- pass 2: those entries into the list
    if (warp_gather(std::false_type{}, bstar << 20) == nlist) {
      select_list(nlist);
      return;
    }
  }
  // ---- pass 2: the keys of B*; levels 2 and 3 over them
  if (in_smem)
    sweep([&](uint32_t key) {
      if ((key >> 20) == bstar) cand[atomicAdd(&sh.ncand, 1)] = key;
    });
  for (int i = tid; i < 1024; i += NT) sh.hist[i] = 0u;
  __syncthreads();
  const int nc = sh.ncand;
  if (in_smem) {
    for (int c = tid; c < nc; c += NT) atomicAdd(&sh.hist[(cand[c] >> 10) & 1023], 1u);
  } else {
    sweep([&](uint32_t key) {
      if ((key >> 20) == bstar) atomicAdd(&sh.hist[(key >> 10) & 1023], 1u);
    });
  }
  __syncthreads();
  {
    int bins[PER2];
#pragma unroll
    for (int i = 0; i < PER2; ++i) bins[i] = (int)sh.hist[1023 - PER2 * tid - i];
    bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, need, sh.scratch, sh.res);
  }
  const uint32_t p2 = (bstar << 10) | (uint32_t)sh.res[0];
  need -= sh.res[1];
  for (int i = tid; i < 1024; i += NT) sh.hist[i] = 0u;
  __syncthreads();
  if (in_smem) {
    for (int c = tid; c < nc; c += NT)
      if ((cand[c] >> 10) == p2) atomicAdd(&sh.hist[cand[c] & 1023], 1u);
  } else {
    sweep([&](uint32_t key) {
      if ((key >> 10) == p2) atomicAdd(&sh.hist[key & 1023], 1u);
    });
  }
  __syncthreads();
  {
    int bins[PER2];
#pragma unroll
    for (int i = 0; i < PER2; ++i) bins[i] = (int)sh.hist[1023 - PER2 * tid - i];
    bin_from_top<NT, PER2>(bins, 1023 - PER2 * tid, need, sh.scratch, sh.res);
  }
  const uint32_t kstar = (p2 << 10) | (uint32_t)sh.res[0];
  const int need_eq = need - sh.res[1];  // entries equal to k* to take, lowest index first

  // ---- pass 3: the selection in index order
  int run_above = 0, run_eq = 0;
  for (int base = 0; base < n; base += NT * kE) {
    const int i0 = base + tid * kE;
    uint32_t above = 0u, eq = 0u;
#pragma unroll
    for (int q = 0; q < kE / 4; ++q) {
      const int e = i0 + 4 * q;
      float f[4];
      if (e + 3 < n) {
        const float4 v = s4[e >> 2];
        f[0] = v.x, f[1] = v.y, f[2] = v.z, f[3] = v.w;
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) f[c] = e + c < n ? scores[e + c] : 0.f;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t key = e + c < n ? score_key(f[c]) : 0u;
        above |= (uint32_t)(key > kstar) << (4 * q + c);
        eq |= (uint32_t)(key == kstar) << (4 * q + c);
      }
    }
    int tot;
    const int before =
        block_excl_scan<NT>(__popc(above) | (__popc(eq) << 16), sh.scratch, &tot);
    const int a_before = before & 0xFFFF, e_before = before >> 16;
    int e_rank = run_eq + e_before;
    int pos = run_above + a_before + min(e_rank, need_eq);
    for (uint32_t m = above | eq; m; m &= m - 1) {
      const int b = __ffs(m) - 1;
      bool take = (above >> b) & 1u;
      if (!take) take = e_rank++ < need_eq;
      if (take) {
        if (pos < a.k) {
          out[pos] = i0 + b;
          if (out_s) out_s[pos] = scores[i0 + b];
        }
        ++pos;
      }
    }
    run_above += tot & 0xFFFF;
    run_eq += tot >> 16;
  }
  if (tid == 0 && run_above + min(run_eq, need_eq) != a.k)
    flag_error(a.err, CSA_EW_BAD_INDEX);  // internal invariant
}

}  // namespace

size_t indexer_topk_workspace_bytes(int n_query, int N_cap) {
  const int qc = n_query < kQueryChunk ? n_query : kQueryChunk;
  return align256((size_t)qc * score_stride(N_cap) * sizeof(float));
}

namespace {

// scores of queries [q0, q0 + qc) into L (row of query q0 + i at i * stride):
// for many tokens per sequence one tensor-core GEMM, else the streaming kernel
cudaError_t launch_scores(const IndexerArgs& a, int q0, int qc, const WsLayout& L,
                          cudaStream_t st) {
  if (a.T > 8 && indexer_gemm_applies(a))
    return launch_indexer_gemm(a, q0, qc, L.scores, L.stride, st);
  // one wave (the CTAs per SM the format fits), fewer when there is little
  // work: at least kChunk entries' worth of groups per CTA on average
  const int64_t groups = (int64_t)qc * ((a.N_cap + 15) / 16);
  int64_t n_cta = (groups * 16 + kChunk - 1) / kChunk;
  const int per_sm = score_ctas_per_sm(a.fp4 ? 2 : a.fp8 ? 1 : 0);
  if (n_cta > per_sm * kNumSMs) n_cta = per_sm * kNumSMs;
  const dim3 g1((unsigned)(n_cta > 0 ? n_cta : 1));
  if (a.fp4) return launch_pdl(indexer_score_kernel<2>, g1, dim3(kThreads), 0, st, a, q0, qc, L);
  if (a.fp8) return launch_pdl(indexer_score_kernel<1>, g1, dim3(kThreads), 0, st, a, q0, qc, L);
  return launch_pdl(indexer_score_kernel<0>, g1, dim3(kThreads), 0, st, a, q0, qc, L);
}

}  // namespace

cudaError_t launch_indexer_scores(const IndexerArgs& a, float* scores, int ld, cudaStream_t st) {
  for (int q0 = 0; q0 < a.n_query; q0 += kQueryChunk) {
    const int qc = (a.n_query - q0 < kQueryChunk) ? a.n_query - q0 : kQueryChunk;
    WsLayout L;
    L.scores = scores + (int64_t)q0 * ld;
    L.stride = ld;
    const cudaError_t e = launch_scores(a, q0, qc, L, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {

// Select launch shape: CTAs of NT threads with E entries per thread, cs per
// query (one cluster).
struct SelPlan {
  int nt, per, cs;
  const void* fn;
};

SelPlan select_plan(int n_query, int n_cap) {
  // few queries: 1024-thread CTAs, the fewest entries per thread (8, 16, 32)
  // that need at most 8 CTAs per query (clusters of 8 still fit two to a GPC)
  SelPlan p;
  p.nt = 1024;
  p.per = n_cap <= 8 * 1024 * 8 ? 8 : n_cap <= 8 * 1024 * 16 ? 16 : 32;
  p.cs = (n_cap + 1024 * p.per - 1) / (1024 * p.per);
  // many queries (several waves of CTAs, each latency-bound): 512-thread
  // CTAs, two per SM, so that one CTA's barriers overlap another's work
  const int64_t ctas = (int64_t)(n_query < kQueryChunk ? n_query : kQueryChunk) * p.cs;
  if (ctas > 2 * kNumSMs && n_cap <= 8 * 512 * 32) {
    p.nt = 512;
    p.per = 32;
    p.cs = (n_cap + 512 * 32 - 1) / (512 * 32);
  }
  p.fn = p.nt == 512   ? (const void*)topk_select_kernel<512, 32>
         : p.per == 8  ? (const void*)topk_select_kernel<1024, 8>
         : p.per == 16 ? (const void*)topk_select_kernel<1024, 16>
                       : (const void*)topk_select_kernel<1024, 32>;
  return p;
}

}  // namespace

cudaError_t launch_indexer_topk(const IndexerArgs& a, void* ws, cudaStream_t st) {
  WsLayout L = carve(ws, a.N_cap);
  const SelPlan p = select_plan(a.n_query, a.N_cap);
  {
    cudaError_t e = ensure_smem_attr(p.fn, sel_smem_bytes(p.nt, p.per), true);
    if (e == cudaSuccess)
      e = ensure_smem_attr((const void*)topk_stream_kernel<512>, (int)sizeof(StreamShared));
    if (e != cudaSuccess) return e;
  }
  for (int q0 = 0; q0 < a.n_query; q0 += kQueryChunk) {
    const int qc = (a.n_query - q0 < kQueryChunk) ? a.n_query - q0 : kQueryChunk;
    cudaError_t e = launch_scores(a, q0, qc, L, st);
    if (e != cudaSuccess) return e;
    if (qc >= kStreamQueries) {  // one CTA per query, streamed from L2
      e = launch_pdl(topk_stream_kernel<512>, dim3((unsigned)qc), dim3(512),
                     sizeof(StreamShared), st, a, q0, L);
      if (e != cudaSuccess) return e;
      continue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.cs, (unsigned)qc);
    cfg.blockDim = dim3((unsigned)p.nt);
    cfg.dynamicSmemBytes = sel_smem_bytes(p.nt, p.per);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (p.nt == 512)
      e = cudaLaunchKernelEx(&cfg, topk_select_kernel<512, 32>, a, q0, L);
    else if (p.per == 8)
      e = cudaLaunchKernelEx(&cfg, topk_select_kernel<1024, 8>, a, q0, L);
    else if (p.per == 16)
      e = cudaLaunchKernelEx(&cfg, topk_select_kernel<1024, 16>, a, q0, L);
    else
      e = cudaLaunchKernelEx(&cfg, topk_select_kernel<1024, 32>, a, q0, L);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa
