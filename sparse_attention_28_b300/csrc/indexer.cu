// indexer.cu -- Lightning-Indexer scores and exact top-k selection.
//
// Method: hyper.ai DeepSeek-V4 page, Method ("A Lightning Indexer then
// selects the top-k compressed KV entries"); aiboss88 DeepSeek-V4 page,
// Technical Principles (index score, then top-k sparse selection; FP8 range
// for the low-precision indexer QK path); elamur.ai page, Summary ("runs
// DeepSeek Sparse Attention"), read as
//     I(t,s) = sum_h w[t][h] * ReLU(q[t][h] . k[s]),  s < n_vis(t).
//
// Pipeline per call (queries processed in chunks that keep the score buffer
// near L2 size):
//   1. memset of the per-query histogram + candidate counter,
//   2. score kernel: streams the compressed indexer keys once (the dominant
//      HBM traffic), computes the 4-head scores with m16n8k16 tensor-core
//      MMAs (entries on M, heads on N), writes fp32 scores and a 4096-bin
//      histogram of the top 12 bits of each score's order-preserving key,
//   3. mark kernel (several CTAs per query): from the histogram finds the
//      threshold bin B*; sets a bitmap bit for every entry above B* and
//      appends the entries of bin B* to a candidate list,
//   4. select kernel (one CTA per query): exact k-th key among the
//      candidates (ties to the lower index), then writes the selected entries
//      in ascending index order from the bitmap.
// Bins, keys and the tie rule give the same set as a full sort on
// (-score, index).
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kDI = 64;
constexpr int kHI = 4;
constexpr int kScoreThreads = 256;
constexpr int kChunk = 2048;       // entries per score CTA
constexpr int kUnroll = 4;         // 16-entry groups in flight per warp
constexpr int kMarkThreads = 256;
constexpr int kMarkSlice = 8192;   // entries per mark CTA
constexpr int kMarkUnroll = 8;     // 32-entry words per warp per run
constexpr int kSelThreads = 512;
constexpr int kQueryChunk = 256;   // queries per pass (bounds the workspace)
constexpr int kHdrWords = kHistBins + 32;  // hist[4096], cand counter, pad

struct WsLayout {
  float* scores;      // [QC][N_cap]
  int32_t* hdr;       // [QC][kHdrWords]
  uint32_t* bitmap;   // [QC][bm_stride]
  uint2* cand;        // [QC][kCandCap] (key, index)
  int bm_stride;
};

__host__ __device__ inline int bitmap_words(int n_cap) { return ((n_cap + 31) / 32 + 3) & ~3; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout carve(void* ws, int qc, int n_cap) {
  WsLayout L;
  uint8_t* p = reinterpret_cast<uint8_t*>(ws);
  L.scores = reinterpret_cast<float*>(p);
  p += align256((size_t)qc * n_cap * sizeof(float));
  L.hdr = reinterpret_cast<int32_t*>(p);
  p += align256((size_t)qc * kHdrWords * sizeof(int32_t));
  L.bm_stride = bitmap_words(n_cap);
  L.bitmap = reinterpret_cast<uint32_t*>(p);
  p += align256((size_t)qc * L.bm_stride * sizeof(uint32_t));
  L.cand = reinterpret_cast<uint2*>(p);
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

// ------------------------------------------------------------------ scores
// Fragment mapping (m16n8k16, A = 16 entries x 16 dims, B = 16 dims x 8
// heads, heads 4..7 are zero).  The contraction order over the 64 dims is
// free, so each thread loads whole 16-byte vectors of a key row and the query
// fragments use the same permutation:
//   bf16: thread (g, c) holds row bytes [16c,16c+16) and [64+16c, 64+16c+16);
//         k-step s takes word s of each vector.
//   E4M3: thread (g, c) holds row bytes [16c, 16c+16) converted to 8 f16x2
//         words (exact); k-step s takes words s and 4+s.
template <bool FP8>
__global__ void __launch_bounds__(kScoreThreads) indexer_score_kernel(IndexerArgs a, int q0,
                                                                     WsLayout L) {
  __shared__ int hist_s[kHistBins];
  const int qid = q0 + blockIdx.y;
  const int lq = blockIdx.y;
  const int64_t nv = visible_entries(a, qid, a.err, blockIdx.x == 0 && threadIdx.x == 0);
  const int64_t e0 = (int64_t)blockIdx.x * kChunk;
  if (e0 >= nv) return;
  const int64_t e1 = (e0 + kChunk < nv) ? e0 + kChunk : nv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  for (int i = tid; i < kHistBins; i += kScoreThreads) hist_s[i] = 0;

  // query fragments (heads g < 4) and head weights (heads 2c, 2c+1 for c < 2)
  uint32_t qb0[4] = {0, 0, 0, 0}, qb1[4] = {0, 0, 0, 0};
  float w0 = 0.f, w1 = 0.f;
  if (g < kHI) {
    if (FP8) {
      const uint8_t* qr = reinterpret_cast<const uint8_t*>(a.q) + ((int64_t)qid * kHI + g) * kDI;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(qr + 16 * c));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t lo = e4m3x2_to_f16x2((uint16_t)(wv[s >> 1] >> ((s & 1) * 16)));
        const uint32_t hi = e4m3x2_to_f16x2((uint16_t)(wv[2 + (s >> 1)] >> ((s & 1) * 16)));
        qb0[s] = lo;
        qb1[s] = hi;
      }
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
  __syncthreads();

  const int b = qid / a.T;
  float* scores = L.scores + (int64_t)lq * a.N_cap;
  const int n_groups = (int)((e1 - e0 + 15) / 16);
  for (int gb = warp * kUnroll; gb < n_groups; gb += (kScoreThreads / 32) * kUnroll) {
    uint4 ra[kUnroll][2], rb[kUnroll][2];  // rows g and g+8 of each group
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t ea = e0 + (int64_t)(gb + u) * 16 + g, eb = ea + 8;
      if (FP8) {
        const uint8_t* kb = reinterpret_cast<const uint8_t*>(a.keys) + (int64_t)b * a.k_bstride;
        ra[u][0] = ea < e1 ? __ldg(reinterpret_cast<const uint4*>(kb + ea * kDI + 16 * c))
                           : make_uint4(0, 0, 0, 0);
        rb[u][0] = eb < e1 ? __ldg(reinterpret_cast<const uint4*>(kb + eb * kDI + 16 * c))
                           : make_uint4(0, 0, 0, 0);
      } else {
        const bf16* kb = reinterpret_cast<const bf16*>(a.keys) + (int64_t)b * a.k_bstride;
        const uint4 z = make_uint4(0, 0, 0, 0);
        ra[u][0] = ea < e1 ? __ldg(reinterpret_cast<const uint4*>(kb + ea * kDI + 8 * c)) : z;
        ra[u][1] = ea < e1 ? __ldg(reinterpret_cast<const uint4*>(kb + ea * kDI + 32 + 8 * c)) : z;
        rb[u][0] = eb < e1 ? __ldg(reinterpret_cast<const uint4*>(kb + eb * kDI + 8 * c)) : z;
        rb[u][1] = eb < e1 ? __ldg(reinterpret_cast<const uint4*>(kb + eb * kDI + 32 + 8 * c)) : z;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (gb + u >= n_groups) break;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (FP8) {
        const uint32_t xa[4] = {ra[u][0].x, ra[u][0].y, ra[u][0].z, ra[u][0].w};
        const uint32_t xb[4] = {rb[u][0].x, rb[u][0].y, rb[u][0].z, rb[u][0].w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint32_t af[4];
          af[0] = e4m3x2_to_f16x2((uint16_t)(xa[s >> 1] >> ((s & 1) * 16)));
          af[1] = e4m3x2_to_f16x2((uint16_t)(xb[s >> 1] >> ((s & 1) * 16)));
          af[2] = e4m3x2_to_f16x2((uint16_t)(xa[2 + (s >> 1)] >> ((s & 1) * 16)));
          af[3] = e4m3x2_to_f16x2((uint16_t)(xb[2 + (s >> 1)] >> ((s & 1) * 16)));
          mma_f16_16816(acc, af, qb0[s], qb1[s]);
        }
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
        if (FP8) sc *= __ldg(a.k_scale + (int64_t)b * a.ks_bstride + e);
        scores[e] = sc;
        atomicAdd(&hist_s[score_key(sc) >> 20], 1);
      }
    }
  }
  __syncthreads();
  int32_t* hist = L.hdr + (int64_t)lq * kHdrWords;
  for (int i = tid; i < kHistBins; i += kScoreThreads) {
    const int v = hist_s[i];
    if (v) atomicAdd(hist + i, v);
  }
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

// Threshold bin: the highest bin B such that the count of keys in bins > B
// is < k <= count in bins >= B.  Returns B, the count above it, its count.
template <int NT>
__device__ void find_threshold_bin(const int32_t* hist, int k, int* scratch, int* res) {
  constexpr int per = kHistBins / NT;
  const int tid = threadIdx.x;
  // thread tid owns bins [kHistBins - (tid+1)*per, kHistBins - tid*per): high bins first
  const int hi = kHistBins - tid * per;
  int local = 0;
  for (int i = 1; i <= per; ++i) local += hist[hi - i];
  int total;
  const int before = block_excl_scan<NT>(local, scratch, &total);  // count in higher bins
  if (before < k && before + local >= k) {
    int run = before;
    for (int i = 1; i <= per; ++i) {
      const int bin = hi - i, cnt = hist[bin];
      if (run + cnt >= k) {
        res[0] = bin;
        res[1] = run;
        res[2] = cnt;
        break;
      }
      run += cnt;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ mark
// grid (slices, queries): bitmap bits for keys above the threshold bin; the
// keys in it are gathered in shared memory and appended to the query's
// candidate list with one global atomic per CTA.
__global__ void __launch_bounds__(kMarkThreads) topk_mark_kernel(IndexerArgs a, int q0,
                                                                 WsLayout L) {
  extern __shared__ __align__(16) uint2 lcand[];  // [kMarkSlice]
  __shared__ int scratch[32];
  __shared__ int res[3];
  __shared__ int n_local, g_base;
  const int qid = q0 + blockIdx.y, lq = blockIdx.y;
  const int64_t nv = visible_entries(a, qid, nullptr, false);
  const int64_t s0 = (int64_t)blockIdx.x * kMarkSlice;
  if (nv <= a.k || s0 >= nv) return;
  if (threadIdx.x == 0) n_local = 0;
  const int32_t* hist = L.hdr + (int64_t)lq * kHdrWords;
  find_threshold_bin<kMarkThreads>(hist, a.k, scratch, res);
  const uint32_t bstar = (uint32_t)res[0];
  const float* scores = L.scores + (int64_t)lq * a.N_cap;
  uint32_t* bm = L.bitmap + (int64_t)lq * L.bm_stride;
  int32_t* counter = L.hdr + (int64_t)lq * kHdrWords + kHistBins;
  uint2* cand = L.cand + (int64_t)lq * kCandCap;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t s1 = (s0 + kMarkSlice < nv) ? s0 + kMarkSlice : nv;
  // each warp takes runs of kMarkUnroll * 32 consecutive entries; all loads of
  // a run are issued before any is used
  for (int64_t run = s0 + (int64_t)warp * kMarkUnroll * 32; run < s1;
       run += (int64_t)kMarkThreads * kMarkUnroll) {
    uint32_t key[kMarkUnroll];
#pragma unroll
    for (int u = 0; u < kMarkUnroll; ++u) {
      const int64_t i = run + u * 32 + lane;
      key[u] = i < s1 ? score_key(scores[i]) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kMarkUnroll; ++u) {
      const int64_t base = run + u * 32;
      if (base >= s1) break;
      const bool in = base + lane < s1;
      const uint32_t bin = key[u] >> 20;
      const unsigned above = __ballot_sync(0xFFFFFFFFu, in && bin > bstar);
      const unsigned at = __ballot_sync(0xFFFFFFFFu, in && bin == bstar);
      if (lane == 0) bm[base >> 5] = above;
      if (at) {
        int slot0 = 0;
        if (lane == 0) slot0 = atomicAdd(&n_local, __popc(at));
        slot0 = __shfl_sync(0xFFFFFFFFu, slot0, 0);
        if ((at >> lane) & 1u)
          lcand[slot0 + __popc(at & ((1u << lane) - 1u))] = make_uint2(key[u], (uint32_t)(base + lane));
      }
    }
  }
  __syncthreads();
  const int n = n_local;
  if (n == 0) return;
  if (threadIdx.x == 0) g_base = atomicAdd(counter, n);
  __syncthreads();
  const int gb = g_base;
  for (int i = threadIdx.x; i < n; i += kMarkThreads)
    if (gb + i < kCandCap) cand[gb + i] = lcand[i];
}

// ------------------------------------------------------------------ select
// One CTA per query.  Dynamic shared memory: bitmap[nw] | eqmap[nw] | hist[1024].
// The exact k-th key inside the threshold bin comes from two 10-bit radix
// passes over the bin's candidate list (or, if it overflowed, over all
// scores); ties at that key go to the lowest indices.
constexpr int kSelUnroll = 8;

template <bool FromCand>
__device__ __forceinline__ void radix_pass(const uint2* cand, const float* scores, int64_t n,
                                           uint32_t pmask, uint32_t prefix, int shift, int* h) {
  for (int64_t i0 = threadIdx.x; i0 < n; i0 += (int64_t)kSelThreads * kSelUnroll) {
    uint32_t key[kSelUnroll];
#pragma unroll
    for (int u = 0; u < kSelUnroll; ++u) {
      const int64_t i = i0 + (int64_t)u * kSelThreads;
      key[u] = i < n ? (FromCand ? __ldcg(&cand[i].x) : score_key(__ldcg(scores + i))) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kSelUnroll; ++u) {
      const int64_t i = i0 + (int64_t)u * kSelThreads;
      if (i < n && (key[u] & pmask) == prefix) atomicAdd(&h[(key[u] >> shift) & 1023], 1);
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(IndexerArgs a, int q0,
                                                                  WsLayout L) {
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ int scratch[32];
  __shared__ int res[3];
  __shared__ uint32_t sel_key;
  __shared__ int sel_need;
  const int qid = q0 + blockIdx.x, lq = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t nv = visible_entries(a, qid, nullptr, false);
  int32_t* out = a.topk_idx + (int64_t)qid * a.k;
  float* out_s = a.topk_score ? a.topk_score + (int64_t)qid * a.k : nullptr;
  const float* scores = L.scores + (int64_t)lq * a.N_cap;

  if (nv <= a.k) {  // every visible entry is selected
    for (int64_t r = tid; r < a.k; r += kSelThreads) {
      out[r] = r < nv ? (int32_t)r : -1;
      if (out_s) out_s[r] = r < nv ? scores[r] : -INFINITY;
    }
    return;
  }

  const int nw = (int)((nv + 31) / 32);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(sm);
  uint32_t* eqmap = bitmap + L.bm_stride;
  int* h = reinterpret_cast<int*>(eqmap + L.bm_stride);

  const int32_t* hist = L.hdr + (int64_t)lq * kHdrWords;
  find_threshold_bin<kSelThreads>(hist, a.k, scratch, res);
  const uint32_t bstar = (uint32_t)res[0];
  const int c_above = res[1], c_bin = res[2];
  const int n_cand_written = hist[kHistBins];
  const uint32_t* bm_g = L.bitmap + (int64_t)lq * L.bm_stride;
  for (int i = tid; i < nw; i += kSelThreads) {
    bitmap[i] = bm_g[i];
    eqmap[i] = 0u;
  }
  const bool fast = c_bin <= kCandCap && n_cand_written == c_bin;
  const uint2* cand = L.cand + (int64_t)lq * kCandCap;
  int need = a.k - c_above;  // to take from the threshold bin, >= 1

  // ---- exact key within the bin: two 10-bit radix passes (bits 19..10, 9..0)
  uint32_t prefix = bstar << 20;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const uint32_t pmask = pass == 0 ? 0xFFF00000u : 0xFFFFFC00u;
    for (int i = tid; i < 1024; i += kSelThreads) h[i] = 0;
    __syncthreads();
    if (fast)
      radix_pass<true>(cand, scores, c_bin, pmask, prefix, shift, h);
    else
      radix_pass<false>(cand, scores, nv, pmask, prefix, shift, h);
    __syncthreads();
    {
      constexpr int per = 1024 / kSelThreads;
      const int hi = 1024 - tid * per;
      int local = 0;
      for (int i = 1; i <= per; ++i) local += h[hi - i];
      int total;
      const int before = block_excl_scan<kSelThreads>(local, scratch, &total);
      if (before < need && before + local >= need) {
        int run = before;
        for (int i = 1; i <= per; ++i) {
          const int bin = hi - i, cnt = h[bin];
          if (run + cnt >= need) {
            res[0] = bin;
            res[1] = run;
            break;
          }
          run += cnt;
        }
      }
      __syncthreads();
      prefix |= (uint32_t)res[0] << shift;
      need -= res[1];
      __syncthreads();
    }
  }
  if (tid == 0) {
    sel_key = prefix;
    sel_need = need;  // how many entries with key == sel_key to take (lowest indices)
  }
  __syncthreads();
  const uint32_t kstar = sel_key;
  const int need_eq = sel_need;

  // ---- mark the threshold-bin entries: above kstar -> bitmap, equal -> eqmap
  if (fast) {
    for (int i = tid; i < c_bin; i += kSelThreads) {
      const uint2 ce = __ldcg(&cand[i]);
      if (ce.x > kstar) atomicOr(&bitmap[ce.y >> 5], 1u << (ce.y & 31));
      else if (ce.x == kstar) atomicOr(&eqmap[ce.y >> 5], 1u << (ce.y & 31));
    }
  } else {
    for (int64_t i0 = tid; i0 < nv; i0 += (int64_t)kSelThreads * kSelUnroll) {
      uint32_t key[kSelUnroll];
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u) {
        const int64_t i = i0 + (int64_t)u * kSelThreads;
        key[u] = i < nv ? score_key(__ldcg(scores + i)) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u) {
        const int64_t i = i0 + (int64_t)u * kSelThreads;
        if (i >= nv || (key[u] >> 20) != bstar) continue;
        if (key[u] > kstar) atomicOr(&bitmap[i >> 5], 1u << (i & 31));
        else if (key[u] == kstar) atomicOr(&eqmap[i >> 5], 1u << (i & 31));
      }
    }
  }
  __syncthreads();

  // ---- ordered emission: thread tid owns words [tid*R, tid*R + R)
  const int R = (nw + kSelThreads - 1) / kSelThreads;
  const int w0 = tid * R, w1 = (w0 + R < nw) ? w0 + R : nw;
  int eqc = 0;
  for (int w = w0; w < w1; ++w) eqc += __popc(eqmap[w]);
  int total;
  int eq_run = block_excl_scan<kSelThreads>(eqc, scratch, &total);
  int selc = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t e = eqmap[w];
    uint32_t take = 0;
    while (e && eq_run < need_eq) {
      const uint32_t low = e & (~e + 1u);
      take |= low;
      e ^= low;
      ++eq_run;
    }
    const uint32_t fin = bitmap[w] | take;
    bitmap[w] = fin;
    selc += __popc(fin);
  }
  int pos = block_excl_scan<kSelThreads>(selc, scratch, &total);
  for (int w = w0; w < w1; ++w) {
    uint32_t fin = bitmap[w];
    while (fin) {
      const int bit = __ffs(fin) - 1;
      fin &= fin - 1;
      const int64_t i = (int64_t)w * 32 + bit;
      if (pos < a.k) {
        out[pos] = (int32_t)i;
        if (out_s) out_s[pos] = scores[i];
      }
      ++pos;
    }
  }
  if (tid == 0 && total != a.k) flag_error(a.err, CSA_EW_BAD_INDEX);  // internal invariant
  for (int r = total + tid; r < a.k; r += kSelThreads) {
    out[r] = -1;
    if (out_s) out_s[r] = -INFINITY;
  }
}

int select_smem_bytes(int n_cap) { return 2 * bitmap_words(n_cap) * 4 + 1024 * 4; }

}  // namespace

size_t indexer_topk_workspace_bytes(int n_query, int N_cap) {
  const int qc = n_query < kQueryChunk ? n_query : kQueryChunk;
  return align256((size_t)qc * N_cap * sizeof(float)) +
         align256((size_t)qc * kHdrWords * sizeof(int32_t)) +
         align256((size_t)qc * bitmap_words(N_cap) * sizeof(uint32_t)) +
         align256((size_t)qc * kCandCap * sizeof(uint2));
}

cudaError_t launch_indexer_topk(const IndexerArgs& a, void* ws, cudaStream_t st) {
  const int qc_max = a.n_query < kQueryChunk ? a.n_query : kQueryChunk;
  WsLayout L = carve(ws, qc_max, a.N_cap);
  const int sel_smem = select_smem_bytes(a.N_cap);
  cudaError_t e = ensure_smem_attr((const void*)topk_select_kernel, select_smem_bytes(kMaxNcap));
  if (e != cudaSuccess) return e;
  e = ensure_smem_attr((const void*)topk_mark_kernel, kMarkSlice * sizeof(uint2));
  if (e != cudaSuccess) return e;
  for (int q0 = 0; q0 < a.n_query; q0 += kQueryChunk) {
    const int qc = (a.n_query - q0 < kQueryChunk) ? a.n_query - q0 : kQueryChunk;
    e = cudaMemsetAsync(L.hdr, 0, (size_t)qc * kHdrWords * sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    dim3 g1((a.N_cap + kChunk - 1) / kChunk, qc);
    if (a.fp8)
      indexer_score_kernel<true><<<g1, kScoreThreads, 0, st>>>(a, q0, L);
    else
      indexer_score_kernel<false><<<g1, kScoreThreads, 0, st>>>(a, q0, L);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g2((a.N_cap + kMarkSlice - 1) / kMarkSlice, qc);
    topk_mark_kernel<<<g2, kMarkThreads, kMarkSlice * sizeof(uint2), st>>>(a, q0, L);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    topk_select_kernel<<<qc, kSelThreads, sel_smem, st>>>(a, q0, L);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace csa
