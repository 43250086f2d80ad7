// attn.cu -- MQA attention over a gathered key set (compressed entries chosen
// by top-k, or all visible ones, plus the raw sliding window) with an
// attention-sink logit, on the fifth-generation tensor cores (tcgen05/TMEM);
// the keys of one query are split across a thread-block cluster and the
// partial results merged through distributed shared memory.
//
// Method: hyper.ai DeepSeek-V4 page, Method (MQA core attention over the
// top-k compressed entries; HCA dense over all entries; sliding-window
// branch); aiboss88 DeepSeek-V4 page, Technical Principles (window + attention
// sink); elamur.ai page, References [20] (flash-decoding: split the key range
// over many CTAs, merge the partial softmax results by log-sum-exp).
//
// One CTA owns one (query token, key split); the splits of a query form one
// cluster.  All H heads share each K/V row (MQA), so the H x 128 query block is
// the M side of the contractions (M = 64 for H <= 64, else 128) and every
// gathered 256-byte K/V row is read from memory once.  Key slots: compressed
// entries [0, n_c), padding to a multiple of 4, then the window.
//
// Keys move in 64-key stages and are contracted in 128-key tiles (two
// consecutive stages).  Shared memory holds four regions (K dims 0-63, K dims
// 64-127, V dims 0-63, V dims 64-127), each a ring of stages of 64 rows x 128
// bytes in the 128-byte swizzled layout, so that the rows of a stage pair are
// contiguous and one MMA descriptor spans 128 keys.
// Warp roles (384 threads):
//   warp 0       one thread issues S = Q K^T (8 MMAs of M x 128 x 16) into one
//                of two TMEM buffers; the warp owns the TMEM allocation
//   warp 1       one thread issues O += P V (8 MMAs of M x 128 x 16)
//   warps 2-3, 8-11  loaders: per stage, one row lookup per key, then one TMA
//                box per region when the 64 rows are contiguous, or 16-byte
//                cp.async row gathers (skipped slots zero-filled)
//   warps 4-7    softmax on the 16-lane TMEM layout: base-2 online softmax
//                with lazy rescaling (O in TMEM is rescaled only when a row's
//                running max grows by more than 2^8); P (bf16) to shared
//                memory.  The exponentials of tile t are computed while the
//                P V of tile t-1 still runs.
// FP8-stored entries (KV8 = true, csa_attn_fp8kv): the loaders copy each
// stage's E4M3 codes, scales and bf16 RoPE channels to a staging slot and,
// two stages later, decode them into the ring: K's rows as bf16 (code *
// scale, nearest even), V's rows as their exact f16 codes, unscaled.  The
// softmax adds log2 of each key's V scale to its logit, so P (f16 here)
// carries the scale into P V, and divides it out of the row sums; the raw
// window rows' V is converted to f16 in place (scale 1).
// Separate S and P V issuers keep the tensor pipe fed while either one waits
// on a barrier.  Every mbarrier wait is bounded; on timeout the CTA records
// CSA_EW_TIMEOUT in the error word, still reaches every barrier, and frees its
// TMEM.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tma.cuh"

namespace csa {

namespace {

constexpr int kD = 128;
constexpr int kStageKeys = 64;   // keys per stage (one row lookup per loader lane)
constexpr int kTileKeys = 128;   // keys per MMA tile (two stages)
constexpr int kBlk = 8192;       // bytes of one stage in one region (64 rows x 128 B)
constexpr int kThreads = 384;
constexpr int kLoadThreads = 192;  // warps 2-3 and 8-11
constexpr int kSoftWarp0 = 4;
constexpr int kSoftThreads = 128;
constexpr int kMaxCluster = 16;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr int kPrefetch = 4;  // stages of top-k entries looked up ahead by the loaders

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;    // S buffer b at column 128 * b
constexpr uint32_t kOCol = 256;  // O accumulator

// FP8-stored compressed entries (KV8): per entry 64 E4M3 codes of K's
// non-RoPE channels, 128 of V, one fp32 scale each; the staging slot of a
// stage holds them (and K's bf16 RoPE channels) for its 64 slots until they
// are decoded into the ring.  Only the decode writes a stage's compressed rows
// into the ring, so the copies of a stage need no free ring slot and run
// ahead of the tensor cores by kS8Lag stages.
constexpr int kS8R = 0;                  // RoPE channels, [64 rows][128 B], 128-byte swizzled
constexpr int kS8K = kS8R + 64 * 128;    // [64 rows][64 B]
constexpr int kS8V = kS8K + 64 * 64;     // [64 rows][128 B]
constexpr int kS8KS = kS8V + 64 * 128;   // fp32 [64]
constexpr int kS8VS = kS8KS + 64 * 4;    // fp32 [64]
constexpr int kS8Bytes = (kS8VS + 64 * 4 + 1023) / 1024 * 1024;  // slots stay 1024-aligned
constexpr int kS8Slots = 3;  // a stage's codes are decoded kS8Lag stages after their copies
constexpr int kS8Lag = 2;

template <int M, bool KV8 = false>
struct Cfg {
  static constexpr int kStages = KV8 ? 4 : M == 64 ? 6 : 4;  // 64-key stages, even
  static constexpr int kPairs = kStages / 2;
  static constexpr int kRegion = kStages * kBlk;
  static constexpr int kQBytes = M * 256;  // 2 K-blocks x [M x 128 B]
  static constexpr int kPBytes = M * 256;  // 2 K-blocks (keys 0-63, 64-127) x [M x 128 B]
  static constexpr int kQOff = 0;
  static constexpr int kK0 = kQBytes;
  static constexpr int kK1 = kK0 + kRegion;
  static constexpr int kV0 = kK1 + kRegion;
  static constexpr int kV1 = kV0 + kRegion;
  static constexpr int kPOff = kV1 + kRegion;
  static constexpr int kMetaOff = kPOff + kPBytes;  // stages x 64 row codes
  static constexpr int kS8Off = kMetaOff + kStages * kStageKeys * 4;
  // KV8: log2 of each key's V scale, per ring stage (the softmax folds the
  // scale into P; V enters the tensor cores as its exact f16 codes)
  static constexpr int kSvOff = kS8Off + (KV8 ? kS8Slots * kS8Bytes : 0);
  static constexpr int kBarOff = kSvOff + (KV8 ? kStages * kStageKeys * 4 : 0);
  static constexpr int kSmemBytes = kBarOff + 512 + 1024;  // + alignment slack
  // after the main loop: own partial O rows (fp32) over the K regions, rows
  // received from the cluster over the V regions (and P); lse values and
  // merge weights over Q
  static constexpr int kPartOff = kK0;
  static constexpr int kRecvOff = kV0;              // [ns][hp][128] fp32
  static constexpr int kPartLseOff = kQOff;         // [H]
  static constexpr int kRecvLseOff = kQOff + 1024;  // [ns][hp]
  static constexpr int kWgtOff = kQOff + 2048;      // [hp][ns]
  static constexpr int kSinkOff = kQOff + 3072;     // [H]
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(2 * kRegion >= M * 512, "partial O fits over the K regions");
  static_assert(2 * kRegion + kPBytes >= (M + kMaxCluster) * 512, "received rows fit");
  static_assert(kQBytes >= 3072 + 4 * 128, "merge scratch and sink logits fit over Q");
};

struct Bars {
  uint64_t kv_full[3];     // per stage pair: both stages landed (one arrival per loader thread
                           // per stage, plus the TMA bytes)
  uint64_t pair_empty[3];  // per stage pair: the P V that read it has completed
  uint64_t meta_full[4];   // per tile t % 4: its stages' validity bits published
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t p_free;
  uint64_t q_full;
  uint32_t tmem_slot;
  int timed_out;
  // per stage j % 8 and loader warp 0/1 (a stage's bits outlive its ring slot:
  // with KV8 the copies of stage j + 4 may start before tile j / 2 is done)
  uint32_t valid[8][2];
  uint32_t dense[8][2];  // its 32 rows continue its lane 0's row
  uint32_t cmp[8][2];    // its 32 rows are all compressed entries
  uint64_t s8_full[kS8Slots];  // KV8: a staging slot's bulk copies landed (one arrival a stage)
};

// Tensor maps: the query block, and boxes of 64 rows that load a whole stage
// of contiguous compressed entries.
struct Maps {
  CUtensorMap q, kc, vc;
  CUtensorMap kr;  // KV8: K's RoPE channels, rows of 64 bf16
};

// Slot -> row code: r >= 0 is row r of the 2-D row view of the compressed
// caches, -1 a skipped slot, -(r + 2) row r of the raw (window) caches.  Row
// counts below 2^31 - 2 are checked on the host.
struct KeySet {
  const int32_t* sel;  // nullptr: dense
  const int32_t* src;  // list read by fetch(): sel, or any valid int32 when there is none
  int n_c, n_c4;
  int n_cap;
  int64_t cmp_row0;  // b * cmp rows per sequence
  int64_t raw_row0;  // b * raw rows per sequence
  int64_t win_row0;  // ring row of the window's first position
  int64_t raw_cap;
  int k_end;

  // The top-k entry behind slot v (meaningless for slots that have none).
  // The value is only consumed by code(), stages later, so the load latency
  // overlaps the stages in between; the address always stays in the list.
  __device__ __forceinline__ int32_t fetch(int v) const {
    return __ldg(src + (sel ? (v < n_c ? v : n_c - 1) : 0));
  }
  __device__ __forceinline__ int32_t code(int v, int32_t s, int32_t* err) const {
    if (v >= k_end) return -1;
    if (v < n_c) {
      int64_t e = v;
      if (sel) {
        if (s < 0 || s >= n_cap) {
          if (s != -1) flag_error(err, CSA_EW_BAD_INDEX);
          return -1;
        }
        e = s;
      }
      return (int32_t)(cmp_row0 + e);
    }
    if (v < n_c4) return -1;  // padding
    int64_t r = win_row0 + (v - n_c4);
    if (r >= raw_cap) r -= raw_cap;
    return (int32_t)(-(raw_row0 + r) - 2);
  }
};

__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, Bars* bars,
                                             int32_t* err) {
  if (tc::mbar_wait(bar, parity, kWaitLimit)) return true;
  atomicExch(&bars->timed_out, 1);
  flag_error(err, CSA_EW_TIMEOUT);
  return false;
}

// AND of a predicate over the loader threads (named barrier 1).
__device__ __forceinline__ bool loaders_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, %2, q;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kLoadThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void loaders_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kLoadThreads) : "memory");
}

// Eight E4M3 codes (c.x low byte first) times the entry's scale, as eight
// bf16 (nearest even): one 16-byte row chunk of the decoded entry.
__device__ __forceinline__ uint4 dequant8(uint2 c, float sc) {
  uint32_t w[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const uint32_t hv = e4m3x2_to_f16x2((uint16_t)(((h < 2) ? c.x : c.y) >> (16 * (h & 1))));
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hv));
    w[h] = pack_bf16x2(f.x * sc, f.y * sc);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// Eight E4M3 codes (c.x low byte first) as eight f16, exact (no scale).
__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 c) {
  return make_uint4(e4m3x2_to_f16x2((uint16_t)c.x), e4m3x2_to_f16x2((uint16_t)(c.x >> 16)),
                    e4m3x2_to_f16x2((uint16_t)c.y), e4m3x2_to_f16x2((uint16_t)(c.y >> 16)));
}
// Eight bf16 as eight f16 (nearest even).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int h = 0; h < 4; ++h)
    o[h] = pack_f16x2(__uint_as_float(w[h] << 16), __uint_as_float(w[h] & 0xFFFF0000u));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int M>
struct RowMap {  // softmax-thread view of the 16-lane TMEM layout
  static constexpr int NG = M / 64;  // 16-lane groups per warp quadrant
  __device__ __forceinline__ static int row(int qd, int g, int r8) {
    return M == 64 ? qd * 16 + r8 : qd * 32 + g * 16 + r8;
  }
  __device__ __forceinline__ static uint32_t lane_field(int qd, int g) {
    return (uint32_t)((qd * 32 + g * 16) << 16);
  }
};

// Split merge of one query whose splits form a cluster and left their
// normalised partial rows and lse values in part_o / part_lse (global
// memory): one cluster barrier (release / acquire at cluster scope) makes
// every split's rows visible, then CTA `split` combines heads
// [split*hp, split*hp + hp) reading them from L2 (ld.global.cg), with the
// weights exp(lse_s - M) / Z of the cluster merge (the sink's term in Z
// only).  Each thread owns four channels of one head: it loads the head's
// lse values and its pieces of the first eight splits' rows together (one
// round trip to L2; a second for splits 8-15), and forms the weights itself.
// sink_s: H floats.
__device__ __forceinline__ void merge_from_global(const AttnArgs& a, int qid, int split, int ns,
                                                  float* sink_s, float sink_mine) {
  constexpr int kRows = 8;  // splits' rows in flight at a time
  const int tid = threadIdx.x, H = a.H;
  if (tid < H) sink_s[tid] = sink_mine;
  tc::cluster_sync();
  const int hp = (H + ns - 1) / ns;
  const int h0 = split * hp;
  const int nh = H - h0 < hp ? (H - h0 > 0 ? H - h0 : 0) : hp;
  const float* plse = a.part_lse + (int64_t)qid * ns * H;  // split s, head h at s * H + h
  const float4* rows = reinterpret_cast<const float4*>(a.part_o + (int64_t)qid * ns * H * kD);
  const int64_t sstride = (int64_t)H * kD / 4;  // float4s between splits
  for (int it = tid; it < nh * 32; it += kThreads) {
    const int hl = it >> 5, d4 = it & 31, h = h0 + hl;
    float ls[kMaxCluster];
    float4 v[kRows];
#pragma unroll
    for (int s = 0; s < kMaxCluster; ++s) ls[s] = s < ns ? __ldcg(plse + s * H + h) : -INFINITY;
#pragma unroll
    for (int s = 0; s < kRows; ++s)
      v[s] = s < ns ? __ldcg(rows + s * sstride + h * 32 + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
    float Mx = a.sink ? sink_s[h] : -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxCluster; ++s) Mx = fmaxf(Mx, ls[s]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse = -INFINITY;
    if (Mx != -INFINITY) {
      float w[kMaxCluster];
      float Z = a.sink ? ex2_approx((sink_s[h] - Mx) * kLog2e) : 0.f;
#pragma unroll
      for (int s = 0; s < kMaxCluster; ++s) {
        w[s] = ls[s] == -INFINITY ? 0.f : ex2_approx((ls[s] - Mx) * kLog2e);
        Z += w[s];
      }
      const float inv = 1.f / Z;
#pragma unroll
      for (int s = 0; s < kRows; ++s) {
        const float ws = w[s] * inv;
        acc.x += ws * v[s].x;
        acc.y += ws * v[s].y;
        acc.z += ws * v[s].z;
        acc.w += ws * v[s].w;
      }
      if (ns > kRows) {
#pragma unroll
        for (int s = 0; s < kMaxCluster - kRows; ++s)
          v[s] = kRows + s < ns ? __ldcg(rows + (kRows + s) * sstride + h * 32 + d4)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < kMaxCluster - kRows; ++s) {
          const float ws = w[kRows + s] * inv;
          acc.x += ws * v[s].x;
          acc.y += ws * v[s].y;
          acc.z += ws * v[s].z;
          acc.w += ws * v[s].w;
        }
      }
      lse = Mx + logf(Z);
    }
    if (d4 == 0 && a.lse) a.lse[(int64_t)qid * H + h] = lse;
    reinterpret_cast<uint2*>(a.out + ((int64_t)qid * H + h) * kD)[d4] =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

template <int M, bool KV8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(AttnArgs a, const __grid_constant__ Maps maps) {
  using C = Cfg<M, KV8>;
  constexpr int kStages = C::kStages;
  constexpr int kPairs = C::kPairs;
  constexpr int NL = kLoadThreads;
  // Everything up to griddepcontrol.wait below reads only what no kernel of
  // this library writes (the queries, positions, entry counts, sink logits)
  // and sets up shared and tensor memory, so it overlaps the end of the
  // previous kernel (the top-k select) under programmatic dependent launch.
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  const uint32_t sbase = smem_u32(sm);
  Bars* bars = reinterpret_cast<Bars*>(sm + C::kBarOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ns = a.n_split;
  const int qid = blockIdx.x / ns, split = blockIdx.x % ns;
  const int b = qid / a.T;
  const int H = a.H;
  const bool is_loader = warp == 2 || warp == 3 || warp >= 8;
  const int lt = warp <= 3 ? tid - 64 : tid - 192;  // loader index (loader warps only)

  // ---- the query's key set and this split's range
  const int64_t t = a.pos_is_len ? (int64_t)__ldg(a.pos + b) - 1 : (int64_t)__ldg(a.pos + qid);
  bool bad_pos = t < 0;  // flagged after the wait (the error word may be the previous kernel's)
  int n_c;
  if (!a.dense) {
    n_c = a.sel_count;
  } else {
    int64_t present = a.n_cmp ? (int64_t)__ldg(a.n_cmp + b) : 0;
    if (present < 0 || present > a.N_cap) {
      bad_pos = true;
      present = present < 0 ? 0 : a.N_cap;
    }
    const int64_t nv = t >= 0 ? (t + 1) / a.m_prime : 0;
    n_c = (int)(nv < present ? nv : present);
  }
  int64_t win_lo = t - a.window + 1;
  if (win_lo < 0) win_lo = 0;
  const int n_w = (a.window > 0 && t >= 0) ? (int)(t - win_lo + 1) : 0;
  const int n_c4 = n_w > 0 ? (n_c + 3) & ~3 : n_c;
  const int n_keys = n_c4 + n_w;
  const int k_begin = split * a.keys_per_split;
  int k_end = k_begin + a.keys_per_split;
  if (k_end > n_keys) k_end = n_keys;
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + kTileKeys - 1) / kTileKeys : 0;
  const int n_stages = 2 * n_tiles;

  // Leading stages whose 64 slots are all compressed entries of a dense key
  // set (HCA) are four TMA boxes each, issued by one thread without per-slot
  // lookups: the thread publishes the stage's slot bits and arrives for the
  // whole loader group.  The first kStages of them (no ring slot to wait
  // for) are issued during the set-up, once the barriers exist.
  int j_fast = 0;
  if (!KV8 && a.dense) {
    const int full = (n_c < k_end ? n_c : k_end) - k_begin;
    j_fast = full > 0 ? full / kStageKeys : 0;
    if (j_fast > n_stages) j_fast = n_stages;
  }
  const int j_pre = j_fast < kStages ? j_fast : kStages;
  auto issue_dense_stage = [&](int j) {
    const int st = j % kStages, pr = (j >> 1) % kPairs;
    bars->valid[j & 7][0] = 0xFFFFFFFFu;
    bars->valid[j & 7][1] = 0xFFFFFFFFu;
    if (j & 1) tc::mbar_arrive(&bars->meta_full[(j >> 1) & 3]);  // both stages' bits
    const int row = (int)((int64_t)b * (a.cmp_bstride / kD) + k_begin + (int64_t)j * kStageKeys);
    const uint32_t off = st * kBlk;
    tma::expect_tx(&bars->kv_full[pr], 4 * kBlk);
    tma::load_box(sbase + C::kK0 + off, &maps.kc, 0, row, &bars->kv_full[pr]);
    tma::load_box(sbase + C::kK1 + off, &maps.kc, 64, row, &bars->kv_full[pr]);
    tma::load_box(sbase + C::kV0 + off, &maps.vc, 0, row, &bars->kv_full[pr]);
    tma::load_box(sbase + C::kV1 + off, &maps.vc, 64, row, &bars->kv_full[pr]);
    tc::mbar_arrive_count(&bars->kv_full[pr], kLoadThreads - 1);
  };

  // ---- set-up: barriers, TMEM, the query block, zero Q rows >= H
  if (warp == 0) {
    tc::tmem_alloc(&bars->tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 32) {
    for (int p = 0; p < kPairs; ++p) {
      tc::mbar_init(&bars->kv_full[p], 2 * kLoadThreads);
      tc::mbar_init(&bars->pair_empty[p], 1);
    }
    // KV8: every code thread arrives once per stage, after its key's V scale
    for (int i = 0; i < 4; ++i) tc::mbar_init(&bars->meta_full[i], KV8 ? 2 * kStageKeys : 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bars->s_full[i], 1);
      tc::mbar_init(&bars->s_free[i], kSoftThreads / 32);  // one arrival per softmax warp
    }
    tc::mbar_init(&bars->p_full, kSoftThreads / 32);
    tc::mbar_init(&bars->p_free, 1);
    tc::mbar_init(&bars->q_full, 1);
    if (KV8)
      for (int i = 0; i < kS8Slots; ++i) tc::mbar_init(&bars->s8_full[i], 1);
    bars->timed_out = 0;
    tc::fence_mbar_init();
    if (n_tiles > 0) {  // H rows of 256 bytes as two K-blocks
      tma::expect_tx(&bars->q_full, 2 * H * 128);
      tma::load_box(sbase + C::kQOff, &maps.q, 0, qid * H, &bars->q_full);
      tma::load_box(sbase + C::kQOff + M * 128, &maps.q, 64, qid * H, &bars->q_full);
    }
    if (j_pre > 0) {
      pdl_wait();  // the entries may be the previous kernel's output
      for (int j = 0; j < j_pre; ++j) issue_dense_stage(j);
    }
  }
  for (int idx = tid; idx < (M - H) * 16; idx += kThreads) {
    const int r = H + (idx >> 4), c16 = idx & 15;
    *reinterpret_cast<uint4*>(sm + C::kQOff + (c16 >> 3) * (M * 128) +
                              tc::sw128_offset(r, c16 & 7)) = make_uint4(0, 0, 0, 0);
  }
  // sink logits: one per thread for the split merge (tid < H), and the
  // softmax threads' own rows for a single split's epilogue
  // (loaded here, first used after the main loop: the loads do not hold up
  // the set-up)
  float sink_mine = -INFINITY;
  if (a.sink && tid < H) sink_mine = __ldg(a.sink + tid);
  float sink_rows[2][2] = {{-INFINITY, -INFINITY}, {-INFINITY, -INFINITY}};
  if (a.sink && warp >= kSoftWarp0 && warp < kSoftWarp0 + 4) {
#pragma unroll
    for (int g = 0; g < RowMap<M>::NG; ++g)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int h = RowMap<M>::row(warp & 3, g, lane >> 2) + 8 * h2;
        if (h < H) sink_rows[g][h2] = __ldg(a.sink + h);
      }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;
  pdl_wait();  // the previous kernel's results (top-k lists, new entries) are visible now
  if (bad_pos && tid == 0 && split == 0) flag_error(a.err, CSA_EW_BAD_POSITION);

  if (n_tiles > 0 && warp == 0) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_bf16(M, kTileKeys, false, false);
      bool ok = wait_or_flag(&bars->q_full, 0, bars, a.err);
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int pr = j % kPairs, sb = j & 1;
        ok = wait_or_flag(&bars->kv_full[pr], (j / kPairs) & 1, bars, a.err);
        if (ok && j >= 2) ok = wait_or_flag(&bars->s_free[sb], ((j - 2) >> 1) & 1, bars, a.err);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t k0 = sbase + C::kK0 + pr * 2 * kBlk;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t ad =
              tc::desc_sw128(sbase + C::kQOff + (kk >> 2) * (M * 128) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd =
              tc::desc_sw128(k0 + (kk >> 2) * C::kRegion + (kk & 3) * 32, 16, 1024);
          tc::mma_ss(tmem + kSCol + sb * kTileKeys, ad, bd, id_s, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bars->s_full[sb]);
      }
    }
    __syncwarp();
  } else if (n_tiles > 0 && warp == 1) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      const uint32_t id_o = KV8 ? tc::idesc_f16(M, kD, false, true) : tc::idesc_bf16(M, kD, false, true);
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int pr = j % kPairs;
        ok = wait_or_flag(&bars->p_full, j & 1, bars, a.err);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t v0 = sbase + C::kV0 + pr * 2 * kBlk;
#pragma unroll
        for (int s = 0; s < kTileKeys / 16; ++s) {
          const uint64_t ad =
              tc::desc_sw128(sbase + C::kPOff + (s >> 2) * (M * 128) + (s & 3) * 32, 16, 1024);
          const uint64_t bd = tc::desc_sw128(v0 + s * 2048, C::kRegion, 1024);
          tc::mma_ss(tmem + kOCol, ad, bd, id_o, (j > 0 || s > 0) ? 1u : 0u);
        }
        tc::mma_commit(&bars->p_free);
        tc::mma_commit(&bars->pair_empty[pr]);
      }
      // drain: the last commit covers every MMA this thread issued
      if (ok)
        wait_or_flag(&bars->pair_empty[(n_tiles - 1) % kPairs], ((n_tiles - 1) / kPairs) & 1,
                     bars, a.err);
    }
    __syncwarp();
  } else if (n_tiles > 0 && is_loader) {
    // ------------------------------------------------------------ loaders
    KeySet ks;
    ks.sel = (a.dense || n_c == 0) ? nullptr : a.sel + (int64_t)qid * a.sel_stride;
    ks.src = ks.sel ? ks.sel : a.pos;
    ks.n_c = n_c;
    ks.n_c4 = n_c4;
    ks.n_cap = a.N_cap;
    ks.cmp_row0 = (int64_t)b * (a.cmp_bstride / kD);
    ks.raw_row0 = (int64_t)b * (a.raw_bstride / kD);
    ks.raw_cap = a.raw_cap > 0 ? a.raw_cap : 1;
    ks.win_row0 = win_lo % ks.raw_cap;
    ks.k_end = k_end;
    const bf16* kc = a.k_cmp;
    const bf16* vc = a.v_cmp;
    const bf16* kr = a.k_raw;
    const bf16* vr = a.v_raw;
    int32_t* codes = reinterpret_cast<int32_t*>(sm + C::kMetaOff);
    // The dense key set's remaining whole-entry stages (the set-up issued the
    // first j_pre): one thread waits for each ring slot and issues them; the
    // group joins at the first stage that needs per-slot lookups (the window).
    int issued = lt == 0 ? j_pre : 0;
    bool fast_ok = true;
    if (j_fast > 0 && lt == 0) {
      for (int j = j_pre; j < j_fast; ++j) {
        const int pr = (j >> 1) % kPairs;
        if (j >= kStages && (j & 1) == 0)
          fast_ok = wait_or_flag(&bars->pair_empty[pr], ((j >> 1) / kPairs - 1) & 1, bars, a.err);
        fast_ok = fast_ok && !*(volatile int*)&bars->timed_out;
        if (!fast_ok) break;
        issue_dense_stage(j);
        issued = j + 1;
      }
    }
    // top-k entries of this thread's slot (lt < 64) for the next kPrefetch
    // stages: pf[i] belongs to stage j + i
    int32_t pf[kPrefetch];
#pragma unroll
    for (int i = 0; i < kPrefetch; ++i)
      pf[i] = lt < kStageKeys ? ks.fetch(k_begin + (j_fast + i) * kStageKeys + lt) : 0;
    // Every loader thread gives one arrival per stage on its pair's kv_full:
    // for a gathered stage once its own copies have landed (cp.async
    // mbarrier tracking, the loader does not block), for a TMA stage at issue
    // (thread 0's arrival carries the transaction count).
    // KV8: a stage's compressed rows go as E4M3 codes and scales to a staging
    // slot (bulk copies when its 64 rows are contiguous, else 16-byte
    // cp.async gathers), RoPE channels (bf16) and raw window rows straight to
    // the ring; kS8Lag stages later every loader decodes its share of the
    // codes into the ring's bf16 rows (code * scale) and gives the stage's
    // kv_full arrival.
    auto kv8_issue = [&](int j, bool dense, bool all_cmp) {
      const int st = j % kStages;
      const uint32_t stg = sbase + C::kS8Off + (j % kS8Slots) * kS8Bytes;
      const uint32_t off = st * kBlk;
      uint64_t* full = &bars->s8_full[j % kS8Slots];
      if (!all_cmp && j >= kStages) {
        // raw window rows and skipped slots go straight to the ring slot
        if (lt == 0)
          wait_or_flag(&bars->pair_empty[(j >> 1) % kPairs], ((j >> 1) / kPairs - 1) & 1, bars,
                       a.err);
        loaders_sync();
      }
      if (dense) {
        // 64 contiguous entries: their codes as two bulk copies, their RoPE
        // channels as one TMA box (thread 0); the scales below
        if (lt == 0) {
          const int32_t row0 = codes[st * kStageKeys];
          tma::expect_tx(full, kStageKeys * (64 + 128 + 128));
          tma::bulk_load(stg + kS8K, a.k8 + (int64_t)row0 * 64, kStageKeys * 64, full);
          tma::bulk_load(stg + kS8V, a.v8 + (int64_t)row0 * 128, kStageKeys * 128, full);
          tma::load_box(stg + kS8R, &maps.kr, 0, row0, full);
        }
      } else if (lt == 0) {
        tc::mbar_arrive(full);
      }
      constexpr int kIss = (kStageKeys * 16 + NL - 1) / NL;
      int32_t cds[kIss];
#pragma unroll
      for (int i = 0; i < kIss; ++i) {
        const int ci = lt + i * NL;
        cds[i] = ci < kStageKeys * 16 ? codes[st * kStageKeys + (ci >> 4)] : -1;
      }
#pragma unroll
      for (int i = 0; i < kIss; ++i) {
        const int ci = lt + i * NL;
        if (dense || ci >= kStageKeys * 16) break;
        const int r = ci >> 4, c16 = ci & 15;
        const int32_t cd = cds[i];
        const uint32_t so = off + ((c16 >> 3) ? C::kRegion : 0) + tc::sw128_offset(r, c16 & 7);
        if (cd >= 0) {
          if (c16 < 4)
            cp_async16(stg + kS8K + r * 64 + c16 * 16, a.k8 + (int64_t)cd * 64 + c16 * 16, 16);
          if (c16 < 8)
            cp_async16(stg + kS8V + r * 128 + c16 * 16, a.v8 + (int64_t)cd * 128 + c16 * 16, 16);
          else
            cp_async16(stg + kS8R + tc::sw128_offset(r, c16 & 7),
                       a.k_rope + (int64_t)cd * 64 + (c16 - 8) * 8, 16);
        } else {
          const bool ok = cd != -1;
          const int64_t goff = (int64_t)(-(cd + 2)) * kD + c16 * 8;
          cp_async16(sbase + C::kK0 + so, ok ? (const void*)(kr + goff) : (const void*)a.q,
                     ok ? 16 : 0);
          cp_async16(sbase + C::kV0 + so, ok ? (const void*)(vr + goff) : (const void*)a.q,
                     ok ? 16 : 0);
        }
      }
      if (lt < kStageKeys) {
        const int32_t cd = codes[st * kStageKeys + lt];
        if (cd >= 0) {
          cp_async4(stg + kS8KS + lt * 4, a.k8_scale + cd, 4);
          cp_async4(stg + kS8VS + lt * 4, a.v8_scale + cd, 4);
        }
      }
      cp_async_commit();
    };
    auto kv8_decode = [&](int s8) {
      if (lt == 0 && s8 >= kStages)  // the ring slot's previous tile is done
        wait_or_flag(&bars->pair_empty[(s8 >> 1) % kPairs], ((s8 >> 1) / kPairs - 1) & 1, bars,
                     a.err);
      loaders_sync();  // every loader's copies of stage s8 have landed
      wait_or_flag(&bars->s8_full[s8 % kS8Slots], (s8 / kS8Slots) & 1, bars, a.err);  // and bulk
      const int st = s8 % kStages, pr = (s8 >> 1) % kPairs;
      const uint8_t* stg = sm + C::kS8Off + (s8 % kS8Slots) * kS8Bytes;
      const float* ksc = reinterpret_cast<const float*>(stg + kS8KS);
      const float* vsc = reinterpret_cast<const float*>(stg + kS8VS);
      const uint32_t off = st * kBlk;
      // Output chunks of 8 channels: 8 per row of K's non-RoPE channels
      // (code * scale -> bf16) and of its RoPE channels (copied), 16 per row
      // of V (code -> f16, or a raw row's bf16 -> f16 in place).  Each thread
      // first loads every row code, scale and source chunk of its outputs,
      // then converts and stores them (no shared-memory load between two
      // stores); the K and V chunks are separate loops, so that a warp's
      // lanes take the same path.
      constexpr int kPerK = (kStageKeys * 8 + NL - 1) / NL;
      constexpr int kPerV = (kStageKeys * 16 + NL - 1) / NL;
      int32_t cdk[kPerK], cdv[kPerV];
      uint2 ck[kPerK], cv[kPerV];
      float scv[kPerK];
      uint4 rope[kPerK];
#pragma unroll
      for (int i = 0; i < kPerK; ++i) {
        const int oc = lt + i * NL;
        const int r = (oc >> 3) & (kStageKeys - 1), part = oc & 7;
        cdk[i] = oc < kStageKeys * 8 ? codes[st * kStageKeys + r] : -1;
        ck[i] = *reinterpret_cast<const uint2*>(stg + kS8K + r * 64 + part * 8);
        scv[i] = ksc[r];
        rope[i] = *reinterpret_cast<const uint4*>(stg + kS8R + tc::sw128_offset(r, part));
      }
#pragma unroll
      for (int i = 0; i < kPerV; ++i) {
        const int oc = lt + i * NL;
        const int r = (oc >> 4) & (kStageKeys - 1), v = oc & 15;
        cdv[i] = oc < kStageKeys * 16 ? codes[st * kStageKeys + r] : -1;
        cv[i] = *reinterpret_cast<const uint2*>(stg + kS8V + r * 128 + v * 8);
      }
#pragma unroll
      for (int i = 0; i < kPerK; ++i) {
        const int oc = lt + i * NL;
        if (cdk[i] >= 0) {
          const uint32_t o = off + tc::sw128_offset(oc >> 3, oc & 7);
          *reinterpret_cast<uint4*>(sm + C::kK0 + o) = dequant8(ck[i], scv[i]);
          *reinterpret_cast<uint4*>(sm + C::kK1 + o) = rope[i];  // same swizzled offsets
        }
      }
#pragma unroll
      for (int i = 0; i < kPerV; ++i) {
        const int oc = lt + i * NL;
        const int r = oc >> 4, v = oc & 15;
        if (cdv[i] == -1) continue;  // skipped slot or past the stage
        uint4* d = reinterpret_cast<uint4*>(sm + C::kV0 + off + (v >> 3) * C::kRegion +
                                            tc::sw128_offset(r, v & 7));
        if (cdv[i] >= 0) *d = e4m3x8_to_f16x8(cv[i]);
        else *d = bf16x8_to_f16x8(*d);
      }
      // log2 of the key's V scale (0 for raw rows, skipped slots and zero scales)
      if (lt < kStageKeys) {
        const float sv = codes[st * kStageKeys + lt] >= 0 ? vsc[lt] : 1.f;
        reinterpret_cast<float*>(sm + C::kSvOff)[st * kStageKeys + lt] =
            sv > 0.f ? __log2f(sv) : 0.f;
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&bars->kv_full[pr]);
      // the stage's validity bits and V scales are published for the softmax
      if (lt < kStageKeys) tc::mbar_arrive(&bars->meta_full[(s8 >> 1) & 3]);
    };
    for (int j = j_fast; j < n_stages; ++j) {
      const int st = j % kStages, pr = (j >> 1) % kPairs;
      bool go = fast_ok;
      if (!KV8 && lt == 0 && j >= kStages && (j & 1) == 0)
        go = wait_or_flag(&bars->pair_empty[pr], ((j >> 1) / kPairs - 1) & 1, bars, a.err);
      go = go && !*(volatile int*)&bars->timed_out;
      // every loader thread takes the same branch: named barrier 1 below
      if (!loaders_all(go)) break;
      if (lt < kStageKeys) {
        const int32_t cd = ks.code(k_begin + j * kStageKeys + lt, pf[0], a.err);
        codes[st * kStageKeys + lt] = cd;
        // contiguous compressed rows within this warp's 32 slots
        const int32_t w0 = __shfl_sync(0xFFFFFFFFu, cd, 0);
        const unsigned vb = __ballot_sync(0xFFFFFFFFu, cd != -1);
        const unsigned cb = __ballot_sync(0xFFFFFFFFu, w0 >= 0 && cd == w0 + (lt & 31));
        const unsigned ab = __ballot_sync(0xFFFFFFFFu, cd >= 0);
        if ((lt & 31) == 0) {
          bars->valid[j & 7][lt >> 5] = vb;
          bars->dense[j & 7][lt >> 5] = cb;
          bars->cmp[j & 7][lt >> 5] = ab;
        }
      }
#pragma unroll
      for (int i = 0; i + 1 < kPrefetch; ++i) pf[i] = pf[i + 1];
      if (lt < kStageKeys)
        pf[kPrefetch - 1] = ks.fetch(k_begin + (j + kPrefetch) * kStageKeys + lt);
      loaders_sync();
      const int32_t base = codes[st * kStageKeys];
      const bool dense_rows = (bars->dense[j & 7][0] & bars->dense[j & 7][1]) == 0xFFFFFFFFu &&
                              codes[st * kStageKeys + 32] == base + 32;
      const bool all_cmp = (bars->cmp[j & 7][0] & bars->cmp[j & 7][1]) == 0xFFFFFFFFu;
      const bool dense = !KV8 && dense_rows;
      if (!KV8 && lt == 0 && (j & 1)) tc::mbar_arrive(&bars->meta_full[(j >> 1) & 3]);  // both stages
      const uint32_t off = st * kBlk;
      if constexpr (KV8) {
        kv8_issue(j, dense_rows, all_cmp);
        if (j >= kS8Lag) {
          cp_async_wait<kS8Lag>();
          kv8_decode(j - kS8Lag);
        }
      } else if (dense) {
        if (lt == 0) {
          tma::expect_tx(&bars->kv_full[pr], 4 * kBlk);
          tma::load_box(sbase + C::kK0 + off, &maps.kc, 0, (int)base, &bars->kv_full[pr]);
          tma::load_box(sbase + C::kK1 + off, &maps.kc, 64, (int)base, &bars->kv_full[pr]);
          tma::load_box(sbase + C::kV0 + off, &maps.vc, 0, (int)base, &bars->kv_full[pr]);
          tma::load_box(sbase + C::kV1 + off, &maps.vc, 64, (int)base, &bars->kv_full[pr]);
        } else {
          tc::mbar_arrive(&bars->kv_full[pr]);
        }
      } else {
        // the row codes of all of this thread's chunks first, then the copies
        // back to back (no shared-memory load between two copies)
        constexpr int kIt = (kStageKeys * 16 + NL - 1) / NL;
        int32_t cds[kIt];
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
          const int ci = lt + i * NL;
          cds[i] = ci < kStageKeys * 16 ? codes[st * kStageKeys + (ci >> 4)] : -1;
        }
#pragma unroll
        for (int i = 0; i < kIt; ++i) {
          const int ci = lt + i * NL;
          if (ci >= kStageKeys * 16) break;
          const int r = ci >> 4, c16 = ci & 15;
          const int32_t cd = cds[i];
          const bool ok = cd != -1;
          const bool raw = cd < -1;
          const int64_t goff = (int64_t)(raw ? -(cd + 2) : cd) * kD + c16 * 8;
          const bf16* kp = ok ? (raw ? kr : kc) + goff : a.q;
          const bf16* vp = ok ? (raw ? vr : vc) + goff : a.q;
          const uint32_t so = off + ((c16 >> 3) ? C::kRegion : 0) + tc::sw128_offset(r, c16 & 7);
          cp_async16(sbase + C::kK0 + so, kp, ok ? 16 : 0);
          cp_async16(sbase + C::kV0 + so, vp, ok ? 16 : 0);
        }
        tc::cp_async_mbar_arrive(&bars->kv_full[pr]);
      }
      issued = j + 1;
    }
    if constexpr (KV8) {
      // the last stages' codes (only when every stage was issued)
      if (issued == n_stages)
        for (int s8 = n_stages > kS8Lag ? n_stages - kS8Lag : 0; s8 < n_stages; ++s8) {
          if (n_stages - 1 - s8 >= 1)
            cp_async_wait<1>();
          else
            cp_async_wait<0>();
          kv8_decode(s8);
        }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    if (KV8 && lt == 0) {
      // bulk copies still in flight after a timeout land before the CTA exits
      tc::mbar_wait(&bars->q_full, 0, kWaitLimit);
      for (int i = issued > kS8Slots ? issued - kS8Slots : 0; i < issued; ++i)
        tc::mbar_wait(&bars->s8_full[i % kS8Slots], (i / kS8Slots) & 1, kWaitLimit);
    } else if (lt == 0) {
      // bulk copies still in flight after a timeout land before the CTA exits
      tc::mbar_wait(&bars->q_full, 0, kWaitLimit);
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; i += 2)
        tc::mbar_wait(&bars->kv_full[(i >> 1) % kPairs], ((i >> 1) / kPairs) & 1, kWaitLimit);
    }
  } else if (warp >= kSoftWarp0 && warp < kSoftWarp0 + 4) {
    // ------------------------------------------------------------ softmax
    using RM = RowMap<M>;
    constexpr int NG = RM::NG;
    const int qd = warp & 3;
    const int r8 = lane >> 2, c4 = lane & 3;
    float m_ref[NG][2], l_sum[NG][2];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      m_ref[g][0] = m_ref[g][1] = -INFINITY;
      l_sum[g][0] = l_sum[g][1] = 0.f;
    }
    uint8_t* pbuf = sm + C::kPOff;
    // KV8: log2 V scale of key 32q + 8u + 2c4 of tile j (stage 2j + q/2)
    const float* svp = reinterpret_cast<const float*>(sm + C::kSvOff);
    auto sv_col = [&](int j, int q, int u) {
      return ((2 * j + (q >> 1)) % kStages) * kStageKeys + 32 * (q & 1) + 8 * u + 2 * c4;
    };
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      // waits are made warp-uniform: tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xFFFFFFFFu, wait_or_flag(&bars->meta_full[j & 3], (j >> 2) & 1, bars, a.err)))
        break;
      const int st0 = (2 * j) & 7;
      const uint32_t vm[4] = {bars->valid[st0][0], bars->valid[st0][1], bars->valid[st0 + 1][0],
                              bars->valid[st0 + 1][1]};
      if (!__all_sync(0xFFFFFFFFu, wait_or_flag(&bars->s_full[sb], (j >> 1) & 1, bars, a.err)))
        break;
      tc::fence_after_sync();
      bool stop = false;
#pragma unroll 1
      for (int g = 0; g < NG; ++g) {
        // sr[q*16 + u*4 + k]: k = 0,1 -> row A cols 32q + 8u + 2c4 (+1);
        //                     k = 2,3 -> row B, same columns
        uint32_t sr[64];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          tc::tmem_ld16x256_x4(tmem + RM::lane_field(qd, g) + kSCol + sb * kTileKeys + q * 32,
                               &sr[q * 16]);
        tc::tmem_ld_wait();
        if (g == NG - 1) {
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bars->s_free[sb]);
        }
        float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            // KV8: log2 of the V scales of keys 32q + 8u + 2c4 (+1), added to
            // their logits so that P carries them (V is the raw codes)
            float2 lv = make_float2(0.f, 0.f);
            if constexpr (KV8) lv = *reinterpret_cast<const float2*>(svp + sv_col(j, q, u));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int bit = 8 * u + 2 * c4 + (k & 1);
              const int i = q * 16 + u * 4 + k;
              const float x = ((vm[q] >> bit) & 1u)
                                  ? __uint_as_float(sr[i]) * a.scale_log2 + ((k & 1) ? lv.y : lv.x)
                                  : -INFINITY;
              sr[i] = __float_as_uint(x);
              mt[k >> 1] = fmaxf(mt[k >> 1], x);
            }
          }
        // lazy rescaling: a row's reference max moves only when the tile max
        // exceeds it by more than 2^8 (or on its first finite tile)
        float f[2];
        bool grow_any = false;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          mt[h2] = fmaxf(mt[h2], __shfl_xor_sync(0xFFFFFFFFu, mt[h2], 1));
          mt[h2] = fmaxf(mt[h2], __shfl_xor_sync(0xFFFFFFFFu, mt[h2], 2));
          const bool move = mt[h2] > m_ref[g][h2] + 8.f;
          const bool grow = move && m_ref[g][h2] != -INFINITY;
          f[h2] = grow ? ex2_approx(m_ref[g][h2] - mt[h2]) : 1.f;
          grow_any |= grow;
          if (move) m_ref[g][h2] = mt[h2];
          l_sum[g][h2] *= f[h2];
        }
        // exponentials (relative to the new reference) while P V of tile j-1 runs
        const float mA = m_ref[g][0] == -INFINITY ? 0.f : m_ref[g][0];
        const float mB = m_ref[g][1] == -INFINITY ? 0.f : m_ref[g][1];
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2_approx(__uint_as_float(sr[4 * i]) - mA);
          const float p1 = ex2_approx(__uint_as_float(sr[4 * i + 1]) - mA);
          const float p2 = ex2_approx(__uint_as_float(sr[4 * i + 2]) - mB);
          const float p3 = ex2_approx(__uint_as_float(sr[4 * i + 3]) - mB);
          if constexpr (KV8) {
            // the row sums exclude the V scales: weights p / scale
            const float2 lv = *reinterpret_cast<const float2*>(svp + sv_col(j, i >> 2, i & 3));
            const float i0 = ex2_approx(-lv.x), i1 = ex2_approx(-lv.y);
            l_sum[g][0] += p0 * i0 + p1 * i1;
            l_sum[g][1] += p2 * i0 + p3 * i1;
            pk[2 * i] = pack_f16x2(p0, p1);
            pk[2 * i + 1] = pack_f16x2(p2, p3);
          } else {
            l_sum[g][0] += p0 + p1;
            l_sum[g][1] += p2 + p3;
            pk[2 * i] = pack_bf16x2(p0, p1);
            pk[2 * i + 1] = pack_bf16x2(p2, p3);
          }
        }
        // the P buffer and O are free once P V of tile j-1 has completed
        if (g == 0 && j >= 1) {
          if (!__all_sync(0xFFFFFFFFu, wait_or_flag(&bars->p_free, (j - 1) & 1, bars, a.err))) {
            stop = true;
            break;
          }
          tc::fence_after_sync();
        }
        if (__any_sync(0xFFFFFFFFu, grow_any)) {
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t o[16];
            const uint32_t ta = tmem + RM::lane_field(qd, g) + kOCol + q * 32;
            tc::tmem_ld16x256_x4(ta, o);
            tc::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * f[(i & 3) >> 1]);
            tc::tmem_st16x256_x4(ta, o);
          }
          tc::tmem_st_wait();
        }
        const int rowA = RM::row(qd, g, r8), rowB = rowA + 8;
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            // key 32q + 8u + 2c4: K-block q/2, 16-byte chunk 4(q%2) + u, byte 4c4
            uint8_t* blk = pbuf + (q >> 1) * (M * 128) + 4 * c4;
            *reinterpret_cast<uint32_t*>(blk + tc::sw128_offset(rowA, 4 * (q & 1) + u)) =
                pk[2 * (q * 4 + u)];
            *reinterpret_cast<uint32_t*>(blk + tc::sw128_offset(rowB, 4 * (q & 1) + u)) =
                pk[2 * (q * 4 + u) + 1];
          }
      }
      if (stop) break;
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bars->p_full);
    }
    // ---- epilogue: O rows after the last P V, normalised
    bool have_o = n_tiles > 0 && !*(volatile int*)&bars->timed_out;
    if (__any_sync(0xFFFFFFFFu, have_o))
      have_o = wait_or_flag(&bars->p_free, (n_tiles - 1) & 1, bars, a.err);
    have_o = __all_sync(0xFFFFFFFFu, have_o);
    tc::fence_after_sync();
#pragma unroll
    for (int g = 0; g < NG; ++g) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        l_sum[g][h2] += __shfl_xor_sync(0xFFFFFFFFu, l_sum[g][h2], 1);
        l_sum[g][h2] += __shfl_xor_sync(0xFFFFFFFFu, l_sum[g][h2], 2);
      }
      const int rowA = RM::row(qd, g, r8);
      float fac[2], lse_r[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const bool any = have_o && l_sum[g][h2] > 0.f;
        if (ns > 1) {
          fac[h2] = any ? 1.f / l_sum[g][h2] : 0.f;
          lse_r[h2] = any ? (m_ref[g][h2] + log2f(l_sum[g][h2])) * kLn2 : -INFINITY;
        } else {
          const float sk = sink_rows[g][h2] * kLog2e;
          float Mx = any ? m_ref[g][h2] : -INFINITY;
          if (a.sink) Mx = fmaxf(Mx, sk);
          fac[h2] = 0.f;
          lse_r[h2] = -INFINITY;
          if (Mx != -INFINITY) {
            const float w = any ? exp2f(m_ref[g][h2] - Mx) : 0.f;
            const float Z = l_sum[g][h2] * w + (a.sink ? exp2f(sk - Mx) : 0.f);
            fac[h2] = w / Z;
            lse_r[h2] = (Mx + log2f(Z)) * kLn2;
          }
        }
      }
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t o[16];
        if (have_o) {
          tc::tmem_ld16x256_x4(tmem + RM::lane_field(qd, g) + kOCol + q * 32, o);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int col = 32 * q + 8 * u + 2 * c4;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int h = rowA + 8 * h2;
            if (h >= H) continue;
            const float v0 = __uint_as_float(o[u * 4 + 2 * h2]) * fac[h2];
            const float v1 = __uint_as_float(o[u * 4 + 2 * h2 + 1]) * fac[h2];
            if (ns > 1 && a.part_o)
              *reinterpret_cast<float2*>(a.part_o + (((int64_t)qid * ns + split) * H + h) * kD +
                                         col) = make_float2(v0, v1);
            else if (ns > 1)
              *reinterpret_cast<float2*>(sm + C::kPartOff + h * 512 + col * 4) =
                  make_float2(v0, v1);
            else
              *reinterpret_cast<uint32_t*>(a.out + ((int64_t)qid * H + h) * kD + col) =
                  pack_bf16x2(v0, v1);
          }
        }
      }
      if (c4 == 0) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int h = rowA + 8 * h2;
          if (h >= H) continue;
          if (ns > 1 && a.part_lse)
            a.part_lse[((int64_t)qid * ns + split) * H + h] = lse_r[h2];
          else if (ns > 1)
            reinterpret_cast<float*>(sm + C::kPartLseOff)[h] = lse_r[h2];
          else if (a.lse)
            a.lse[(int64_t)qid * H + h] = lse_r[h2];
        }
      }
    }
  }

  // ---- teardown: every role is done with TMEM
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (ns <= 1 || (a.part_o && !a.xch)) return;  // one split, or merged by attn_merge_kernel
  if (a.xch) {
    merge_from_global(a, qid, split, ns, reinterpret_cast<float*>(sm + C::kSinkOff), sink_mine);
    return;
  }

  // ---- split merge inside the cluster.  CTA `split` combines heads
  // [split*hp, split*hp + hp).  After the first cluster barrier no CTA uses
  // its stages again, so every CTA pushes its partial rows and lse values for
  // those heads into the owner's shared memory (remote stores, no round
  // trips); after the second barrier each CTA combines its heads locally.
  if (tid < H) reinterpret_cast<float*>(sm + C::kSinkOff)[tid] = sink_mine;
  tc::cluster_sync();
  const int hp = (H + ns - 1) / ns;
  {
    const float* part = reinterpret_cast<const float*>(sm + C::kPartOff);
    const float* part_lse = reinterpret_cast<const float*>(sm + C::kPartLseOff);
    for (int it = tid; it < H * 32; it += kThreads) {
      const int h = it >> 5, d4 = it & 31;
      const int owner = h / hp, slot = split * hp + (h - owner * hp);
      const float4 v = *reinterpret_cast<const float4*>(part + h * kD + d4 * 4);
      tc::st_cluster_f32x4(tc::map_shared(sbase + C::kRecvOff + slot * 512 + d4 * 16, owner), v);
    }
    for (int h = tid; h < H; h += kThreads) {
      const int owner = h / hp, slot = split * hp + (h - owner * hp);
      tc::st_cluster_f32(tc::map_shared(sbase + C::kRecvLseOff + slot * 4, owner), part_lse[h]);
    }
  }
  tc::cluster_sync();
  const int h0 = split * hp;
  const int nh = H - h0 < hp ? (H - h0 > 0 ? H - h0 : 0) : hp;
  const float* rlse = reinterpret_cast<const float*>(sm + C::kRecvLseOff);  // [ns][hp]
  const float* rrow = reinterpret_cast<const float*>(sm + C::kRecvOff);     // [ns][hp][128]
  float* wgt = reinterpret_cast<float*>(sm + C::kWgtOff);                  // [nh][ns]
  const float* sink_s = reinterpret_cast<const float*>(sm + C::kSinkOff);
  for (int hl = tid; hl < nh; hl += kThreads) {
    const int h = h0 + hl;
    float Mx = sink_s[h];
    for (int s = 0; s < ns; ++s) Mx = fmaxf(Mx, rlse[s * hp + hl]);
    float lse = -INFINITY;
    if (Mx != -INFINITY) {
      float Z = a.sink ? expf(sink_s[h] - Mx) : 0.f;
      for (int s = 0; s < ns; ++s) {
        const float ls = rlse[s * hp + hl];
        const float w = ls == -INFINITY ? 0.f : expf(ls - Mx);
        wgt[hl * ns + s] = w;
        Z += w;
      }
      const float inv = 1.f / Z;
      for (int s = 0; s < ns; ++s) wgt[hl * ns + s] *= inv;
      lse = Mx + logf(Z);
    } else {
      for (int s = 0; s < ns; ++s) wgt[hl * ns + s] = 0.f;
    }
    if (a.lse) a.lse[(int64_t)qid * H + h] = lse;
  }
  __syncthreads();
  for (int it = tid; it < nh * 32; it += kThreads) {
    const int hl = it >> 5, d4 = it & 31, h = h0 + hl;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ns; ++s) {
      const float w = wgt[hl * ns + s];
      const float4 v = *reinterpret_cast<const float4*>(rrow + (s * hp + hl) * kD + d4 * 4);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    reinterpret_cast<uint2*>(a.out + ((int64_t)qid * H + h) * kD)[d4] =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

// Split merge through global memory (a6), for splits run without a cluster:
// grid (queries, ceil(H / 4)), warp w of CTA (q, y) merges head 4y + w.  The
// same combination as the cluster merge: weights exp(lse_s - M) / Z over the
// splits, the sink's exp(sink - M) in Z only.  The lanes read the splits'
// lse values in parallel, and the partial rows are loaded eight splits at a
// time, so that the loads overlap.
__global__ void __launch_bounds__(128) attn_merge_kernel(AttnArgs a) {
  pdl_trigger();
  const int qid = blockIdx.x, lane = threadIdx.x & 31;
  const int h = blockIdx.y * 4 + (threadIdx.x >> 5);
  const int ns = a.n_split, H = a.H;
  if (h >= H) return;
  const float sink_h = a.sink ? __ldg(a.sink + h) : -INFINITY;  // an input: before the wait
  pdl_wait();
  const float* lse_p = a.part_lse + (int64_t)qid * ns * H + h;  // split s at s * H
  const float4* row = reinterpret_cast<const float4*>(a.part_o + ((int64_t)qid * ns * H + h) * kD);
  const int64_t rstride = (int64_t)H * kD / 4;  // float4s between splits
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse = -INFINITY;
  if (ns <= 32) {
    // lane j holds split j's lse; the first kRows splits' rows are loaded at
    // the same time (one round trip for both), the rest kRows at a time
    constexpr int kRows = 16;
    const float ls = lane < ns ? lse_p[(int64_t)lane * H] : -INFINITY;
    float4 v[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j)
      v[j] = j < ns ? row[j * rstride + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    float Mx = fmaxf(sink_h, ls);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xFFFFFFFFu, Mx, o));
    if (Mx != -INFINITY) {
      const float wl = ls == -INFINITY ? 0.f : expf(ls - Mx);
      float zl = wl;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) zl += __shfl_xor_sync(0xFFFFFFFFu, zl, o);
      const float Z = zl + (a.sink ? expf(sink_h - Mx) : 0.f);
      const float inv = 1.f / Z;
      for (int s0 = 0; s0 < ns; s0 += kRows) {
        if (s0 > 0) {
#pragma unroll
          for (int j = 0; j < kRows; ++j)
            v[j] = s0 + j < ns ? row[(s0 + j) * rstride + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const float w = __shfl_sync(0xFFFFFFFFu, wl, (s0 + j) & 31) * inv;
          if (s0 + j < ns) {
            acc.x += w * v[j].x;
            acc.y += w * v[j].y;
            acc.z += w * v[j].z;
            acc.w += w * v[j].w;
          }
        }
      }
      lse = Mx + logf(Z);
    }
    reinterpret_cast<uint2*>(a.out + ((int64_t)qid * H + h) * kD)[lane] =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    if (lane == 0 && a.lse) a.lse[(int64_t)qid * H + h] = lse;
    return;
  }
  // the splits' lse values, all lanes at once (lane j holds splits j, j + 32, ..)
  float Mx = sink_h;
  for (int s = lane; s < ns; s += 32) Mx = fmaxf(Mx, lse_p[(int64_t)s * H]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xFFFFFFFFu, Mx, o));
  if (Mx != -INFINITY) {
    float zl = 0.f;  // this lane's share of Z
    for (int s = lane; s < ns; s += 32) {
      const float ls = lse_p[(int64_t)s * H];
      zl += ls == -INFINITY ? 0.f : expf(ls - Mx);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zl += __shfl_xor_sync(0xFFFFFFFFu, zl, o);
    const float Z = zl + (a.sink ? expf(sink_h - Mx) : 0.f);
    const float inv = 1.f / Z;
    // the partial rows, eight splits' loads in flight at a time
    constexpr int kBatch = 8;
    for (int s0 = 0; s0 < ns; s0 += kBatch) {
      float4 v[kBatch];
      float w[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int s = s0 + j;
        const float ls = s < ns ? lse_p[(int64_t)s * H] : -INFINITY;
        w[j] = ls == -INFINITY ? 0.f : expf(ls - Mx) * inv;
        v[j] = s < ns ? row[s * rstride + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        acc.x += w[j] * v[j].x;
        acc.y += w[j] * v[j].y;
        acc.z += w[j] * v[j].z;
        acc.w += w[j] * v[j].w;
      }
    }
    lse = Mx + logf(Z);
  }
  reinterpret_cast<uint2*>(a.out + ((int64_t)qid * H + h) * kD)[lane] =
      make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  if (lane == 0 && a.lse) a.lse[(int64_t)qid * H + h] = lse;
}

// attr: room for two attributes (cluster shape; programmatic launch if pdl)
template <int M, bool KV8>
cudaLaunchConfig_t launch_cfg(int n_split, int n_query, cudaStream_t st,
                              cudaLaunchAttribute* attr, bool pdl, bool cluster = true) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)n_split * (unsigned)n_query);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<M, KV8>::kSmemBytes;
  cfg.stream = st;
  unsigned n = 0;
  if (n_split > 1 && cluster) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)n_split;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) set_pdl(attr[n++]);
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cfg;
}

// Clusters of size n the device keeps resident at once (cached per device).
template <int M, bool KV8>
int active_clusters(int n) {
  static std::mutex mu;  // callers may be on several host threads
  static int cache[16][kMaxCluster + 1];
  static bool init = false;
  if (n <= 1) return 1 << 20;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 16) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (auto& row : cache)
      for (int& v : row) v = -1;
    init = true;
  }
  int& c = cache[dev][n];
  if (c < 0) {
    ensure_smem_attr((const void*)attn_tc_kernel<M, KV8>, Cfg<M, KV8>::kSmemBytes, true);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_cfg<M, KV8>(n, 1, nullptr, attr, false);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, attn_tc_kernel<M, KV8>, &cfg) != cudaSuccess)
      clusters = 0;
    cudaGetLastError();
    c = clusters;
  }
  return c;
}

template <int M, bool KV8>
cudaError_t launch_tc(AttnArgs a, const Maps& maps, void* ws, cudaStream_t st) {
  cudaError_t e =
      ensure_smem_attr((const void*)attn_tc_kernel<M, KV8>, Cfg<M, KV8>::kSmemBytes, true);
  if (e != cudaSuccess) return e;
  // Pick the split count: at most one cluster of splits per query, every
  // cluster resident at once (one wave), about one CTA per SM in total.
  int ns = 1, kps = 0;
  if (a.fixed_kps > 0) {
    // batch-invariant: the split depends on the key count only, so a query's
    // partials and their merge order do not depend on the other queries
    kps = (a.fixed_kps + kStageKeys - 1) / kStageKeys * kStageKeys;
    ns = (a.n_keys_max + 3 + kps - 1) / kps;
    if (ns > kMaxCluster) return cudaErrorInvalidValue;  // checked on the host first
    ws = nullptr;
  } else {
    for (int cap = kMaxCluster; cap >= 1; --cap) {
      attn_plan(a.n_query, a.n_keys_max, cap, &ns, &kps);
      if (ns <= 1 || (long)active_clusters<M, KV8>(ns) >= (long)a.n_query) break;
    }
  }
  // Where clusters that large cannot all be resident and a workspace is
  // given, run more splits without a cluster and merge them in a second
  // kernel (partials through L2) instead.
  bool free_splits = false;
  if (ws && a.n_query * ns < (kNumSMs * 4) / 5) {
    int ns_f = 1, kps_f = 0;
    attn_plan(a.n_query, a.n_keys_max, kNumSMs, &ns_f, &kps_f);
    if (ns_f * 5 > ns * 6) {
      ns = ns_f;
      kps = kps_f;
      free_splits = true;
    }
  }
  a.n_split = ns;
  a.keys_per_split = kps;
  a.xch = 0;
  if (ns > 1 && ws) {
    // partial rows through the workspace: merged by a second kernel (free
    // splits) or by the cluster itself after one barrier
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_lse = a.part_o + (int64_t)a.n_query * ns * a.H * kD;
    a.xch = free_splits ? 0 : 1;
  }
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_cfg<M, KV8>(ns, a.n_query, st, attr, true, !free_splits);
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<M, KV8>, a, maps);
  if (e != cudaSuccess || !free_splits) return e;
  return launch_pdl(attn_merge_kernel, dim3((unsigned)a.n_query, (unsigned)((a.H + 3) / 4)),
                    dim3(128), 0, st, a);
}

}  // namespace

// Split plan: the splits of a query run as one cluster of at most
// max_cluster CTAs; about one CTA per SM in total.  Splits hold a multiple of
// 64 key slots (one stage); the key count includes up to 3 padding slots
// after the compressed entries.
void attn_plan(int n_query, int n_keys_max, int max_cluster, int* n_split, int* keys_per_split) {
  n_keys_max += 3;
  int ns = kNumSMs / (n_query > 0 ? n_query : 1);
  const int max_tiles = (n_keys_max + kTileKeys - 1) / kTileKeys;
  if (ns > max_tiles) ns = max_tiles;
  if (ns > max_cluster) ns = max_cluster;
  if (ns < 1) ns = 1;
  int kps = (n_keys_max + ns - 1) / ns;
  kps = (kps + kStageKeys - 1) / kStageKeys * kStageKeys;
  ns = (n_keys_max + kps - 1) / kps;
  if (ns < 1) ns = 1;
  *n_split = ns;
  *keys_per_split = kps;
}

// Workspace for splits without a cluster (partial rows and lse values of
// every split of every query); 0 when a query would get a single split.
size_t attn_workspace_bytes(int n_query, int H, int n_keys_max) {
  int ns = 1, kps = 0;
  attn_plan(n_query, n_keys_max, kNumSMs, &ns, &kps);
  if (ns <= 1) return 0;
  const size_t bytes = (size_t)n_query * ns * H * (kD + 1) * sizeof(float);
  return (bytes + 255) & ~size_t(255);
}

cudaError_t launch_attention(AttnArgs a, void* ws, cudaStream_t st) {
  // 2-D row views (rows of 128 elements) of the query block and the compressed caches
  Maps maps;
  const void* dummy = a.q;
  cudaError_t e = tma::encode_rows128(&maps.q, a.q, (uint64_t)a.n_query * a.H, (uint32_t)a.H);
  if (e != cudaSuccess) return e;
  const bool has_c = a.k_cmp && a.N_cap > 0 && !a.kv8;
  const uint64_t crow = has_c ? (uint64_t)(a.n_batch - 1) * (a.cmp_bstride / kD) + a.N_cap : 1;
  e = tma::encode_rows128(&maps.kc, has_c ? a.k_cmp : dummy, crow, kStageKeys);
  if (e == cudaSuccess) e = tma::encode_rows128(&maps.vc, has_c ? a.v_cmp : dummy, crow, kStageKeys);
  if (e != cudaSuccess) return e;
  if (a.kv8) {
    if (a.H > 64) return cudaErrorInvalidValue;  // checked on the host first
    const uint64_t rrow = a.N_cap > 0 ? (uint64_t)a.n_batch * a.N_cap : 1;
    e = tma::encode_rows(&maps.kr, a.N_cap > 0 ? (const void*)a.k_rope : dummy, 64, rrow,
                         kStageKeys);
    if (e != cudaSuccess) return e;
    return launch_tc<64, true>(a, maps, ws, st);
  }
  if (a.H <= 64) return launch_tc<64, false>(a, maps, ws, st);
  return launch_tc<128, false>(a, maps, ws, st);
}

}  // namespace csa
