// attn.cu -- MQA attention over a gathered key set (compressed entries chosen
// by top-k or all visible ones, plus the raw sliding window), with an
// attention-sink logit; split over keys, merged by log-sum-exp.
//
// Method: hyper.ai DeepSeek-V4 page, Method (MQA core attention over the
// top-k compressed entries; HCA dense over all entries; sliding-window
// branch); aiboss88 DeepSeek-V4 page, Technical Principles (window + attention
// sink); elamur.ai page, References [20] (flash-decoding: split the key range
// over many CTAs, merge the partial softmax results by their log-sum-exp).
//
// Design (B300): all H heads of one query token share every K/V row (MQA), so
// the H x D query block is the M side of a tensor-core contraction and each
// gathered 256-byte K/V row is read from HBM once per (query, split).  A CTA
// owns one (query, key split); warp w owns heads 16w..16w+15.  K/V rows are
// gathered by 16-byte cp.async into an XOR-swizzled, double-buffered shared
// tile of 64 keys; S = Q K^T and O += P V use m16n8k16 bf16 MMAs with fp32
// accumulators; the online softmax runs in the base-2 domain.
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kTileKeys = 64;
constexpr int kD = 128;
constexpr int kRowBytes = kD * 2;                   // 256
constexpr int kTileBytes = kTileKeys * kRowBytes;   // 16 KB
constexpr int kStageBytes = 2 * kTileBytes;         // K + V

// Virtual key slot v of a query -> (pointer to K row, pointer to V row), or
// invalid.  Slots [0, n_c) are compressed entries, [n_c, n_c + n_w) the raw
// window rows win_lo .. t.
struct KeySource {
  const bf16* kc;
  const bf16* vc;
  const bf16* kr;
  const bf16* vr;
  const int32_t* sel;  // nullptr: dense (slot v -> entry v)
  int n_c;
  int n_cap;
  int64_t win_lo;
  int32_t* err;

  __device__ __forceinline__ bool row(int v, int64_t& off, bool& raw) const {
    if (v < n_c) {
      int64_t e = v;
      if (sel) {
        int32_t s = __ldg(sel + v);
        if (s < 0) {
          if (s != -1) flag_error(err, CSA_EW_BAD_INDEX);
          return false;
        }
        if (s >= n_cap) {
          flag_error(err, CSA_EW_BAD_INDEX);
          return false;
        }
        e = s;
      }
      off = e * kD;
      raw = false;
      return true;
    }
    off = (win_lo + (v - n_c)) * kD;
    raw = true;
    return true;
  }
};

template <int NW>
__global__ void __launch_bounds__(NW * 32) attn_partial_kernel(AttnArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int qid = blockIdx.y;
  const int split = blockIdx.x;
  const int b = qid / a.T;

  // ---- the query's key set
  const int64_t t = a.pos_is_len ? (int64_t)__ldg(a.pos + b) - 1 : (int64_t)__ldg(a.pos + qid);
  // the window part needs the position inside the raw cache; visibility of
  // compressed entries only needs t >= 0
  const bool win_ok = a.window > 0 && t >= 0 && t < a.raw_cap;
  if (tid == 0 && (t < 0 || (a.window > 0 && t >= a.raw_cap)))
    flag_error(a.err, CSA_EW_BAD_POSITION);
  int n_c;
  if (!a.dense) {
    n_c = a.sel_count;
  } else {
    int64_t present = a.n_cmp ? (int64_t)__ldg(a.n_cmp + b) : 0;
    if (present < 0 || present > a.N_cap) {
      if (tid == 0) flag_error(a.err, CSA_EW_BAD_POSITION);
      present = present < 0 ? 0 : a.N_cap;
    }
    const int64_t nv = t >= 0 ? (t + 1) / a.m_prime : 0;
    n_c = (int)(nv < present ? nv : present);
  }
  int64_t win_lo = t - a.window + 1;
  if (win_lo < 0) win_lo = 0;
  const int n_w = win_ok ? (int)(t - win_lo + 1) : 0;
  const int n_keys = n_c + n_w;
  const int k_begin = split * a.keys_per_split;
  int k_end = k_begin + a.keys_per_split;
  if (k_end > n_keys) k_end = n_keys;
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + kTileKeys - 1) / kTileKeys : 0;

  KeySource src;
  src.kc = a.k_cmp + (int64_t)b * a.cmp_bstride;
  src.vc = a.v_cmp + (int64_t)b * a.cmp_bstride;
  src.kr = a.k_raw + (int64_t)b * a.raw_bstride;
  src.vr = a.v_raw + (int64_t)b * a.raw_bstride;
  src.sel = a.dense ? nullptr : a.sel + (int64_t)qid * a.sel_stride;
  src.n_c = n_c;
  src.n_cap = a.N_cap;
  src.win_lo = win_lo;
  src.err = a.err;

  uint32_t* valid_mask = reinterpret_cast<uint32_t*>(smem + 2 * kStageBytes);  // [2][2]
  const uint32_t smem_base = smem_u32(smem);

  // Loader: chunk ci = tid + i*NT covers row ci/16, 16-byte column ci%16;
  // 16 consecutive threads copy one 256-byte row.
  auto load_tile = [&](int stage, int tile) {
    const int v0 = k_begin + tile * kTileKeys;
    const uint32_t kbase = smem_base + stage * kStageBytes;
    const uint32_t vbase = kbase + kTileBytes;
#pragma unroll
    for (int i = 0; i < (kTileKeys * 16) / NT; ++i) {
      const int ci = tid + i * NT;
      const int r = ci >> 4, col = ci & 15;
      const int v = v0 + r;
      int64_t off = 0;
      bool raw = false;
      bool ok = v < k_end && src.row(v, off, raw);
      // zero-fill copies read nothing; their source is any valid address
      const bf16* kp = ok ? (raw ? src.kr : src.kc) + off + col * 8 : a.q;
      const bf16* vp = ok ? (raw ? src.vr : src.vc) + off + col * 8 : a.q;
      const uint32_t so = r * kRowBytes + ((col ^ (r & 7)) << 4);
      cp_async16(kbase + so, kp, ok ? 16 : 0);
      cp_async16(vbase + so, vp, ok ? 16 : 0);
    }
    // validity words for rows 0..31 and 32..63 (warp w handles word w, w+NW, ..)
    for (int wd = warp; wd < 2; wd += NW) {
      const int v = v0 + wd * 32 + lane;
      int64_t off;
      bool raw;
      const bool ok = v < k_end && src.row(v, off, raw);
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
      if (lane == 0) valid_mask[stage * 2 + wd] = bal;
    }
  };

  // ---- Q fragments for this warp's 16 heads (rows g and g+8), 8 k-steps
  uint32_t qa[8][4];
  {
    const int h0 = warp * 16 + g;
    const uint32_t* q0 = reinterpret_cast<const uint32_t*>(a.q + ((int64_t)qid * a.H + h0) * kD);
    const uint32_t* q1 = q0 + 8 * kD / 2;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      qa[kk][0] = __ldg(q0 + kk * 8 + c);
      qa[kk][1] = __ldg(q1 + kk * 8 + c);
      qa[kk][2] = __ldg(q0 + kk * 8 + 4 + c);
      qa[kk][3] = __ldg(q1 + kk * 8 + 4 + c);
    }
  }

  float acc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running max (log2 domain), rows g, g+8
  float l0 = 0.f, l1 = 0.f;              // per-thread partial sums

  if (n_tiles > 0) {
    load_tile(0, 0);
    cp_async_commit();
  }
  for (int tile = 0; tile < n_tiles; ++tile) {
    const int stage = tile & 1;
    if (tile + 1 < n_tiles) {
      load_tile(stage ^ 1, tile + 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const uint32_t kbase = smem_base + stage * kStageBytes;
    const uint32_t vbase = kbase + kTileBytes;
    const uint32_t vm0 = valid_mask[stage * 2], vm1 = valid_mask[stage * 2 + 1];

    // ---- S = Q K^T for 16 heads x 64 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        const int key = jp * 16 + ri + ((mi >> 1) << 3);
        const int chunk = kk * 2 + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kbase + key * kRowBytes + ((chunk ^ (key & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * jp], qa[kk], b0, b1);
        mma_bf16_16816(s[2 * jp + 1], qa[kk], b2, b3);
      }
    }

    // ---- mask, online softmax (base 2)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int slot = j * 8 + 2 * c + e;
        const bool ok = ((slot < 32 ? vm0 >> slot : vm1 >> (slot - 32)) & 1u) != 0;
        s[j][e] = ok ? s[j][e] * a.scale_log2 : -INFINITY;
        s[j][2 + e] = ok ? s[j][2 + e] * a.scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[j][e]);
        mx1 = fmaxf(mx1, s[j][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float use0 = mn0 == -INFINITY ? 0.f : mn0;
    const float use1 = mn1 == -INFINITY ? 0.f : mn1;
    const float corr0 = exp2f(m0 - use0), corr1 = exp2f(m1 - use1);
    m0 = mn0;
    m1 = mn1;
    l0 *= corr0;
    l1 *= corr1;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      acc[j][0] *= corr0;
      acc[j][1] *= corr0;
      acc[j][2] *= corr1;
      acc[j][3] *= corr1;
    }
    uint32_t pa[4][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p0 = exp2f(s[j][0] - use0), p1 = exp2f(s[j][1] - use0);
      const float p2 = exp2f(s[j][2] - use1), p3 = exp2f(s[j][3] - use1);
      l0 += p0 + p1;
      l1 += p2 + p3;
      pa[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
      pa[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }

    // ---- O += P V  (P: 16 heads x 64 keys, V: 64 keys x 128 dims)
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const int key = kk2 * 16 + ri + ((mi & 1) << 3);
        const int chunk = np * 2 + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + key * kRowBytes + ((chunk ^ (key & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(acc[2 * np], pa[kk2], b0, b1);
        mma_bf16_16816(acc[2 * np + 1], pa[kk2], b2, b3);
      }
    }
    __syncthreads();  // the stage is overwritten by the load two tiles ahead
  }

  // ---- finish: row sums across the 4 threads of a row group
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);

  const int h_lo = warp * 16 + g, h_hi = h_lo + 8;
  if (a.n_split > 1) {
    // partial result of this split: normalised o and its lse (natural log)
    const int64_t base = ((int64_t)qid * a.n_split + split) * a.H;
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    float* o0 = a.part_o + (base + h_lo) * kD;
    float* o1 = a.part_o + (base + h_hi) * kD;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      *reinterpret_cast<float2*>(o0 + j * 8 + 2 * c) = make_float2(acc[j][0] * inv0, acc[j][1] * inv0);
      *reinterpret_cast<float2*>(o1 + j * 8 + 2 * c) = make_float2(acc[j][2] * inv1, acc[j][3] * inv1);
    }
    if (c == 0) {
      a.part_lse[base + h_lo] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
      a.part_lse[base + h_hi] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
    }
    return;
  }
  // single split: fold in the sink and write the final output
  float M0 = m0, M1 = m1;
  float sk0 = -INFINITY, sk1 = -INFINITY;
  if (a.sink) {
    sk0 = __ldg(a.sink + h_lo) * kLog2e;
    sk1 = __ldg(a.sink + h_hi) * kLog2e;
    M0 = fmaxf(M0, sk0);
    M1 = fmaxf(M1, sk1);
  }
  float f0 = 0.f, f1 = 0.f, lse0 = -INFINITY, lse1 = -INFINITY;
  if (M0 != -INFINITY) {
    const float w = l0 > 0.f ? exp2f(m0 - M0) : 0.f;
    const float Z = l0 * w + (a.sink ? exp2f(sk0 - M0) : 0.f);
    f0 = w / Z;
    lse0 = (M0 + log2f(Z)) * kLn2;
  }
  if (M1 != -INFINITY) {
    const float w = l1 > 0.f ? exp2f(m1 - M1) : 0.f;
    const float Z = l1 * w + (a.sink ? exp2f(sk1 - M1) : 0.f);
    f1 = w / Z;
    lse1 = (M1 + log2f(Z)) * kLn2;
  }
  uint32_t* out0 = reinterpret_cast<uint32_t*>(a.out + ((int64_t)qid * a.H + h_lo) * kD);
  uint32_t* out1 = reinterpret_cast<uint32_t*>(a.out + ((int64_t)qid * a.H + h_hi) * kD);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    out0[j * 4 + c] = pack_bf16x2(acc[j][0] * f0, acc[j][1] * f0);
    out1[j * 4 + c] = pack_bf16x2(acc[j][2] * f1, acc[j][3] * f1);
  }
  if (a.lse && c == 0) {
    a.lse[(int64_t)qid * a.H + h_lo] = lse0;
    a.lse[(int64_t)qid * a.H + h_hi] = lse1;
  }
}

// One warp per (query, head): merge the n_split partials with the sink.
__global__ void __launch_bounds__(256) attn_merge_kernel(AttnArgs a) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int total = a.n_query * a.H;
  if (warp_global >= total) return;
  const int qid = warp_global / a.H, h = warp_global % a.H;
  const int64_t base = (int64_t)qid * a.n_split * a.H + h;
  float M = a.sink ? __ldg(a.sink + h) : -INFINITY;
  for (int s = 0; s < a.n_split; ++s) M = fmaxf(M, a.part_lse[base + (int64_t)s * a.H]);
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse = -INFINITY;
  if (M != -INFINITY) {
    float Z = a.sink ? expf(__ldg(a.sink + h) - M) : 0.f;
    for (int s = 0; s < a.n_split; ++s) {
      const float ls = a.part_lse[base + (int64_t)s * a.H];
      if (ls == -INFINITY) continue;
      const float w = expf(ls - M);
      Z += w;
      const float4 v =
          reinterpret_cast<const float4*>(a.part_o + (base + (int64_t)s * a.H) * kD)[lane];
      o.x += w * v.x;
      o.y += w * v.y;
      o.z += w * v.z;
      o.w += w * v.w;
    }
    const float inv = 1.f / Z;
    o.x *= inv;
    o.y *= inv;
    o.z *= inv;
    o.w *= inv;
    lse = M + logf(Z);
  }
  uint2 packed = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
  reinterpret_cast<uint2*>(a.out + ((int64_t)qid * a.H + h) * kD)[lane] = packed;
  if (a.lse && lane == 0) a.lse[(int64_t)qid * a.H + h] = lse;
}

template <int NW>
cudaError_t launch_partial(const AttnArgs& a, cudaStream_t st) {
  const int smem = 2 * kStageBytes + 16;
  cudaError_t e = ensure_smem_attr((const void*)attn_partial_kernel<NW>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_split, a.n_query);
  attn_partial_kernel<NW><<<grid, NW * 32, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

void attn_plan(int n_query, int n_keys_max, int* n_split, int* keys_per_split) {
  int max_split = (n_keys_max + kTileKeys - 1) / kTileKeys;
  if (max_split < 1) max_split = 1;
  const int target = 2 * kNumSMs;
  int ns = (target + n_query - 1) / n_query;
  if (ns > max_split) ns = max_split;
  if (ns < 1) ns = 1;
  int kps = (n_keys_max + ns - 1) / ns;
  kps = ((kps + kTileKeys - 1) / kTileKeys) * kTileKeys;
  if (kps < kTileKeys) kps = kTileKeys;
  ns = (n_keys_max + kps - 1) / kps;
  if (ns < 1) ns = 1;
  *n_split = ns;
  *keys_per_split = kps;
}

size_t attn_workspace_bytes(int n_query, int H, int n_keys_max) {
  int ns, kps;
  attn_plan(n_query, n_keys_max, &ns, &kps);
  if (ns <= 1) return 0;
  const size_t parts = (size_t)n_query * ns * H;
  return parts * kD * sizeof(float) + parts * sizeof(float) + 256;
}

cudaError_t launch_attention(AttnArgs a, void* ws, cudaStream_t st) {
  int ns, kps;
  attn_plan(a.n_query, a.n_keys_max, &ns, &kps);
  a.n_split = ns;
  a.keys_per_split = kps;
  if (ns > 1) {
    const size_t parts = (size_t)a.n_query * ns * a.H;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_lse = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + parts * kD * sizeof(float));
  }
  cudaError_t e;
  switch (a.H) {
    case 16: e = launch_partial<1>(a, st); break;
    case 32: e = launch_partial<2>(a, st); break;
    case 64: e = launch_partial<4>(a, st); break;
    case 128: e = launch_partial<8>(a, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess || ns <= 1) return e;
  const int warps = a.n_query * a.H;
  attn_merge_kernel<<<(warps * 32 + 255) / 256, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace csa
