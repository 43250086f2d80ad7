// api.cu -- the extern "C" boundary of libcsa.so (declared in include/csa.h).
// Validates every argument on the host, then launches the kernels on the
// caller's stream.  Nothing here allocates device memory or synchronises.
#include <mutex>
#include <set>
#include <tuple>

#include "common.cuh"
#include "kernels.h"

namespace csa {

// Function attributes are per device: set once per (function, device, size),
// under a lock (the library may be called from several host threads).
cudaError_t ensure_smem_attr(const void* func, int bytes, bool big_clusters) {
  static std::mutex mu;
  static std::set<std::tuple<const void*, int, int, bool>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(std::make_tuple(func, dev, bytes, big_clusters))) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && big_clusters)
    e = cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done.insert(std::make_tuple(func, dev, bytes, big_clusters));
  return e;
}

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CSA_OK;
  return CSA_ERR_CUDA;
}

constexpr int kD = 128;

bool heads_supported(int H) { return H == 16 || H == 32 || H == 64 || H == 128; }

// Shared validation of the attention calls.
int check_attention_common(const void* q, const void* k_cmp, const void* v_cmp,
                           int64_t cmp_bstride, int N_cap, const void* k_raw, const void* v_raw,
                           int64_t raw_bstride, int64_t raw_cap, int window, const float* sink,
                           int B, int T, int H, int D, const void* out, const float* lse) {
  if (B < 0 || T < 0 || H <= 0 || D <= 0 || window < 0 || N_cap < 0 || raw_cap < 0)
    return CSA_ERR_INVALID_ARG;
  if (D != kD || !heads_supported(H)) return CSA_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return CSA_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return CSA_ERR_INVALID_ARG;
  // caches are read as 2-D views of 256-byte rows spanning all sequences
  if (N_cap > 0) {
    if (!k_cmp || !v_cmp || !aligned16(k_cmp) || !aligned16(v_cmp)) return CSA_ERR_INVALID_ARG;
    if (cmp_bstride % D != 0 || cmp_bstride < (int64_t)N_cap * D) return CSA_ERR_INVALID_ARG;
    if ((B - 1) * (cmp_bstride / D) + N_cap >= (int64_t(1) << 31)) return CSA_ERR_UNSUPPORTED;
  }
  if (window > 0) {
    if (!k_raw || !v_raw || !aligned16(k_raw) || !aligned16(v_raw)) return CSA_ERR_INVALID_ARG;
    if (raw_cap < window || raw_bstride % D != 0 || raw_bstride < raw_cap * D)
      return CSA_ERR_INVALID_ARG;
    if ((B - 1) * (raw_bstride / D) + raw_cap >= (int64_t(1) << 31) - 2) return CSA_ERR_UNSUPPORTED;
  }
  if ((int64_t)B * T * H >= (int64_t(1) << 31)) return CSA_ERR_UNSUPPORTED;
  if (sink && !aligned4(sink)) return CSA_ERR_INVALID_ARG;
  if (lse && !aligned4(lse)) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" {

const char* csa_status_str(int status) {
  switch (status) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID_ARG: return "CSA_ERR_INVALID_ARG: invalid argument";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED: size or dtype not supported";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE: workspace too small";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA: CUDA launch failed";
    case CSA_ERR_TIMEOUT: return "CSA_ERR_TIMEOUT: bounded device wait expired";
    default: return "unknown status";
  }
}

int csa_abi_version(void) { return 1; }

// ---------------------------------------------------------------- a1
int csa_compress_kv_span(const void* raw, int64_t raw_bstride, int64_t raw_cap, int B, int d,
                         int m, int span, int block_begin, int n_blocks, const void* W,
                         const float* pos_bias, void* out, int64_t out_bstride, int out_dtype,
                         float* out_scale, int64_t scale_bstride, int32_t* err_word,
                         void* stream) {
  (void)err_word;
  if (B < 0 || d <= 0 || m <= 0 || span < m || block_begin < 0 || n_blocks < 0)
    return CSA_ERR_INVALID_ARG;
  if (out_dtype != CSA_BF16 && out_dtype != CSA_FP8_E4M3 && out_dtype != CSA_FP4_E2M1)
    return CSA_ERR_UNSUPPORTED;
  if ((d != 64 && d != 128) || span > 256) return CSA_ERR_UNSUPPORTED;
  if (B == 0 || n_blocks == 0) return CSA_OK;
  if (!raw || !W || !pos_bias || !out) return CSA_ERR_INVALID_ARG;
  if (!aligned16(raw) || !aligned16(W) || !aligned4(pos_bias)) return CSA_ERR_INVALID_ARG;
  const int64_t end_block = (int64_t)block_begin + n_blocks;
  if (raw_cap < span || raw_bstride % 8 != 0 || raw_cap * d > raw_bstride)
    return CSA_ERR_INVALID_ARG;
  if (end_block * d > out_bstride) return CSA_ERR_INVALID_ARG;
  if (out_dtype != CSA_BF16) {
    if (!out_scale || !aligned4(out_scale) || end_block > scale_bstride) return CSA_ERR_INVALID_ARG;
  }
  if (out_dtype == CSA_FP4_E2M1 && out_bstride % 32 != 0) return CSA_ERR_INVALID_ARG;
  CompressArgs a = {};
  a.raw = reinterpret_cast<const bf16*>(raw);
  a.raw_bstride = raw_bstride;
  a.raw_cap = raw_cap;
  a.B = B;
  a.d = d;
  a.m = m;
  a.span = span;
  a.block_begin = block_begin;
  a.n_blocks = n_blocks;
  a.W = reinterpret_cast<const bf16*>(W);
  a.pos_bias = pos_bias;
  a.out = out;
  a.out_bstride = out_bstride;
  a.fp8 = out_dtype == CSA_FP8_E4M3;
  a.fp4 = out_dtype == CSA_FP4_E2M1;
  a.out_scale = out_scale;
  a.scale_bstride = scale_bstride;
  return cuda_status(launch_compress(a, reinterpret_cast<cudaStream_t>(stream)));
}

int csa_compress_kv(const void* raw, int64_t raw_bstride, int64_t raw_cap, int B, int d, int m,
                    int block_begin, int n_blocks, const void* W, const float* pos_bias, void* out,
                    int64_t out_bstride, int out_dtype, float* out_scale, int64_t scale_bstride,
                    int32_t* err_word, void* stream) {
  return csa_compress_kv_span(raw, raw_bstride, raw_cap, B, d, m, m, block_begin, n_blocks, W,
                              pos_bias, out, out_bstride, out_dtype, out_scale, scale_bstride,
                              err_word, stream);
}

int csa_compress_kv_mixed(const void* raw, int64_t raw_bstride, int64_t raw_cap, int B, int d,
                          int m, int span, int block_begin, int n_blocks, const void* W,
                          const float* pos_bias, void* out_codes, int64_t codes_bstride,
                          float* out_scale, int64_t scale_bstride, void* out_rope,
                          int64_t rope_bstride, int n_rope, int32_t* err_word, void* stream) {
  (void)err_word;
  if (B < 0 || d <= 0 || m <= 0 || span < m || block_begin < 0 || n_blocks < 0)
    return CSA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || span > 256) return CSA_ERR_UNSUPPORTED;
  if (n_rope <= 0 || n_rope >= d || n_rope % 8 != 0 || (d - n_rope) % 16 != 0)
    return CSA_ERR_INVALID_ARG;
  if (B == 0 || n_blocks == 0) return CSA_OK;
  if (!raw || !W || !pos_bias || !out_codes || !out_scale || !out_rope) return CSA_ERR_INVALID_ARG;
  if (!aligned16(raw) || !aligned16(W) || !aligned4(pos_bias) || !aligned4(out_scale))
    return CSA_ERR_INVALID_ARG;
  const int64_t end_block = (int64_t)block_begin + n_blocks;
  if (raw_cap < span || raw_bstride % 8 != 0 || raw_cap * d > raw_bstride)
    return CSA_ERR_INVALID_ARG;
  if (end_block * (d - n_rope) > codes_bstride || end_block * n_rope > rope_bstride ||
      end_block > scale_bstride)
    return CSA_ERR_INVALID_ARG;
  CompressArgs a = {};
  a.raw = reinterpret_cast<const bf16*>(raw);
  a.raw_bstride = raw_bstride;
  a.raw_cap = raw_cap;
  a.B = B;
  a.d = d;
  a.m = m;
  a.span = span;
  a.block_begin = block_begin;
  a.n_blocks = n_blocks;
  a.W = reinterpret_cast<const bf16*>(W);
  a.pos_bias = pos_bias;
  a.out = out_codes;
  a.out_bstride = codes_bstride;
  a.fp8 = 1;
  a.out_scale = out_scale;
  a.scale_bstride = scale_bstride;
  a.fp8_dims = d - n_rope;
  a.out_hi = reinterpret_cast<bf16*>(out_rope);
  a.out_hi_bstride = rope_bstride;
  return cuda_status(launch_compress(a, reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- a2 + a3
size_t csa_indexer_topk_workspace(int B, int T, int N_cap, int k) {
  (void)k;
  if (B <= 0 || T <= 0 || N_cap <= 0) return 0;
  return indexer_topk_workspace_bytes(B * T, N_cap);
}

namespace {

// checks shared by the indexer calls (status, or -1 when the call may go on)
int indexer_checks(const void* q_idx, const float* q_scale, const float* w, const void* k_idx,
                   int64_t k_bstride, const float* k_scale, int64_t ks_bstride, int idx_dtype,
                   const int32_t* q_pos, const int32_t* n_cmp, int B, int T, int H_I, int d_I,
                   int N_cap, int m) {
  if (B < 0 || T < 0 || N_cap < 0 || m <= 0) return CSA_ERR_INVALID_ARG;
  if (idx_dtype != CSA_BF16 && idx_dtype != CSA_FP8_E4M3 && idx_dtype != CSA_FP4_E2M1)
    return CSA_ERR_UNSUPPORTED;
  if (H_I != 4 || d_I != 64) return CSA_ERR_UNSUPPORTED;
  if (N_cap > kMaxNcap) return CSA_ERR_UNSUPPORTED;
  if (B == 0 || T == 0) return CSA_OK;
  if (N_cap == 0) return CSA_ERR_INVALID_ARG;
  if ((int64_t)B * T > (1 << 30)) return CSA_ERR_UNSUPPORTED;
  if (!q_idx || !w || !k_idx || !q_pos || !n_cmp) return CSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned4(w) || !aligned4(q_pos) ||
      !aligned4(n_cmp))
    return CSA_ERR_INVALID_ARG;
  if (idx_dtype == CSA_FP8_E4M3) {
    if (!q_scale || !k_scale || !aligned4(q_scale) || !aligned4(k_scale))
      return CSA_ERR_INVALID_ARG;
    if (k_bstride % 16 != 0 || ks_bstride < N_cap) return CSA_ERR_INVALID_ARG;
  } else if (idx_dtype == CSA_FP4_E2M1) {
    // codes: 32 bytes per entry; scales: 4 E4M3 bytes per entry / query head
    if (!q_scale || !k_scale || !aligned4(q_scale) || !aligned4(k_scale))
      return CSA_ERR_INVALID_ARG;
    if (k_bstride % 32 != 0 || ks_bstride < N_cap) return CSA_ERR_INVALID_ARG;
  } else if (k_bstride % 8 != 0) {
    return CSA_ERR_INVALID_ARG;
  }
  if (k_bstride < (int64_t)N_cap * d_I) return CSA_ERR_INVALID_ARG;
  return -1;
}

IndexerArgs indexer_args(const void* q_idx, const float* q_scale, const float* w,
                         const void* k_idx, int64_t k_bstride, const float* k_scale,
                         int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
                         const int32_t* n_cmp, int B, int T, int N_cap, int m, int k,
                         int32_t* err_word) {
  IndexerArgs a = {};
  a.q = q_idx;
  a.q_scale = q_scale;
  a.w = w;
  a.keys = k_idx;
  a.k_bstride = k_bstride;
  a.k_scale = k_scale;
  a.ks_bstride = ks_bstride;
  a.fp8 = idx_dtype == CSA_FP8_E4M3;
  a.fp4 = idx_dtype == CSA_FP4_E2M1;
  a.q_pos = q_pos;
  a.n_cmp = n_cmp;
  a.T = T;
  a.n_query = B * T;
  a.N_cap = N_cap;
  a.m = m;
  a.k = k;
  a.err = err_word;
  return a;
}

}  // namespace

}  // extern "C"

namespace csa {

// Every argument check of csa_indexer_topk except the workspace: a status to
// return, or -1 when the call may go on (shared with the static-scratch
// entry point, so that both give the same status for the same arguments).
int indexer_topk_arg_status(const void* q_idx, const float* q_scale, const float* w,
                            const void* k_idx, int64_t k_bstride, const float* k_scale,
                            int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
                            const int32_t* n_cmp, int B, int T, int H_I, int d_I, int N_cap,
                            int m, int k, const int32_t* topk_idx, const float* topk_score) {
  if (k <= 0) return CSA_ERR_INVALID_ARG;
  const int c = indexer_checks(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride, idx_dtype,
                               q_pos, n_cmp, B, T, H_I, d_I, N_cap, m);
  if (c >= 0) return c;
  if (k > N_cap) return CSA_ERR_INVALID_ARG;
  if (!topk_idx || !aligned4(topk_idx)) return CSA_ERR_INVALID_ARG;
  if (topk_score && !aligned4(topk_score)) return CSA_ERR_INVALID_ARG;
  return -1;
}

}  // namespace csa

extern "C" {

int csa_indexer_scores(const void* q_idx, const float* q_scale, const float* w, const void* k_idx,
                       int64_t k_bstride, const float* k_scale, int64_t ks_bstride, int idx_dtype,
                       const int32_t* q_pos, const int32_t* n_cmp, int B, int T, int H_I, int d_I,
                       int N_cap, int m, float* scores, int64_t ld, int32_t* err_word,
                       void* stream) {
  const int c = indexer_checks(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride, idx_dtype,
                               q_pos, n_cmp, B, T, H_I, d_I, N_cap, m);
  if (c >= 0) return c;
  if (!scores || !aligned4(scores) || ld < N_cap || ld > INT32_MAX) return CSA_ERR_INVALID_ARG;
  IndexerArgs a = indexer_args(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride, idx_dtype,
                               q_pos, n_cmp, B, T, N_cap, m, 1, err_word);
  return cuda_status(
      launch_indexer_scores(a, scores, (int)ld, reinterpret_cast<cudaStream_t>(stream)));
}

int csa_indexer_topk(const void* q_idx, const float* q_scale, const float* w, const void* k_idx,
                     int64_t k_bstride, const float* k_scale, int64_t ks_bstride, int idx_dtype,
                     const int32_t* q_pos, const int32_t* n_cmp, int B, int T, int H_I, int d_I,
                     int N_cap, int m, int k, int32_t* topk_idx, float* topk_score, void* ws,
                     size_t ws_bytes, int32_t* err_word, void* stream) {
  const int c = indexer_topk_arg_status(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride,
                                        idx_dtype, q_pos, n_cmp, B, T, H_I, d_I, N_cap, m, k,
                                        topk_idx, topk_score);
  if (c >= 0) return c;
  const size_t need = indexer_topk_workspace_bytes(B * T, N_cap);
  if (!ws || ws_bytes < need || !aligned16(ws)) return CSA_ERR_WORKSPACE;
  IndexerArgs a = indexer_args(q_idx, q_scale, w, k_idx, k_bstride, k_scale, ks_bstride, idx_dtype,
                               q_pos, n_cmp, B, T, N_cap, m, k, err_word);
  a.topk_idx = topk_idx;
  a.topk_score = topk_score;
  return cuda_status(launch_indexer_topk(a, ws, reinterpret_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------- a4 / a5 / a6
size_t csa_attn_workspace(int B, int T, int H, int n_keys_max) {
  if (B <= 0 || T <= 0 || H <= 0 || n_keys_max <= 0) return 0;
  return attn_workspace_bytes(B * T, H, n_keys_max);
}

static int run_attention(AttnArgs& a, void* ws, size_t ws_bytes, void* stream) {
  if (a.n_query == 0) return CSA_OK;
  // the workspace is optional: without it (or if it is too small) the key
  // splits of a query always merge inside a cluster
  const size_t need = attn_workspace_bytes(a.n_query, a.H, a.n_keys_max);
  if (ws && !aligned16(ws)) return CSA_ERR_WORKSPACE;
  void* use = (need > 0 && ws && ws_bytes >= need) ? ws : nullptr;
  return cuda_status(launch_attention(a, use, reinterpret_cast<cudaStream_t>(stream)));
}

static void fill_common(AttnArgs& a, const void* q, const void* k_cmp, const void* v_cmp,
                        int64_t cmp_bstride, int N_cap, const void* k_raw, const void* v_raw,
                        int64_t raw_bstride, int64_t raw_cap, int window, const float* sink,
                        float softmax_scale, int H, void* out, float* lse, int32_t* err_word) {
  a = AttnArgs();
  a.q = reinterpret_cast<const bf16*>(q);
  a.k_cmp = reinterpret_cast<const bf16*>(k_cmp);
  a.v_cmp = reinterpret_cast<const bf16*>(v_cmp);
  a.cmp_bstride = cmp_bstride;
  a.N_cap = N_cap;
  // with no window, raw pointers may be NULL: point the (never dereferenced)
  // raw source at the compressed cache so address arithmetic stays defined
  a.k_raw = reinterpret_cast<const bf16*>(window > 0 ? k_raw : k_cmp);
  a.v_raw = reinterpret_cast<const bf16*>(window > 0 ? v_raw : v_cmp);
  a.raw_bstride = window > 0 ? raw_bstride : 0;
  a.raw_cap = raw_cap;
  a.window = window;
  a.sink = sink;
  a.scale_log2 = softmax_scale * kLog2e;
  a.H = H;
  a.out = reinterpret_cast<bf16*>(out);
  a.lse = lse;
  a.err = err_word;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.fixed_kps = 0;
  a.n_cmp = nullptr;
  a.m_prime = 1;
  a.dense = 0;
  a.sel = nullptr;
  a.sel_count = 0;
  a.sel_stride = 0;
}

int csa_sparse_attn_decode(const void* q, const void* k_cmp, const void* v_cmp,
                           int64_t cmp_bstride, int N_cap, const int32_t* topk_idx, int k,
                           const void* k_raw, const void* v_raw, int64_t raw_bstride,
                           int64_t raw_cap, const int32_t* seq_len, int window, const float* sink,
                           float softmax_scale, int B, int H, int D, void* out, float* lse,
                           void* ws, size_t ws_bytes, int32_t* err_word, void* stream) {
  int st = check_attention_common(q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride,
                                  raw_cap, window, sink, B, 1, H, D, out, lse);
  if (st != CSA_OK || B == 0) return st;
  if (k < 0 || (k > 0 && (!topk_idx || !aligned4(topk_idx) || N_cap <= 0))) return CSA_ERR_INVALID_ARG;
  if (!seq_len || !aligned4(seq_len)) return CSA_ERR_INVALID_ARG;
  if (k + window <= 0) return CSA_ERR_INVALID_ARG;
  AttnArgs a;
  fill_common(a, q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride, raw_cap, window,
              sink, softmax_scale, H, out, lse, err_word);
  a.sel = topk_idx;
  a.sel_count = k;
  a.sel_stride = k;
  a.pos = seq_len;
  a.pos_is_len = 1;
  a.T = 1;
  a.n_batch = B;
  a.n_query = B;
  a.n_keys_max = k + window;
  return run_attention(a, ws, ws_bytes, stream);
}

int csa_sparse_attn_prefill(const void* q, const void* k_cmp, const void* v_cmp,
                            int64_t cmp_bstride, int N_cap, const int32_t* topk_idx, int k,
                            const void* k_raw, const void* v_raw, int64_t raw_bstride,
                            int64_t raw_cap, const int32_t* q_pos, int window, const float* sink,
                            float softmax_scale, int B, int T, int H, int D, void* out,
                            float* lse, void* ws, size_t ws_bytes, int32_t* err_word,
                            void* stream) {
  int st = check_attention_common(q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride,
                                  raw_cap, window, sink, B, T, H, D, out, lse);
  if (st != CSA_OK || B == 0 || T == 0) return st;
  if (k < 0 || (k > 0 && (!topk_idx || !aligned4(topk_idx) || N_cap <= 0))) return CSA_ERR_INVALID_ARG;
  if (!q_pos || !aligned4(q_pos)) return CSA_ERR_INVALID_ARG;
  if (k + window <= 0) return CSA_ERR_INVALID_ARG;
  if ((int64_t)B * T > (1 << 30)) return CSA_ERR_UNSUPPORTED;
  AttnArgs a;
  fill_common(a, q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride, raw_cap, window,
              sink, softmax_scale, H, out, lse, err_word);
  a.sel = topk_idx;
  a.sel_count = k;
  a.sel_stride = k;
  a.pos = q_pos;
  a.pos_is_len = 0;
  a.T = T;
  a.n_batch = B;
  a.n_query = B * T;
  a.n_keys_max = k + window;
  return run_attention(a, ws, ws_bytes, stream);
}

int csa_sparse_attn_batch_invariant(const void* q, const void* k_cmp, const void* v_cmp,
                                    int64_t cmp_bstride, int N_cap, const int32_t* topk_idx,
                                    int k, const void* k_raw, const void* v_raw,
                                    int64_t raw_bstride, int64_t raw_cap, const int32_t* q_pos,
                                    int window, const float* sink, float softmax_scale, int B,
                                    int T, int H, int D, void* out, float* lse,
                                    int keys_per_split, int32_t* err_word, void* stream) {
  int st = check_attention_common(q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride,
                                  raw_cap, window, sink, B, T, H, D, out, lse);
  if (st != CSA_OK || B == 0 || T == 0) return st;
  if (k < 0 || (k > 0 && (!topk_idx || !aligned4(topk_idx) || N_cap <= 0))) return CSA_ERR_INVALID_ARG;
  if (!q_pos || !aligned4(q_pos)) return CSA_ERR_INVALID_ARG;
  if (k + window <= 0) return CSA_ERR_INVALID_ARG;
  if ((int64_t)B * T > (1 << 30)) return CSA_ERR_UNSUPPORTED;
  // at most 16 splits (one cluster) of keys_per_split slots, rounded up to 64
  if (keys_per_split <= 0 || keys_per_split > (1 << 24)) return CSA_ERR_INVALID_ARG;
  const int64_t kps = ((int64_t)keys_per_split + 63) / 64 * 64;
  if ((k + window + 3 + kps - 1) / kps > 16) return CSA_ERR_INVALID_ARG;
  AttnArgs a;
  fill_common(a, q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride, raw_cap, window,
              sink, softmax_scale, H, out, lse, err_word);
  a.sel = topk_idx;
  a.sel_count = k;
  a.sel_stride = k;
  a.pos = q_pos;
  a.pos_is_len = 0;
  a.T = T;
  a.n_batch = B;
  a.n_query = B * T;
  a.n_keys_max = k + window;
  a.fixed_kps = keys_per_split;
  return cuda_status(launch_attention(a, nullptr, reinterpret_cast<cudaStream_t>(stream)));
}

int hca_dense_attn_decode(const void* q, const void* k_cmp, const void* v_cmp,
                          int64_t cmp_bstride, int N_cap, const int32_t* n_cmp, int m_prime,
                          const void* k_raw, const void* v_raw, int64_t raw_bstride,
                          int64_t raw_cap, const int32_t* seq_len, int window, const float* sink,
                          float softmax_scale, int B, int H, int D, void* out, float* lse,
                          void* ws, size_t ws_bytes, int32_t* err_word, void* stream) {
  int st = check_attention_common(q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride,
                                  raw_cap, window, sink, B, 1, H, D, out, lse);
  if (st != CSA_OK || B == 0) return st;
  if (m_prime <= 0 || !seq_len || !aligned4(seq_len)) return CSA_ERR_INVALID_ARG;
  if (N_cap > 0 && (!n_cmp || !aligned4(n_cmp))) return CSA_ERR_INVALID_ARG;
  if (N_cap + window <= 0) return CSA_ERR_INVALID_ARG;
  AttnArgs a;
  fill_common(a, q, k_cmp, v_cmp, cmp_bstride, N_cap, k_raw, v_raw, raw_bstride, raw_cap, window,
              sink, softmax_scale, H, out, lse, err_word);
  a.dense = 1;
  a.n_cmp = n_cmp;
  a.m_prime = m_prime;
  a.pos = seq_len;
  a.pos_is_len = 1;
  a.T = 1;
  a.n_batch = B;
  a.n_query = B;
  a.n_keys_max = N_cap + window;
  return run_attention(a, ws, ws_bytes, stream);
}

int csa_attn_fp8kv(const void* q, const void* k_nope, const float* k_scale, const void* k_rope,
                   const void* v, const float* v_scale, int N_cap, const int32_t* topk_idx, int k,
                   const int32_t* n_cmp, int m_prime, const void* k_raw, const void* v_raw,
                   int64_t raw_bstride, int64_t raw_cap, const int32_t* q_pos, int window,
                   const float* sink, float softmax_scale, int B, int T, int H, int D, void* out,
                   float* lse, void* ws, size_t ws_bytes, int32_t* err_word, void* stream) {
  int st = check_attention_common(q, k_nope, v, (int64_t)N_cap * kD, N_cap, k_raw, v_raw,
                                  raw_bstride, raw_cap, window, sink, B, T, H, D, out, lse);
  if (st != CSA_OK || B == 0 || T == 0) return st;
  if (H > 64) return CSA_ERR_UNSUPPORTED;
  if (!q_pos || !aligned4(q_pos)) return CSA_ERR_INVALID_ARG;
  if ((int64_t)B * T > (1 << 30)) return CSA_ERR_UNSUPPORTED;
  if (N_cap > 0 && (!k_scale || !v_scale || !k_rope || !aligned4(k_scale) ||
                    !aligned4(v_scale) || !aligned16(k_rope)))
    return CSA_ERR_INVALID_ARG;
  const bool dense = topk_idx == nullptr;
  if (dense) {
    if (m_prime <= 0 || (N_cap > 0 && (!n_cmp || !aligned4(n_cmp)))) return CSA_ERR_INVALID_ARG;
    if (N_cap + window <= 0) return CSA_ERR_INVALID_ARG;
  } else {
    if (k <= 0 || N_cap <= 0 || !aligned4(topk_idx)) return CSA_ERR_INVALID_ARG;
  }
  AttnArgs a;
  fill_common(a, q, k_nope, v, (int64_t)N_cap * kD, N_cap, k_raw, v_raw, raw_bstride, raw_cap,
              window, sink, softmax_scale, H, out, lse, err_word);
  a.kv8 = 1;
  a.k8 = reinterpret_cast<const uint8_t*>(k_nope);
  a.k8_scale = k_scale;
  a.k_rope = reinterpret_cast<const bf16*>(k_rope);
  a.v8 = reinterpret_cast<const uint8_t*>(v);
  a.v8_scale = v_scale;
  if (dense) {
    a.dense = 1;
    a.n_cmp = n_cmp;
    a.m_prime = m_prime;
    a.n_keys_max = N_cap + window;
  } else {
    a.sel = topk_idx;
    a.sel_count = k;
    a.sel_stride = k;
    a.n_keys_max = k + window;
  }
  a.pos = q_pos;
  a.pos_is_len = 0;
  a.T = T;
  a.n_batch = B;
  a.n_query = B * T;
  return run_attention(a, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------- output projection
int csa_grouped_out_proj(const void* o, const void* W, void* y, int n, int H, int D, int G,
                         int d_g, int32_t* err_word, void* stream) {
  if (n < 0 || H <= 0 || D <= 0 || G <= 0 || d_g <= 0 || H % G != 0) return CSA_ERR_INVALID_ARG;
  const int64_t K = (int64_t)(H / G) * D;
  if (K % 64 != 0 || d_g % 128 != 0 || (int64_t)H * D > (1 << 20)) return CSA_ERR_UNSUPPORTED;
  if (n == 0) return CSA_OK;
  if (!o || !W || !y) return CSA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(W) || !aligned16(y)) return CSA_ERR_INVALID_ARG;
  OutProjArgs a;
  a.o = reinterpret_cast<const bf16*>(o);
  a.W = reinterpret_cast<const bf16*>(W);
  a.y = reinterpret_cast<bf16*>(y);
  a.n = n;
  a.H = H;
  a.D = D;
  a.G = G;
  a.d_g = d_g;
  a.err = err_word;
  return cuda_status(launch_out_proj(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
