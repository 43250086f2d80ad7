// kernels.h -- internal launch interface between the C ABI layer (api.cu)
// and the kernels.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda_bf16.h>

namespace csa {

// Sets the dynamic shared-memory limit of a kernel once per device.
// sets the dynamic shared memory limit (and, with big_clusters, permission
// for clusters above 8 CTAs) once per function and device; thread-safe
cudaError_t ensure_smem_attr(const void* func, int bytes, bool big_clusters = false);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  const __nv_bfloat16* q;  // [n_query][H][128]
  const __nv_bfloat16* k_cmp;
  const __nv_bfloat16* v_cmp;
  int64_t cmp_bstride;
  int N_cap;
  int dense;           // 1: compressed rows 0 .. n_vis-1 (HCA); 0: rows from sel
  const int32_t* sel;  // [n_query][sel_stride] compressed rows (sparse)
  int sel_count;
  int64_t sel_stride;
  const int32_t* n_cmp;  // dense: entries present per sequence
  int m_prime;           // dense: compression ratio for the visibility rule
  const __nv_bfloat16* k_raw;
  const __nv_bfloat16* v_raw;
  int64_t raw_bstride;
  int64_t raw_cap;  // ring of raw_cap rows: position p at row p % raw_cap
  const int32_t* pos;  // pos_is_len ? seq_len[B] : q_pos[n_query]
  int pos_is_len;
  int T;  // query tokens per sequence (query q belongs to sequence q / T)
  int window;
  const float* sink;
  float scale_log2;  // softmax_scale * log2(e)
  int H;
  int n_batch;  // sequences (rows of the caches' 2-D views span all of them)
  int n_query;
  int n_keys_max;
  int fixed_kps;  // > 0: every query's keys split into ranges of this many slots
  // FP8-stored compressed entries (kv8 != 0; k_cmp / v_cmp unused): K's 64
  // non-RoPE channels as E4M3 codes [rows][64] with fp32 scales [rows], its 64
  // RoPE channels bf16 [rows][64]; V as E4M3 codes [rows][128] with scales.
  // Row = b * N_cap + entry.  H <= 64.
  int kv8;
  const uint8_t* k8;
  const float* k8_scale;
  const __nv_bfloat16* k_rope;
  const uint8_t* v8;
  const float* v8_scale;
  // filled by launch_attention
  int n_split;
  int keys_per_split;
  float* part_o;
  float* part_lse;
  // 1: the splits of a query are one cluster and exchange their partial rows
  // through part_o / part_lse (global memory, L2) instead of distributed
  // shared memory; 0 with part_o set: splits without a cluster, merged by a
  // second kernel
  int xch;
  __nv_bfloat16* out;
  float* lse;
  int32_t* err;
};

// ---------------------------------------------------------------- output projection
struct OutProjArgs {
  const __nv_bfloat16* o;  // [n][H * D]
  const __nv_bfloat16* W;  // [G][d_g][(H / G) * D]
  __nv_bfloat16* y;        // [n][G * d_g]
  int n, H, D, G, d_g;
  int32_t* err;
};
cudaError_t launch_out_proj(const OutProjArgs& a, cudaStream_t st);

void attn_plan(int n_query, int n_keys_max, int max_cluster, int* n_split, int* keys_per_split);
size_t attn_workspace_bytes(int n_query, int H, int n_keys_max);  // 0: splits merge on chip
cudaError_t launch_attention(AttnArgs a, void* ws, cudaStream_t st);

// ---------------------------------------------------------------- indexer + top-k
constexpr int kHistBins = 4096;  // top 12 bits of the order-preserving score key
constexpr int kMaxNcap = 1 << 19;

struct IndexerArgs {
  const void* q;  // [n_query][4][64] bf16 or E4M3
  const float* q_scale;
  const float* w;
  const void* keys;  // [B][k_bstride] rows of 64 (bf16 or E4M3)
  int64_t k_bstride;
  const float* k_scale;
  int64_t ks_bstride;
  int fp8;
  int fp4;  // E2M1 codes with E4M3 block scales (one per 16 channels)
  const int32_t* q_pos;
  const int32_t* n_cmp;
  int T;
  int n_query;
  int N_cap;
  int m;
  int k;
  int32_t* err;
  // outputs
  int32_t* topk_idx;
  float* topk_score;
};

size_t indexer_topk_workspace_bytes(int n_query, int N_cap);
// Host checks of csa_indexer_topk's arguments other than the workspace: a
// CSA_* status to return, or -1 when the call may go on.
int indexer_topk_arg_status(const void* q_idx, const float* q_scale, const float* w,
                            const void* k_idx, int64_t k_bstride, const float* k_scale,
                            int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
                            const int32_t* n_cmp, int B, int T, int H_I, int d_I, int N_cap,
                            int m, int k, const int32_t* topk_idx, const float* topk_score);
cudaError_t launch_indexer_topk(const IndexerArgs& a, void* ws, cudaStream_t st);
// the scores alone: query q's row at scores + q * ld (entries < n_vis)
cudaError_t launch_indexer_scores(const IndexerArgs& a, float* scores, int ld, cudaStream_t st);
// tensor-core scorer for many bf16 query tokens per sequence (T a multiple of
// 64): scores of queries [q0, q0 + qc) into scores[(q - q0) * stride + entry]
bool indexer_gemm_applies(const IndexerArgs& a);
cudaError_t launch_indexer_gemm(const IndexerArgs& a, int q0, int qc, float* scores, int stride,
                                cudaStream_t st);

// ---------------------------------------------------------------- compression
struct CompressArgs {
  const __nv_bfloat16* raw;
  int64_t raw_bstride;
  int64_t raw_cap;  // ring of raw_cap rows: position p at row p % raw_cap
  int B, d, m, block_begin, n_blocks;
  int span;  // raw tokens per block, ending at its last token (span >= m; m: no overlap)
  const __nv_bfloat16* W;
  const float* pos_bias;
  void* out;
  int64_t out_bstride;
  int fp8;
  int fp4;  // E2M1 codes with E4M3 block scales (one per 16 channels)
  float* out_scale;
  int64_t scale_bstride;
  // mixed storage (fp8 != 0, 0 < fp8_dims < d): channels [0, fp8_dims) as
  // E4M3 rows of fp8_dims bytes in out, the rest bf16 rows of d - fp8_dims in
  // out_hi (batch stride out_hi_bstride elements)
  int fp8_dims;
  __nv_bfloat16* out_hi;
  int64_t out_hi_bstride;
};

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t st);

}  // namespace csa
