/*
 * csa.h -- C ABI of libcsa.so: the CSA / HCA attention hot path on one GPU.
 *
 * The method (page "DeepSeek-V4: Towards Highly Efficient Million-Token
 * Context Intelligence", hyper.ai, Method):
 *   CSA compresses every m raw KV tokens into one entry, scores the entries
 *   with a Lightning Indexer, keeps the top-k, and runs MQA attention over
 *   them (plus a sliding window of raw tokens and an attention sink, aiboss88
 *   DeepSeek-V4 page, Technical Principles).  HCA compresses by m' >> m
 *   without overlap and attends densely over every compressed entry, also
 *   with the window branch.
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; nothing is
 *     allocated, freed or retained by the library.  Scratch memory is passed in
 *     (`ws`, sized by the *_workspace queries).
 *   - Tensors are row-major and contiguous inside a sequence; the distance
 *     between sequences ("bstride") is given in ELEMENTS of the tensor's type.
 *     bf16 tensors and their bstrides must be 16-byte aligned (bstride a
 *     multiple of 8 elements); FP8 tensors 16-byte aligned (bstride a multiple
 *     of 16); fp32 / int32 tensors 4-byte aligned.
 *   - Each call is asynchronous and stream-ordered on `stream` (a
 *     cudaStream_t; NULL = legacy default stream).  No call synchronises the
 *     device or the host.  Calls with disjoint outputs and workspaces may run
 *     concurrently on different streams.
 *   - Host-side validation runs first; on any error nothing is launched and a
 *     non-zero status is returned.
 *   - `err_word` (optional, device int32) receives bit flags OR-ed in by the
 *     kernels when they meet an input they cannot honour (they skip it and
 *     never trap): CSA_EW_BAD_INDEX (a top-k index outside [-1, N_cap)),
 *     CSA_EW_BAD_POSITION (a position or length outside the cache or < 0),
 *     CSA_EW_TIMEOUT (an internal pipeline wait expired; outputs invalid).
 *     The word is never cleared by the library; the caller reads it when it
 *     chooses.
 *   - Numbers: bf16 inputs, fp32 accumulation, bf16 outputs rounded to
 *     nearest even.  FP8 is OCP E4M3 ("e4m3fn") with one fp32 scale per row.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA_API __attribute__((visibility("default")))
#else
#define CSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define CSA_OK 0
#define CSA_ERR_INVALID_ARG 1 /* null pointer, bad shape / stride / alignment, k > N_cap ... */
#define CSA_ERR_UNSUPPORTED 2 /* a size or dtype this build has no kernel for */
#define CSA_ERR_WORKSPACE 3   /* ws too small (or NULL while needed) */
#define CSA_ERR_CUDA 4        /* a launch failed; the CUDA error was consumed */
#define CSA_ERR_TIMEOUT 5     /* reserved for bounded device-side waits */

/* err_word bits */
#define CSA_EW_BAD_INDEX 1
#define CSA_EW_BAD_POSITION 2
#define CSA_EW_TIMEOUT 4 /* a bounded device-side wait gave up (should never happen) */

/* element types */
#define CSA_BF16 0
#define CSA_FP8_E4M3 1
/* OCP FP4 E2M1 codes, two per byte (channel 2i in the low nibble), with one
 * E4M3 scale byte per 16 channels (value = code value * block scale): the
 * pages' FP4 indexer path, its dynamic range extended with FP8.  Indexer
 * vectors only (d_I = 64: 32 code bytes and 4 scale bytes per vector). */
#define CSA_FP4_E2M1 2

/* Human-readable name of a status code (static string, never NULL). */
CSA_API const char* csa_status_str(int status);

/* Version of this ABI (bumped on any signature change). */
CSA_API int csa_abi_version(void);

/* ------------------------------------------------------------------------
 * a1. Block compression (CSA ratio m, HCA ratio m').
 *
 * Source: hyper.ai DeepSeek-V4 page, Method -- "compresses every m tokens
 * into a single entry using learnable compression weights and positional
 * biases"; HCA: "without overlapping compression".  The operator is this
 * library's reading of that sentence: for block j of sequence b, channel c,
 *     g[i][c] = sum_e W[c][e] * x[j*m+i][e] + pos_bias[i][c],  i < m
 *     y[j][c] = sum_i softmax_i(g[.][c])[i] * x[j*m+i][c]
 * Blocks [block_begin, block_begin + n_blocks) of every sequence are written.
 *
 *   raw       bf16 [B][raw_bstride]: token rows of d, a ring of raw_cap rows:
 *             position p is row p mod raw_cap; block j reads positions
 *             j*m .. j*m+m-1 (raw_cap >= m).
 *   W         bf16 [d][d] (row = output channel), pos_bias fp32 [m][d].
 *   out       out_dtype == CSA_BF16: bf16 [B][out_bstride], row j of d.
 *             out_dtype == CSA_FP4_E2M1: bytes, row j of d/2 (out_bstride
 *             counts channels: a multiple of 32), plus out_scale pointing to
 *             E4M3 bytes [B][scale_bstride][d/16]: per block of 16 channels
 *             the nearest E4M3 value of amax / 6 (1 if all zero; at least
 *             2^-9), codes the nearest E2M1 value of y / scale (ties to
 *             even, saturating at 6).
 *             out_dtype == CSA_FP8_E4M3: E4M3 bytes, row j of d, plus
 *             out_scale fp32 [B][scale_bstride]: scale = max_c |y| / 448
 *             (1 when all zero), code = nearest-even E4M3 of y / scale,
 *             saturating at 448.
 *   d in {64, 128}; 1 <= m <= 256.
 * ---------------------------------------------------------------------- */
CSA_API int csa_compress_kv(const void* raw, int64_t raw_bstride, int64_t raw_cap, int B, int d,
                    int m, int block_begin, int n_blocks, const void* W, const float* pos_bias,
                    void* out, int64_t out_bstride, int out_dtype, float* out_scale,
                    int64_t scale_bstride, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * a1 with overlapping blocks.  The hyper.ai DeepSeek-V4 page (Method, HCA
 * paragraph) says HCA compresses "without overlapping compression", which
 * this library reads as: CSA's blocks may overlap.  Block j keeps its stride
 * m, its position in the output and its visibility rule (it ends at token
 * j*m + m - 1), but is compressed from the `span` raw tokens ending there:
 *     p_i = j*m + m - span + i,  0 <= i < span,  negative positions left out
 *     g[i][c] = sum_e W[c][e] x[p_i][e] + pos_bias[i][c];  softmax over i
 *     y[j][c] = sum_i a[i][c] x[p_i][c]
 * Arguments as csa_compress_kv, plus span (m <= span <= 256) with
 * pos_bias fp32 [span][d] (row i belongs to position p_i).  The raw ring
 * must hold the span: raw_cap >= span.  span == m is csa_compress_kv.
 * ---------------------------------------------------------------------- */
CSA_API int csa_compress_kv_span(const void* raw, int64_t raw_bstride, int64_t raw_cap, int B,
                                 int d, int m, int span, int block_begin, int n_blocks,
                                 const void* W, const float* pos_bias, void* out,
                                 int64_t out_bstride, int out_dtype, float* out_scale,
                                 int64_t scale_bstride, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * a1 into mixed-precision storage.  The hyper.ai DeepSeek-V4 page (Method)
 * stores the KV entries in FP8 except their RoPE dimensions, which stay
 * BF16.  Reading: the last n_rope channels of an entry are its RoPE
 * channels.  The operator is that of csa_compress_kv_span; its output y is
 * stored as
 *     channels [0, d - n_rope):  E4M3 codes, row j of d - n_rope bytes in
 *                                out_codes [B][codes_bstride], with
 *                                out_scale fp32 [B][scale_bstride]: scale =
 *                                max |y| over these channels / 448 (1 when
 *                                all zero), code = nearest-even E4M3 of
 *                                y / scale, saturating;
 *     channels [d - n_rope, d):  bf16 (nearest even), row j of n_rope in
 *                                out_rope [B][rope_bstride].
 * Other arguments as csa_compress_kv_span.  0 < n_rope < d, n_rope a
 * multiple of 8, d - n_rope a multiple of 16; codes_bstride counts bytes,
 * rope_bstride bf16 elements.  A K stream with RoPE channels uses this call;
 * a V stream (no RoPE channels) uses csa_compress_kv_span with
 * CSA_FP8_E4M3.  Status: as csa_compress_kv_span.
 * ---------------------------------------------------------------------- */
CSA_API int csa_compress_kv_mixed(const void* raw, int64_t raw_bstride, int64_t raw_cap, int B,
                                  int d, int m, int span, int block_begin, int n_blocks,
                                  const void* W, const float* pos_bias, void* out_codes,
                                  int64_t codes_bstride, float* out_scale, int64_t scale_bstride,
                                  void* out_rope, int64_t rope_bstride, int n_rope,
                                  int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * a2 + a3. Lightning-Indexer scores and exact top-k.
 *
 * Sources: hyper.ai DeepSeek-V4 page, Method ("A Lightning Indexer then
 * selects the top-k compressed KV entries"); aiboss88 page, Technical
 * Principles (index score, then top-k; FP8 range for the low-precision
 * indexer QK path); elamur.ai page, Summary ("runs DeepSeek Sparse
 * Attention") -- read as the score
 *     I(t,s) = sum_h w[t][h] * ReLU(q[t][h] . k[s]),    s < n_vis(t)
 *     n_vis(t) = min(n_cmp[b], floor((t + 1) / m))   (block-causal)
 * FP8: q[t][h] . k[s] = q_scale[t][h] * k_scale[s] * sum_d q8[d] * k8[d].
 * FP4 (idx_dtype CSA_FP4_E2M1): q_idx [B][T][H_I][d_I/2] and k_idx rows of
 * d_I/2 bytes (k_bstride still counts channels: a multiple of 32); q_scale
 * and k_scale then point to E4M3 block-scale bytes, [B][T][H_I][d_I/16] and
 * [B][ks_bstride][d_I/16]; the dot product is over code * scale values.
 * Selection: the min(k, n_vis) largest scores, ties to the lower index,
 * written in ascending index order and padded with -1.
 *
 *   q_idx     [B][T][H_I][d_I] (bf16, or E4M3 bytes with q_scale fp32
 *             [B][T][H_I]); w fp32 [B][T][H_I].
 *   k_idx     [B][k_bstride] rows of d_I (bf16 or E4M3 bytes), with
 *             k_scale fp32 [B][ks_bstride] for E4M3.
 *   q_pos     int32 [B][T] absolute positions; n_cmp int32 [B] entries present
 *             (<= N_cap).
 *   topk_idx  int32 [B][T][k] out; topk_score fp32 [B][T][k] out (optional,
 *             the selected entries' scores, -inf in padded slots).
 *   ws        csa_indexer_topk_workspace(B, T, N_cap, k) bytes.
 *   H_I == 4, d_I == 64; 1 <= k <= N_cap.
 * ---------------------------------------------------------------------- */
CSA_API size_t csa_indexer_topk_workspace(int B, int T, int N_cap, int k);
CSA_API int csa_indexer_topk(const void* q_idx, const float* q_scale, const float* w,
                     const void* k_idx, int64_t k_bstride, const float* k_scale,
                     int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
                     const int32_t* n_cmp, int B, int T, int H_I, int d_I, int N_cap, int m,
                     int k, int32_t* topk_idx, float* topk_score, void* ws, size_t ws_bytes,
                     int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * a2 alone: the Lightning-Indexer scores I(t,s) of csa_indexer_topk (same
 * sources, reading and arguments), written out instead of selected from.
 *
 *   scores    fp32 [B*T][ld] out: row b*T + t holds I(t,s) at column s for
 *             s < n_vis(t); columns from n_vis(t) on are unspecified (they may
 *             be written).  ld >= N_cap.
 *   No workspace.  Errors: as csa_indexer_topk (k is not an argument here).
 * ---------------------------------------------------------------------- */
CSA_API int csa_indexer_scores(const void* q_idx, const float* q_scale, const float* w,
                               const void* k_idx, int64_t k_bstride, const float* k_scale,
                               int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
                               const int32_t* n_cmp, int B, int T, int H_I, int d_I, int N_cap,
                               int m, float* scores, int64_t ld, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * a4 + a6, batch-invariant.  The elamur.ai DeepSeek-V4 page (Key points,
 * infrastructure) and the myWiki DeepSeek-V4 notes (Infrastructure
 * Highlights) list batch-invariant, deterministic kernels for bitwise
 * reproducibility.  csa_sparse_attn_prefill splits each query's keys
 * according to how many queries share the call, so the fp32 summation order
 * of a query's result changes with B and T.  This call fixes the split by the
 * key count alone: ranges of keys_per_split slots (rounded up to 64), at most
 * 16 of them (one thread-block cluster per query), merged in split order.  A
 * query's output and lse are then bitwise the same whatever else is in the
 * batch, and from run to run.
 *
 * Arguments as csa_sparse_attn_prefill (T query tokens per sequence at
 * q_pos, so T = 1 is decode with q_pos = seq_len - 1, and T = 2 a two-token
 * multi-token-prediction step), without a workspace, plus keys_per_split
 * > 0 with ceil((k + window + 3) / round64(keys_per_split)) <= 16, else
 * CSA_ERR_INVALID_ARG.  The clusters need not all be resident at once (a
 * large batch may run in several waves).
 * ---------------------------------------------------------------------- */
CSA_API int csa_sparse_attn_batch_invariant(const void* q, const void* k_cmp, const void* v_cmp,
                                            int64_t cmp_bstride, int N_cap,
                                            const int32_t* topk_idx, int k, const void* k_raw,
                                            const void* v_raw, int64_t raw_bstride,
                                            int64_t raw_cap, const int32_t* q_pos, int window,
                                            const float* sink, float softmax_scale, int B, int T,
                                            int H, int D, void* out, float* lse,
                                            int keys_per_split, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * a4 / a5 over FP8-stored compressed entries.  The hyper.ai DeepSeek-V4 page
 * (Method) keeps the KV cache in FP8 apart from the RoPE dimensions, which
 * stay BF16.  Reading (D = 128): K's channels 0-63 are its non-RoPE channels,
 * stored as E4M3 codes with one fp32 scale per entry, channels 64-127 its
 * RoPE channels in bf16; V has no RoPE channels: 128 E4M3 codes with its own
 * per-entry scale.  The attention is that of csa_sparse_attn_prefill (or
 * hca_dense_attn_decode) over the decoded entries, code * scale; on the GPU
 * each decoded value is rounded to bf16 (nearest even) before the tensor
 * cores use it.  The raw window rows stay bf16.
 *
 *   q        bf16 [B][T][H][128]; q_pos int32 [B][T] absolute positions
 *            (T = 1, q_pos = seq_len - 1 for decode).
 *   k_nope   E4M3 bytes [B][N_cap][64];  k_scale fp32 [B][N_cap];
 *   k_rope   bf16 [B][N_cap][64];
 *   v        E4M3 bytes [B][N_cap][128]; v_scale fp32 [B][N_cap]
 *            (all contiguous: entry e of sequence b is row b * N_cap + e).
 *   topk_idx int32 [B][T][k]: CSA, the selected entries (-1 = none).
 *            NULL: HCA, every visible entry 0 .. n_vis - 1 with
 *            n_vis = min(n_cmp[b], floor((q_pos + 1) / m_prime)).
 *   k_raw, v_raw, raw_bstride, raw_cap, window, sink, softmax_scale, out,
 *   lse, ws, ws_bytes: as csa_sparse_attn_prefill (workspace sized by
 *   csa_attn_workspace(B, T, H, k + window), or N_cap + window for HCA).
 *   H <= 64, D == 128, else CSA_ERR_UNSUPPORTED; other statuses as the
 *   bf16 calls.
 * ---------------------------------------------------------------------- */
CSA_API int csa_attn_fp8kv(const void* q, const void* k_nope, const float* k_scale,
                           const void* k_rope, const void* v, const float* v_scale, int N_cap,
                           const int32_t* topk_idx, int k, const int32_t* n_cmp, int m_prime,
                           const void* k_raw, const void* v_raw, int64_t raw_bstride,
                           int64_t raw_cap, const int32_t* q_pos, int window, const float* sink,
                           float softmax_scale, int B, int T, int H, int D, void* out, float* lse,
                           void* ws, size_t ws_bytes, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * Grouped output projection after the MQA core attention.  The hyper.ai
 * DeepSeek-V4 page (Method, CSA paragraph) follows the core attention with
 * "a grouped output projection"; read as: the H heads of a query's output are
 * split into G groups of H/G consecutive heads, and group g's K = (H/G) * D
 * values are projected by its own matrix W_g:
 *     y[q][g*d_g + r] = sum_{j < K} W[g][r][j] * o[q][g*K + j]
 * fp32 accumulation, bf16 output (nearest even).
 *
 *   o    bf16 [n][H][D] (the attention output, contiguous);
 *   W    bf16 [G][d_g][K] (row = output channel), caller-owned weights;
 *   y    bf16 [n][G * d_g] out.
 *   H % G == 0; K a multiple of 64; d_g a multiple of 128; all three
 *   pointers 16-byte aligned.  Status as the other calls (1 invalid
 *   argument, 2 unsupported shape, 4 CUDA); timeouts of the kernel's bounded
 *   waits set CSA_EW_TIMEOUT in err_word.
 * ---------------------------------------------------------------------- */
CSA_API int csa_grouped_out_proj(const void* o, const void* W, void* y, int n, int H, int D,
                                 int G, int d_g, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * a3, without caller scratch.  An integration variant: the DeepSeek-V4 pages
 * have no counterpart to it; it computes exactly what csa_indexer_topk does.
 *
 * For callers that cannot allocate device memory at the point of the call:
 * a decode loop that reserved its HBM up front and must not call the device
 * allocator (which can synchronise the device) inside the step, or a host
 * runtime that has no device allocator of its own to hand out scratch.  The
 * scratch is a fixed array of CSA_INDEXER_STATIC_SCRATCH_BYTES in the
 * library's own device memory (one per device), so the call allocates
 * nothing: no cudaMalloc / cudaFree, no allocating library routine.
 *
 * Arguments, layouts, ownership and results are those of csa_indexer_topk,
 * without ws / ws_bytes.
 *   Limit: csa_indexer_topk_workspace(B, T, N_cap, k) must not exceed
 *   CSA_INDEXER_STATIC_SCRATCH_BYTES (16 MiB).  The workspace is one fp32
 *   score per compressed entry for up to 256 queries at a time, so this covers
 *   any number of queries over 16384 entries, 32 queries over 131072, or 8 over
 *   524288; a larger problem returns CSA_ERR_WORKSPACE before anything runs.
 *   Statuses: the argument checks of csa_indexer_topk come first and give
 *   its statuses; the capacity check follows; both before any CUDA call.
 *   Set-up: the first call on a device (the device current on the calling
 *   thread) looks up the array's device address (cudaGetSymbolAddress) and
 *   caches it with the id of the current context; that lookup can load the
 *   library's kernels, so make the first call per device before any stream
 *   capture.  A device reset (cudaDeviceReset) creates a new context in which
 *   the array may sit elsewhere: the next call sees the new context id and
 *   looks the address up again (again outside any capture, then).  A failed
 *   lookup returns CSA_ERR_CUDA.
 *   Zeroing: nothing in the array has to start at zero; each call writes
 *   every score it later reads, before reading it, on `stream`.
 *   Overlap: all calls on one device share the one array.  Calls ordered on
 *   one stream are safe; two calls that can run at the same time (different
 *   streams without an event between them, or several host threads) race on
 *   the scratch and give undefined results.
 * ---------------------------------------------------------------------- */
#define CSA_INDEXER_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
CSA_API int csa_indexer_topk_static(const void* q_idx, const float* q_scale, const float* w,
                                    const void* k_idx, int64_t k_bstride, const float* k_scale,
                                    int64_t ks_bstride, int idx_dtype, const int32_t* q_pos,
                                    const int32_t* n_cmp, int B, int T, int H_I, int d_I,
                                    int N_cap, int m, int k, int32_t* topk_idx,
                                    float* topk_score, int32_t* err_word, void* stream);

/* ------------------------------------------------------------------------
 * Self-test of the bounded device waits.  Not part of the method (the pages
 * have no counterpart): every pipelined kernel of this library waits on its
 * mbarriers with an iteration limit and, when a wait gives up, sets
 * CSA_EW_TIMEOUT in err_word and returns instead of hanging.  This call runs
 * that same wait on a barrier in a one-thread kernel with nothing else in
 * flight (no bulk copy, MMA or tensor memory), so a caller can check the
 * give-up path on its GPU without faulting or hanging it.
 *
 *   arrive    0: nobody arrives at the barrier, the wait gives up after
 *             `limit` polls and CSA_EW_TIMEOUT is ORed into *err_word;
 *             nonzero: the one expected arrival comes first, the wait returns
 *             at once and *err_word is left as it was.
 *   limit     polls before giving up, 1 .. 2^20 (each poll blocks for a
 *             bounded, hardware-defined time, so the kernel ends within
 *             milliseconds).
 *   err_word  device int32, 4-byte aligned, required; read it after the
 *             stream has reached the call.
 * Status: 0 launched, 1 bad argument (nothing launched), 4 launch failed.
 * The kernel leaves the device usable: later calls of the library run
 * normally.
 * ---------------------------------------------------------------------- */
CSA_API int csa_selftest_bounded_wait(int arrive, uint32_t limit, int32_t* err_word,
                                      void* stream);

/* ------------------------------------------------------------------------
 * Feed probes (measurement only: nothing of the method).  They time the two
 * ways the hot path reads memory, for the rooflines the kernels are judged
 * against: a contiguous stream read once (the indexer keys) and 512-byte row
 * gathers into shared memory (the attention's top-k K/V rows).
 *
 * csa_probe_stream_read: 148 * ctas_per_sm CTAs (1..4) of 512 threads each
 *   read an equal contiguous share of src with 16-byte loads, in_flight
 *   (1, 4 or 8) loads per thread issued before any is used.  src: device,
 *   16-byte aligned, `bytes` readable (the remainder below one vector per
 *   CTA is not read).  sink: device float, written only if the XOR of all
 *   data read equals a fixed constant (it is there so that the loads stay).
 * csa_probe_row_gather: n_ctas CTAs; CTA c reads `stages` (1..64) stages
 *   of 64 rows of 512 bytes, row r of stage s at index
 *   idx[(c * stages + s) * 64 + r] of the table (n_rows < 2^31 rows;
 *   indices are clamped into [0, n_rows)), into a ring of `ring` (2, 4 or
 *   6) stages of 32 KB of shared memory.  Each CTA first copies its
 *   stages * 64 indices into shared memory, so no copy waits on an index
 *   load.  mode 0: 16-byte cp.async copies by each of 256 threads and a
 *   block barrier per stage; mode 2: the same with 512 threads; mode 1: TMA
 *   tile::gather4 (four 128-byte pieces of four rows per instruction, 128-
 *   byte swizzled; each 512-byte row read as 4 x 128 bytes) issued by one
 *   warp of 256 threads, with a full and an empty mbarrier per ring slot
 *   (bounded waits: sink = 2 if one gave up); mode 3: the same issued by
 *   four warps; mode 4: by eight warps (384 threads).  table: device,
 *   16-byte aligned; idx: device int32,
 *   n_ctas * stages * 64 entries; sink as above.
 * Both return CSA_OK, CSA_ERR_INVALID_ARG (checked before any launch) or
 * CSA_ERR_CUDA; they are asynchronous on `stream`.
 * ---------------------------------------------------------------------- */
CSA_API int csa_probe_stream_read(const void* src, int64_t bytes, int ctas_per_sm, int in_flight,
                                  float* sink, void* stream);
CSA_API int csa_probe_row_gather(const void* table, int64_t n_rows, const int32_t* idx, int n_ctas,
                                 int stages, int ring, int mode, float* sink, void* stream);

/* ------------------------------------------------------------------------
 * a4 / a5 / a6. Attention over compressed entries + window + sink.
 *
 * Sources: hyper.ai DeepSeek-V4 page, Method (MQA core attention with shared
 * keys and values over the top-k entries; HCA dense over all entries; both
 * with a sliding-window branch); aiboss88 page, Technical Principles
 * (sliding window and attention sink); elamur.ai page, References [20]
 * (flash-decoding: split the keys, merge partial results by log-sum-exp).
 * For query token t of sequence b and head h, over the key set
 *     S = {compressed rows selected for t} u {raw rows max(0,t-window+1)..t}
 *     l_j = softmax_scale * q_h . K_j,  M = max(max_j l_j, sink_h)
 *     Z   = exp(sink_h - M) + sum_j exp(l_j - M)
 *     out_h = sum_j exp(l_j - M) V_j / Z,   lse_h = M + ln Z
 * (no sink term when sink == NULL; empty S without sink gives out = 0,
 * lse = -inf).  K and V are shared by all H heads (MQA).  They may alias
 * (k_cmp == v_cmp, k_raw == v_raw).
 *
 *   q         bf16 [B][H][D] (decode) or [B][T][H][D] (prefill).
 *   k_cmp, v_cmp  bf16 [B][cmp_bstride], rows of D; N_cap rows per sequence;
 *             cmp_bstride a multiple of D (the caches are read as one 2-D
 *             array of 256-byte rows).
 *   k_raw, v_raw  bf16 [B][raw_bstride]: a ring of raw_cap rows per
 *             sequence, position p at row p mod raw_cap (raw_cap >= window;
 *             a cache at full length is the case raw_cap > every position);
 *             raw_bstride a multiple of D.
 *   seq_len   int32 [B] (decode: t = seq_len - 1, the token's own K/V is
 *             already in the raw cache); q_pos int32 [B][T] (prefill).
 *   out       bf16, same shape as q; lse fp32 [B][(T)][H] (optional).
 *   ws        optional: csa_attn_workspace(B, T, H, n_keys_max) bytes (16-byte
 *             aligned), where n_keys_max is the largest key-set size (k +
 *             window for CSA; the largest n_vis + window for HCA).  Without it
 *             (NULL, or fewer bytes) the key splits of a query run as one
 *             thread-block cluster and merge through distributed shared
 *             memory.  With it, when clusters that large cannot all be
 *             resident at once (few queries, many keys), the keys are split
 *             further without a cluster and the partial results merged by a
 *             second kernel through this buffer.  Either way the result is
 *             the same combination; a misaligned ws returns CSA_ERR_WORKSPACE.
 *   H in {16, 32, 64, 128}; D == 128.
 * ---------------------------------------------------------------------- */
CSA_API size_t csa_attn_workspace(int B, int T, int H, int n_keys_max);

/* CSA decode: one query token per sequence; compressed rows = topk_idx[b][.]
 * (entries < 0 are skipped). */
CSA_API int csa_sparse_attn_decode(const void* q, const void* k_cmp, const void* v_cmp,
                           int64_t cmp_bstride, int N_cap, const int32_t* topk_idx, int k,
                           const void* k_raw, const void* v_raw, int64_t raw_bstride,
                           int64_t raw_cap, const int32_t* seq_len, int window,
                           const float* sink, float softmax_scale, int B, int H, int D,
                           void* out, float* lse, void* ws, size_t ws_bytes, int32_t* err_word,
                           void* stream);

/* CSA prefill: T query tokens per sequence at positions q_pos; compressed
 * rows = topk_idx[b][t][.]. */
CSA_API int csa_sparse_attn_prefill(const void* q, const void* k_cmp, const void* v_cmp,
                            int64_t cmp_bstride, int N_cap, const int32_t* topk_idx, int k,
                            const void* k_raw, const void* v_raw, int64_t raw_bstride,
                            int64_t raw_cap, const int32_t* q_pos, int window,
                            const float* sink, float softmax_scale, int B, int T, int H, int D,
                            void* out, float* lse, void* ws, size_t ws_bytes,
                            int32_t* err_word, void* stream);

/* HCA decode: compressed rows 0 .. n_vis-1 with
 * n_vis = min(n_cmp[b], floor(seq_len[b] / m_prime)). */
CSA_API int hca_dense_attn_decode(const void* q, const void* k_cmp, const void* v_cmp,
                          int64_t cmp_bstride, int N_cap, const int32_t* n_cmp, int m_prime,
                          const void* k_raw, const void* v_raw, int64_t raw_bstride,
                          int64_t raw_cap, const int32_t* seq_len, int window,
                          const float* sink, float softmax_scale, int B, int H, int D,
                          void* out, float* lse, void* ws, size_t ws_bytes, int32_t* err_word,
                          void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H_ */
