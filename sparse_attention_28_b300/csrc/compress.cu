// compress.cu -- block compression of raw KV / indexer-key rows.
//
// Method: hyper.ai DeepSeek-V4 page, Method -- CSA "compresses every m tokens
// into a single entry using learnable compression weights and positional
// biases"; HCA consolidates every m' tokens "without overlapping
// compression" (read as: CSA's blocks may overlap).  Operator (this
// library's reading of those sentences): block j (stride m) is compressed
// from the span >= m raw tokens ending at its last token, positions
// p_i = j*m + m - span + i (the non-negative ones); for channel c
//     g[i][c] = sum_e W[c][e] x[p_i][e] + pos_bias[i][c]
//     y[j][c] = sum_i softmax_i(g[.][c])[i] * x[p_i][c]
// span = m is the non-overlapping operator.  Output: bf16 (nearest even), or
// E4M3 with one fp32 scale per entry, scale = max_c |y| / 448 (1 if all
// zero), code = nearest-even E4M3 of y / scale, saturating.  Mixed storage
// (the same page keeps the RoPE channels of the KV entries in BF16 and the
// rest in FP8): channels below fp8_dims as E4M3 with the scale taken over
// them alone, the others bf16 into a second array.
//
// One CTA per (block, sequence), one thread per output channel.  The
// block's span raw rows (fp32) are staged in shared memory; each thread
// reads its own W row straight from global memory (all of it in flight at
// once: no other thread uses it) and forms its channel's gate logits 4
// positions at a time (x rows as shared-memory broadcasts), folded into an
// online softmax.
#include "common.cuh"
#include "kernels.h"

namespace csa {

namespace {

constexpr int kPosChunk = 4;  // positions whose gate logits are formed together

template <int D>
__global__ void __launch_bounds__(D) compress_kernel(CompressArgs a) {
  // The reads below (raw rows, W, position biases) touch only what no kernel
  // of this library writes, so they are issued before griddepcontrol.wait and
  // all at once (one memory latency for the kernel, not one per position);
  // the output is written after the wait.
  pdl_trigger();
  extern __shared__ __align__(16) float xs[];  // [span][D]
  __shared__ float red[D / 32];
  const int c = threadIdx.x;
  const int b = blockIdx.y;
  const int64_t j = (int64_t)a.block_begin + blockIdx.x;
  const int m = a.m;
  // this channel's W row: D bf16 as D/8 16-byte vectors
  uint4 wrow[D / 8];
#pragma unroll
  for (int e8 = 0; e8 < D / 8; ++e8)
    wrow[e8] = __ldg(reinterpret_cast<const uint4*>(a.W + (int64_t)c * D) + e8);
  const bf16* xb = a.raw + (int64_t)b * a.raw_bstride;
  // the span's tokens: bias row i belongs to position j*m + m - span + i; rows
  // of negative positions are left out (k counts the rows that remain)
  const int64_t p0 = j * m + m - a.span;
  const int i_off = p0 < 0 ? (int)(-p0) : 0;
  const int np = a.span - i_off;
  const int64_t r0 = (p0 + i_off) % a.raw_cap;  // ring row of the first token
  const float* bias = a.pos_bias + (int64_t)i_off * D;
  float bnext[kPosChunk];  // position biases of this channel for the next chunk
#pragma unroll
  for (int ii = 0; ii < kPosChunk; ++ii) bnext[ii] = ii < np ? __ldg(bias + (int64_t)ii * D + c) : 0.f;
  constexpr int kRowBatch = 8;  // raw rows in flight per thread
  for (int k0 = 0; k0 < np; k0 += kRowBatch) {
    bf16 xr[kRowBatch];
#pragma unroll
    for (int kk = 0; kk < kRowBatch; ++kk) {
      int64_t r = r0 + k0 + kk;
      if (r >= a.raw_cap) r -= a.raw_cap;
      if (k0 + kk < np) xr[kk] = xb[r * D + c];
    }
#pragma unroll
    for (int kk = 0; kk < kRowBatch; ++kk)
      if (k0 + kk < np) xs[(k0 + kk) * D + c] = __bfloat162float(xr[kk]);
  }
  __syncthreads();

  float mx = -INFINITY, den = 0.f, num = 0.f;
  for (int i0 = 0; i0 < np; i0 += kPosChunk) {
    const int n = (np - i0 < kPosChunk) ? np - i0 : kPosChunk;
    float bv[kPosChunk];
#pragma unroll
    for (int ii = 0; ii < kPosChunk; ++ii) {  // this chunk's biases; the next chunk's requested
      bv[ii] = bnext[ii];
      const int in = i0 + kPosChunk + ii;
      bnext[ii] = in < np ? __ldg(bias + (int64_t)in * D + c) : 0.f;
    }
    float gl[kPosChunk];
#pragma unroll
    for (int ii = 0; ii < kPosChunk; ++ii) gl[ii] = 0.f;
#pragma unroll
    for (int e8 = 0; e8 < D / 8; ++e8) {
      const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wrow[e8]);
      float wf[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(w2[q]);
        wf[2 * q] = f.x;
        wf[2 * q + 1] = f.y;
      }
#pragma unroll
      for (int ii = 0; ii < kPosChunk; ++ii) {
        if (ii < n) {
          const float* xr = xs + (i0 + ii) * D + e8 * 8;
#pragma unroll
          for (int q = 0; q < 8; ++q) gl[ii] = fmaf(wf[q], xr[q], gl[ii]);
        }
      }
    }
#pragma unroll
    for (int ii = 0; ii < kPosChunk; ++ii) {
      if (ii < n) {
        const float gi = gl[ii] + bv[ii];
        const float xv = xs[(i0 + ii) * D + c];
        if (gi > mx) {
          const float r = expf(mx - gi);
          den = den * r + 1.f;
          num = num * r + xv;
          mx = gi;
        } else {
          const float p = expf(gi - mx);
          den += p;
          num += p * xv;
        }
      }
    }
  }
  const float y = num / den;
  pdl_wait();  // outputs only from here on

  if (a.fp4) {
    // FP4: per 16 channels one E4M3 scale, the nearest to amax / 6 (1 if the
    // block is zero, at least the smallest positive E4M3 value), and E2M1
    // codes of y / scale, two per byte
    float am = fabsf(y);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
    uint32_t sc = am > 0.f ? (uint32_t)__nv_cvt_float_to_fp8(am / 6.f, __NV_SATFINITE, __NV_E4M3)
                           : 0x38u;  // E4M3 1.0
    float scv = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sc, __NV_E4M3)));
    if (scv == 0.f) {
      sc = 1u;  // 2^-9
      scv = __half2float(__half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)1, __NV_E4M3)));
    }
    const uint32_t q = (uint32_t)__nv_cvt_float_to_fp4(y / scv, __NV_E2M1, cudaRoundNearest) & 0xFu;
    const uint32_t q1 = __shfl_down_sync(0xFFFFFFFFu, q, 1);
    uint8_t* out = reinterpret_cast<uint8_t*>(a.out) + (int64_t)b * (a.out_bstride / 2) + j * (D / 2);
    if ((c & 1) == 0) out[c >> 1] = static_cast<uint8_t>(q | (q1 << 4));
    if ((c & 15) == 0)
      reinterpret_cast<uint8_t*>(a.out_scale)[((int64_t)b * a.scale_bstride + j) * (D / 16) +
                                              (c >> 4)] = static_cast<uint8_t>(sc);
    return;
  }
  if (!a.fp8) {
    bf16* out = reinterpret_cast<bf16*>(a.out) + (int64_t)b * a.out_bstride + j * D;
    out[c] = __float2bfloat16_rn(y);
    return;
  }
  // E4M3 with a per-entry scale (channels below dl; mixed storage: the rest bf16)
  const int dl = (a.fp8_dims > 0 && a.fp8_dims < D) ? a.fp8_dims : D;
  float am = c < dl ? fabsf(y) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
  if ((c & 31) == 0) red[c >> 5] = am;
  __syncthreads();
  float amax = 0.f;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  if (c < dl) {
    uint8_t* out = reinterpret_cast<uint8_t*>(a.out) + (int64_t)b * a.out_bstride + j * dl;
    out[c] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(y / scale, __NV_SATFINITE, __NV_E4M3));
  } else {
    bf16* hi = a.out_hi + (int64_t)b * a.out_hi_bstride + j * (D - dl);
    hi[c - dl] = __float2bfloat16_rn(y);
  }
  if (c == 0) a.out_scale[(int64_t)b * a.scale_bstride + j] = scale;
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, cudaStream_t st) {
  if (a.n_blocks == 0 || a.B == 0) return cudaSuccess;
  dim3 grid(a.n_blocks, a.B);
  cudaError_t e;
  if (a.d == 128) {
    e = ensure_smem_attr((const void*)compress_kernel<128>, 256 * 128 * 4);
    if (e != cudaSuccess) return e;
    e = launch_pdl(compress_kernel<128>, grid, dim3(128), a.span * 128 * 4, st, a);
  } else {
    e = ensure_smem_attr((const void*)compress_kernel<64>, 256 * 64 * 4);
    if (e != cudaSuccess) return e;
    e = launch_pdl(compress_kernel<64>, grid, dim3(64), a.span * 64 * 4, st, a);
  }
  return e;
}

}  // namespace csa
