// CUDA-core split-K contraction: one CTA per (32-row block, 256-column slice).
//
// It realises the stock engine's split-K layout from the hc_fused page
// (docstring: "80 K slices of 256, one CTA per slice and row block, every
// slice's [rows, 24] partial written to memory"): each CTA writes its slice's
// per-row totals (24 mix values and the sum of squares) to the workspace, and
// hcmix_reduce_kernel adds the slices in slice order.  It serves the
// small-M regime, where the W read (1.97 MB) and launch latency dominate and a
// 128-row tensor-core tile would be mostly empty.
//
// Thread layout: 128 threads = 32 rows x 4 output quarters (6 outputs each).
// Per chunk the CTA stages W[24, 64] in shared memory as (W, w0, W - w0), the
// grid-aligned split described in hcmix_common.cuh; each thread splits its
// row's 64 x values into x0 / x - x0 and runs three FFMA chains per output:
//   top  += x0 * w0                     (exact)
//   rest += x0 * (W - w0); rest += (x - x0) * W
// and the chunk dot is fl32(top + rest).
#pragma once

#include "hcmix_common.cuh"

namespace hcmix {

constexpr int kSimtRows = 32;
constexpr int kSimtThreads = 128;

__global__ void __launch_bounds__(kSimtThreads)
hcmix_simt_slice_kernel(const uint16_t* __restrict__ x, int64_t x_stride,
                        const float* __restrict__ W, int64_t w_stride, int M, int Mpad,
                        float* __restrict__ part) {
  // rows padded to 68 floats: the four output quarters of a warp then read
  // four different banks (6 * 68 = 408 = 24 mod 32)
  __shared__ __align__(16) float s_w[kMix][kChunk + 4];
  __shared__ float s_w0[kMix][kChunk + 4];
  __shared__ float s_rw[kMix][kChunk + 4];

  const int s = blockIdx.y;
  const int64_t k_slice = (int64_t)s * kSlice;
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int rloc = t >> 2, q = t & 3;
  const int row = blockIdx.x * kSimtRows + rloc;
  const bool active = row < M;
  const uint16_t* xr = x + (int64_t)(active ? row : 0) * x_stride + k_slice;

  float acc[6];
#pragma unroll
  for (int jj = 0; jj < 6; ++jj) acc[jj] = 0.0f;
  float sqs = 0.0f;

  for (int c = 0; c < kChunksPerSlice; ++c) {
    const int64_t k0 = k_slice + (int64_t)c * kChunk;
    // stage W[:, k0:k0+64]: 24 rows x 16 float4
    for (int i = t; i < kMix * (kChunk / 4); i += kSimtThreads) {
      const int j = i / (kChunk / 4), v4 = i % (kChunk / 4);
      const float4 v = *reinterpret_cast<const float4*>(W + (int64_t)j * w_stride + k0 + 4 * v4);
      *reinterpret_cast<float4*>(&s_w[j][4 * v4]) = v;
    }
    __syncthreads();
    // grid split per output row of the chunk: one warp per output
    for (int j = warp; j < kMix; j += kSimtThreads / 32) {
      const float a = s_w[j][lane], b = s_w[j][lane + 32];
      uint32_t m = max(__float_as_uint(a) & 0x7fffffffu, __float_as_uint(b) & 0x7fffffffu);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float magic = grid_magic_from_exp_field(m >> 23);
      const float a0 = grid_round(a, magic), b0 = grid_round(b, magic);
      s_w0[j][lane] = a0;
      s_w0[j][lane + 32] = b0;
      s_rw[j][lane] = __fsub_rn(a, a0);
      s_rw[j][lane + 32] = __fsub_rn(b, b0);
    }
    __syncthreads();

    if (active) {
      uint32_t xw[32];
      const uint4* src = reinterpret_cast<const uint4*>(xr + c * kChunk);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = src[i];
        xw[4 * i] = v.x; xw[4 * i + 1] = v.y; xw[4 * i + 2] = v.z; xw[4 * i + 3] = v.w;
      }
      const float xmagic = grid_magic_from_exp_field(bf16x64_max_exp_field(xw));
      float top[6], rest[6];
#pragma unroll
      for (int jj = 0; jj < 6; ++jj) { top[jj] = 0.0f; rest[jj] = 0.0f; }
#pragma unroll 4
      for (int i = 0; i < 32; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int k = 2 * i + h;
          const float xf = h ? bf16_hi(xw[i]) : bf16_lo(xw[i]);
          const float x0 = grid_round(xf, xmagic);
          const float x1 = __fsub_rn(xf, x0);
#pragma unroll
          for (int jj = 0; jj < 6; ++jj) {
            const int j = 6 * q + jj;
            top[jj] = __fmaf_rn(x0, s_w0[j][k], top[jj]);
            rest[jj] = __fmaf_rn(x0, s_rw[j][k], rest[jj]);
            rest[jj] = __fmaf_rn(x1, s_w[j][k], rest[jj]);
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < 6; ++jj) acc[jj] = __fadd_rn(acc[jj], __fadd_rn(top[jj], rest[jj]));
      if (q == 0) sqs = __fadd_rn(sqs, sq_tree64(xw));
    }
    __syncthreads();  // s_w* are rewritten for the next chunk
  }

  if (active) {
#pragma unroll
    for (int jj = 0; jj < 6; ++jj)
      part[((int64_t)s * kPartStride + 6 * q + jj) * Mpad + row] = acc[jj];
    if (q == 0) part[((int64_t)s * kPartStride + kMix) * Mpad + row] = sqs;
  }
}

}  // namespace hcmix
