// CUDA-core contraction kernels: the hc_fused page's two designs on the same
// per-chunk arithmetic.
//
// hcmix_simt_slice_kernel, one CTA per (32-row block, 256-column slice), is
// the stock engine's split-K layout described in the page's module docstring:
// every (slice, row block) pair has its own CTA, which stores that slice's
// per-row totals (24 mix values and the sum of squares) in the workspace, and
// hcmix_reduce_kernel then adds the slices in slice order.
//
// hcmix_simt_fullk_kernel, one CTA per 32-row block walking every slice, is
// the page's own fused design: a CTA covers the whole of K for its rows and
// carries a running total instead of storing per-slice partials.  It adds
// each slice total into that running total in slice order, starting from
// zero, and writes only the total, as the single "slice" that
// hcmix_reduce_kernel then turns into the epilogue (the page likewise hands
// its total to the stock reduce+Sinkhorn kernel as a one-slice input).  The
// addition order is the split-K path's, so both kernels give bit-identical
// statistics; they exist side by side as an A/B of the two designs on GB300.
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

struct SimtSmem {
  // rows padded to 68 floats: the four output quarters of a warp then read
  // four different banks (6 * 68 = 408 = 24 mod 32)
  __align__(16) float w[kMix][kChunk + 4];
  float w0[kMix][kChunk + 4];
  float rw[kMix][kChunk + 4];
};

// One 256-column slice for the CTA's 32 rows: acc[jj] receives the slice
// total of output 6q + jj (chunk dots added in chunk order from zero) and,
// for q == 0, sqs the slice's sum of squares.  Every thread of the CTA calls
// it (it synchronises the CTA); inactive rows compute nothing.
__device__ __forceinline__ void simt_slice(const uint16_t* __restrict__ xr, bool active,
                                           const float* __restrict__ W, int64_t w_stride,
                                           int64_t k_slice, SimtSmem& sm, float (&acc)[6],
                                           float& sqs) {
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int q = t & 3;
#pragma unroll
  for (int jj = 0; jj < 6; ++jj) acc[jj] = 0.0f;
  sqs = 0.0f;

  for (int c = 0; c < kChunksPerSlice; ++c) {
    const int64_t k0 = k_slice + (int64_t)c * kChunk;
    // stage W[:, k0:k0+64]: 24 rows x 16 float4
    for (int i = t; i < kMix * (kChunk / 4); i += kSimtThreads) {
      const int j = i / (kChunk / 4), v4 = i % (kChunk / 4);
      const float4 v = *reinterpret_cast<const float4*>(W + (int64_t)j * w_stride + k0 + 4 * v4);
      *reinterpret_cast<float4*>(&sm.w[j][4 * v4]) = v;
    }
    __syncthreads();
    // grid split per output row of the chunk: one warp per output
    for (int j = warp; j < kMix; j += kSimtThreads / 32) {
      const float a = sm.w[j][lane], b = sm.w[j][lane + 32];
      uint32_t m = max(__float_as_uint(a) & 0x7fffffffu, __float_as_uint(b) & 0x7fffffffu);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      const float magic = grid_magic_from_exp_field(m >> 23);
      const float a0 = grid_round(a, magic), b0 = grid_round(b, magic);
      sm.w0[j][lane] = a0;
      sm.w0[j][lane + 32] = b0;
      sm.rw[j][lane] = __fsub_rn(a, a0);
      sm.rw[j][lane + 32] = __fsub_rn(b, b0);
    }
    __syncthreads();

    if (active) {
      uint32_t xw[32];
      const uint4* src = reinterpret_cast<const uint4*>(xr + k0);
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
            top[jj] = __fmaf_rn(x0, sm.w0[j][k], top[jj]);
            rest[jj] = __fmaf_rn(x0, sm.rw[j][k], rest[jj]);
            rest[jj] = __fmaf_rn(x1, sm.w[j][k], rest[jj]);
          }
        }
      }
#pragma unroll
      for (int jj = 0; jj < 6; ++jj) acc[jj] = __fadd_rn(acc[jj], __fadd_rn(top[jj], rest[jj]));
      if (q == 0) sqs = __fadd_rn(sqs, sq_tree64(xw));
    }
    __syncthreads();  // the staged W is rewritten for the next chunk
  }
}

// Writes one row's 6 outputs (and, for q == 0, the sum of squares) into
// workspace slot `slot` of the partial layout part[(slot * 25 + j) * Mpad + row].
__device__ __forceinline__ void simt_store(float* __restrict__ part, int64_t slot, int Mpad,
                                           int row, int q, const float (&v)[6], float sqv) {
#pragma unroll
  for (int jj = 0; jj < 6; ++jj) part[(slot * kPartStride + 6 * q + jj) * Mpad + row] = v[jj];
  if (q == 0) part[(slot * kPartStride + kMix) * Mpad + row] = sqv;
}

__global__ void __launch_bounds__(kSimtThreads)
hcmix_simt_slice_kernel(const uint16_t* __restrict__ x, int64_t x_stride,
                        const float* __restrict__ W, int64_t w_stride, int M, int Mpad,
                        float* __restrict__ part) {
  __shared__ SimtSmem sm;
  const int s = blockIdx.y;
  const int t = threadIdx.x;
  const int row = blockIdx.x * kSimtRows + (t >> 2);
  const bool active = row < M;
  const uint16_t* xr = x + (int64_t)(active ? row : 0) * x_stride;
  float acc[6], sqs;
  simt_slice(xr, active, W, w_stride, (int64_t)s * kSlice, sm, acc, sqs);
  if (active) simt_store(part, s, Mpad, row, t & 3, acc, sqs);
}

__global__ void __launch_bounds__(kSimtThreads)
hcmix_simt_fullk_kernel(const uint16_t* __restrict__ x, int64_t x_stride,
                        const float* __restrict__ W, int64_t w_stride, int M, int Mpad,
                        int n_slices, float* __restrict__ part) {
  __shared__ SimtSmem sm;
  const int t = threadIdx.x;
  const int row = blockIdx.x * kSimtRows + (t >> 2);
  const bool active = row < M;
  const uint16_t* xr = x + (int64_t)(active ? row : 0) * x_stride;
  float tot[6], sqt = 0.0f;
#pragma unroll
  for (int jj = 0; jj < 6; ++jj) tot[jj] = 0.0f;
  for (int s = 0; s < n_slices; ++s) {
    float acc[6], sqs;
    simt_slice(xr, active, W, w_stride, (int64_t)s * kSlice, sm, acc, sqs);
#pragma unroll
    for (int jj = 0; jj < 6; ++jj) tot[jj] = __fadd_rn(tot[jj], acc[jj]);
    sqt = __fadd_rn(sqt, sqs);
  }
  if (active) simt_store(part, 0, Mpad, row, t & 3, tot, sqt);
}

}  // namespace hcmix
