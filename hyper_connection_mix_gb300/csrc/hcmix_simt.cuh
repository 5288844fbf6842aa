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
// Per slice the CTA stages W[24, 256] and its rows of x in shared memory with
// cp.async and splits W per (output, chunk) into (W, w0, W - w0), the
// grid-aligned split described in hcmix_common.cuh; per chunk each thread
// splits its row's 64 x values into x0 / x - x0 and runs three FFMA chains per
// output:
//   top  += x0 * w0                     (exact)
//   rest += x0 * (W - w0); rest += (x - x0) * W
// and the chunk dot is fl32(top + rest).
#pragma once

#include "hcmix_common.cuh"

namespace hcmix {

constexpr int kSimtRows = 32;
constexpr int kSimtThreads = 128;
constexpr int kSimtWStride = kSlice + 4;  // floats per staged W row
constexpr int kSimtXStride = kSlice + 8;  // bf16 per staged x row (528 bytes)

// A whole slice is staged at once: W[24, 256] as (W, w0, W - w0) and the
// CTA's 32 rows of x, so a CTA waits for memory once per slice rather than
// once per chunk.  W rows are padded to 260 floats: the four output quarters
// of a warp then read four different banks (6 * 260 = 24 mod 32); x rows to
// 528 bytes, so the eight rows a warp reads at once fall in different banks.
struct SimtSmem {
  __align__(16) float w[kMix][kSimtWStride];
  __align__(16) float w0[kMix][kSimtWStride];
  __align__(16) float rw[kMix][kSimtWStride];
  __align__(16) uint16_t x[kSimtRows][kSimtXStride];
};
constexpr size_t kSimtSmemBytes = sizeof(SimtSmem);

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// One 256-column slice for the CTA's 32 rows starting at row0 (nrows of them
// exist): acc[jj] receives the slice total of output 6q + jj (chunk dots
// added in chunk order from zero) and, for q == 0, sqs the slice's sum of
// squares.  Every thread of the CTA calls it (it synchronises the CTA);
// threads of rows past the end compute nothing.
__device__ __forceinline__ void simt_slice(const uint16_t* __restrict__ x, int64_t x_stride,
                                           int row0, int nrows, const float* __restrict__ W,
                                           int64_t w_stride, int64_t k_slice, SimtSmem& sm,
                                           float (&acc)[6], float& sqs) {
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const int q = t & 3, rloc = t >> 2;
#pragma unroll
  for (int jj = 0; jj < 6; ++jj) acc[jj] = 0.0f;
  sqs = 0.0f;

  // every load of the slice in flight at once: W[24][256] and x[rows][256]
  for (int i = t; i < kMix * (kSlice / 4); i += kSimtThreads) {
    const int j = i / (kSlice / 4), v4 = i % (kSlice / 4);
    cp_async16(&sm.w[j][4 * v4], W + (int64_t)j * w_stride + k_slice + 4 * v4);
  }
  for (int i = t; i < nrows * (kSlice / 8); i += kSimtThreads) {
    const int r = i / (kSlice / 8), v8 = i % (kSlice / 8);
    cp_async16(&sm.x[r][8 * v8], x + (int64_t)(row0 + r) * x_stride + k_slice + 8 * v8);
  }
  cp_async_wait_all();
  __syncthreads();
  // grid split per (output, chunk): one warp per task, two columns per lane
  for (int task = warp; task < kMix * kChunksPerSlice; task += kSimtThreads / 32) {
    const int j = task / kChunksPerSlice, c0 = (task % kChunksPerSlice) * kChunk;
    const float a = sm.w[j][c0 + lane], b = sm.w[j][c0 + lane + 32];
    uint32_t m = max(__float_as_uint(a) & 0x7fffffffu, __float_as_uint(b) & 0x7fffffffu);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float magic = grid_magic_from_exp_field(m >> 23);
    const float a0 = grid_round(a, magic), b0 = grid_round(b, magic);
    sm.w0[j][c0 + lane] = a0;
    sm.w0[j][c0 + lane + 32] = b0;
    sm.rw[j][c0 + lane] = __fsub_rn(a, a0);
    sm.rw[j][c0 + lane + 32] = __fsub_rn(b, b0);
  }
  __syncthreads();

  if (rloc < nrows) {
    for (int c = 0; c < kChunksPerSlice; ++c) {
      const int c0 = c * kChunk;
      uint32_t xw[32];
      const uint4* src = reinterpret_cast<const uint4*>(&sm.x[rloc][c0]);
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
          const int k = c0 + 2 * i + h;
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
  }
  __syncthreads();  // the staged slice is overwritten by the next call
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
  extern __shared__ __align__(16) uint8_t simt_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(simt_raw);
  const int s = blockIdx.y;
  const int t = threadIdx.x;
  const int row0 = blockIdx.x * kSimtRows;
  const int nrows = min(kSimtRows, M - row0);
  const int row = row0 + (t >> 2);
  float acc[6], sqs;
  simt_slice(x, x_stride, row0, nrows, W, w_stride, (int64_t)s * kSlice, sm, acc, sqs);
  if (row < M) simt_store(part, s, Mpad, row, t & 3, acc, sqs);
}

__global__ void __launch_bounds__(kSimtThreads)
hcmix_simt_fullk_kernel(const uint16_t* __restrict__ x, int64_t x_stride,
                        const float* __restrict__ W, int64_t w_stride, int M, int Mpad,
                        int n_slices, float* __restrict__ part) {
  extern __shared__ __align__(16) uint8_t simt_raw[];
  SimtSmem& sm = *reinterpret_cast<SimtSmem*>(simt_raw);
  const int t = threadIdx.x;
  const int row0 = blockIdx.x * kSimtRows;
  const int nrows = min(kSimtRows, M - row0);
  const int row = row0 + (t >> 2);
  float tot[6], sqt = 0.0f;
#pragma unroll
  for (int jj = 0; jj < 6; ++jj) tot[jj] = 0.0f;
  for (int s = 0; s < n_slices; ++s) {
    float acc[6], sqs;
    simt_slice(x, x_stride, row0, nrows, W, w_stride, (int64_t)s * kSlice, sm, acc, sqs);
#pragma unroll
    for (int jj = 0; jj < 6; ++jj) tot[jj] = __fadd_rn(tot[jj], acc[jj]);
    sqt = __fadd_rn(sqt, sqs);
  }
  if (row < M) simt_store(part, 0, Mpad, row, t & 3, tot, sqt);
}

}  // namespace hcmix
