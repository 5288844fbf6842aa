// Ordered cross-slice reduction and the fused epilogue.
//
// The stock reduce+Sinkhorn kernel of the hc_fused page sums the per-slice
// partials in slice order, starting from zero, and then runs the epilogue;
// this kernel does the same from the workspace partials
// part[(slice * 25 + j) * Mpad + row] (j < 24: mix, j = 24: sum of squares).
//
// Layout: 32 rows per CTA and one warp per output j (25 warps, one row per
// lane), so every load of a (slice, j) pair is 32 consecutive floats.  Each
// lane issues its slice loads in batches of 40 before adding them in slice
// order, so the L2 latency is paid per batch rather than per slice.  The
// first 512 threads then run the epilogue, 16 per row.
#pragma once

#include "hcmix_common.cuh"

namespace hcmix {

constexpr int kReduceRows = 32;
constexpr int kReduceThreads = 32 * kPartStride;
constexpr int kReduceBatch = 40;

// Epilogue of the CTA's 32 rows from their totals in shared memory
// (s_tot[j][r]: j < 24 mix, j = 24 sum of squares): 16 threads per row,
// thread e owns comb entry e = 4i + j and, for e < 8, logit e of pre (e < 4)
// or post.  Sinkhorn sums are gathered with shuffles and added in index
// order, as one thread per row would.  The CTA's first nrows rows are done
// (nrows <= 32 and nrows * 16 a multiple of 32, so that whole warps take
// part in the shuffles); threads nrows * 16 and up do nothing.
__device__ __forceinline__ void epilogue16(const float (&s_tot)[kPartStride][kReduceRows + 1],
                                           int row0, int nrows, int M, float inv_k,
                                           const float* __restrict__ hc_scale,
                                           const float* __restrict__ hc_base, int iters,
                                           float rms_eps, float hc_eps, float* __restrict__ pre,
                                           float* __restrict__ post, float* __restrict__ comb) {
  const int tid = threadIdx.x;
  if (tid >= nrows * kHc * kHc) return;
  const int rloc = tid >> 4, e = tid & 15;
  const int row = row0 + rloc;
  const int gbase = threadIdx.x & 16;  // first lane of this row's 16-lane group
  const float sq = s_tot[kMix][rloc];
  const float v = __fadd_rn(__fmul_rn(sq, inv_k), rms_eps);
  const float rr = __fdiv_rn(1.0f, __fsqrt_rn(v));
  if (e < 2 * kHc) {
    const float sc = e < kHc ? hc_scale[0] : hc_scale[1];
    const float lg = __fadd_rn(__fmul_rn(__fmul_rn(s_tot[e][rloc], rr), sc), hc_base[e]);
    const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-lg)));
    if (row < M) {
      if (e < kHc) pre[(int64_t)row * kHc + e] = sg;
      else post[(int64_t)row * kHc + (e - kHc)] = __fmul_rn(2.0f, sg);
    }
  }
  const float lgc = __fadd_rn(__fmul_rn(__fmul_rn(s_tot[2 * kHc + e][rloc], rr), hc_scale[2]),
                              hc_base[2 * kHc + e]);
  float c = expf(lgc);
  const int ci = e >> 2, cj = e & 3;
  for (int it = 0; it < iters; ++it) {
    float s = __shfl_sync(0xffffffffu, c, gbase + 4 * ci);
    s = __fadd_rn(s, __shfl_sync(0xffffffffu, c, gbase + 4 * ci + 1));
    s = __fadd_rn(s, __shfl_sync(0xffffffffu, c, gbase + 4 * ci + 2));
    s = __fadd_rn(s, __shfl_sync(0xffffffffu, c, gbase + 4 * ci + 3));
    c = __fdiv_rn(c, __fadd_rn(s, hc_eps));
    s = __shfl_sync(0xffffffffu, c, gbase + cj);
    s = __fadd_rn(s, __shfl_sync(0xffffffffu, c, gbase + 4 + cj));
    s = __fadd_rn(s, __shfl_sync(0xffffffffu, c, gbase + 8 + cj));
    s = __fadd_rn(s, __shfl_sync(0xffffffffu, c, gbase + 12 + cj));
    c = __fdiv_rn(c, __fadd_rn(s, hc_eps));
  }
  if (row < M) comb[(int64_t)row * kHc * kHc + e] = c;
}

__global__ void __launch_bounds__(kReduceThreads)
hcmix_reduce_kernel(const float* __restrict__ part, int n_slices, int Mpad, int M, float inv_k,
                    const float* __restrict__ hc_scale, const float* __restrict__ hc_base,
                    int iters, float rms_eps, float hc_eps, float* __restrict__ pre,
                    float* __restrict__ post, float* __restrict__ comb,
                    float* __restrict__ mix_out, float* __restrict__ sq_out, int do_epilogue) {
  __shared__ float s_tot[kPartStride][kReduceRows + 1];
  const int lane = threadIdx.x & 31, out = threadIdx.x >> 5;  // out: mix index or 24 (sq)
  const int lrow = blockIdx.x * kReduceRows + lane;
  float t = 0.0f;
  if (lrow < M) {
    const float* p = part + (int64_t)out * Mpad + lrow;
    const int64_t step = (int64_t)kPartStride * Mpad;
    int s = 0;
    for (; s + kReduceBatch <= n_slices; s += kReduceBatch) {
      float v[kReduceBatch];
#pragma unroll
      for (int q = 0; q < kReduceBatch; ++q) v[q] = __ldg(p + (int64_t)(s + q) * step);
#pragma unroll
      for (int q = 0; q < kReduceBatch; ++q) t = __fadd_rn(t, v[q]);
    }
    for (; s < n_slices; ++s) t = __fadd_rn(t, __ldg(p + (int64_t)s * step));
  }
  s_tot[out][lane] = t;
  __syncthreads();
  const int tid = threadIdx.x;
  const int row0 = blockIdx.x * kReduceRows;
  if (mix_out != nullptr && tid < kReduceRows * kMix) {
    const int r = tid / kMix, jj = tid % kMix;
    if (row0 + r < M) mix_out[(int64_t)(row0 + r) * kMix + jj] = s_tot[jj][r];
  }
  if (sq_out != nullptr && tid < kReduceRows && row0 + tid < M) sq_out[row0 + tid] = s_tot[kMix][tid];
  if (!do_epilogue) return;
  epilogue16(s_tot, row0, kReduceRows, M, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps, pre, post, comb);
}

// Small-M variant (decode batches): 2 rows per CTA and one warp per output j.
// All 32 lanes fetch the (row, j) values of the slices they own (slice s to
// lane s % 32), so every load of a CTA is in flight at once; the values are
// parked in shared memory and lane r of the warp then adds row r's slices in
// slice order from zero.  Then the same 16-threads-per-row epilogue.
constexpr int kReduceSmallRows = 2;
constexpr int kReduceSmallMaxSlices = 128;  // slices held in shared memory (K <= 32768)

__global__ void __launch_bounds__(kReduceThreads)
hcmix_reduce_small_kernel(const float* __restrict__ part, int n_slices, int Mpad, int M,
                          float inv_k, const float* __restrict__ hc_scale,
                          const float* __restrict__ hc_base, int iters, float rms_eps,
                          float hc_eps, float* __restrict__ pre, float* __restrict__ post,
                          float* __restrict__ comb, float* __restrict__ mix_out,
                          float* __restrict__ sq_out, int do_epilogue) {
  __shared__ float s_val[kPartStride][kReduceSmallRows][kReduceSmallMaxSlices];
  __shared__ float s_tot[kPartStride][kReduceRows + 1];
  const int lane = threadIdx.x & 31, out = threadIdx.x >> 5;  // out: mix index or 24 (sq)
  const int row0 = blockIdx.x * kReduceSmallRows;
  const int64_t step = (int64_t)kPartStride * Mpad;
#pragma unroll
  for (int r = 0; r < kReduceSmallRows; ++r) {
    if (row0 + r >= M) continue;
    const float* p = part + (int64_t)out * Mpad + row0 + r;
    float v[kReduceSmallMaxSlices / 32];
#pragma unroll
    for (int i = 0; i < kReduceSmallMaxSlices / 32; ++i) {
      const int sl = lane + 32 * i;
      v[i] = sl < n_slices ? __ldg(p + (int64_t)sl * step) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < kReduceSmallMaxSlices / 32; ++i) s_val[out][r][lane + 32 * i] = v[i];
  }
  __syncwarp();
  float t = 0.0f;
  if (lane < kReduceSmallRows && row0 + lane < M)
    for (int sl = 0; sl < n_slices; ++sl) t = __fadd_rn(t, s_val[out][lane][sl]);
  if (lane < kReduceSmallRows) s_tot[out][lane] = t;
  __syncthreads();
  const int tid = threadIdx.x;
  if (mix_out != nullptr && tid < kReduceSmallRows * kMix) {
    const int r = tid / kMix, jj = tid % kMix;
    if (row0 + r < M) mix_out[(int64_t)(row0 + r) * kMix + jj] = s_tot[jj][r];
  }
  if (sq_out != nullptr && tid < kReduceSmallRows && row0 + tid < M)
    sq_out[row0 + tid] = s_tot[kMix][tid];
  if (!do_epilogue) return;
  epilogue16(s_tot, row0, kReduceSmallRows, M, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps,
             pre, post, comb);
}

// The epilogue alone from caller-provided mix[M, 24] and sq[M]: 32 rows per
// CTA staged in shared memory in the reduce kernel's layout, then the same
// 16-threads-per-row epilogue.
constexpr int kEpilogueThreads = kReduceRows * kHc * kHc;

__global__ void __launch_bounds__(kEpilogueThreads)
hcmix_epilogue_kernel(const float* __restrict__ mix, const float* __restrict__ sq, int M,
                      float inv_k, const float* __restrict__ hc_scale,
                      const float* __restrict__ hc_base, int iters, float rms_eps, float hc_eps,
                      float* __restrict__ pre, float* __restrict__ post,
                      float* __restrict__ comb) {
  __shared__ float s_tot[kPartStride][kReduceRows + 1];
  const int row0 = blockIdx.x * kReduceRows;
  const int rows = min(kReduceRows, M - row0);
  for (int i = threadIdx.x; i < kReduceRows * kMix; i += kEpilogueThreads) {
    const int r = i / kMix, j = i % kMix;
    s_tot[j][r] = r < rows ? mix[(int64_t)(row0 + r) * kMix + j] : 0.0f;
  }
  if (threadIdx.x < kReduceRows)
    s_tot[kMix][threadIdx.x] = (int)threadIdx.x < rows ? sq[row0 + threadIdx.x] : 0.0f;
  __syncthreads();
  epilogue16(s_tot, row0, kReduceRows, M, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps, pre, post, comb);
}

}  // namespace hcmix
