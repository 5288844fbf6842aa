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
// first 32 threads then run the epilogue, one row each.
#pragma once

#include "hcmix_common.cuh"

namespace hcmix {

constexpr int kReduceRows = 32;
constexpr int kReduceThreads = 32 * kPartStride;
constexpr int kReduceBatch = 40;

// 1 / s for a Sinkhorn normalisation, by which the row's (column's) four
// entries are then multiplied: the approximate reciprocal (within 1 ulp over
// the whole range, subnormal s included, since the non-.ftz form keeps
// subnormals; with the product, each entry is within 2 ulp of c / s, and the
// iteration's own contraction keeps the result within a few ulp of the
// correctly rounded sequence).  No branch: a data-dependent branch around a
// division here made each Sinkhorn round ~10x slower.
__device__ __forceinline__ float sinkhorn_rcp(float s) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// The epilogue of one row, by one thread, from the row's totals (s_tot[j][r]:
// j < 24 mix, j = 24 sum of squares): r = 1/sqrt(sq (1/K) + rms_eps); logit
// j = mix_j r scale[g(j)] + base_j; pre = sigmoid, post = 2 sigmoid;
// Sinkhorn on exp of the 16 comb logits, rows then columns, sums in index
// order.  The row and column reciprocals of a normalisation are taken once
// (sinkhorn_rcp) and multiplied in.  Rows at or past
// row_end are not written.
__device__ __forceinline__ void epilogue_row(const float (&s_tot)[kPartStride][kReduceRows + 1],
                                             int r, int row, int row_end, float inv_k,
                                             const float* __restrict__ hc_scale,
                                             const float* __restrict__ hc_base, int iters,
                                             float rms_eps, float hc_eps,
                                             float* __restrict__ pre, float* __restrict__ post,
                                             float* __restrict__ comb) {
  const float v = __fadd_rn(__fmul_rn(s_tot[kMix][r], inv_k), rms_eps);
  const float rr = __fdiv_rn(1.0f, __fsqrt_rn(v));
  float pp[2 * kHc];
#pragma unroll
  for (int e = 0; e < 2 * kHc; ++e) {
    const float sc = e < kHc ? hc_scale[0] : hc_scale[1];
    const float lg = __fadd_rn(__fmul_rn(__fmul_rn(s_tot[e][r], rr), sc), hc_base[e]);
    pp[e] = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-lg)));
  }
  float c[kHc][kHc];
#pragma unroll
  for (int i = 0; i < kHc; ++i)
#pragma unroll
    for (int jj = 0; jj < kHc; ++jj) {
      const int e = 2 * kHc + kHc * i + jj;
      c[i][jj] = expf(__fadd_rn(__fmul_rn(__fmul_rn(s_tot[e][r], rr), hc_scale[2]), hc_base[e]));
    }
  // every sum is of positive values, so s + 0 = s: the eps add is skipped at 0
  const bool add_eps = hc_eps != 0.0f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kHc; ++i) {
      float s = __fadd_rn(__fadd_rn(__fadd_rn(c[i][0], c[i][1]), c[i][2]), c[i][3]);
      if (add_eps) s = __fadd_rn(s, hc_eps);
      const float rs = sinkhorn_rcp(s);
#pragma unroll
      for (int jj = 0; jj < kHc; ++jj) c[i][jj] = __fmul_rn(c[i][jj], rs);
    }
#pragma unroll
    for (int jj = 0; jj < kHc; ++jj) {
      float s = __fadd_rn(__fadd_rn(__fadd_rn(c[0][jj], c[1][jj]), c[2][jj]), c[3][jj]);
      if (add_eps) s = __fadd_rn(s, hc_eps);
      const float rs = sinkhorn_rcp(s);
#pragma unroll
      for (int i = 0; i < kHc; ++i) c[i][jj] = __fmul_rn(c[i][jj], rs);
    }
  }
  if (row >= row_end) return;
#pragma unroll
  for (int e = 0; e < kHc; ++e) {
    pre[(int64_t)row * kHc + e] = pp[e];
    post[(int64_t)row * kHc + e] = __fmul_rn(2.0f, pp[kHc + e]);
  }
#pragma unroll
  for (int i = 0; i < kHc; ++i)
#pragma unroll
    for (int jj = 0; jj < kHc; ++jj) comb[(int64_t)row * kHc * kHc + kHc * i + jj] = c[i][jj];
}

// The epilogue of the CTA's first nrows (<= 32) rows: one thread per row.
__device__ __forceinline__ void epilogue_rows(const float (&s_tot)[kPartStride][kReduceRows + 1],
                                              int row0, int nrows, int row_end, float inv_k,
                                              const float* __restrict__ hc_scale,
                                              const float* __restrict__ hc_base, int iters,
                                              float rms_eps, float hc_eps,
                                              float* __restrict__ pre, float* __restrict__ post,
                                              float* __restrict__ comb) {
  const int t = threadIdx.x;
  if (t < nrows)
    epilogue_row(s_tot, t, row0 + t, row_end, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps,
                 pre, post, comb);
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
  epilogue_rows(s_tot, row0, kReduceRows, M, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps, pre, post,
                comb);
}

// Small-M variant (decode batches): 2 rows per CTA and one warp per output j.
// All 32 lanes fetch the (row, j) values of the slices they own (slice s to
// lane s % 32), so every load of a CTA is in flight at once; the values are
// parked in shared memory and lane r of the warp then adds row r's slices in
// slice order from zero.  Then the same one-thread-per-row epilogue.
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
  epilogue_rows(s_tot, row0, kReduceSmallRows, M, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps,
                pre, post, comb);
}

// The epilogue alone from caller-provided mix[M, 24] and sq[M]: 32 rows per
// CTA staged in shared memory in the reduce kernel's layout, then the same
// one-thread-per-row epilogue.
constexpr int kEpilogueThreads = kReduceRows;

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
  epilogue_rows(s_tot, row0, kReduceRows, M, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps, pre, post,
                comb);
}

}  // namespace hcmix
