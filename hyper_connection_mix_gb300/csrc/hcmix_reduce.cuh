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

// Fast transcendentals of the epilogue.  Each is within a few ulp of the
// exact value, far inside the 1e-5 absolute tolerance of pre / post / comb
// (values of order 1); the GPU tests hold the results to that tolerance
// against the oracle.
//   * rcp_fast: the approximate reciprocal (max error 1 ulp; a subnormal
//     input flushes to zero and gives an infinity, which the callers exclude
//     or redo);
//   * exp_fast(x) = 2^(x log2 e), the product x log2 e carried to double
//     length (its rounding error e enters as the factor 1 + e ln 2), then the
//     approximate 2^t (max relative error 2^-22.5);
//   * rsqrt_fast: the approximate 1/sqrt (max relative error 2^-22.9).
__device__ __forceinline__ float rcp_fast(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}
__device__ __forceinline__ float exp_fast(float x) {
  constexpr float kLog2e = 1.44269502f, kLog2eLo = 1.92596299e-08f;  // log2 e = kLog2e + kLog2eLo
  constexpr float kLn2 = 0.693147182f;
  const float t = __fmul_rn(x, kLog2e);
  const float e = __fadd_rn(__fmaf_rn(x, kLog2e, -t), __fmul_rn(x, kLog2eLo));
  float p;
  asm("ex2.approx.f32 %0, %1;" : "=f"(p) : "f"(t));  // (subnormal results kept)
  return __fmul_rn(p, __fmaf_rn(e, kLn2, 1.0f));
}
__device__ __forceinline__ float rsqrt_fast(float v) {
  float r;
  asm("rsqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// Sinkhorn rounds (row normalisation, then column normalisation, sums in
// index order, the reciprocal of each sum multiplied in) on the comb matrix
// held as row-major pairs P[i][h] = (c[i][2h], c[i][2h+1]), so that the
// column sums and every scaling run on packed pairs.  With kEps, hc_eps is
// added to every sum (every sum is of non-negative values, so without it the
// sums are unchanged).  A sum below the normal range gives an infinite
// reciprocal, which leaves an infinity or NaN in the matrix: the caller checks
// for that and redoes the rounds with kDivide, which divides each entry by
// its sum (IEEE, as the oracle does) instead.
// The same rounds (hc_eps = 0) in scaling form: the matrix A = exp of the
// logits stays as it is and the rounds update a row scale u and a column
// scale v instead, u_i = 1 / sum_j A_ij v_j, then v_j = 1 / sum_i A_ij u_i;
// after the last round the result is A_ij u_i v_j.  In exact arithmetic this
// is the row-then-column normalisation above: after every step the
// normalised matrix is A_ij u_i v_j, and normalising its rows (columns) sets
// u (v) as written.  It leaves one reciprocal per sum and no per-entry
// scaling in the chain, so a round is ~10% shorter.  Each sum is formed in
// pairs, (A_i0 v_0 + A_i2 v_2) + (A_i1 v_1 + A_i3 v_3).  A scale that is not
// a positive finite number (a sum that overflowed, or reached 2^126, where the
// approximate reciprocal flushes to zero, or fell below the normal range)
// turns the result into NaN, so that the caller's check redoes the rounds
// with kDivide.
__device__ __forceinline__ void sinkhorn_rounds_scaled(float2 (&P)[kHc][kHc / 2], int iters) {
  static_assert(kHc == 4, "four-by-four comb");
  float u[kHc] = {1.0f, 1.0f, 1.0f, 1.0f};
  float2 v[kHc / 2] = {make_float2(1.0f, 1.0f), make_float2(1.0f, 1.0f)};
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kHc; ++i) {
      const float2 t = __ffma2_rn(P[i][1], v[1], __fmul2_rn(P[i][0], v[0]));
      u[i] = rcp_fast(__fadd_rn(t.x, t.y));
    }
#pragma unroll
    for (int h = 0; h < kHc / 2; ++h) {
      const float2 a = __ffma2_rn(P[1][h], make_float2(u[1], u[1]),
                                  __fmul2_rn(P[0][h], make_float2(u[0], u[0])));
      const float2 b = __ffma2_rn(P[3][h], make_float2(u[3], u[3]),
                                  __fmul2_rn(P[2][h], make_float2(u[2], u[2])));
      const float2 c = __fadd2_rn(a, b);
      v[h] = make_float2(rcp_fast(c.x), rcp_fast(c.y));
    }
  }
  if (iters > 0) {
    bool good = true;
#pragma unroll
    for (int i = 0; i < kHc; ++i) good = good && u[i] > 0.0f && u[i] <= 3.40282347e38f;
#pragma unroll
    for (int h = 0; h < kHc / 2; ++h)
      good = good && v[h].x > 0.0f && v[h].x <= 3.40282347e38f && v[h].y > 0.0f &&
             v[h].y <= 3.40282347e38f;
    if (!good) u[0] = __int_as_float(0x7fc00000);  // NaN: the caller redoes the rounds
#pragma unroll
    for (int i = 0; i < kHc; ++i)
#pragma unroll
      for (int h = 0; h < kHc / 2; ++h)
        P[i][h] = __fmul2_rn(__fmul2_rn(P[i][h], make_float2(u[i], u[i])), v[h]);
  }
}

template <bool kDivide, bool kEps>
__device__ __forceinline__ void sinkhorn_rounds(float2 (&P)[kHc][kHc / 2], int iters, float hc_eps) {
  static_assert(kHc == 4, "four-by-four comb");
  const float2 eps2 = make_float2(hc_eps, hc_eps);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kHc; ++i) {
      float s = __fadd_rn(__fadd_rn(__fadd_rn(P[i][0].x, P[i][0].y), P[i][1].x), P[i][1].y);
      if constexpr (kEps) s = __fadd_rn(s, hc_eps);
      if constexpr (kDivide) {
#pragma unroll
        for (int h = 0; h < kHc / 2; ++h)
          P[i][h] = make_float2(__fdiv_rn(P[i][h].x, s), __fdiv_rn(P[i][h].y, s));
      } else {
        const float rs = rcp_fast(s);
        const float2 rs2 = make_float2(rs, rs);
        P[i][0] = __fmul2_rn(P[i][0], rs2);
        P[i][1] = __fmul2_rn(P[i][1], rs2);
      }
    }
#pragma unroll
    for (int h = 0; h < kHc / 2; ++h) {
      float2 s = __fadd2_rn(__fadd2_rn(__fadd2_rn(P[0][h], P[1][h]), P[2][h]), P[3][h]);
      if constexpr (kEps) s = __fadd2_rn(s, eps2);
      if constexpr (kDivide) {
#pragma unroll
        for (int i = 0; i < kHc; ++i)
          P[i][h] = make_float2(__fdiv_rn(P[i][h].x, s.x), __fdiv_rn(P[i][h].y, s.y));
      } else {
        const float2 rs = make_float2(rcp_fast(s.x), rcp_fast(s.y));
#pragma unroll
        for (int i = 0; i < kHc; ++i) P[i][h] = __fmul2_rn(P[i][h], rs);
      }
    }
  }
}

// The epilogue of one row, from the row's totals (s_tot[j][r]: j < 24 mix,
// j = 24 sum of squares): r = 1/sqrt(sq (1/K) + rms_eps); logit j = mix_j r
// scale[g(j)] + base_j; pre = sigmoid, post = 2 sigmoid; Sinkhorn on exp of
// the 16 comb logits, rows then columns, sums in index order.  (hc_eps is
// added to every sum; the workloads use 0.)  Four consecutive lanes share a
// row: lane q computes pre q, post q and row q of exp(comb logits); lane 0
// gathers the 16 values and runs the rounds (a chain of dependent steps that
// does not split well).  Every lane of the warp calls this (the shuffles need
// them all); `active` is the same for the four lanes of a row, and rows at or
// past row_end are not written.
__device__ __forceinline__ void epilogue_row4(const float (&s_tot)[kPartStride][kReduceRows + 1],
                                              int r, bool active, int row, int row_end, float inv_k,
                                              const float* __restrict__ hc_scale,
                                              const float* __restrict__ hc_base, int iters,
                                              float rms_eps, float hc_eps,
                                              float* __restrict__ pre, float* __restrict__ post,
                                              float* __restrict__ comb) {
  const int q = threadIdx.x & 3, base = (threadIdx.x & 31) & ~3;
  const int rr_row = active ? r : 0;
  const float v = __fadd_rn(__fmul_rn(s_tot[kMix][rr_row], inv_k), rms_eps);
  const float rr = rsqrt_fast(v);
  auto logit = [&](int e, float sc) {
    return __fadd_rn(__fmul_rn(__fmul_rn(s_tot[e][rr_row], rr), sc), hc_base[e]);
  };
  const float p_pre = rcp_fast(__fadd_rn(1.0f, exp_fast(-logit(q, hc_scale[0]))));  // (>= 1: no subnormal)
  const float p_post = rcp_fast(__fadd_rn(1.0f, exp_fast(-logit(kHc + q, hc_scale[1]))));
  float c[kHc];  // row q of the comb matrix
#pragma unroll
  for (int jj = 0; jj < kHc; ++jj) c[jj] = exp_fast(logit(2 * kHc + kHc * q + jj, hc_scale[2]));
  float2 P[kHc][kHc / 2];  // P[i][h] = (c[i][2h], c[i][2h+1]), gathered on lane q == 0
#pragma unroll
  for (int i = 0; i < kHc; ++i)
#pragma unroll
    for (int h = 0; h < kHc / 2; ++h)
      P[i][h] = make_float2(__shfl_sync(0xffffffffu, c[2 * h], base + i),
                            __shfl_sync(0xffffffffu, c[2 * h + 1], base + i));
  const bool write = active && row < row_end;
  if (write) {
    pre[(int64_t)row * kHc + q] = p_pre;
    post[(int64_t)row * kHc + q] = __fmul_rn(2.0f, p_post);
  }
  if (q != 0 || !active) return;
  if (hc_eps != 0.0f)
    sinkhorn_rounds<false, true>(P, iters, hc_eps);
  else
    sinkhorn_rounds_scaled(P, iters);
  float check = 0.0f;
#pragma unroll
  for (int i = 0; i < kHc; ++i) check += (P[i][0].x + P[i][0].y) + (P[i][1].x + P[i][1].y);
  if (!isfinite(check)) {
    // a sum fell below the normal range (or the inputs hold an infinity or
    // NaN): again from exp of the logits, dividing by the sums
#pragma unroll
    for (int i = 0; i < kHc; ++i)
#pragma unroll
      for (int h = 0; h < kHc / 2; ++h)
        P[i][h] = make_float2(exp_fast(logit(2 * kHc + kHc * i + 2 * h, hc_scale[2])),
                              exp_fast(logit(2 * kHc + kHc * i + 2 * h + 1, hc_scale[2])));
    sinkhorn_rounds<true, true>(P, iters, hc_eps);
  }
  if (!write) return;
#pragma unroll
  for (int i = 0; i < kHc; ++i)
#pragma unroll
    for (int h = 0; h < kHc / 2; ++h) {
      comb[(int64_t)row * kHc * kHc + kHc * i + 2 * h] = P[i][h].x;
      comb[(int64_t)row * kHc * kHc + kHc * i + 2 * h + 1] = P[i][h].y;
    }
}

// The epilogue of the CTA's first nrows (<= 32) rows: four lanes per row, the
// first 4 * 32 threads (every lane of those warps takes part).
constexpr int kEpilogueLanes = 4 * kReduceRows;
__device__ __forceinline__ void epilogue_rows(const float (&s_tot)[kPartStride][kReduceRows + 1],
                                              int row0, int nrows, int row_end, float inv_k,
                                              const float* __restrict__ hc_scale,
                                              const float* __restrict__ hc_base, int iters,
                                              float rms_eps, float hc_eps,
                                              float* __restrict__ pre, float* __restrict__ post,
                                              float* __restrict__ comb) {
  const int t = threadIdx.x;
  if (t < kEpilogueLanes)
    epilogue_row4(s_tot, t >> 2, (t >> 2) < nrows, row0 + (t >> 2), row_end, inv_k, hc_scale,
                  hc_base, iters, rms_eps, hc_eps, pre, post, comb);
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
constexpr int kEpilogueThreads = kEpilogueLanes;

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
