// Ordered cross-slice reduction and the fused epilogue.
//
// The stock reduce+Sinkhorn kernel of the hc_fused page sums the per-slice
// partials "in slice order" starting from zero and then runs the epilogue;
// this kernel does the same from the workspace partials
// part[(slice * 25 + j) * Mpad + row] (j < 24: mix, j = 24: sum of squares).
//
// Layout: 32 rows per CTA and one warp per output j (25 warps, one row per
// lane), so every load of a (slice, j) pair is 32 consecutive floats.  Each
// lane issues its slice loads in batches of 40 before adding them in slice
// order, so the L2 latency is paid per batch rather than per slice.  Warp 0
// then runs the epilogue, one row per lane.
#pragma once

#include "hcmix_common.cuh"

namespace hcmix {

constexpr int kReduceRows = 32;
constexpr int kReduceThreads = 32 * kPartStride;
constexpr int kReduceBatch = 40;

__global__ void __launch_bounds__(kReduceThreads)
hcmix_reduce_kernel(const float* __restrict__ part, int n_slices, int Mpad, int M, float inv_k,
                    const float* __restrict__ hc_scale, const float* __restrict__ hc_base,
                    int iters, float rms_eps, float hc_eps, float* __restrict__ pre,
                    float* __restrict__ post, float* __restrict__ comb,
                    float* __restrict__ mix_out, float* __restrict__ sq_out, int do_epilogue) {
  __shared__ float s_tot[kPartStride][kReduceRows + 1];
  const int lane = threadIdx.x & 31, out = threadIdx.x >> 5;  // out: mix index or 24 (sq)
  const int row = blockIdx.x * kReduceRows + lane;
  float t = 0.0f;
  if (row < M) {
    const float* p = part + (int64_t)out * Mpad + row;
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
  if (out != 0 || row >= M) return;
  float mixv[kMix];
#pragma unroll
  for (int j = 0; j < kMix; ++j) mixv[j] = s_tot[j][lane];
  const float sq = s_tot[kMix][lane];
  if (mix_out != nullptr) {
#pragma unroll
    for (int j = 0; j < kMix; ++j) mix_out[(int64_t)row * kMix + j] = mixv[j];
  }
  if (sq_out != nullptr) sq_out[row] = sq;
  if (do_epilogue) {
    epilogue_row(mixv, sq, inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps,
                 pre + (int64_t)row * kHc, post + (int64_t)row * kHc,
                 comb + (int64_t)row * kHc * kHc);
  }
}

// The epilogue alone from caller-provided mix[M, 24] and sq[M].
__global__ void __launch_bounds__(128)
hcmix_epilogue_kernel(const float* __restrict__ mix, const float* __restrict__ sq, int M,
                      float inv_k, const float* __restrict__ hc_scale,
                      const float* __restrict__ hc_base, int iters, float rms_eps, float hc_eps,
                      float* __restrict__ pre, float* __restrict__ post,
                      float* __restrict__ comb) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= M) return;
  float mixv[kMix];
#pragma unroll
  for (int j = 0; j < kMix; ++j) mixv[j] = mix[(int64_t)row * kMix + j];
  epilogue_row(mixv, sq[row], inv_k, hc_scale, hc_base, iters, rms_eps, hc_eps,
               pre + (int64_t)row * kHc, post + (int64_t)row * kHc,
               comb + (int64_t)row * kHc * kHc);
}

}  // namespace hcmix
