// Ordered cross-slice reduction and the fused epilogue.
//
// The stock reduce+Sinkhorn kernel of the hc_fused page sums the per-slice
// partials "in slice order" starting from zero and then runs the epilogue;
// this kernel does the same from the workspace partials
// part[(slice * 25 + j) * Mpad + row] (j < 24: mix, j = 24: sum of squares).
//
// Layout: 256 threads per CTA, 32 rows per CTA.  Warp w sums outputs
// j = w, w + 8, w + 16 (and warp 0 also j = 24) for the 32 rows, one row per
// lane, so every load of a (slice, j) pair is 32 consecutive floats.  Warp 0
// then runs the epilogue, one row per lane.
#pragma once

#include "hcmix_common.cuh"

namespace hcmix {

constexpr int kReduceRows = 32;
constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads)
hcmix_reduce_kernel(const float* __restrict__ part, int n_slices, int Mpad, int M, float inv_k,
                    const float* __restrict__ hc_scale, const float* __restrict__ hc_base,
                    int iters, float rms_eps, float hc_eps, float* __restrict__ pre,
                    float* __restrict__ post, float* __restrict__ comb,
                    float* __restrict__ mix_out, float* __restrict__ sq_out, int do_epilogue) {
  __shared__ float s_tot[kPartStride][kReduceRows + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = blockIdx.x * kReduceRows + lane;
  for (int j = warp; j < kPartStride; j += kReduceThreads / 32) {
    float t = 0.0f;
    if (row < M) {
      const float* p = part + (int64_t)j * Mpad + row;
      const int64_t step = (int64_t)kPartStride * Mpad;
#pragma unroll 8
      for (int s = 0; s < n_slices; ++s) t = __fadd_rn(t, p[s * step]);
    }
    s_tot[j][lane] = t;
  }
  __syncthreads();
  if (warp != 0 || row >= M) return;
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
