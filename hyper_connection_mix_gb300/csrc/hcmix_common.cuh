// Shared device helpers for the hyper-connection mix-statistics kernels.
//
// Numerics (hc_fused page, module docstring, bullets 1 and 3): every 64-wide
// chunk dot d is produced as fp32 and then added into a slice total that starts
// from zero; slice totals are added into the grand total in slice order.  The
// kernels produce d as the exact chunk dot rounded once to fp32, computed as
//
//   d = fl32(top + rest),  top  = sum_k x0[k] * w0[k]           (exact in fp32)
//                          rest = sum_k (x - x0)[k] * W[k] + x0[k] * (W - w0)[k]
//
// where x0 is x rounded to the grid 2^(ex-7) (ex = exponent of the chunk's
// largest |x| in this row) and w0 is W rounded to the grid 2^(ew-7) (ew = the
// exponent of the chunk's largest |W| in this output).  Both have at most 8
// significant bits and share a grid, so every partial sum of x0*w0 over 64
// terms is a multiple of 2^(ex+ew-14) below 2^(ex+ew+8): it fits the 24-bit
// fp32 significand and no fp32 accumulator (FFMA or tensor core) rounds it.
// rest is ~2^-8 of top, so its own rounding sits ~2^-8 ulp below d's last bit
// and d equals the correctly rounded chunk dot except in rare near-tie cases.
#pragma once

#include <cstdint>

namespace hcmix {

constexpr int kChunk = 64;
constexpr int kSlice = 256;
constexpr int kChunksPerSlice = kSlice / kChunk;
constexpr int kMix = 24;
constexpr int kHc = 4;
constexpr int kPartStride = kMix + 1;  // 24 mix partials + 1 sum-of-squares partial

// Device error codes written to the workspace error word (first write wins).
enum DeviceError : uint32_t {
  kDevOk = 0,
  kDevWaitTimeout = 1,
  kDevBadState = 2,
};

__device__ __forceinline__ void record_device_error(uint32_t* err, uint32_t code) {
  if (err != nullptr) atomicCAS(err, 0u, code);
}

// Magic constant 1.5 * 2^(e - 7 + 23) for the largest-magnitude bit pattern
// `absbits_exp_field` (the biased exponent field of the largest |value|, 0..255).
// (v + magic) - magic rounds v to a multiple of 2^(e - 7).  Returns 0 (no split)
// when the magic constant would not be a finite normal number.
__device__ __forceinline__ float grid_magic_from_exp_field(uint32_t field) {
  uint32_t f = field < 1u ? 1u : field;
  if (f > 238u) return 0.0f;
  return __uint_as_float(((f + 16u) << 23) | 0x00400000u);
}

__device__ __forceinline__ float grid_round(float v, float magic) {
  return __fsub_rn(__fadd_rn(v, magic), magic);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Largest |bf16| exponent field over 32 packed words (64 values).
__device__ __forceinline__ uint32_t bf16x64_max_exp_field(const uint32_t (&w)[32]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    uint32_t a = w[i] & 0x7fff7fffu;
    uint32_t lo = a & 0xffffu, hi = a >> 16;
    m = max(m, max(lo, hi));
  }
  return m >> 7;
}

// The page's fixed sum-of-squares tree over one 64-column chunk held as 32
// packed bf16 words (word i = columns 2i, 2i+1): combine columns differing in
// bit 4, then bits 3, 2, 1, 0, then the two 32-column halves (_sq_tree).
__device__ __forceinline__ float sq_tree64(const uint32_t (&w)[32]) {
  float v[64];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = bf16_lo(w[i]), b = bf16_hi(w[i]);
    v[2 * i] = __fmul_rn(a, a);
    v[2 * i + 1] = __fmul_rn(b, b);
  }
#pragma unroll
  for (int i = 0; i < 64; ++i)
    if ((i & 16) == 0) v[i] = __fadd_rn(v[i], v[i | 16]);
#pragma unroll
  for (int i = 0; i < 64; ++i)
    if ((i & 24) == 0) v[i] = __fadd_rn(v[i], v[i | 8]);
#pragma unroll
  for (int i = 0; i < 64; ++i)
    if ((i & 28) == 0) v[i] = __fadd_rn(v[i], v[i | 4]);
#pragma unroll
  for (int i = 0; i < 64; ++i)
    if ((i & 30) == 0) v[i] = __fadd_rn(v[i], v[i | 2]);
#pragma unroll
  for (int i = 0; i < 64; ++i)
    if ((i & 31) == 0) v[i] = __fadd_rn(v[i], v[i | 1]);
  return __fadd_rn(v[0], v[32]);
}

}  // namespace hcmix
