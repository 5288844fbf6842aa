// Tensor-core (tcgen05) contraction path for sm_103a.
//
// Work: the rows are cut into 128-row tiles and K into 256-column slices (the
// hc_fused page's slice grid); a unit is one (tile, slice) pair, numbered
// slice-major.  Each CTA of a grid of min(#SMs, #units) takes a contiguous
// range of units, so its units mostly share one slice, and writes, for each
// unit, the slice totals of its 128 rows (24 mix values and the sum of
// squares) to the workspace partials; hcmix_reduce_kernel then adds the
// slices in slice order.
//
// Per 64-column chunk (see hcmix_common.cuh for the numerics):
//   * warp 0 (one thread) loads x with TMA, two chunks of a tile (32 KB) per
//     load, into a 3-stage ring; warp 2 (one thread) loads the four W limbs of
//     a slice [96 rows x 64 per chunk] into the B buffers of a warpgroup when
//     that warpgroup reaches a new slice (128-byte swizzle for both).  The
//     limbs come from hcmix_pack_limbs_kernel, except when every CTA owns one
//     unit (small batches): the CTA then splits its slice of W into the B
//     buffers itself during set-up;
//   * a compute warpgroup (one thread per row) reads its row from shared
//     memory, sums the squares with the page's tree, splits x into the limbs
//     x0 (grid-aligned) and x1 = x - x0, and stores both into its TMEM A area;
//   * the warpgroup's MMA warp (warp 1 for warpgroup 0, the last warp for
//     warpgroup 1) issues 8 MMAs of M=128, N=96, K=16 with A in TMEM and B in
//     shared memory:  B rows [0 | w0 | w1 | w2] against x1, then
//     [w0 | w1 | w2 | w3] against x0, accumulating into the warpgroup's TMEM D:
//       D = [x0.w0 | x0.w1 + x1.w0 | x0.w2 + x1.w1 | x0.w3 + x1.w2]
//     (the first 24 columns are exact; x1.w3 ~ 2^-34 relative is dropped);
//     the whole warp runs the issue loop and one elected lane issues a
//     chunk's MMAs and commit from one inline-assembly block, which keeps the
//     loop warp-uniform and the issuer's instruction count small;
//   * the warpgroup reads D and forms the chunk dot fl32(top + rest).
// Two warpgroups work on two units at a time.  Each is software-pipelined: it
// transforms chunk k+1 into its second TMEM A buffer before it waits for the
// MMAs of chunk k, so the MMA latency hides behind the next transform; D is
// released together with A(k+1).  TMEM holds 2 x (2 x 64 A + 96 D) columns.
//
// tf32x3 mode (hcmix_tc_kernel<true>): the hc_fused page's own chunk
// arithmetic instead of the exact limbs.  W is packed as big = W rounded to
// tf32 (nearest, ties away: the page's _tf32_rna) and small = W - big; x
// (exact in tf32) goes to TMEM as fp32; per chunk the MMA warp issues, in the
// page's order, dot(x, small) from zero and then dot(x, big) on top of it:
// 2 x 8 MMAs of M=128, N=32 (24 outputs + 8 zero rows), K=8, kind::tf32, and
// D's first 24 columns are the chunk dot.  The rest of the pipeline (units,
// stages, barriers, sum of squares, partials) is the same.  The tensor
// core's own rounding inside each MMA decides the last bits of every chunk
// dot, so this mode is not exact; the page gives no bound either.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hcmix.h"
#include "hcmix_common.cuh"
#include "hcmix_sm100.cuh"

namespace hcmix {
namespace tc {

constexpr int kXStages = 3;                                 // x stages in flight
constexpr int kChunksPerStage = 2;  // an x stage holds two chunks of a tile (one 32 KB load)
constexpr int kWG = 2;
// Units run slice-major, so a CTA's units mostly share one slice and the W
// limbs of a slice (one B buffer per chunk) stay in shared memory across
// them; each warpgroup has its own set, reloaded when its slice changes.
constexpr int kBStages = kWG * kChunksPerSlice;
constexpr int kFirstComputeWarp = 3;  // warp 0: x loads, 1: MMAs of warpgroup 0, 2: W loads
// one MMA-issuing warp per warpgroup: warp 1 for warpgroup 0, the last warp
// for warpgroup 1
constexpr int kWarps = kFirstComputeWarp + 4 * kWG + 1;
constexpr int kMmaWarp1 = kWarps - 1;
constexpr int kThreads = kWarps * 32;
constexpr int kTileM = 128;
constexpr uint32_t kRowBytes = 128;                       // 64 bf16 per smem row
constexpr uint32_t kXChunkBytes = kTileM * kRowBytes;     // one chunk of a tile
constexpr uint32_t kXBytes = kChunksPerStage * kXChunkBytes;  // x stage
constexpr uint32_t kBRows = 120;                          // exact-mode B rows the MMAs read
constexpr uint32_t kLimbRows = 4 * kMix;                  // w0..w3, 24 rows each
constexpr uint32_t kLimbRowOffset = kMix;                 // limbs occupy B rows 24..119
constexpr uint32_t kXTxBytes = kXBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = 64;  // exact: x0 and x1, 32 columns each; tf32x3: 64 fp32 x
constexpr uint32_t kTf32Rows = 32;  // tf32x3 B rows per part: 24 outputs + 8 zero rows
constexpr uint64_t kWaitLimitNs = 2000000000ull;          // 2 s per wait
constexpr uint64_t kDrainLimitNs = 500000000ull;
constexpr uint32_t kWarpArrivals = 4;                      // one arrive per warp of a warpgroup

struct Bookkeeping {
  uint64_t full_x[kXStages];
  uint64_t empty_x[kXStages];
  uint64_t full_b[kBStages];
  uint64_t empty_b[kBStages];
  uint64_t a_ready[kWG];
  uint64_t d_ready[kWG];
  uint64_t drain[kWG];
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: the abort flag of waits that must not be cut short
};

// Per-mode B buffer (one per chunk of a warpgroup's slice), MMA shape and
// TMEM use.
template <bool kTf32>
struct Mode;
template <>
struct Mode<false> {  // exact limbs: 24 zero rows, then w0..w3 (96 rows), bf16
  static constexpr uint32_t kBBytes = kBRows * kRowBytes;
  static constexpr uint32_t kBTxBytes = kLimbRows * kRowBytes;
  static constexpr uint32_t kN = 96;
  static constexpr uint32_t kIdesc = sm100::idesc_bf16_f32(128, kN);
};
template <>
struct Mode<true> {  // tf32x3: [big, small][two 32-column halves][32 rows][128 B], fp32
  static constexpr uint32_t kBBytes = 2 * 2 * kTf32Rows * kRowBytes;
  static constexpr uint32_t kBTxBytes = kBBytes;  // one TMA box, zero rows included
  static constexpr uint32_t kN = kTf32Rows;
  static constexpr uint32_t kIdesc = sm100::idesc_tf32_f32(128, kN);
};
template <bool kTf32>
constexpr uint32_t kWGCols = 2 * kACols + Mode<kTf32>::kN;  // two A buffers and one D per warpgroup
template <bool kTf32>
constexpr size_t kRingBytes = (size_t)kXStages * kXBytes + (size_t)kBStages * Mode<kTf32>::kBBytes;
template <bool kTf32>
constexpr size_t kSmemBytes = kRingBytes<kTf32> + 1024 + 1024;

static_assert(kWG * kWGCols<false> <= kTmemCols && kWG * kWGCols<true> <= kTmemCols, "TMEM budget");
static_assert(sizeof(Bookkeeping) <= 1024, "bookkeeping area");
static_assert(kChunksPerSlice % kChunksPerStage == 0, "x stages hold chunks of one slice");
static_assert(kSmemBytes<false> <= 232448 && kSmemBytes<true> <= 232448, "dynamic shared memory");
static_assert(Mode<false>::kBBytes % 1024 == 0 && Mode<true>::kBBytes % 1024 == 0 &&
                  kLimbRowOffset + kLimbRows <= kBRows, "B buffer layout");

// ---------------------------------------------------------------- W limbs

// W[24, K] fp32 -> limbs[4][24][K] bf16 with W = w0 + w1 + w2 + w3 exactly:
// w0 = W rounded to the grid 2^(ew-7) of its (output, chunk), then three
// round-to-nearest bf16 pieces of the remainder.  16 lanes per (output,
// chunk), four consecutive columns per lane.
constexpr int kPackThreads = 256;
constexpr int kPackTasksPerBlock = kPackThreads / 16;

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

// Largest |W| bit pattern over a 16-lane group's 64 values (four per lane);
// every lane of the warp takes part.
__device__ __forceinline__ uint32_t max_abs_bits16(float4 v) {
  uint32_t m = max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                   max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// The four bf16 limbs of four consecutive W values of one (output, chunk)
// whose largest |W| has the bit pattern m: out[p] holds limb p of the four
// values as two packed bf16 pairs.
__device__ __forceinline__ void split_limbs4(float4 v, uint32_t m, uint32_t (&out)[4][2]) {
  const float magic = grid_magic_from_exp_field(m >> 23);
  const float in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float w0 = grid_round(in[e], magic);
    const float r1 = __fsub_rn(in[e], w0);
    const float w1 = __bfloat162float(__float2bfloat16_rn(r1));
    const float r2 = __fsub_rn(r1, w1);
    const float w2 = __bfloat162float(__float2bfloat16_rn(r2));
    const float w3 = __fsub_rn(r2, w2);
    const uint32_t b[4] = {bf16_bits(w0), bf16_bits(w1), bf16_bits(w2), bf16_bits(w3)};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      if (e % 2 == 0) out[p][e / 2] = b[p];
      else out[p][e / 2] |= b[p] << 16;
    }
  }
}

__global__ void __launch_bounds__(kPackThreads)
hcmix_pack_limbs_kernel(const float* __restrict__ W, int64_t w_stride, int K,
                        uint16_t* __restrict__ limbs) {
  sm100::grid_launch_dependents();  // the contraction may start streaming x now
  const int sub = threadIdx.x & 15;
  const int task = blockIdx.x * kPackTasksPerBlock + (threadIdx.x >> 4);
  const int nch = K / kChunk;
  const bool active = task < kMix * nch;
  const int j = active ? task / nch : 0, c = active ? task % nch : 0;
  const int64_t k = (int64_t)c * kChunk + 4 * sub;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (active) v = *reinterpret_cast<const float4*>(W + (int64_t)j * w_stride + k);
  const uint32_t m = max_abs_bits16(v);
  if (!active) return;
  uint32_t out[4][2];
  split_limbs4(v, m, out);
#pragma unroll
  for (int p = 0; p < 4; ++p)
    *reinterpret_cast<uint2*>(limbs + ((int64_t)p * kMix + j) * K + k) =
        make_uint2(out[p][0], out[p][1]);
}

// W[24, K] fp32 -> parts[2][24][K] fp32 for the tf32x3 mode: part 0 is
// big = W rounded to tf32 (nearest, ties away from zero), part 1 is
// small = W - big, exact in fp32 and passed to the MMAs as it is (the page
// hands the unrounded difference to its tf32 dot).  One float4 per thread.
__global__ void __launch_bounds__(kPackThreads)
hcmix_pack_tf32_kernel(const float* __restrict__ W, int64_t w_stride, int K,
                       float* __restrict__ parts) {
  sm100::grid_launch_dependents();  // the contraction may start streaming x now
  const int64_t per_row = K / 4;
  const int64_t i = (int64_t)blockIdx.x * kPackThreads + threadIdx.x;
  if (i >= kMix * per_row) return;
  const int j = (int)(i / per_row);
  const int64_t k = (i % per_row) * 4;
  const float4 v = *reinterpret_cast<const float4*>(W + (int64_t)j * w_stride + k);
  const float4 big = make_float4(sm100::cvt_rna_tf32(v.x), sm100::cvt_rna_tf32(v.y),
                                 sm100::cvt_rna_tf32(v.z), sm100::cvt_rna_tf32(v.w));
  const float4 small = make_float4(__fsub_rn(v.x, big.x), __fsub_rn(v.y, big.y),
                                   __fsub_rn(v.z, big.z), __fsub_rn(v.w, big.w));
  *reinterpret_cast<float4*>(parts + (int64_t)j * K + k) = big;
  *reinterpret_cast<float4*>(parts + (int64_t)(kMix + j) * K + k) = small;
}

// ---------------------------------------------------------------- main kernel

constexpr uint32_t kBf16x2One = 0x3f803f80u;

// Both halves of the bf16 magic constant 1.5 * 2^(ex+2) for the chunk's
// largest |x| (exponent ex).  (x + magic) - magic rounds x to the grid
// 2^(ex-5).  0 (no split) when the constant would not be a finite bf16.
__device__ __forceinline__ uint32_t bf16x2_split_magic(const uint32_t (&w)[32]) {
  uint32_t t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = sm100::bf16x2_max_abs(w[i], w[i + 16]);
#pragma unroll
  for (int n = 8; n > 0; n >>= 1) {
#pragma unroll
    for (int i = 0; i < n; ++i) t[i] = sm100::bf16x2_max_abs(t[i], t[i + n]);
  }
  const uint32_t m = t[0];
  uint32_t f = max((m >> 7) & 0xffu, (m >> 23) & 0xffu);
  f = f < 1u ? 1u : f;
  if (f > 252u) return 0u;
  const uint32_t h = ((f + 2u) << 7) | 0x40u;
  return h | (h << 16);
}

// The page's sum-of-squares tree (column bits 4, 3, 2, 1, 0, then the two
// halves) on 32 packed words: word w holds columns 2w (low half) and 2w+1
// (high half), so columns differing in bit b >= 1 sit in words differing in
// bit b-1 at the same half.  The bit-4 level fl(x_c^2 + x_{c+16}^2) is one
// mixed-precision FMA on an exact square; the pair sums of bits 3..1 are done
// two at a time.
__device__ __forceinline__ float sq_tree64_f32x2(const uint32_t (&w)[32]) {
  float h[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t* q = w + 16 * half;
    float2 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)  // column bit 4: words i and i + 8
      v[i] = make_float2(sm100::fma_sq_bf16_lo(q[i], sm100::fma_sq_bf16_lo(q[i + 8], 0.0f)),
                         sm100::fma_sq_bf16_hi(q[i], sm100::fma_sq_bf16_hi(q[i + 8], 0.0f)));
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __fadd2_rn(v[i], v[i + 4]);  // bit 3
#pragma unroll
    for (int i = 0; i < 2; ++i) v[i] = __fadd2_rn(v[i], v[i + 2]);  // bit 2
    v[0] = __fadd2_rn(v[0], v[1]);                                   // bit 1
    h[half] = __fadd_rn(v[0].x, v[0].y);                             // bit 0
  }
  return __fadd_rn(h[0], h[1]);                                      // the two halves
}

// One chunk's MMAs and the commit to `bar` from one asm block: the whole
// (converged) warp runs it and the lane that elect.sync picks issues every
// instruction, so the issuer spends a few instructions per MMA.  `a` is the
// chunk's TMEM A buffer, `bdesc` the descriptor of its B buffer; a K-step
// advances the B start address by 32 bytes (2 descriptor units).
//
// Exact limbs: x1 (A columns 32..63) against B rows 0..95 = [0 | w0 | w1 | w2]
// from zero, then x0 (A columns 0..31) against rows 24..119 = [w0 | w1 | w2 |
// w3] (+3072 bytes = 192 units), four K-steps of 16 each.
__device__ __forceinline__ void mma_chunk_exact(uint32_t d, uint32_t a, uint64_t bdesc,
                                                uint32_t idesc, uint32_t bar) {
  asm volatile(
      "{\n\t"
      ".reg .pred e, pz, pa;\n\t"
      ".reg .b32 ta;\n\t"
      ".reg .b64 tb;\n\t"
      "setp.ne.b32 pz, %1, %1;\n\t"
      "setp.eq.b32 pa, %1, %1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "add.u32 ta, %1, 32;\n\t"
      "add.u64 tb, %2, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pz;\n\t"
      "add.u32 ta, %1, 40;\n\t"
      "add.u64 tb, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 48;\n\t"
      "add.u64 tb, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 56;\n\t"
      "add.u64 tb, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 0;\n\t"
      "add.u64 tb, %2, 192;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 8;\n\t"
      "add.u64 tb, %2, 194;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 16;\n\t"
      "add.u64 tb, %2, 196;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 24;\n\t"
      "add.u64 tb, %2, 198;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], tb, %3, pa;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t}"
      ::"r"(d), "r"(a), "l"(bdesc), "r"(idesc), "r"(bar)
      : "memory");
}

// tf32x3: dot(x, small) from zero, then + dot(x, big); eight K-steps of 8
// columns each (A columns 8q..), K-step q in half q / 4 (+4096 bytes = 256
// units) at 32 bytes per step, the small part 8192 bytes (512 units) after
// the big one.
__device__ __forceinline__ void mma_chunk_tf32x3(uint32_t d, uint32_t a, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t bar) {
  asm volatile(
      "{\n\t"
      ".reg .pred e, pz, pa;\n\t"
      ".reg .b32 ta;\n\t"
      ".reg .b64 tb;\n\t"
      "setp.ne.b32 pz, %1, %1;\n\t"
      "setp.eq.b32 pa, %1, %1;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "add.u32 ta, %1, 0;\n\t"
      "add.u64 tb, %2, 512;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pz;\n\t"
      "add.u32 ta, %1, 8;\n\t"
      "add.u64 tb, %2, 514;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 16;\n\t"
      "add.u64 tb, %2, 516;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 24;\n\t"
      "add.u64 tb, %2, 518;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 32;\n\t"
      "add.u64 tb, %2, 768;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 40;\n\t"
      "add.u64 tb, %2, 770;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 48;\n\t"
      "add.u64 tb, %2, 772;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 56;\n\t"
      "add.u64 tb, %2, 774;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 0;\n\t"
      "add.u64 tb, %2, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 8;\n\t"
      "add.u64 tb, %2, 2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 16;\n\t"
      "add.u64 tb, %2, 4;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 24;\n\t"
      "add.u64 tb, %2, 6;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 32;\n\t"
      "add.u64 tb, %2, 256;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 40;\n\t"
      "add.u64 tb, %2, 258;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 48;\n\t"
      "add.u64 tb, %2, 260;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 56;\n\t"
      "add.u64 tb, %2, 262;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t}"
      ::"r"(d), "r"(a), "l"(bdesc), "r"(idesc), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fail(Bookkeeping& bk, uint32_t* err) {
  record_device_error(err, kDevWaitTimeout);
  *reinterpret_cast<volatile int*>(&bk.abort) = 1;
}

template <bool kTf32>
__global__ void __launch_bounds__(kThreads, 1)
hcmix_tc_kernel(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w, int n_tiles, int Mpad,
                int64_t n_units, float* __restrict__ part, uint32_t* __restrict__ err,
                const float* __restrict__ w_src, int64_t w_stride) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  using MD = Mode<kTf32>;
  constexpr uint32_t kWGC = kWGCols<kTf32>;
  Bookkeeping& bk = *reinterpret_cast<Bookkeeping*>(smem + kRingBytes<kTf32>);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int64_t G = gridDim.x, b = blockIdx.x;
  const int64_t u_begin = b * n_units / G;
  const int n = (int)((b + 1) * n_units / G - u_begin);

  auto x_smem = [&](int st) { return smem + (size_t)st * kXBytes; };
  auto b_smem = [&](int st) { return smem + (size_t)kXStages * kXBytes + (size_t)st * MD::kBBytes; };

  // units are slice-major: unit u is tile u % n_tiles of slice u / n_tiles
  auto unit_tile = [&](int64_t u) { return (int)(u % n_tiles); };
  auto unit_slice = [&](int64_t u) { return (int)(u / n_tiles); };

  // x loads in the producer's order (round, chunk pair, warpgroup); load i
  // fills stage i % kXStages, each stage two chunks of one unit, released by
  // its warpgroup.  Issues the loads numbered [from, to) and returns how many
  // loads were issued in total; ok turns false when a wait for a free stage
  // gives up.  Loads below kXStages need no free stage.
  auto x_loads = [&](int from, int to, uint64_t pol, const volatile int* abort_flag,
                     bool& ok) -> int {
    int i = 0;
    for (int r = 0; kWG * r < n; ++r) {
      const int act = min(kWG, n - kWG * r);
      for (int c = 0; c < kChunksPerSlice; c += kChunksPerStage) {
        for (int g = 0; g < act; ++g, ++i) {
          if (i < from) continue;
          if (i >= to) return i;
          const int64_t unit = u_begin + kWG * r + g;
          const int st = i % kXStages;
          const uint32_t ph = (uint32_t)(i / kXStages) & 1u;
          if (i >= kXStages &&
              !mbar_wait(smem_u32(&bk.empty_x[st]), ph ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            return i;
          }
          const uint32_t full = smem_u32(&bk.full_x[st]);
          mbar_arrive_expect_tx(full, kXTxBytes);
          tma_load_3d(smem_u32(x_smem(st)), &tmap_x, 0, unit_tile(unit) * kTileM,
                      unit_slice(unit) * kChunksPerSlice + c, full, pol);
        }
      }
    }
    return i;
  };

  // ---- set-up: barriers, the zero rows of every B buffer, TMEM.  Thread 0,
  // which is also the x producer, starts the first x loads as soon as the
  // barriers exist, so their DRAM latency overlaps the rest of the set-up.
  if (threadIdx.x == 0) {
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(smem_u32(&bk.full_x[s]), 1);
      mbar_init(smem_u32(&bk.empty_x[s]), kWarpArrivals);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(smem_u32(&bk.full_b[s]), 1);
      mbar_init(smem_u32(&bk.empty_b[s]), 1);
    }
    for (int g = 0; g < kWG; ++g) {
      mbar_init(smem_u32(&bk.a_ready[g]), kWarpArrivals);
      mbar_init(smem_u32(&bk.d_ready[g]), 1);
    }
    for (int g = 0; g < kWG; ++g) mbar_init(smem_u32(&bk.drain[g]), 1);
    bk.abort = 0;
    bk.never = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&tmap_x);
    bool ok = true;
    x_loads(0, kXStages, l2_policy_evict_first(), &bk.never, ok);
  }
  if constexpr (!kTf32) {
    // rows 0..23 of each B buffer stay zero (the limbs are loaded to rows 24..119;
    // the tf32x3 boxes bring their own zero rows)
    constexpr int kUnits = kLimbRowOffset * kRowBytes / 16;
    for (int idx = threadIdx.x; idx < kBStages * kUnits; idx += kThreads) {
      const int s = idx / kUnits, u = idx % kUnits;
      sts128(smem_u32(b_smem(s)) + (uint32_t)u * 16, make_uint4(0, 0, 0, 0));
    }
    if (w_src != nullptr) {
      // every CTA owns one unit (small batches): the whole CTA splits that
      // unit's slice of W straight into warpgroup 0's four B buffers, in the
      // layout the TMA would give (row r of a buffer: 128 bytes, 16-byte
      // piece i stored at piece i ^ (r & 7)), instead of a separate pack
      // kernel writing limbs for every slice
      const int64_t k_slice = (int64_t)(u_begin / n_tiles) * kSlice;
      const int sub = threadIdx.x & 15;
      constexpr int kTasks = kMix * kChunksPerSlice;  // (output, chunk) pairs, 16 lanes each
      constexpr int kGroups = kThreads / 16;
      constexpr int kRounds = (kTasks + kGroups - 1) / kGroups;
      float4 wv[kRounds];  // every W load of this lane in flight at once
#pragma unroll
      for (int q = 0; q < kRounds; ++q) {
        const int task = q * kGroups + (threadIdx.x >> 4);
        wv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (task < kTasks)
          wv[q] = *reinterpret_cast<const float4*>(
              w_src + (int64_t)(task / kChunksPerSlice) * w_stride + k_slice +
              (task % kChunksPerSlice) * kChunk + 4 * sub);
      }
#pragma unroll
      for (int q = 0; q < kRounds; ++q) {  // uniform trip count
        const int task = q * kGroups + (threadIdx.x >> 4);
        const bool active = task < kTasks;
        const int j = active ? task / kChunksPerSlice : 0, c = active ? task % kChunksPerSlice : 0;
        const float4 v = wv[q];
        const uint32_t m = max_abs_bits16(v);
        if (!active) continue;
        uint32_t out[4][2];
        split_limbs4(v, m, out);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t r = kLimbRowOffset + (uint32_t)(p * kMix + j);
          const uint32_t addr = smem_u32(b_smem(c)) + r * kRowBytes +
                                ((((uint32_t)sub >> 1) ^ (r & 7u)) << 4) + ((uint32_t)sub & 1u) * 8;
          asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(out[p][0]),
                       "r"(out[p][1])
                       : "memory");
        }
      }
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bk.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bk.tmem_base;
  const volatile int* abort_flag = &bk.abort;
  const volatile int* never = &bk.never;

  if (warp == 0) {
    // ---------------- x producer (thread 0): the loads after the first
    // kXStages, each once its stage has been released
    if (lane == 0) {
      bool ok = true;
      const int i = x_loads(kXStages, 1 << 30, l2_policy_evict_first(), abort_flag, ok);
      if (!ok) fail(bk, err);
      // drain: the loads still in flight complete before the CTA can exit
      for (int j = max(0, i - kXStages); j < i; ++j)
        mbar_wait(smem_u32(&bk.full_x[j % kXStages]), (uint32_t)(j / kXStages) & 1u, never,
                  kDrainLimitNs);
    }
  } else if (warp == 2) {
    // ---------------- W producer: when warpgroup g reaches a new slice, its
    // four B buffers are reloaded with that slice's limbs, once the MMAs of
    // its previous slice have released them (empty_b, committed after their
    // last use)
    if (lane == 0 && w_src != nullptr) {
      // the set-up filled warpgroup 0's buffers with the CTA's only slice
      for (int c = 0; c < kChunksPerSlice; ++c) mbar_arrive(smem_u32(&bk.full_b[c]));
    } else if (lane == 0) {
      prefetch_tensormap(&tmap_w);
      grid_dependency_wait();  // the limbs come from the pack kernel launched before
      const uint64_t pol = l2_policy_evict_last();
      int loads[kWG] = {0, 0}, cur[kWG] = {-1, -1};
      bool ok = true;
      for (int r = 0; ok && kWG * r < n; ++r) {
        const int act = min(kWG, n - kWG * r);
#pragma unroll
        for (int g = 0; g < kWG; ++g) {
          if (!ok || g >= act) continue;
          const int sl = unit_slice(u_begin + kWG * r + g);
          if (sl == cur[g]) continue;
          cur[g] = sl;
          for (int c = 0; c < kChunksPerSlice; ++c) {
            const int j = g * kChunksPerSlice + c;
            if (loads[g] > 0 && !mbar_wait(smem_u32(&bk.empty_b[j]),
                                           (uint32_t)(loads[g] - 1) & 1u, abort_flag,
                                           kWaitLimitNs)) {
              fail(bk, err);
              ok = false;
              break;
            }
            const uint32_t full = smem_u32(&bk.full_b[j]);
            mbar_arrive_expect_tx(full, MD::kBTxBytes);
            if constexpr (kTf32)  // both parts, both 32-column halves of the chunk
              tma_load_4d(smem_u32(b_smem(j)), &tmap_w, 0, 0,
                          2 * (sl * kChunksPerSlice + c), 0, full, pol);
            else
              tma_load_2d(smem_u32(b_smem(j)) + kLimbRowOffset * kRowBytes, &tmap_w,
                          (sl * kChunksPerSlice + c) * kChunk, 0, full, pol);
          }
          ++loads[g];
        }
      }
      // drain
#pragma unroll
      for (int g = 0; g < kWG; ++g)
        if (loads[g] > 0)
          for (int c = 0; c < kChunksPerSlice; ++c)
            mbar_wait(smem_u32(&bk.full_b[g * kChunksPerSlice + c]), (uint32_t)(loads[g] - 1) & 1u,
                      never, kDrainLimitNs);
    }
  } else if (warp == 1 || warp == kMmaWarp1) {
    // ---------------- MMA issuer of warpgroup gm, its chunks in sequence
    // order (round, chunk).  One issuer per warpgroup: an issuing thread
    // spends ~45 cycles per MMA and, once MMAs are queued, a few hundred
    // cycles in any shared-memory access (its mbarrier waits included), so a
    // single issuer for both warpgroups left the tensor pipe idle between
    // chunks.  Each commit tracks the MMAs of the thread that issues it, so
    // the two issuers' commits are independent.  Chunk i needs its
    // warpgroup's x limbs (a_ready) and the W limb tile of its slice (full_b,
    // phase = the warpgroup's slice count).  In order, each wait depends only
    // on earlier chunks, so no wait can close a cycle.  The whole warp runs the loop, the waits are warp votes and one
    // elected lane issues each MMA and commit: a loop whose control flow the
    // compiler cannot prove warp-uniform issued MMAs at about half the rate.
    // per warpgroup: slice of its current unit, B loads so far, and whether
    // this round's unit is the last of its slice (tracked incrementally: the
    // units of a round are consecutive)
    const int gm = warp == 1 ? 0 : 1;
    int64_t u_tile = u_begin % n_tiles, u_slice = u_begin / n_tiles;  // of unit u_begin + kWG * r
    int loads[kWG] = {0, 0}, cur[kWG] = {-1, -1};
    bool ok = true;
    for (int r = 0; ok && kWG * r < n; ++r) {
      const int act = min(kWG, n - kWG * r);
      int sl[kWG];
      bool fresh[kWG], last_use[kWG];
      {
        int64_t t = u_tile, sv = u_slice;
#pragma unroll
        for (int g = 0; g < kWG; ++g) {
          sl[g] = (int)sv;
          fresh[g] = g < act && sl[g] != cur[g];
          if (fresh[g]) {
            cur[g] = sl[g];
            ++loads[g];
          }
          if (++t == n_tiles) { t = 0; ++sv; }
        }
        u_tile = t;
        u_slice = sv;
        // unit + kWG of warpgroup g is unit kWG * (r + 1) + g: its slice
#pragma unroll
        for (int g = 0; g < kWG; ++g) {
          int64_t t2 = t, s2 = sv;
          for (int q = 0; q < g; ++q)
            if (++t2 == n_tiles) { t2 = 0; ++s2; }
          last_use[g] = kWG * (r + 1) + g >= n || (int)s2 != sl[g];
        }
      }
      for (int c = 0; ok && c < kChunksPerSlice; ++c) {
#pragma unroll
        for (int g = 0; g < kWG; ++g) {
          if (!ok || g >= act || g != gm) continue;
          const int j = g * kChunksPerSlice + c;
          const uint32_t aph = (uint32_t)(r * kChunksPerSlice + c) & 1u;
          // the W buffer is waited for at its first use in a slice only
          ok = __all_sync(0xffffffffu,
                          mbar_wait(smem_u32(&bk.a_ready[g]), aph, abort_flag, kWaitLimitNs) &&
                              (!fresh[g] ||
                               mbar_wait(smem_u32(&bk.full_b[j]), (uint32_t)(loads[g] - 1) & 1u,
                                         abort_flag, kWaitLimitNs)));
          if (!ok) break;
          tc_fence_after();
          const uint32_t a = tmem + (uint32_t)g * kWGC + aph * kACols;
          const uint32_t d = tmem + (uint32_t)g * kWGC + 2 * kACols;
          const uint64_t bdesc = smem_desc_sw128(smem_u32(b_smem(j)));
          if constexpr (kTf32)
            mma_chunk_tf32x3(d, a, bdesc, MD::kIdesc, smem_u32(&bk.d_ready[g]));
          else
            mma_chunk_exact(d, a, bdesc, MD::kIdesc, smem_u32(&bk.d_ready[g]));
          if (last_use[g]) umma_commit_warp(smem_u32(&bk.empty_b[j]));
        }
      }
    }
    if (!ok && lane == 0) fail(bk, err);
    umma_commit_warp(smem_u32(&bk.drain[gm]));
    mbar_wait(smem_u32(&bk.drain[gm]), 0, never, kDrainLimitNs);
  } else {
    // ---------------- compute warpgroups: one thread per tile row
    const int g = (warp - kFirstComputeWarp) >> 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t a_base = tmem + (uint32_t)g * kWGC;
    const uint32_t d_col = a_base + 2 * kACols;
    // byte offsets of the row's 16-byte pieces p in a swizzled x tile
    uint32_t xoff[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) xoff[p] = (uint32_t)row * kRowBytes + ((uint32_t)(p ^ (row & 7)) << 4);
    const int my_units = (n - g + kWG - 1) / kWG;
    const int my_chunks = kChunksPerSlice * my_units;

    // transform of this warpgroup's chunk k: sum of squares and the x limbs
    // into A buffer k % 2; returns the chunk's sum of squares
    auto transform = [&](int k, float& tsq) -> bool {
      const int r = k / kChunksPerSlice, c = k % kChunksPerSlice;
      const int act = min(kWG, n - kWG * r);
      // x stage of this chunk: rounds before r loaded kWG * kChunksPerSlice /
      // kChunksPerStage stages each
      const int i = r * kWG * (kChunksPerSlice / kChunksPerStage) + (c / kChunksPerStage) * act + g;
      const int st = i % kXStages;
      const uint32_t ph = (uint32_t)(i / kXStages) & 1u;
      bool ok = mbar_wait(smem_u32(&bk.full_x[st]), ph, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return false;
      const uint32_t xt = smem_u32(x_smem(st)) + (uint32_t)(c % kChunksPerStage) * kXChunkBytes;
      uint32_t xw[32];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint4 v = lds128(xt + xoff[p]);
        xw[4 * p] = v.x; xw[4 * p + 1] = v.y; xw[4 * p + 2] = v.z; xw[4 * p + 3] = v.w;
      }
      tsq = sq_tree64_f32x2(xw);
      const uint32_t a_col = a_base + (uint32_t)(k & 1) * kACols;
      if constexpr (kTf32) {
        // x as fp32 (bf16 is exact in tf32), column c = chunk column c
        uint32_t lo[32], hi[32];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          lo[2 * t] = xw[t] << 16;
          lo[2 * t + 1] = xw[t] & 0xffff0000u;
          hi[2 * t] = xw[16 + t] << 16;
          hi[2 * t + 1] = xw[16 + t] & 0xffff0000u;
        }
        tmem_st32(lanes | a_col, lo);
        tmem_st32(lanes | (a_col + 32), hi);
      } else {
        // x0 = x rounded to the grid 2^(ex-5) with the bf16 magic constant
        // 1.5 * 2^(ex+2) (x + magic stays in one binade, so one bf16 rounding
        // puts x on the grid); x1 = x - x0 is exact.  Both are bf16, <= 8 bits.
        const uint32_t magic = bf16x2_split_magic(xw);
        uint32_t w0[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          w0[t] = bf16x2_sub(bf16x2_fma(xw[t], kBf16x2One, magic), magic);
          xw[t] = bf16x2_sub(xw[t], w0[t]);  // x1, in place
        }
        // the stores complete in the background; tcgen05.wait::st comes
        // before the A buffer is handed to the MMA warp
        tmem_st32(lanes | a_col, w0);
        tmem_st32(lanes | (a_col + 32), xw);
      }
      if (c % kChunksPerStage == kChunksPerStage - 1) {  // both chunks of the stage read
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bk.empty_x[st]));
      }
      return true;
    };

    float2 acc[kMix / 2];
#pragma unroll
    for (int j = 0; j < kMix / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
    float sqs = 0.0f, tsq_cur = 0.0f, tsq_next = 0.0f;
    bool ok = my_chunks > 0 ? transform(0, tsq_cur) : true;
    if (ok && my_chunks > 0) {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bk.a_ready[g]));
    }
    for (int k = 0; ok && k < my_chunks; ++k) {
      if (k + 1 < my_chunks) {
        ok = transform(k + 1, tsq_next);
        if (!ok) break;
      }
      ok = mbar_wait(smem_u32(&bk.d_ready[g]), (uint32_t)k & 1u, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // exact: D = [top | r1 | r2 | r3]; chunk dot = top + ((r1 + r2) + r3), in
      // output pairs; all 96 columns in one TMEM round trip.  tf32x3: D's first
      // 24 columns are the chunk dot.
      uint32_t dv[kTf32 ? kMix : 4 * kMix];
      if constexpr (kTf32) {
        tmem_ld16(lanes | d_col, dv);
        tmem_ld8(lanes | (d_col + 16), dv + 16);
      } else {
        tmem_ld32(lanes | d_col, dv);
        tmem_ld32(lanes | (d_col + 32), dv + 32);
        tmem_ld32(lanes | (d_col + 64), dv + 64);
      }
      tmem_wait_ld();
      // A(k+1) is written and D has been read: the MMAs of chunk k+1 may run
      // while this chunk's dot is formed
      if (k + 1 < my_chunks) {
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bk.a_ready[g]));
      }
#pragma unroll
      for (int j = 0; j < kMix / 2; ++j) {
        const float2 top = make_float2(__uint_as_float(dv[2 * j]), __uint_as_float(dv[2 * j + 1]));
        if constexpr (kTf32) {
          acc[j] = __fadd2_rn(acc[j], top);
        } else {
          const float2 u = make_float2(__uint_as_float(dv[kMix + 2 * j]), __uint_as_float(dv[kMix + 2 * j + 1]));
          const float2 v = make_float2(__uint_as_float(dv[2 * kMix + 2 * j]), __uint_as_float(dv[2 * kMix + 2 * j + 1]));
          const float2 w = make_float2(__uint_as_float(dv[3 * kMix + 2 * j]), __uint_as_float(dv[3 * kMix + 2 * j + 1]));
          acc[j] = __fadd2_rn(acc[j], __fadd2_rn(top, __fadd2_rn(__fadd2_rn(u, v), w)));
        }
      }
      sqs = __fadd_rn(sqs, tsq_cur);
      tsq_cur = tsq_next;
      if (k % kChunksPerSlice == kChunksPerSlice - 1) {
        const int64_t unit = u_begin + kWG * (k / kChunksPerSlice) + g;
        const int tile = unit_tile(unit), s = unit_slice(unit);
        // the reduce kernel reads the partials next: keep them in L2 while x
        // streams through it with evict_first
        float* p = part + (int64_t)s * kPartStride * Mpad + (int64_t)tile * kTileM + row;
        const uint64_t keep = l2_policy_evict_last();
#pragma unroll
        for (int j = 0; j < kMix / 2; ++j) {
          stg_f32_hint(p + (int64_t)(2 * j) * Mpad, acc[j].x, keep);
          stg_f32_hint(p + (int64_t)(2 * j + 1) * Mpad, acc[j].y, keep);
          acc[j] = make_float2(0.0f, 0.0f);
        }
        stg_f32_hint(p + (int64_t)kMix * Mpad, sqs, keep);
        sqs = 0.0f;
      }
    }
    if (!ok) fail(bk, err);
  }

  // ---- teardown: every role has finished (or given up); free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D bf16 tensor map: `inner` contiguous elements, `rows` rows `row_bytes`
// apart; boxes of box_inner x box_rows with the 128-byte swizzle; reads past
// the tensor return zeros.
inline bool make_map_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                             uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
            box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a row-major bf16 matrix [rows, inner] as [inner / 64 chunks]
// [rows][64]: one box is `box_chunks` consecutive 64-column chunks of
// `box_rows` rows, stored in shared memory as box_chunks [box_rows x 128 B]
// tiles with the 128-byte swizzle; reads past the rows return zeros.
inline bool make_map_bf16_3d_chunks(CUtensorMap* map, const void* base, uint64_t inner,
                                    uint64_t rows, uint64_t row_bytes, uint32_t box_rows,
                                    uint32_t box_chunks) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kChunk, rows, inner / kChunk};
  const cuuint64_t strides[2] = {row_bytes, (cuuint64_t)kChunk * 2};
  const cuuint32_t box[3] = {(cuuint32_t)kChunk, box_rows, box_chunks};
  const cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D view of the tf32x3 parts[2][24][K] (fp32) as [part][K / 32 halves]
// [24 rows][32]: one box is both parts of two consecutive 32-column halves
// (one chunk) with 32 rows, stored in shared memory as [part][half][32 rows x
// 128 B] with the 128-byte swizzle; rows 24..31 lie past the tensor and are
// filled with zeros.
inline bool make_map_tf32_parts(CUtensorMap* map, const float* parts, uint64_t K) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {32, (cuuint64_t)kMix, K / 32, 2};
  const cuuint64_t strides[3] = {K * 4, 128, (cuuint64_t)kMix * K * 4};
  const cuuint32_t box[4] = {32, kTf32Rows, 2, 2};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(parts), dims, strides,
            box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kTf32>
hcmix_status launch_main(const CUtensorMap& mx, const CUtensorMap& mw, int64_t M, int64_t K,
                         float* part, int Mpad, uint32_t* err, const float* w_src,
                         int64_t w_stride, bool dependent, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  const int64_t n_tiles = (M + kTileM - 1) / kTileM;
  const int64_t n_units = n_tiles * (K / kSlice);
  const int64_t grid = n_units < sms ? n_units : sms;
  if (cudaFuncSetAttribute(hcmix_tc_kernel<kTf32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes<kTf32>) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  // launched as a programmatic dependent of the pack kernel: x streams while
  // W is being packed; the W producer waits for the pack grid
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes<kTf32>;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, hcmix_tc_kernel<kTf32>, mx, mw, (int)n_tiles, Mpad, n_units, part,
                         err, w_src, w_stride) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? HCMIX_OK : HCMIX_ERR_CUDA;
}

}  // namespace tc

// Packs W (exact limbs, or the tf32x3 big / small parts), then runs the
// tensor-core contraction into `part`.  `packed` is the workspace area of
// 4 * 24 * K * 2 bytes (= 2 * 24 * K * 4) that holds the packed W.  With W
// null (exact mode only), `packed` already holds limbs written by
// hcmix_pack_limbs_kernel and nothing is packed.
inline hcmix_status tc_launch(const uint16_t* x, int64_t x_stride, const float* W,
                              int64_t w_stride, int64_t M, int64_t K, void* packed,
                              float* part, int Mpad, uint32_t* err, cudaStream_t stream,
                              bool tf32x3) {
  if (W == nullptr && tf32x3) return HCMIX_ERR_INVALID_ARG;  // prepacked W: exact limbs only
  CUtensorMap mx, mw;
  if (!tc::make_map_bf16_3d_chunks(&mx, x, (uint64_t)K, (uint64_t)M, (uint64_t)x_stride * 2,
                                    tc::kTileM, tc::kChunksPerStage))
    return HCMIX_ERR_CUDA;
  if (tf32x3) {
    float* parts = static_cast<float*>(packed);
    const int64_t n4 = kMix * (K / 4);
    tc::hcmix_pack_tf32_kernel<<<(unsigned)((n4 + tc::kPackThreads - 1) / tc::kPackThreads),
                                 tc::kPackThreads, 0, stream>>>(W, w_stride, (int)K, parts);
    if (cudaGetLastError() != cudaSuccess) return HCMIX_ERR_CUDA;
    if (!tc::make_map_tf32_parts(&mw, parts, (uint64_t)K)) return HCMIX_ERR_CUDA;
    return tc::launch_main<true>(mx, mw, M, K, part, Mpad, err, nullptr, 0, true, stream);
  }
  uint16_t* limbs = static_cast<uint16_t*>(packed);
  if (!tc::make_map_bf16_2d(&mw, limbs, (uint64_t)K, tc::kLimbRows, (uint64_t)K * 2, kChunk,
                            tc::kLimbRows))
    return HCMIX_ERR_CUDA;
  if (W == nullptr)  // limbs packed ahead of the call
    return tc::launch_main<false>(mx, mw, M, K, part, Mpad, err, nullptr, 0, false, stream);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  const int64_t n_units = (M + tc::kTileM - 1) / tc::kTileM * (K / kSlice);
  if (n_units <= sms)  // one unit per CTA: each CTA splits its own slice of W
    return tc::launch_main<false>(mx, mw, M, K, part, Mpad, err, W, w_stride, false, stream);
  const int nch = (int)(K / kChunk);
  const int pack_blocks = (kMix * nch + tc::kPackTasksPerBlock - 1) / tc::kPackTasksPerBlock;
  tc::hcmix_pack_limbs_kernel<<<pack_blocks, tc::kPackThreads, 0, stream>>>(W, w_stride, (int)K,
                                                                           limbs);
  if (cudaGetLastError() != cudaSuccess) return HCMIX_ERR_CUDA;
  return tc::launch_main<false>(mx, mw, M, K, part, Mpad, err, nullptr, 0, true, stream);
}

// W[24, K] fp32 -> limbs[4][24][K] bf16, the tensor-core kernel's B operand.
inline hcmix_status tc_pack_limbs(const float* W, int64_t w_stride, int64_t K, uint16_t* limbs,
                                  cudaStream_t stream) {
  const int nch = (int)(K / kChunk);
  const int pack_blocks = (kMix * nch + tc::kPackTasksPerBlock - 1) / tc::kPackTasksPerBlock;
  tc::hcmix_pack_limbs_kernel<<<pack_blocks, tc::kPackThreads, 0, stream>>>(W, w_stride, (int)K,
                                                                           limbs);
  return cudaGetLastError() == cudaSuccess ? HCMIX_OK : HCMIX_ERR_CUDA;
}

}  // namespace hcmix
