// Tensor-core (tcgen05) path for sm_103a: the whole hc_mix_fused call in one
// persistent kernel.
//
// Work: the rows are cut into 128-row tiles and K into 256-column slices (the
// hc_fused page's slice grid); a unit is one (tile, slice) pair, numbered
// slice-major.  Each CTA of a grid of min(#SMs, #units) takes a contiguous
// range of units, so its units come from at most two consecutive slices at the
// workload sizes (more only when K exceeds 152 slices), and the W operand of
// those slices stays in shared memory for the whole range.
//
// One CTA = 24 warps with fixed roles, each role a stage of a pipeline over
// the CTA's 64-column chunks (k = 0, 1, ... in unit order, four per unit).
// Warp w runs on sub-partition w % 4 and may touch TMEM lanes 32 (w % 4)..:
//   * warps 0..2, the MMA issuers: warp t issues the chunks with k % 3 == t,
//     8 MMAs each (M=128, N=96, K=16, A in TMEM, B in shared memory) into
//     TMEM D buffer t: B rows [0 | w0 | w1 | w2] against x1, then [w0 | w1 |
//     w2 | w3] against x0, so that
//       D = [x0.w0 | x0.w1 + x1.w0 | x0.w2 + x1.w1 | x0.w3 + x1.w2]
//     (the first 24 columns exact; x1.w3 ~ 2^-34 relative is dropped);
//   * warp 3 (one lane), the x producer: it initialises the x barriers,
//     TMA-loads the fp32 W of the CTA's first two slices (staged in slot 1's
//     buffers) and then x, one chunk of a tile (16 KB, 128-byte swizzle) per
//     load into a 6-stage ring.  It issues nothing else, so no other role's
//     shared-memory accesses queue behind its copies;
//   * warps 4..15, the transform warps, three thirds of four (one per
//     quadrant): third t takes the chunks with k % 3 == t.  Each thread reads
//     its row of the chunk from the x stage, sums its squares by the page's
//     fixed tree, splits x into the limbs x0 (grid-aligned) and x1 = x - x0
//     and stores both into TMEM A buffer t (x as fp32 in tf32x3 mode), and
//     the chunk's sum of squares into TMEM column 480 + k % 6;
//   * warps 16..23, the accumulate warps, two halves of four (one per
//     quadrant): half dh takes the units with i % 2 == dh, so that two
//     units' reads are in flight at once.  They read D (TMEM round trips of
//     4 x 8 columns, and the sum-of-squares column), form the chunk dots
//     fl32(top + ((r1 + r2) + r3)), add them into the slice totals (chunks in
//     order, from zero), add the chunk's sum of squares likewise, and store the 24 + 1 slice totals per
//     row to the workspace partials at the end of the unit.  Before that they
//     convert the staged fp32 W into the exact bf16 limbs (or the tf32x3 big
//     / small parts) in shared memory, and they refill a slot when the CTA
//     covers more slices (or TMA-load limbs that hc_mix_pack_w wrote ahead);
//   * warp 2 also initialises the hand-off barriers during set-up.
// The A and D rings are three deep, so that neither hand-off loop (A buffer:
// written, MMAs issued and completed, rewritten; D buffer: MMAs completed,
// read, next MMAs issued) spans fewer than three chunks.  Every mbarrier wait
// is by a waiter that has seen the barrier's previous phase, as a parity wait
// needs: each D barrier (per buffer and accumulate half) and x stage slot
// has fixed waiters that see every phase (the MMA commit that completes a D
// barrier also frees the chunk's A buffer, for the transform third that
// wrote it).  The sums of squares need no barrier of
// their own: column 480 + k % 6 is written with chunk k's A (before its MMAs
// are issued) and read with its D (after they complete), and it is written
// again for chunk k + 6 only after the MMAs of chunk k + 3 completed, which
// were issued only after the accumulate warps had read chunk k's D, and with
// it the column.
//
// Tail (same kernel): once every CTA has stored its partials (a grid-wide
// barrier; the launch is cooperative, so every CTA is resident), CTA b adds
// the slice totals of rows [b M / G, (b + 1) M / G) in slice order from zero
// and, for hc_mix_fused, runs the epilogue (rms, logits, pre / post, Sinkhorn)
// on them; hc_mix_stats writes mix / sq instead.
//
// tf32x3 mode (hcmix_tc_kernel<true>): the hc_fused page's own chunk
// arithmetic instead of the exact limbs.  W is split as big = W rounded to
// tf32 (nearest, ties away: the page's _tf32_rna) and small = W - big; x
// (exact in tf32) goes to TMEM as fp32; per chunk the MMA warp issues, in the
// page's order, dot(x, small) from zero and then dot(x, big) on top of it:
// 2 x 8 MMAs of M=128, N=32, K=8, kind::tf32.  D's first 24 columns are the
// chunk dot (columns 24..31 come from B rows past the 24 outputs and are never
// read).  The tensor core's own rounding inside each MMA decides the last bits
// of every chunk dot, so this mode is not exact; the page gives no bound either.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hcmix.h"
#include "hcmix_common.cuh"
#include "hcmix_reduce.cuh"
#include "hcmix_sm100.cuh"

namespace hcmix {
namespace tc {

// x stages in flight, each one chunk of a tile (one 16 KB load): stage k % 6
// holds chunk k, so each stage serves one transform third.  (Three stages of
// two chunks stream as fast; the smaller first loads land sooner.)
constexpr int kXStages = 6;
constexpr int kChunksPerStage = 1;
constexpr int kNumA = 3;   // TMEM A buffers: chunk k uses A buffer k % 3 (transform third k % 3)
constexpr int kNumD = 3;   // TMEM D buffers: chunk k uses D buffer k % 3
constexpr int kNumSq = 6;  // sum-of-squares TMEM columns: chunk k uses kSqCol0 + k % 6
constexpr int kSlots = 2;  // W slots: a CTA's consecutive slices alternate between them
constexpr int kWBufs = kSlots * kChunksPerSlice;
constexpr int kMmaWarp0 = 0, kTmemWarp = 1;
constexpr int kNumMma = 3;  // MMA-issuing warps 0..2: chunk k to warp k % 3 (its A and D buffers)
constexpr int kXWarp = 3;   // the x producer (one lane)
constexpr int kFirstTWarp = 4;   // transform warps 4..15: three thirds of four, chunks k % 3
constexpr int kNumTWarps = 12;
constexpr int kFirstDWarp = 16;  // accumulate warps 16..23: warp 16 + 4 dh + q, quadrant q, units i % 2 == dh
constexpr int kNumDWarps = 8;
constexpr int kFirstWorkWarp = 4;  // transform and accumulate warps: kFirstWorkWarp ..
constexpr int kWarps = kFirstWorkWarp + kNumTWarps + kNumDWarps;
constexpr int kThreads = kWarps * 32;
// registers per thread: the register file of a sub-partition (16K) over its warps
constexpr int kMaxRegs = (16384 / (((kWarps + 3) / 4) * 32)) / 8 * 8;
constexpr int kDRounds = kMaxRegs >= 96 ? 2 : 3;  // TMEM round trips per chunk for D
constexpr int kTileM = 128;
constexpr uint32_t kRowBytes = 128;                           // 64 bf16 per smem row
constexpr uint32_t kXChunkBytes = kTileM * kRowBytes;         // one chunk of a tile
constexpr uint32_t kXBytes = kChunksPerStage * kXChunkBytes;  // x stage
constexpr uint32_t kLimbRows = 4 * kMix;                      // w0..w3, 24 rows each
constexpr uint32_t kLimbRowOffset = kMix;                     // limbs occupy B rows 24..119
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = 64;  // exact: x0 and x1, 32 columns each; tf32x3: 64 fp32 x
constexpr uint32_t kDCol0 = kNumA * kACols;  // first D column
constexpr uint32_t kSqCol0 = 480;             // the sums of squares, past the D buffers
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainLimitNs = 500000000ull;

// Per-mode W buffer (one per chunk of a slot), MMA shape and D width.
template <bool kTf32>
struct Mode;
template <>
struct Mode<false> {  // exact limbs: 24 zero rows, then w0..w3 (96 rows), bf16
  static constexpr uint32_t kBBytes = (kLimbRowOffset + kLimbRows) * kRowBytes;
  static constexpr uint32_t kBTxBytes = kLimbRows * kRowBytes;
  static constexpr uint32_t kN = 96;
  static constexpr uint32_t kIdesc = sm100::idesc_bf16_f32(128, kN);
};
template <>
struct Mode<true> {  // tf32x3: [big, small][two 32-column halves][24 rows x 128 B], fp32
  static constexpr uint32_t kBlockBytes = kMix * kRowBytes;  // 3 KB, 1 KB aligned
  static constexpr uint32_t kBBytes = 4 * kBlockBytes;
  static constexpr uint32_t kBTxBytes = 0;  // no TMA path
  // N = 32: rows 24..31 of a block are the first rows of the next one (or the
  // shared memory after the last buffer); D columns 24..31 are never read
  static constexpr uint32_t kN = 32;
  static constexpr uint32_t kIdesc = sm100::idesc_tf32_f32(128, kN);
};
template <bool kTf32>
constexpr uint32_t kDCols = Mode<kTf32>::kN;

template <bool kTf32>
constexpr size_t kXOff = 0;
template <bool kTf32>
constexpr size_t kWOff = (size_t)kXStages * kXBytes;
template <bool kTf32>
constexpr size_t kBkOff = kWOff<kTf32> + (size_t)kWBufs * Mode<kTf32>::kBBytes;
template <bool kTf32>
constexpr size_t kSmemBytes = kBkOff<kTf32> + 1024 + 1024;  // bookkeeping + base alignment

struct Bookkeeping {
  uint64_t full_x[kXStages];
  uint64_t empty_x[kXStages];
  uint64_t mma_ready[kNumMma];  // chunk k (issuer k % 3): A(k) written and D(k - 3) read
  uint64_t d_full[kNumD * 2];  // [b * 2 + (k / 4) % 2]: D buffer b holds chunk k, of accumulate half (k / 4) % 2
  uint64_t w_full[kWBufs];
  uint64_t w_stage;  // the fp32 W of the first two slices has landed in slot 1 (TMA)
  uint64_t drain[kNumMma];
  uint64_t tail_bar[6];  // the tail's copy slots (kTailSlots)
  uint64_t refill_done[2];  // per accumulate half: its four warps have converted a refilled slot
  uint32_t tmem_base;
  unsigned long long gbar_base;  // the grid barrier's counter before this CTA arrived, rounded down
  int abort;
  int never;  // stays 0: the abort flag of waits that must not be cut short
  int tail_owner;  // one row group: this CTA's arrival completed the count
};

static_assert(kDCol0 + kNumD * kDCols<false> <= kSqCol0 &&
                  kDCol0 + kNumD * kDCols<true> <= kSqCol0 && kSqCol0 + kNumSq <= kTmemCols,
              "TMEM budget");
static_assert(sizeof(Bookkeeping) <= 1024, "bookkeeping area");
static_assert(3 + 6 + 6 <= 30,
              "one barrier (pair) per lane of the initialising warp; lanes 30 and 31 do the rest");
static_assert(kChunksPerSlice % kChunksPerStage == 0, "x stages hold chunks of one unit");
static_assert(kSmemBytes<false> <= 232448 && kSmemBytes<true> <= 232448, "dynamic shared memory");
static_assert(Mode<false>::kBBytes % 1024 == 0 && Mode<true>::kBlockBytes % 1024 == 0,
              "W buffers keep the 1 KB swizzle atoms aligned");
static_assert(kNumTWarps == 3 * 4 && kFirstTWarp % 4 == 0 && kFirstDWarp % 4 == 0 &&
                  kFirstTWarp >= kFirstWorkWarp && kFirstDWarp >= kFirstWorkWarp &&
                  kFirstTWarp + kNumTWarps <= kWarps && kFirstDWarp + kNumDWarps <= kWarps &&
                  (kFirstTWarp + kNumTWarps <= kFirstDWarp || kFirstDWarp + kNumDWarps <= kFirstTWarp),
              "warp roles");
static_assert(kNumMma == 3 && kNumA == 3 && kNumD == 3 && kNumTWarps == 12 && kNumDWarps == 8 &&
                  kNumSq % 3 == 0 && kXStages * kChunksPerStage == 6 &&
                  kXWarp < kFirstWorkWarp && kMmaWarp0 + kNumMma <= kFirstWorkWarp &&
                  (kXWarp < kMmaWarp0 || kXWarp >= kMmaWarp0 + kNumMma),
              "issuer k % 3 and transform third k % 3 own A buffer k % 3 (so a stage slot "
              "always holds the chunks of the same two thirds); the accumulate warps are two "
              "halves by unit");

// A CTA's unit i (tile, slice), for loops that visit the units in order.
struct UnitCursor {
  int i, tile, slice;
  __device__ __forceinline__ void advance_to(int to, int n_tiles) {
    while (i < to) {
      ++i;
      if (++tile == n_tiles) {
        tile = 0;
        ++slice;
      }
    }
  }
};

// Parameters of one launch (passed by value as a __grid_constant__).
struct TcParams {
  int n_tiles;     // 128-row tiles
  int n_slices;    // K / 256
  int M, Mpad;
  int64_t n_units;  // < 2^31 (the host checks)
  int units_q, units_r;  // n_units = units_q * grid + units_r
  float* part;     // workspace partials, groups of 1 << g_shift rows (see part_index)
  int g_shift;     // log2 of the rows per partial group: 3, or fewer for M < 5
  uint32_t* err;   // device error word
  unsigned long long* gbar;  // the grid barrier's counter (workspace header)
  const float* w_src;  // fp32 W, converted in-kernel; null: limbs come by TMA
  int64_t w_stride;
  int tail;        // 0: partials only; 1: + mix / sq; 2: + epilogue (mix / sq optional)
  float inv_k;
  const float* hc_scale;
  const float* hc_base;
  int iters;
  float rms_eps, hc_eps;
  float *pre, *post, *comb, *mix_out, *sq_out;
};

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
// values as two packed bf16 pairs.  Pairs of values go through the packed
// fp32 -> bf16x2 conversion together.
__device__ __forceinline__ void split_limbs4(float4 v, uint32_t m, uint32_t (&out)[4][2]) {
  const float magic = grid_magic_from_exp_field(m >> 23);
  const float in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; e += 2) {
    const float2 w0 = make_float2(grid_round(in[e], magic), grid_round(in[e + 1], magic));
    const float2 r1 = make_float2(__fsub_rn(in[e], w0.x), __fsub_rn(in[e + 1], w0.y));
    const __nv_bfloat162 b1 = __floats2bfloat162_rn(r1.x, r1.y);
    const float2 w1 = __bfloat1622float2(b1);
    const float2 r2 = make_float2(__fsub_rn(r1.x, w1.x), __fsub_rn(r1.y, w1.y));
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(r2.x, r2.y);
    const float2 w2 = __bfloat1622float2(b2);
    const __nv_bfloat162 b3 = __floats2bfloat162_rn(__fsub_rn(r2.x, w2.x), __fsub_rn(r2.y, w2.y));
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(w0.x, w0.y);  // w0 has <= 8 bits: exact
    out[0][e / 2] = *reinterpret_cast<const uint32_t*>(&b0);
    out[1][e / 2] = *reinterpret_cast<const uint32_t*>(&b1);
    out[2][e / 2] = *reinterpret_cast<const uint32_t*>(&b2);
    out[3][e / 2] = *reinterpret_cast<const uint32_t*>(&b3);
  }
}

// Limbs written once for hc_mix_pack_w (the pack-once API); the kernel below
// TMA-loads them instead of converting fp32 W itself.
__global__ void __launch_bounds__(kPackThreads)
hcmix_pack_limbs_kernel(const float* __restrict__ W, int64_t w_stride, int K,
                        uint16_t* __restrict__ limbs) {
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

// One (output j, chunk) task of the in-kernel W conversion: the 16 lanes of a
// half-warp hold four consecutive columns each (lane `sub`: columns 4 sub ..)
// and write them into W buffer `buf` in the layout the MMAs read (128-byte
// rows, 16-byte piece i of row r stored at piece i ^ (r & 7)).  Exact mode:
// limb p of output j in row 24 + 24 p + j.  tf32x3 mode: big and small of
// output j in row j of blocks [part][half].  Every lane of the warp calls it
// (the maximum is a half-warp shuffle); `active` lanes store.
template <bool kTf32>
__device__ __forceinline__ void convert_w4(float4 v, int j, int sub, uint32_t buf, bool active) {
  if constexpr (kTf32) {
    if (!active) return;
    const float4 big = make_float4(sm100::cvt_rna_tf32(v.x), sm100::cvt_rna_tf32(v.y),
                                   sm100::cvt_rna_tf32(v.z), sm100::cvt_rna_tf32(v.w));
    const float4 small = make_float4(__fsub_rn(v.x, big.x), __fsub_rn(v.y, big.y),
                                     __fsub_rn(v.z, big.z), __fsub_rn(v.w, big.w));
    const uint32_t half = (uint32_t)sub >> 3, piece = (uint32_t)sub & 7u, r = (uint32_t)j;
    const uint32_t off = half * Mode<true>::kBlockBytes + r * kRowBytes + ((piece ^ (r & 7u)) << 4);
    sm100::sts128(buf + off, make_uint4(__float_as_uint(big.x), __float_as_uint(big.y),
                                        __float_as_uint(big.z), __float_as_uint(big.w)));
    sm100::sts128(buf + 2 * Mode<true>::kBlockBytes + off,
                  make_uint4(__float_as_uint(small.x), __float_as_uint(small.y),
                             __float_as_uint(small.z), __float_as_uint(small.w)));
  } else {
    const uint32_t m = max_abs_bits16(v);
    if (!active) return;
    uint32_t out[4][2];
    split_limbs4(v, m, out);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t r = kLimbRowOffset + (uint32_t)(p * kMix + j);
      const uint32_t addr =
          buf + r * kRowBytes + ((((uint32_t)sub >> 1) ^ (r & 7u)) << 4) + ((uint32_t)sub & 1u) * 8;
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(out[p][0]), "r"(out[p][1])
                   : "memory");
    }
  }
}

// ---------------------------------------------------------------- x transform

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

// ---------------------------------------------------------------- MMA issue

// One chunk's MMAs and the commit to `bar` from one asm block: the whole
// (converged) warp runs it and the lane that elect.sync picks issues every
// instruction, so the issuer spends a few instructions per MMA.  `a` is the
// chunk's TMEM A buffer, `bdesc` the descriptor of its W buffer; a K-step
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
// columns each (A columns 8q..), K-step q in half q / 4 (+3072 bytes = 192
// units) at 32 bytes per step, the small part 6144 bytes (384 units) after
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
      "add.u64 tb, %2, 384;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pz;\n\t"
      "add.u32 ta, %1, 8;\n\t"
      "add.u64 tb, %2, 386;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 16;\n\t"
      "add.u64 tb, %2, 388;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 24;\n\t"
      "add.u64 tb, %2, 390;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 32;\n\t"
      "add.u64 tb, %2, 576;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 40;\n\t"
      "add.u64 tb, %2, 578;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 48;\n\t"
      "add.u64 tb, %2, 580;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 56;\n\t"
      "add.u64 tb, %2, 582;\n\t"
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
      "add.u64 tb, %2, 192;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 40;\n\t"
      "add.u64 tb, %2, 194;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 48;\n\t"
      "add.u64 tb, %2, 196;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "add.u32 ta, %1, 56;\n\t"
      "add.u64 tb, %2, 198;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], [ta], tb, %3, pa;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t}"
      ::"r"(d), "r"(a), "l"(bdesc), "r"(idesc), "r"(bar)
      : "memory");
}

// CTA-wide barrier for code in which the lanes of a warp have taken
// different paths (one lane producing, the others idle): the warp first
// reconverges, so that the barrier sees whole warps, as it requires.
__device__ __forceinline__ void cta_barrier() {
  __syncwarp();
  __syncthreads();
}

__device__ __forceinline__ void fail(Bookkeeping& bk, uint32_t* err) {
  record_device_error(err, kDevWaitTimeout);
  *reinterpret_cast<volatile int*>(&bk.abort) = 1;
}

// Grid-wide barrier on a monotonic 64-bit counter in the workspace header.
// Every launch that has a tail adds exactly kBarrierQuantum to it, so at the
// start of a launch it is a multiple of kBarrierQuantum, and any value a
// thread reads before its own arrival lies below the next multiple: `base`
// is that value rounded down, and the barrier opens when the counter reaches
// base + kBarrierQuantum.  Arrivals are release adds at GPU scope (each
// publishes the stores its thread has made or synchronised with).  Above
// eight rows each of a CTA's eight accumulate warps arrives (lane 0, after a
// warp sync) as soon as it has stored its last partials, 1 each, and the
// first of CTA 0 also adds the kBarrierQuantum - 8 G of the warps the grid
// does not have; one thread per CTA then waits (grid_barrier_wait: a bounded
// loop of acquire loads).  Up to eight rows one thread per CTA adds the CTA's
// share (grid_barrier_add) after a CTA barrier.  Every CTA must be resident
// (cooperative launch).
constexpr unsigned long long kBarrierQuantum = 8192;  // above 8 x any grid size

__device__ __forceinline__ unsigned long long grid_barrier_add(int64_t b, int64_t nblocks) {
  return b == 0 ? 1 + kBarrierQuantum - (unsigned long long)nblocks : 1;
}
__device__ __forceinline__ unsigned long long grid_barrier_warp_add(int64_t b, int dtid,
                                                                    int64_t nblocks) {
  return b == 0 && dtid == 0 ? 1 + kBarrierQuantum - 8 * (unsigned long long)nblocks : 1;
}
// Returns false when the wait ran out.
__device__ __forceinline__ bool grid_barrier_wait(const unsigned long long* counter,
                                                  unsigned long long base, uint64_t limit_ns) {
  const unsigned long long target = base + kBarrierQuantum;
  const uint64_t t0 = sm100::global_timer_ns();
  for (uint32_t i = 0; sm100::ld_acquire_gpu_u64(counter) < target; ++i) {
    if ((i & 63u) == 63u && sm100::global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- partials

// The tensor-core path stores the slice totals of R-row groups contiguously
// (R = 8, or the power of two at or above M when M < 5), so that the rows a
// CTA reduces arrive in a few bulk copies: value j (24 mix values, then the
// sum of squares) of slice s for row r sits at
//   part[((r / R * n_slices + s) * 25 + j) * R + r % R].
// With R = 8 a warp's 32 rows of one (s, j) are four full 32-byte sectors;
// the narrower groups keep a decode call's reduce from reading the partials
// of rows that do not exist.
__device__ __forceinline__ int64_t part_index(int row, int s, int j, int n_slices, int gs) {
  return ((((int64_t)(row >> gs) * n_slices + s) * kPartStride + j) << gs) +
         (row & ((1 << gs) - 1));
}
__host__ __device__ inline int part_group_shift(int64_t M) {
  return M >= 5 ? 3 : M >= 3 ? 2 : M == 2 ? 1 : 0;
}

constexpr int kTailSlices = 40;                                      // slices per bulk copy
constexpr uint32_t kTailSlotBytes = kTailSlices * kPartStride * 8 * 4;  // 32000
constexpr int kTailSlotsPerHalf = 3;
constexpr int kTailSlots = 2 * kTailSlotsPerHalf;                    // three per half of the CTA
static_assert(sizeof(Bookkeeping::tail_bar) == kTailSlots * sizeof(uint64_t), "tail slots");
constexpr size_t kTailTotOff = (size_t)kTailSlots * kTailSlotBytes;
constexpr size_t kTailParOff = kTailTotOff + (size_t)kPartStride * (kReduceRows + 1) * 4;
constexpr size_t kTailBytes = (kTailParOff + 32 * 4 + 15) / 16 * 16;  // shared memory the tail uses
constexpr int kTailThreads = 512;
// the tail reuses the x / W buffers; the bookkeeping (its barriers) lies past them
static_assert(kTailBytes <= kBkOff<false> && kTailBytes <= kBkOff<true>, "tail shared memory");

// The tail of a call for CTA b of G: the row groups [b n / G, (b + 1) n / G)
// of the n = ceil(M / R) groups of R = 1 << P.g_shift rows.  Each half of the
// CTA (256 threads) takes every other group; its thread t < 25 R owns value
// j = t / R of row t % R and adds that value's slice totals in slice order
// from zero, reading them from bulk copies of up to 40 R' slices, R' = 8 / R
// (three slots per half, all in flight from the start, each refilled once
// added up).  Every 4 groups (at most 32 rows) the CTA writes mix / sq (when
// asked for) and, with P.tail == 2, runs the epilogue on those rows, four
// lanes per row.  `tb`: kTailBytes of shared memory (16-byte aligned);
// `tbar`: kTailSlots mbarriers, initialised with count 1.  Its three steps:
//   tail_params   (threads 0..26) hc_scale and hc_base into shared memory;
//   tail_start    (one thread, after the partials are visible) the first
//                 copies of both halves;
//   tc_tail       (every thread, after a CTA barrier) the rest;
// all three from the same TailPlan, which every thread can make beforehand.
struct TailPlan {
  int gs, R, n_grp, o0, o1, ns, per_piece, n_pieces;
  __device__ TailPlan(const TcParams& P, int64_t b, int64_t G) {
    gs = P.g_shift;
    R = 1 << gs;
    n_grp = (P.M + R - 1) >> gs;
    o0 = (int)(b * n_grp / G);
    o1 = (int)((b + 1) * n_grp / G);
    ns = P.n_slices;
    per_piece = kTailSlices << (3 - gs);  // a slot holds 40 slices of 8 rows
    n_pieces = (ns + per_piece - 1) / per_piece;
  }
  __device__ int groups_of_half(int h) const {  // groups o0 + h, o0 + h + 2, ...
    return h < 2 && o1 - o0 > h ? (o1 - o0 - h + 1) / 2 : 0;
  }
  // item i of half h (group, piece) into its slot i % 3
  __device__ void issue(const TcParams& P, uint8_t* tb, uint64_t* tbar, int h, int i) const {
    using namespace sm100;
    const int grp = o0 + h + 2 * (i / n_pieces), s0 = (i % n_pieces) * per_piece;
    // (rounded up to whole 16-byte units: the extra bytes lie inside the
    // workspace, which holds 128 rows per tile, and are never read)
    const uint32_t bytes =
        ((uint32_t)min(per_piece, ns - s0) * (kPartStride * 4 << gs) + 15) & ~15u;
    const int slot = kTailSlotsPerHalf * h + i % kTailSlotsPerHalf;
    const uint32_t bar = smem_u32(&tbar[slot]);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(smem_u32(tb) + (uint32_t)slot * kTailSlotBytes,
              P.part + ((((int64_t)grp * ns + s0) * kPartStride) << gs), bytes, bar,
              l2_policy_evict_first());
  }
};
static_assert(kTailSlices * kPartStride * 8 * 4 == (int)kTailSlotBytes, "a slot: 40 slices of 8 rows");

__device__ __forceinline__ void tail_params(const TcParams& P, uint8_t* tb) {
  float* s_par = reinterpret_cast<float*>(tb + kTailParOff);  // hc_scale[3], hc_base[24]
  const int tid = threadIdx.x;
  if (P.tail == 2 && tid < 3 + kMix) s_par[tid] = tid < 3 ? P.hc_scale[tid] : P.hc_base[tid - 3];
}

__device__ __forceinline__ void tail_start(const TcParams& P, const TailPlan& T, uint8_t* tb,
                                           uint64_t* tbar) {
  // the partials were written by other CTAs through the generic proxy, and
  // the slots were last used through it
  asm volatile("fence.proxy.async.global;" ::: "memory");
  sm100::fence_proxy_async_smem();
  for (int h = 0; h < 2; ++h) {
    const int n_items = T.groups_of_half(h) * T.n_pieces;
    for (int i = 0; i < kTailSlotsPerHalf && i < n_items; ++i) T.issue(P, tb, tbar, h, i);
  }
}

// A shared-memory load for the tail's slice adds.  Not volatile, so that the
// compiler issues a batch of them back to back; the memory clobber keeps each
// after the wait for its copy (a volatile form made the compiler treat the
// kernel's main loops less well, 2.5 µs slower; plain C++ loads were issued
// one at a time, each paying the shared-memory latency).
__device__ __forceinline__ float lds_f32_batch(uint32_t addr) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void tc_tail(const TcParams& P, const TailPlan& T, uint8_t* tb,
                                        uint64_t* tbar, const volatile int* never) {
  using namespace sm100;
  const int tid = threadIdx.x;
  const int gs = T.gs;
  auto& s_tot = *reinterpret_cast<float (*)[kPartStride][kReduceRows + 1]>(tb + kTailTotOff);
  const float* s_par = reinterpret_cast<const float*>(tb + kTailParOff);
  // threads past the two halves (the kernel has more warps) only join the CTA barriers
  const int h = min(tid >> 8, 2), t = tid & 255;
  const int my_grps = T.groups_of_half(h);
  const int n_items = my_grps * T.n_pieces;  // item = (group, piece)
  const int j = t >> gs, r8 = t & (T.R - 1);
  const bool adder = h < 2 && t < (kPartStride << gs);
  const int vstride = kPartStride << gs;  // one slice
  const int n_groups = (T.o1 - T.o0 + 3) / 4;
  int i = 0;
  for (int g = 0; g < n_groups; ++g) {
    for (int q = 0; q < 2; ++q) {
      const int m = 2 * g + q;  // this half's m-th group
      if (m >= my_grps) continue;
      float tot = 0.0f;
      for (int p = 0; p < T.n_pieces; ++p, ++i) {
        const int slot = kTailSlotsPerHalf * h + i % kTailSlotsPerHalf;
        if (!mbar_wait(smem_u32(&tbar[slot]), (uint32_t)(i / kTailSlotsPerHalf) & 1u, never,
                       kWaitLimitNs))
          record_device_error(P.err, kDevWaitTimeout);
        if (adder) {
          // slice s of value j of row r8 at ((s 25 + j) R + r8); eight loads
          // at a time, then their adds in slice order
          const float* v0 = reinterpret_cast<const float*>(tb + (size_t)slot * kTailSlotBytes) +
                            (j << gs) + r8;
          const int cnt = min(T.per_piece, T.ns - p * T.per_piece);
          int s = 0;
          for (; s + 8 <= cnt; s += 8) {
            float v[8];
            const uint32_t va = sm100::smem_u32(v0 + s * vstride);
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = lds_f32_batch(va + (uint32_t)(u * vstride) * 4u);
#pragma unroll
            for (int u = 0; u < 8; ++u) tot = __fadd_rn(tot, v[u]);
          }
          for (; s < cnt; ++s) tot = __fadd_rn(tot, v0[s * vstride]);
        }
        named_bar_sync(1 + h, 256);  // the half has read the slot
        if (t == 0 && i + kTailSlotsPerHalf < n_items) T.issue(P, tb, tbar, h, i + kTailSlotsPerHalf);
      }
      if (adder) s_tot[j][((h + 2 * q) << gs) + r8] = tot;
    }
    cta_barrier();
    const int r0 = (T.o0 + 4 * g) << gs;
    const int nr = min(min(4 << gs, (T.o1 - T.o0 - 4 * g) << gs), P.M - r0);
    if (P.mix_out != nullptr)
      for (int e = tid; e < nr * kMix; e += blockDim.x)
        P.mix_out[(int64_t)(r0 + e / kMix) * kMix + e % kMix] = s_tot[e % kMix][e / kMix];
    if (P.sq_out != nullptr && tid < nr) P.sq_out[r0 + tid] = s_tot[kMix][tid];
    if (P.tail == 2)
      epilogue_rows(s_tot, r0, nr, r0 + nr, P.inv_k, s_par, s_par + 3, P.iters, P.rms_eps,
                    P.hc_eps, P.pre, P.post, P.comb);
    cta_barrier();
  }
}

// ---------------------------------------------------------------- the kernel

template <bool kTf32>
__global__ void __maxnreg__(kMaxRegs)
hcmix_tc_kernel(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ TcParams P) {
  using namespace sm100;
  using MD = Mode<kTf32>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bookkeeping& bk = *reinterpret_cast<Bookkeeping*>(smem + kBkOff<kTf32>);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int64_t G = gridDim.x, b = blockIdx.x;
  // units [b n_units / G, (b + 1) n_units / G), in 32-bit arithmetic:
  // floor(b (q G + r) / G) = b q + floor(b r / G), with b r < G^2
  const uint32_t ub = (uint32_t)b, ug = (uint32_t)G;
  const uint32_t u_begin = ub * (uint32_t)P.units_q + ub * (uint32_t)P.units_r / ug;
  const uint32_t u_end = (ub + 1) * (uint32_t)P.units_q + (ub + 1) * (uint32_t)P.units_r / ug;
  const int n = (int)(u_end - u_begin);  // units of this CTA, >= 1
  const int n_chunks = kChunksPerSlice * n;
  const int n_loads = n_chunks / kChunksPerStage;
  const uint32_t n_tiles = (uint32_t)P.n_tiles;
  const int s_first = (int)(u_begin / n_tiles);
  const int n_sl = (int)((u_end - 1) / n_tiles) - s_first + 1;  // slices of this CTA

  const uint32_t x_base = smem_u32(smem + kXOff<kTf32>);
  const uint32_t w_base = smem_u32(smem + kWOff<kTf32>);
  auto wbuf = [&](int slot, int c) {
    return w_base + (uint32_t)(slot * kChunksPerSlice + c) * MD::kBBytes;
  };
  // unit i of this CTA: tile (u % n_tiles) of slice (u / n_tiles), u = u_begin + i
  // (32-bit arithmetic from the CTA's first unit: i < n, and n_tiles fits)
  const int tile0 = (int)(u_begin % n_tiles);
  auto unit_tile = [&](int i) { return (tile0 + i) % P.n_tiles; };
  auto unit_slice = [&](int i) { return s_first + (tile0 + i) / P.n_tiles; };
  // the same for loops that visit the units in order: a cursor moved one unit
  // at a time (no division per chunk)
  const UnitCursor cursor0{0, tile0, s_first};

  // x load L fills stage L % kXStages with chunks kChunksPerStage L .. (unit
  // L / kLoadsPerUnit, at which `u` stands)
  constexpr int kLoadsPerUnit = kChunksPerSlice / kChunksPerStage;
  auto issue_x_load = [&](int L, const UnitCursor& u, uint64_t pol) {
    const int st = L % kXStages;
    const uint32_t full = smem_u32(&bk.full_x[st]);
    mbar_arrive_expect_tx(full, kXBytes);
    tma_load_3d(x_base + (uint32_t)st * kXBytes, &tmap_x, 0, u.tile * kTileM,
                u.slice * kChunksPerSlice + (L % kLoadsPerUnit) * kChunksPerStage, full, pol);
  };
  // limbs of chunk c of slice s into W buffer (slot, c) by TMA (exact mode)
  auto issue_w_load = [&](int slot, int c, int s, uint64_t pol) {
    const uint32_t full = smem_u32(&bk.w_full[slot * kChunksPerSlice + c]);
    mbar_arrive_expect_tx(full, MD::kBTxBytes);
    tma_load_2d(wbuf(slot, c) + kLimbRowOffset * kRowBytes, &tmap_w, (s * kChunksPerSlice + c) * kChunk,
                0, full, pol);
  };
  // the fp32 W of slice index j (slot j % 2), converted by the `nthreads`
  // threads numbered `tid` from 0, a batch of each thread's W loads in flight
  // at once.  (A CTA's first two slices come by TMA instead, staged in slot
  // 1's buffers: see convert_staged.)
  auto convert_slice = [&](int j, int tid, int nthreads) {
    constexpr int kTasks = kMix * kChunksPerSlice;  // (output, chunk) pairs, 16 lanes each
    const int groups = nthreads / 16, sub = tid & 15;
    constexpr int kMaxRounds = 12;  // 96 tasks over at least 8 groups
    constexpr int kBatch = 6;       // rounds whose loads are in flight together
#pragma unroll
    for (int q0 = 0; q0 < kMaxRounds; q0 += kBatch) {
      if (q0 * groups >= kTasks) break;
      float4 wv[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int task = (q0 + q) * groups + (tid >> 4);
        wv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (task < kTasks)
          wv[q] = *reinterpret_cast<const float4*>(
              P.w_src + (int64_t)(task / kChunksPerSlice) * P.w_stride +
              (int64_t)(s_first + j) * kSlice + (task % kChunksPerSlice) * kChunk + 4 * sub);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {  // uniform trip count: the shuffles need whole warps
        const int task = (q0 + q) * groups + (tid >> 4);
        if ((q0 + q) * groups >= kTasks) break;
        const bool active = task < kTasks;
        const int t = active ? task : 0;
        convert_w4<kTf32>(wv[q], t / kChunksPerSlice, sub, wbuf(j % kSlots, t % kChunksPerSlice),
                          active);
      }
    }
  };

  // The first two slices' fp32 W, TMA-staged as [slice][24 rows][256] fp32 at
  // the start of slot 1's buffers, converted by the 256 accumulate threads
  // into slot j % 2 (thread `tid`; one batch: every load of a thread is made
  // before any of its stores).  Slice 1 overwrites its own staging, so all
  // threads first read it, then meet at a named barrier, then write (and the
  // exact mode's zero rows of slot 1 come only then).
  const uint32_t w_stage_base = wbuf(1, 0);
  auto convert_staged = [&](int j, int tid) {
    constexpr int kTasks = kMix * kChunksPerSlice;  // (output, chunk) pairs, 16 lanes each
    constexpr int kThr = kNumDWarps * 32, kGroups = kThr / 16, kRounds = kTasks / kGroups;
    static_assert(kTasks % kGroups == 0 && kRounds <= 8, "one batch of staged loads");
    const int sub = tid & 15;
    float4 wv[kRounds];
#pragma unroll
    for (int q = 0; q < kRounds; ++q) {
      const int task = q * kGroups + (tid >> 4);
      const uint4 v = lds128(w_stage_base + (uint32_t)j * (kMix * kSlice * 4) +
                             (uint32_t)(task / kChunksPerSlice) * (kSlice * 4) +
                             (uint32_t)(task % kChunksPerSlice) * (kChunk * 4) + (uint32_t)sub * 16);
      wv[q] = make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                          __uint_as_float(v.w));
    }
    if (j == 1) {
      named_bar_sync(1, kThr);  // every thread has read slice 1's staging
      if constexpr (!kTf32) {
        constexpr int kUnits = kLimbRowOffset * kRowBytes / 16;
        for (int idx = tid; idx < kChunksPerSlice * kUnits; idx += kThr) {
          const int c = idx / kUnits, u = idx % kUnits;
          sts128(wbuf(1, c) + (uint32_t)u * 16, make_uint4(0, 0, 0, 0));
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kRounds; ++q) {
      const int task = q * kGroups + (tid >> 4);
      convert_w4<kTf32>(wv[q], task / kChunksPerSlice, sub, wbuf(j, task % kChunksPerSlice), true);
    }
  };

  // ---- set-up.  Lane 0 of the x producer initialises the barriers (the x
  // ones first) and starts the W staging and the first x load (and, with
  // prepacked limbs, the W loads of the first two slices); warp 1 allocates
  // TMEM; the transform and accumulate warps zero the W buffers' zero rows.
  // The other first x loads leave once set-up is done: with every CTA's first
  // loads in flight at once, each load lands only when nearly all of them
  // have, so fewer at first bring the first chunk in sooner.
  if (warp == kXWarp) {
    if (lane == 0) {
      prefetch_tensormap(&tmap_x);
      prefetch_tensormap(&tmap_w);  // the fp32 W, or the packed limbs
      mbar_init(smem_u32(&bk.w_stage), 1);
      for (int s = 0; s < kXStages; ++s) {
        mbar_init(smem_u32(&bk.full_x[s]), 1);
        mbar_init(smem_u32(&bk.empty_x[s]), kChunksPerStage * 4);  // the four transform warps of each chunk
      }
      fence_mbarrier_init();
      if (P.w_src != nullptr) {  // the first two slices' fp32 W, ahead of the x loads
        const int nw = min(kSlots, n_sl);
        const uint64_t wpol = l2_policy_evict_last();
        mbar_arrive_expect_tx(smem_u32(&bk.w_stage), (uint32_t)nw * (kMix * kSlice * 4));
        for (int j = 0; j < nw; ++j)
          tma_load_2d(w_stage_base + (uint32_t)j * (kMix * kSlice * 4), &tmap_w,
                      (s_first + j) * kSlice, 0, smem_u32(&bk.w_stage), wpol);
      }
      {
        const uint64_t pol = l2_policy_evict_first();
        if (n_loads > 0) issue_x_load(0, cursor0, pol);
      }
      for (int w = 0; w < kWBufs; ++w) mbar_init(smem_u32(&bk.w_full[w]), 1);
      fence_mbarrier_init();
      if constexpr (!kTf32) {
        if (P.w_src == nullptr) {
          const uint64_t wpol = l2_policy_evict_last();
          for (int j = 0; j < kSlots && j < n_sl; ++j)
            for (int c = 0; c < kChunksPerSlice; ++c) issue_w_load(j, c, s_first + j, wpol);
        }
      }
    }
  } else if (warp == kMmaWarp0 + 2) {
    // the other barriers, one or two per lane, while the producer's loads leave
    if (lane < kNumMma) {
      // mma_ready[k % 3]: the four transform warps of chunk k and the four
      // accumulate warps that have read chunk k - 3 (for the first three
      // chunks, those four arrivals are made here)
      mbar_init(smem_u32(&bk.mma_ready[lane]), 8);
      for (int q = 0; q < 4; ++q) mbar_arrive(smem_u32(&bk.mma_ready[lane]));
      mbar_init(smem_u32(&bk.drain[lane]), 1);
    } else if (lane < kNumMma + 2 * kNumD) {
      mbar_init(smem_u32(&bk.d_full[lane - kNumMma]), 1);  // MMA commit
    } else if (lane < kNumMma + 2 * kNumD + kTailSlots) {
      mbar_init(smem_u32(&bk.tail_bar[lane - kNumMma - 2 * kNumD]), 1);
    } else if (lane == 30) {
      for (int h = 0; h < 2; ++h) mbar_init(smem_u32(&bk.refill_done[h]), 4);  // the half's four warps
    } else if (lane == 31) {
      bk.abort = 0;
      bk.never = 0;
    }
    fence_mbarrier_init();
  } else if (warp == kTmemWarp) {
    tmem_alloc(smem_u32(&bk.tmem_base), kTmemCols);
    tmem_relinquish();
  } else if (warp >= kFirstWorkWarp) {
    // the zero rows of the exact-mode W buffers (the fp32 W itself is
    // converted by the accumulate warps after set-up, while the transform
    // warps already work on the first x loads)
    // (slot 1 holds the staged fp32 W at first: its zero rows come later)
    const int tid = threadIdx.x - kFirstWorkWarp * 32, nthr = kThreads - kFirstWorkWarp * 32;
    if constexpr (!kTf32) {
      constexpr int kUnits = kLimbRowOffset * kRowBytes / 16;
      const int nbufs = P.w_src != nullptr ? kChunksPerSlice : kWBufs;
      for (int idx = tid; idx < nbufs * kUnits; idx += nthr) {
        const int w = idx / kUnits, u = idx % kUnits;
        sts128(w_base + (uint32_t)w * MD::kBBytes + (uint32_t)u * 16, make_uint4(0, 0, 0, 0));
      }
    }
    fence_proxy_async_smem();  // generic-proxy stores -> the MMAs' (async proxy) reads
  }
  tc_fence_before();
  cta_barrier();
  tc_fence_after();
  const uint32_t tmem = bk.tmem_base;
  const volatile int* abort_flag = &bk.abort;
  const volatile int* never = &bk.never;

  if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kNumMma) {
    // ---------------- MMA issuers: warp t issues the chunks k with k % 3 ==
    // t, into A and D buffer t.  Chunk k needs its A buffer written and its D
    // buffer read (both on mma_ready[t], one poll) and its W buffer filled
    // (w_full: once filled it stays so until every MMA of the slice is done,
    // so the wait returns at once after the first).  mma_ready[t] is this
    // warp's own barrier, so it has seen every earlier phase, as a parity
    // wait needs; a W barrier's earlier fill has always completed before any
    // issuer waits for its next one.  Each chunk commits once, on d_full:
    // D complete and A free again.  The whole warp runs the loop, the waits
    // are warp votes and one elected lane issues each MMA and the commit.
    const int t = warp - kMmaWarp0;
    bool ok = true;
    UnitCursor u = cursor0;
    for (int k = t; ok && k < n_chunks; k += kNumMma) {
      const int i = k / kChunksPerSlice, c = k % kChunksPerSlice;
      u.advance_to(i, P.n_tiles);
      const int j = u.slice - s_first, slot = j % kSlots;
      bool got = mbar_wait(smem_u32(&bk.mma_ready[t]), (uint32_t)(k / kNumMma) & 1u, abort_flag,
                           kWaitLimitNs);
      got = got && mbar_wait(smem_u32(&bk.w_full[slot * kChunksPerSlice + c]),
                             (uint32_t)(j / kSlots) & 1u, abort_flag, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, got);
      if (!ok) break;
      tc_fence_after();
      const uint32_t a = tmem + (uint32_t)t * kACols;
      const uint32_t d = tmem + kDCol0 + (uint32_t)t * kDCols<kTf32>;
      const uint64_t bdesc = smem_desc_sw128(wbuf(slot, c));
      if constexpr (kTf32)
        mma_chunk_tf32x3(d, a, bdesc, MD::kIdesc, smem_u32(&bk.d_full[t * 2 + (i & 1)]));
      else
        mma_chunk_exact(d, a, bdesc, MD::kIdesc, smem_u32(&bk.d_full[t * 2 + (i & 1)]));
    }
    if (!ok && lane == 0) fail(bk, P.err);
    // every MMA this warp issued completes before TMEM is released
    umma_commit_warp(smem_u32(&bk.drain[t]));
    mbar_wait(smem_u32(&bk.drain[t]), 0, never, kDrainLimitNs);
  } else if (warp == kXWarp) {
    // ---------------- x producer: the loads after the first, each (after the
    // first kXStages) once the transform warps have read the stage's previous
    // load
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      UnitCursor u = cursor0;
      int L = 1;
      for (; L < n_loads; ++L) {
        const int st = L % kXStages;
        u.advance_to(L / kLoadsPerUnit, P.n_tiles);
        if (L >= kXStages && !mbar_wait(smem_u32(&bk.empty_x[st]), (uint32_t)(L / kXStages - 1) & 1u, abort_flag,
                       kWaitLimitNs)) {
          fail(bk, P.err);
          break;
        }
        issue_x_load(L, u, pol);
      }
      // drain: the loads still in flight complete before the CTA can exit
      for (int j = max(0, min(L, n_loads) - kXStages); j < min(L, n_loads); ++j)
        mbar_wait(smem_u32(&bk.full_x[j % kXStages]), (uint32_t)(j / kXStages) & 1u, never,
                  kDrainLimitNs);
    }
  } else if (warp >= kFirstTWarp && warp < kFirstTWarp + kNumTWarps) {
    // ---------------- transform warps, three thirds of four (one warp per
    // quadrant each): third tt takes the chunks k with k % 3 == tt, from x
    // load k (stage k % 6), into A buffer tt.  A parity wait for phase p of an
    // mbarrier is only sound when the waiter already knows phase p - 1
    // complete: earlier, the wait cannot tell p - 2 (same parity) from p and
    // returns at once.  Every wait below follows that rule: stage k % 6 always
    // holds chunks of the same third, so this third waits for every phase of
    // the stages it uses; and
    // the MMAs of its own previous chunk k - 3 complete on d_full[tt][h], h =
    // ((k - 3) / 4) % 2: every phase of d_full[tt][0] and [1] is a chunk of
    // this third, waited for in order, and none can complete past chunk k - 3
    // before this third has written chunk k's A.
    const int tt = (warp - kFirstTWarp) >> 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t a_col = tmem + (uint32_t)tt * kACols;
    const uint32_t row_sw = (uint32_t)row * kRowBytes + ((uint32_t)(row & 7) << 4);
    uint32_t ae_par = 0;  // bit h: parity of the next phase of d_full[tt][h] this third waits for
    bool ok = true;
    for (int k = tt; k < n_chunks; k += kNumA) {
      const int L = k / kChunksPerStage, st = L % kXStages;
      const int s = k % kNumSq;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bk.full_x[st]),
                                             (uint32_t)(L / kXStages) & 1u, abort_flag,
                                             kWaitLimitNs));
      if (!ok) break;
      // the row's 16-byte piece p sits at piece p ^ (row & 7) of its 128-byte
      // row; the row starts on a 128-byte boundary, so that address is
      // (row start + (row & 7) * 16) ^ p * 16
      const uint32_t xt = x_base + (uint32_t)st * kXBytes + (uint32_t)(k % kChunksPerStage) * kXChunkBytes +
                          row_sw;
      uint32_t xw[32];
#pragma unroll
      for (int p = 0; p < 8; ++p) {
        const uint4 v = lds128(xt ^ ((uint32_t)p << 4));
        xw[4 * p] = v.x; xw[4 * p + 1] = v.y; xw[4 * p + 2] = v.z; xw[4 * p + 3] = v.w;
      }
      // the row is in registers: this warp's part of the stage is released
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bk.empty_x[st]));
      const float tsq = sq_tree64_f32x2(xw);
      uint32_t lo[32];  // exact: x0; tf32x3: x[0:32] as fp32.  xw becomes x1 / x[32:64].
      if constexpr (kTf32) {
        uint32_t hi[32];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          lo[2 * t] = xw[t] << 16;
          lo[2 * t + 1] = xw[t] & 0xffff0000u;
          hi[2 * t] = xw[16 + t] << 16;
          hi[2 * t + 1] = xw[16 + t] & 0xffff0000u;
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) xw[t] = hi[t];
      } else {
        // x0 = x rounded to the grid 2^(ex-5) with the bf16 magic constant
        // 1.5 * 2^(ex+2) (x + magic stays in one binade, so one bf16 rounding
        // puts x on the grid); x1 = x - x0 is exact.  Both are bf16, <= 8 bits.
        const uint32_t magic = bf16x2_split_magic(xw);
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          lo[t] = bf16x2_sub(bf16x2_fma(xw[t], kBf16x2One, magic), magic);
          xw[t] = bf16x2_sub(xw[t], lo[t]);  // x1, in place
        }
      }
      // A buffer tt is free once the MMAs of chunk k - 3 are done; so is sum
      // column s: the accumulate warps read chunk k - 6's column before they
      // freed D for chunk k - 3's MMAs
      if (k >= kNumA) {
        const int h = ((k - kNumA) / kChunksPerSlice) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bk.d_full[tt * 2 + h]),
                                               (ae_par >> h) & 1u, abort_flag, kWaitLimitNs));
        ae_par ^= 1u << h;
        if (!ok) break;
      }
      tc_fence_after();
      tmem_st32(lanes | a_col, lo);
      tmem_st32(lanes | (a_col + 32), xw);
      tmem_st1(lanes | (tmem + kSqCol0 + (uint32_t)s), __float_as_uint(tsq));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bk.mma_ready[tt]));
    }
    if (!ok) fail(bk, P.err);
  } else if (warp >= kFirstDWarp && warp < kFirstDWarp + kNumDWarps) {
    // ---------------- accumulate warps, two halves of four (one warp per
    // quadrant each): half dh reads the units i with i % 2 == dh, all 24
    // outputs, so that two units' chunk reads (TMEM round trips, adds,
    // partial stores) are in flight at once.  First all eight convert the W
    // of the CTA's first two slices, which the MMAs need before any D is
    // ready to read.
    const int dh = (warp - kFirstDWarp) >> 2;
    const int dtid = threadIdx.x - kFirstDWarp * 32;  // 0..255
    const int htid = dtid & 127;                       // within the half
    if (dtid == 0 && P.tail != 0)  // (read before this CTA arrives; used after the teardown barrier)
      bk.gbar_base = ld_relaxed_gpu_u64(P.gbar) / kBarrierQuantum * kBarrierQuantum;
    if (P.w_src != nullptr) {
      // the first two slices' W, once their TMA has landed (the MMAs of
      // each wait for its w_full)
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bk.w_stage), 0, abort_flag, kWaitLimitNs)))
        fail(bk, P.err);
      for (int j = 0; j < kSlots && j < n_sl; ++j) {
        convert_staged(j, dtid);
        fence_proxy_async_smem();
        named_bar_sync(1, kNumDWarps * 32);
        if (dtid == 0)
          for (int c = 0; c < kChunksPerSlice; ++c)
            mbar_arrive(smem_u32(&bk.w_full[j * kChunksPerSlice + c]));
      }
    }
    // A CTA with more than two slices reuses the slots: once a half has read
    // the last chunk of slice j - 2, every MMA of that slice is complete, and
    // that half fills slice j's slot (j % 2) before reading on.  Each of its
    // four warps arrives on refill_done[dh] once its share is converted; the
    // half's first warp alone waits there (a bounded wait: a warp that gave
    // up on an earlier wait cannot hold the others) and marks the slot full.
    // Refills of a half lie at least two units apart and no warp of the half
    // runs more than three chunks ahead of another (the D ring), so the first
    // warp has waited for every phase before the next one completes.
    uint32_t refill_par = 0;  // parity of the next phase of refill_done[dh]
    auto refill = [&](int jn) {
      const int slot = jn % kSlots;
      if (P.w_src != nullptr) {
        convert_slice(jn, htid, 4 * 32);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bk.refill_done[dh]));
        if (htid < 32) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bk.refill_done[dh]), refill_par,
                                                 abort_flag, kWaitLimitNs)))
            fail(bk, P.err);
          else if (htid == 0)
            for (int c = 0; c < kChunksPerSlice; ++c)
              mbar_arrive(smem_u32(&bk.w_full[slot * kChunksPerSlice + c]));
        }
        refill_par ^= 1u;
      } else if constexpr (!kTf32) {
        if (htid == 0)
          for (int c = 0; c < kChunksPerSlice; ++c)
            issue_w_load(slot, c, s_first + jn, l2_policy_evict_last());
      }
    };
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t keep = l2_policy_evict_last();  // the tail reads the partials next
    // the parity of the next phase this half waits for on d_full[b][dh] (this
    // half waits for every phase of those barriers, in order)
    uint32_t dpar = 0;
    bool ok = true;
    for (int i = dh; ok && i < n; i += 2) {
      float2 acc[kMix / 2];
#pragma unroll
      for (int j = 0; j < kMix / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
      float sqs = 0.0f;
      for (int c = 0; c < kChunksPerSlice; ++c) {
        const int k = kChunksPerSlice * i + c, b = k % kNumD;
        // D of chunk k complete (and with it the chunk's sum of squares)
        const int sl = k % kNumSq;
        const bool got = mbar_wait(smem_u32(&bk.d_full[b * 2 + dh]), (dpar >> b) & 1u,
                                   abort_flag, kWaitLimitNs);
        dpar ^= 1u << b;
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d_col = tmem + kDCol0 + (uint32_t)b * kDCols<kTf32>;
        uint32_t tsq;  // (in hand at the first wait::ld below)
        tmem_ld1(lanes | (tmem + kSqCol0 + (uint32_t)sl), tsq);
        if constexpr (kTf32) {
          uint32_t dv[kMix];
          tmem_ld16(lanes | d_col, dv);
          tmem_ld8(lanes | (d_col + 16), dv + 16);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&bk.mma_ready[b]));  // D buffer b free for chunk k + 3
          }
#pragma unroll
          for (int j = 0; j < kMix / 2; ++j)
            acc[j] = __fadd2_rn(acc[j], make_float2(__uint_as_float(dv[2 * j]),
                                                    __uint_as_float(dv[2 * j + 1])));
        } else {
          // D = [top | r1 | r2 | r3] (24 columns each); chunk dot = top + ((r1
          // + r2) + r3).  Outputs in kDRounds TMEM round trips of 24 / kDRounds
          // (to stay within the registers); the D buffer is handed back once
          // the last round is in registers.
          constexpr int kCols = kMix / kDRounds;
#pragma unroll
          for (int r = 0; r < kDRounds; ++r) {
            uint32_t dv[4][kCols];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              tmem_ld8(lanes | (d_col + kMix * g + kCols * r), dv[g]);
              if constexpr (kCols == 12) tmem_ld4(lanes | (d_col + kMix * g + kCols * r + 8), dv[g] + 8);
            }
            tmem_wait_ld();
            if (r == kDRounds - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                mbar_arrive(smem_u32(&bk.mma_ready[b]));  // D buffer b free for chunk k + 3
              }
            }
#pragma unroll
            for (int j = 0; j < kCols / 2; ++j) {
              const float2 top = make_float2(__uint_as_float(dv[0][2 * j]), __uint_as_float(dv[0][2 * j + 1]));
              const float2 u = make_float2(__uint_as_float(dv[1][2 * j]), __uint_as_float(dv[1][2 * j + 1]));
              const float2 v = make_float2(__uint_as_float(dv[2][2 * j]), __uint_as_float(dv[2][2 * j + 1]));
              const float2 w = make_float2(__uint_as_float(dv[3][2 * j]), __uint_as_float(dv[3][2 * j + 1]));
              const int a = kCols / 2 * r + j;
              acc[a] = __fadd2_rn(acc[a], __fadd2_rn(top, __fadd2_rn(__fadd2_rn(u, v), w)));
            }
          }
        }
        sqs = __fadd_rn(sqs, __uint_as_float(tsq));
      }
      if (!ok) break;
      const int grow = unit_tile(i) * kTileM + row;
      if (grow < P.M) {  // (the rows past M of the last tile are zeros: not stored)
        const int gs = P.g_shift;
        float* p = P.part + part_index(grow, unit_slice(i), 0, P.n_slices, gs);
#pragma unroll
        for (int j = 0; j < kMix / 2; ++j) {
          stg_f32_hint(p + ((2 * j) << gs), acc[j].x, keep);
          stg_f32_hint(p + ((2 * j + 1) << gs), acc[j].y, keep);
        }
        stg_f32_hint(p + (kMix << gs), sqs, keep);
      }
      // the last unit of slice j done: slice j + 2 (if any) may take its slot
      const int j = unit_slice(i) - s_first;
      if (j + kSlots < n_sl && (i == n - 1 || unit_slice(i + 1) != unit_slice(i)))
        refill(j + kSlots);
    }
    if (!ok) fail(bk, P.err);
    if (P.tail != 0 && P.M > 8) {  // this warp's arrival at the grid barrier
      static_assert(kNumDWarps == 8, "eight arrivals per CTA");
      __syncwarp();
      if (lane == 0) red_add_release_gpu_u64(P.gbar, grid_barrier_warp_add(b, dtid, G));
    }
    if constexpr (!kTf32) {
      // the TMA loads of prepacked limbs complete before the CTA can exit
      if (P.w_src == nullptr && dtid == 0)
        for (int j = max(0, n_sl - kSlots); j < n_sl; ++j)
          for (int c = 0; c < kChunksPerSlice; ++c)
            mbar_wait(smem_u32(&bk.w_full[(j % kSlots) * kChunksPerSlice + c]),
                      (uint32_t)(j / kSlots) & 1u, never, kDrainLimitNs);
    }
  }

  // ---- every role has finished (or given up); TMEM is no longer needed
  tc_fence_before();
  cta_barrier();
  if (warp == kTmemWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (P.tail == 0) return;

  if (P.M <= 8) {
    // ---- one row group (decode sizes): no CTA waits.  Each adds its share
    // to the same counter with one acquire-release atomic; the CTA whose add
    // completes the launch's quantum has seen every other CTA's partials and
    // runs the whole tail, the others are done.
    if (threadIdx.x == 0) {
      const unsigned long long add = grid_barrier_add(b, G);
      const unsigned long long old = atom_add_acq_rel_gpu_u64(P.gbar, add);
      bk.tail_owner = old + add == bk.gbar_base + kBarrierQuantum;
    }
    cta_barrier();
    if (!bk.tail_owner) return;
    tail_params(P, smem);
    const TailPlan T(P, G - 1, G);  // the plan of the CTA that holds the only group
    if (threadIdx.x == 0) tail_start(P, T, smem, bk.tail_bar);
    cta_barrier();
    tc_tail(P, T, smem, bk.tail_bar, never);
    return;
  }

  // ---- tail: once every CTA's partials are stored (grid barrier) this CTA
  // adds the slices of its rows in slice order and runs the epilogue; the x
  // and W buffers are idle now and hold the tail's copies (the epilogue's
  // parameters are loaded while the barrier waits, the first copies leave as
  // soon as it opens)
  tail_params(P, smem);
  const TailPlan T(P, b, G);
  if (threadIdx.x == 0) {
    if (!grid_barrier_wait(P.gbar, bk.gbar_base, kWaitLimitNs))
      record_device_error(P.err, kDevWaitTimeout);
    tail_start(P, T, smem, bk.tail_bar);
  }
  cta_barrier();
  tc_tail(P, T, smem, bk.tail_bar, never);
}

// The tail alone (HCMIX_PATH_TC_STAGED): the same reduce and epilogue as the
// fused kernel's, as a kernel of its own after the contraction.
__global__ void __launch_bounds__(kTailThreads, 1) hcmix_tc_tail_kernel(const __grid_constant__ TcParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tb = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  uint64_t* tbar = reinterpret_cast<uint64_t*>(tb + kTailBytes);
  __shared__ int never;
  tail_params(P, tb);
  const TailPlan T(P, blockIdx.x, gridDim.x);
  if (threadIdx.x == 0) {
    never = 0;
    for (int q = 0; q < kTailSlots; ++q) sm100::mbar_init(sm100::smem_u32(&tbar[q]), 1);
    sm100::fence_mbarrier_init();
    tail_start(P, T, tb, tbar);
  }
  __syncthreads();
  tc_tail(P, T, tb, tbar, &never);
}
constexpr size_t kTailKernelSmem = kTailBytes + kTailSlots * 8 + 128;

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

// 2-D fp32 tensor map: `inner` contiguous elements, `rows` rows `row_bytes`
// apart; boxes of box_inner x box_rows, no swizzle (row-major in shared memory).
inline bool make_map_f32_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                            uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

// The tail kernel of the staged path: the same CTA count as the contraction.
inline hcmix_status launch_tail(const TcParams& P, int64_t grid, cudaStream_t stream) {
  if (cudaFuncSetAttribute(hcmix_tc_tail_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kTailKernelSmem) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  hcmix_tc_tail_kernel<<<(unsigned)grid, kTailThreads, kTailKernelSmem, stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? HCMIX_OK : HCMIX_ERR_CUDA;
}

template <bool kTf32>
hcmix_status launch_main(const CUtensorMap& mx, const CUtensorMap& mw, const TcParams& P,
                         int64_t grid, cudaStream_t stream) {
  if (cudaFuncSetAttribute(hcmix_tc_kernel<kTf32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes<kTf32>) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  // cooperative: every CTA is resident at once, which the grid barrier before
  // the tail relies on (one CTA per SM, grid <= #SMs)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes<kTf32>;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, hcmix_tc_kernel<kTf32>, mx, mw, P) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? HCMIX_OK : HCMIX_ERR_CUDA;
}

}  // namespace tc

// What the tensor-core kernel does after its contraction.
struct TcTail {
  int tail;  // 0: partials only; 1: + mix / sq; 2: + epilogue
  float inv_k;
  const float* hc_scale;
  const float* hc_base;
  int iters;
  float rms_eps, hc_eps;
  float *pre, *post, *comb, *mix_out, *sq_out;
};

// The tensor-core path in one launch: contraction into `part`, then the tail.
// W given: converted inside the kernel (exact limbs, or the tf32x3 big /
// small parts).  W null (exact mode only): `packed` holds limbs written by
// hcmix_pack_limbs_kernel, loaded with TMA.  `header` is the workspace header
// (error word at 0, grid-barrier words at 64 and 128 bytes).  `staged`: the
// tail runs as a second kernel instead (HCMIX_PATH_TC_STAGED).
inline hcmix_status tc_launch(const uint16_t* x, int64_t x_stride, const float* W,
                              int64_t w_stride, int64_t M, int64_t K, const void* packed,
                              float* part, int Mpad, uint32_t* header, const TcTail& t,
                              cudaStream_t stream, bool tf32x3, bool staged = false) {
  if (W == nullptr && (tf32x3 || packed == nullptr)) return HCMIX_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  CUtensorMap mx, mw;
  if (!tc::make_map_bf16_3d_chunks(&mx, x, (uint64_t)K, (uint64_t)M, (uint64_t)x_stride * 2,
                                    tc::kTileM, tc::kChunksPerStage))
    return HCMIX_ERR_CUDA;
  if (W == nullptr) {
    if (!tc::make_map_bf16_2d(&mw, packed, (uint64_t)K, tc::kLimbRows, (uint64_t)K * 2, kChunk,
                              tc::kLimbRows))
      return HCMIX_ERR_CUDA;
  } else if (!tc::make_map_f32_2d(&mw, W, (uint64_t)K, kMix, (uint64_t)w_stride * 4, kSlice, kMix)) {
    return HCMIX_ERR_CUDA;  // the fp32 W, TMA-staged for the first two slices of each CTA
  }
  tc::TcParams P = {};
  P.n_tiles = (int)((M + tc::kTileM - 1) / tc::kTileM);
  P.n_slices = (int)(K / kSlice);
  P.M = (int)M;
  P.g_shift = tc::part_group_shift(M);
  P.Mpad = Mpad;
  P.n_units = (int64_t)P.n_tiles * P.n_slices;
  P.part = part;
  P.err = header;
  P.gbar = reinterpret_cast<unsigned long long*>(header + 16);
  P.w_src = W;
  P.w_stride = w_stride;
  P.tail = t.tail;
  P.inv_k = t.inv_k;
  P.hc_scale = t.hc_scale;
  P.hc_base = t.hc_base;
  P.iters = t.iters;
  P.rms_eps = t.rms_eps;
  P.hc_eps = t.hc_eps;
  P.pre = t.pre;
  P.post = t.post;
  P.comb = t.comb;
  P.mix_out = t.mix_out;
  P.sq_out = t.sq_out;
  const int64_t grid = P.n_units < sms ? P.n_units : sms;
  if (P.n_units >= ((int64_t)1 << 31) || grid > 1024) return HCMIX_ERR_UNSUPPORTED;
  P.units_q = (int)(P.n_units / grid);
  P.units_r = (int)(P.n_units % grid);
  if (staged) P.tail = 0;
  const hcmix_status st = tf32x3 ? tc::launch_main<true>(mx, mw, P, grid, stream)
                                 : tc::launch_main<false>(mx, mw, P, grid, stream);
  if (st != HCMIX_OK || !staged || t.tail == 0) return st;
  P.tail = t.tail;
  return tc::launch_tail(P, grid, stream);
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
