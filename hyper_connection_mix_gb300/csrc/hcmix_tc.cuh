// Tensor-core (tcgen05) contraction path for sm_103a.
//
// Work: the rows are cut into 128-row tiles and K into 256-column slices (the
// hc_fused page's slice grid); a unit is one (tile, slice) pair.  Each CTA of
// a grid of min(#SMs, #units) takes a contiguous range of units and writes,
// for each unit, the slice totals of its 128 rows (24 mix values and the sum
// of squares) to the workspace partials; hcmix_reduce_kernel then adds the
// slices in slice order.
//
// Per 64-column chunk (see hcmix_common.cuh for the numerics):
//   * warp 0 (one thread) loads the x tile [128 rows x 64] and the four W limbs
//     [96 rows x 64] with TMA (128-byte swizzle) into one of 6 stages;
//   * a compute warpgroup (one thread per row) reads its row from shared
//     memory, sums the squares with the page's tree, splits x into the limbs
//     x0 (grid-aligned) and x1 = x - x0, and stores both into its TMEM A area;
//   * warp 1 (one thread) issues 8 MMAs of M=128, N=96, K=16 with A in TMEM
//     and B in shared memory:  B rows [0 | w0 | w1 | w2] against x1, then
//     [w0 | w1 | w2 | w3] against x0, accumulating into the warpgroup's TMEM D:
//       D = [x0.w0 | x0.w1 + x1.w0 | x0.w2 + x1.w1 | x0.w3 + x1.w2]
//     (the first 24 columns are exact; x1.w3 ~ 2^-34 relative is dropped);
//   * the warpgroup reads D and forms the chunk dot fl32(top + rest).
// Three warpgroups work on three units at a time, so transforms, MMAs and
// epilogues of different units overlap; TMEM holds 3 x (64 A + 96 D) columns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hcmix.h"
#include "hcmix_common.cuh"
#include "hcmix_sm100.cuh"

namespace hcmix {
namespace tc {

constexpr int kStages = 6;
constexpr int kWG = 3;
constexpr int kWarps = 2 + 4 * kWG;
constexpr int kThreads = kWarps * 32;
constexpr int kTileM = 128;
constexpr uint32_t kRowBytes = 128;                       // 64 bf16 per smem row
constexpr uint32_t kXBytes = kTileM * kRowBytes;          // x tile
constexpr uint32_t kBBytes = 128 * kRowBytes;             // B buffer, 128 rows
constexpr uint32_t kLimbRows = 4 * kMix;                  // w0..w3, 24 rows each
constexpr uint32_t kLimbRowOffset = kMix;                 // limbs occupy B rows 24..119
constexpr uint32_t kStageBytes = kXBytes + kBBytes;
constexpr uint32_t kTxBytes = kXBytes + kLimbRows * kRowBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = 64;                           // x0: 32 columns, x1: 32 columns
constexpr uint32_t kN = 96;
constexpr uint32_t kWGCols = kACols + kN;
constexpr uint32_t kIdesc = sm100::idesc_bf16_f32(128, kN);
constexpr uint64_t kWaitLimitNs = 2000000000ull;          // 2 s per wait
constexpr uint64_t kDrainLimitNs = 500000000ull;
constexpr uint32_t kWarpArrivals = 4;                      // one arrive per warp of a warpgroup

struct Bookkeeping {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t a_ready[kWG];
  uint64_t d_ready[kWG];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: the abort flag of waits that must not be cut short
};

constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024 + 1024;

static_assert(kWG * kWGCols <= kTmemCols, "TMEM budget");
static_assert(sizeof(Bookkeeping) <= 1024, "bookkeeping area");

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
  uint32_t m = max(max(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu),
                   max(__float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (!active) return;
  const float magic = grid_magic_from_exp_field(m >> 23);
  const float in[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[4][2];
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
#pragma unroll
  for (int p = 0; p < 4; ++p)
    *reinterpret_cast<uint2*>(limbs + ((int64_t)p * kMix + j) * K + k) =
        make_uint2(out[p][0], out[p][1]);
}

// ---------------------------------------------------------------- main kernel

constexpr uint32_t kBf16x2One = 0x3f803f80u;

// Both halves of the bf16 magic constant 1.5 * 2^(ex+2) for the chunk's
// largest |x| (exponent ex).  (x + magic) - magic rounds x to the grid
// 2^(ex-5).  0 (no split) when the constant would not be a finite bf16.
__device__ __forceinline__ uint32_t bf16x2_split_magic(const uint32_t (&w)[32]) {
  uint32_t m = w[0];
#pragma unroll
  for (int i = 1; i < 32; ++i) m = sm100::bf16x2_max_abs(m, w[i]);
  uint32_t f = max((m >> 7) & 0xffu, (m >> 23) & 0xffu);
  f = f < 1u ? 1u : f;
  if (f > 252u) return 0u;
  const uint32_t h = ((f + 2u) << 7) | 0x40u;
  return h | (h << 16);
}

// The page's sum-of-squares tree (column bits 4, 3, 2, 1, 0, then the two
// halves) on 32 packed words, with the pair sums of bits 4..1 done two at a
// time: word w holds columns 2w (low half) and 2w+1 (high half), so columns
// differing in bit b >= 1 sit in words differing in bit b-1 at the same half.
__device__ __forceinline__ float sq_tree64_f32x2(const uint32_t (&w)[32]) {
  float2 v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float2 u = make_float2(bf16_lo(w[i]), bf16_hi(w[i]));
    v[i] = __fmul2_rn(u, u);
  }
  float h[2];
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    float2* q = v + 16 * half;
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fadd2_rn(q[i], q[i + 8]);  // column bit 4
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = __fadd2_rn(q[i], q[i + 4]);  // bit 3
#pragma unroll
    for (int i = 0; i < 2; ++i) q[i] = __fadd2_rn(q[i], q[i + 2]);  // bit 2
    q[0] = __fadd2_rn(q[0], q[1]);                                   // bit 1
    h[half] = __fadd_rn(q[0].x, q[0].y);                             // bit 0
  }
  return __fadd_rn(h[0], h[1]);                                      // the two halves
}

__device__ __forceinline__ void fail(Bookkeeping& bk, uint32_t* err) {
  record_device_error(err, kDevWaitTimeout);
  *reinterpret_cast<volatile int*>(&bk.abort) = 1;
}

// Sequence index of chunk c of round r for warpgroup g (rounds before the last
// are full, so they hold kWG * kChunksPerSlice chunks each).
__device__ __forceinline__ int seq_index(int r, int c, int g, int act) {
  return r * kWG * kChunksPerSlice + c * act + g;
}

__global__ void __launch_bounds__(kThreads, 1)
hcmix_tc_kernel(const __grid_constant__ CUtensorMap tmap_x,
                const __grid_constant__ CUtensorMap tmap_w, int n_slices, int Mpad,
                int64_t n_units, float* __restrict__ part, uint32_t* __restrict__ err) {
  using namespace sm100;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bookkeeping& bk = *reinterpret_cast<Bookkeeping*>(smem + (size_t)kStages * kStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int64_t G = gridDim.x, b = blockIdx.x;
  const int64_t u_begin = b * n_units / G;
  const int n = (int)((b + 1) * n_units / G - u_begin);

  auto x_smem = [&](int st) { return smem + (size_t)st * kStageBytes; };
  auto b_smem = [&](int st) { return smem + (size_t)st * kStageBytes + kXBytes; };

  // ---- set-up: barriers, the zero rows of every B buffer, TMEM
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bk.full[s]), 1);
      mbar_init(smem_u32(&bk.empty[s]), kWarpArrivals + 1);
    }
    for (int g = 0; g < kWG; ++g) {
      mbar_init(smem_u32(&bk.a_ready[g]), kWarpArrivals);
      mbar_init(smem_u32(&bk.d_ready[g]), 1);
    }
    mbar_init(smem_u32(&bk.drain), 1);
    bk.abort = 0;
    bk.never = 0;
    fence_mbarrier_init();
  }
  {
    // rows 0..23 (3072 B) and 120..127 (1024 B) of each B buffer stay zero
    constexpr int kUnits = (3072 + 1024) / 16;
    for (int idx = threadIdx.x; idx < kStages * kUnits; idx += kThreads) {
      const int s = idx / kUnits, u = idx % kUnits;
      const uint32_t off = u < 192 ? (uint32_t)u * 16 : 120 * kRowBytes + (uint32_t)(u - 192) * 16;
      *reinterpret_cast<uint4*>(b_smem(s) + off) = make_uint4(0, 0, 0, 0);
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
    // ---------------- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tmap_x);
      prefetch_tensormap(&tmap_w);
      const uint64_t pol_x = l2_policy_evict_first();
      const uint64_t pol_w = l2_policy_evict_last();
      int i = 0;
      bool ok = true;
      for (int r = 0; ok && kWG * r < n; ++r) {
        const int act = min(kWG, n - kWG * r);
        for (int c = 0; ok && c < kChunksPerSlice; ++c) {
          for (int g = 0; g < act; ++g, ++i) {
            const int64_t unit = u_begin + kWG * r + g;
            const int tile = (int)(unit / n_slices), s = (int)(unit % n_slices);
            const int k0 = s * kSlice + c * kChunk;
            const int st = i % kStages;
            const uint32_t ph = (uint32_t)(i / kStages) & 1u;
            if (i >= kStages &&
                !mbar_wait(smem_u32(&bk.empty[st]), ph ^ 1u, abort_flag, kWaitLimitNs)) {
              fail(bk, err);
              ok = false;
              break;
            }
            const uint32_t full = smem_u32(&bk.full[st]);
            mbar_arrive_expect_tx(full, kTxBytes);
            tma_load_2d(smem_u32(x_smem(st)), &tmap_x, k0, tile * kTileM, full, pol_x);
            tma_load_2d(smem_u32(b_smem(st)) + kLimbRowOffset * kRowBytes, &tmap_w, k0, 0, full,
                        pol_w);
          }
        }
      }
      // drain: the loads still in flight complete before the CTA can exit
      for (int j = max(0, i - kStages); j < i; ++j)
        mbar_wait(smem_u32(&bk.full[j % kStages]), (uint32_t)(j / kStages) & 1u, never,
                  kDrainLimitNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      int cnt[kWG] = {0, 0, 0};
      int i = 0;
      bool ok = true;
      for (int r = 0; ok && kWG * r < n; ++r) {
        const int act = min(kWG, n - kWG * r);
        for (int c = 0; ok && c < kChunksPerSlice; ++c) {
          for (int g = 0; g < act; ++g, ++i) {
            const int st = i % kStages;
            const uint32_t ph = (uint32_t)(i / kStages) & 1u;
            if (!mbar_wait(smem_u32(&bk.a_ready[g]), (uint32_t)cnt[g] & 1u, abort_flag,
                           kWaitLimitNs) ||
                !mbar_wait(smem_u32(&bk.full[st]), ph, abort_flag, kWaitLimitNs)) {
              fail(bk, err);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a = tmem + (uint32_t)g * kWGCols;
            const uint32_t d = a + kACols;
            const uint32_t bb = smem_u32(b_smem(st));
#pragma unroll
            for (int q = 0; q < 4; ++q)  // x1 against [0 | w0 | w1 | w2]
              umma_bf16_ts(d, a + 32 + 8 * q, smem_desc_sw128(bb + 32 * q), kIdesc, q > 0);
#pragma unroll
            for (int q = 0; q < 4; ++q)  // x0 against [w0 | w1 | w2 | w3]
              umma_bf16_ts(d, a + 8 * q,
                           smem_desc_sw128(bb + kLimbRowOffset * kRowBytes + 32 * q), kIdesc, 1);
            umma_commit(smem_u32(&bk.d_ready[g]));
            umma_commit(smem_u32(&bk.empty[st]));
            ++cnt[g];
          }
        }
      }
      umma_commit(smem_u32(&bk.drain));
      mbar_wait(smem_u32(&bk.drain), 0, never, kDrainLimitNs);
    }
  } else {
    // ---------------- compute warpgroups: one thread per tile row
    const int g = (warp - 2) >> 2;
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t a_col = tmem + (uint32_t)g * kWGCols;
    const uint32_t d_col = a_col + kACols;
    int cnt = 0;
    bool ok = true;
    for (int r = 0; ok && kWG * r + g < n; ++r) {
      const int act = min(kWG, n - kWG * r);
      const int64_t unit = u_begin + kWG * r + g;
      const int tile = (int)(unit / n_slices), s = (int)(unit % n_slices);
      float2 acc[kMix / 2];
#pragma unroll
      for (int j = 0; j < kMix / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
      float sqs = 0.0f;
      for (int c = 0; c < kChunksPerSlice; ++c) {
        const int i = seq_index(r, c, g, act);
        const int st = i % kStages;
        const uint32_t ph = (uint32_t)(i / kStages) & 1u;
        ok = mbar_wait(smem_u32(&bk.full[st]), ph, abort_flag, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        // the row's 64 values: 16-byte piece p sits at p ^ (row & 7) (128-byte swizzle)
        const uint8_t* xrow = x_smem(st) + row * kRowBytes;
        uint32_t xw[32];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const uint4 v = *reinterpret_cast<const uint4*>(xrow + ((p ^ (row & 7)) << 4));
          xw[4 * p] = v.x; xw[4 * p + 1] = v.y; xw[4 * p + 2] = v.z; xw[4 * p + 3] = v.w;
        }
        sqs = __fadd_rn(sqs, sq_tree64_f32x2(xw));
        // x0 = x rounded to the grid 2^(ex-5) with the bf16 magic constant
        // 1.5 * 2^(ex+2) (x + magic stays in one binade, so one bf16 rounding puts
        // x on the grid); x1 = x - x0 is exact.  Both are bf16 with <= 8 bits.
        const uint32_t magic = bf16x2_split_magic(xw);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const uint32_t wd = xw[16 * half + t];
            w0[t] = bf16x2_sub(bf16x2_fma(wd, kBf16x2One, magic), magic);
            w1[t] = bf16x2_sub(wd, w0[t]);
          }
          tmem_st16(lanes | (a_col + 16 * half), w0);
          tmem_st16(lanes | (a_col + 32 + 16 * half), w1);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&bk.a_ready[g]));
          mbar_arrive(smem_u32(&bk.empty[st]));
        }
        ok = mbar_wait(smem_u32(&bk.d_ready[g]), (uint32_t)cnt & 1u, abort_flag, kWaitLimitNs);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++cnt;
        tc_fence_after();
        // D = [top | r1 | r2 | r3]; chunk dot = top + ((r1 + r2) + r3), in output pairs
        uint32_t top[kMix], t[kMix];
        float2 rest[kMix / 2];
        tmem_ld16(lanes | d_col, top);
        tmem_ld8(lanes | (d_col + 16), top + 16);
        tmem_ld16(lanes | (d_col + 24), t);
        tmem_ld8(lanes | (d_col + 40), t + 16);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kMix / 2; ++j)
          rest[j] = make_float2(__uint_as_float(t[2 * j]), __uint_as_float(t[2 * j + 1]));
        tmem_ld16(lanes | (d_col + 48), t);
        tmem_ld8(lanes | (d_col + 64), t + 16);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kMix / 2; ++j)
          rest[j] = __fadd2_rn(
              rest[j], make_float2(__uint_as_float(t[2 * j]), __uint_as_float(t[2 * j + 1])));
        tmem_ld16(lanes | (d_col + 72), t);
        tmem_ld8(lanes | (d_col + 88), t + 16);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kMix / 2; ++j) {
          rest[j] = __fadd2_rn(
              rest[j], make_float2(__uint_as_float(t[2 * j]), __uint_as_float(t[2 * j + 1])));
          const float2 d = __fadd2_rn(
              make_float2(__uint_as_float(top[2 * j]), __uint_as_float(top[2 * j + 1])), rest[j]);
          acc[j] = __fadd2_rn(acc[j], d);
        }
      }
      if (!ok) {
        fail(bk, err);
        break;
      }
      float* p = part + (int64_t)s * kPartStride * Mpad + (int64_t)tile * kTileM + row;
#pragma unroll
      for (int j = 0; j < kMix / 2; ++j) {
        p[(int64_t)(2 * j) * Mpad] = acc[j].x;
        p[(int64_t)(2 * j + 1) * Mpad] = acc[j].y;
      }
      p[(int64_t)kMix * Mpad] = sqs;
    }
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

}  // namespace tc

// Packs W into limbs, then runs the tensor-core contraction into `part`.
inline hcmix_status tc_launch(const uint16_t* x, int64_t x_stride, const float* W,
                              int64_t w_stride, int64_t M, int64_t K, uint16_t* limbs,
                              float* part, int Mpad, uint32_t* err, cudaStream_t stream) {
  const int nch = (int)(K / kChunk);
  const int pack_blocks = (kMix * nch + tc::kPackTasksPerBlock - 1) / tc::kPackTasksPerBlock;
  tc::hcmix_pack_limbs_kernel<<<pack_blocks, tc::kPackThreads, 0, stream>>>(W, w_stride, (int)K,
                                                                           limbs);
  if (cudaGetLastError() != cudaSuccess) return HCMIX_ERR_CUDA;

  CUtensorMap mx, mw;
  if (!tc::make_map_bf16_2d(&mx, x, (uint64_t)K, (uint64_t)M, (uint64_t)x_stride * 2, kChunk,
                            tc::kTileM) ||
      !tc::make_map_bf16_2d(&mw, limbs, (uint64_t)K, tc::kLimbRows, (uint64_t)K * 2, kChunk,
                            tc::kLimbRows))
    return HCMIX_ERR_CUDA;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  const int64_t n_tiles = (M + tc::kTileM - 1) / tc::kTileM;
  const int64_t n_units = n_tiles * (K / kSlice);
  const int64_t grid = n_units < sms ? n_units : sms;
  if (cudaFuncSetAttribute(tc::hcmix_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc::kSmemBytes) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  tc::hcmix_tc_kernel<<<(unsigned)grid, tc::kThreads, tc::kSmemBytes, stream>>>(
      mx, mw, (int)(K / kSlice), Mpad, n_units, part, err);
  return cudaGetLastError() == cudaSuccess ? HCMIX_OK : HCMIX_ERR_CUDA;
}

}  // namespace hcmix
