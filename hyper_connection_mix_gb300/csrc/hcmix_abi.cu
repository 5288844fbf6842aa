// C ABI of libhcmix.so (declared in include/hcmix.h).
//
// Host side only: argument validation in the style of the hc_fused page's
// `eligible` gate (2-D bf16 x with unit inner stride, fp32 W of 24 rows, K of
// the slice grid, hc == 4), workspace layout, kernel dispatch and status
// reporting.  Every step of the computation runs in the kernels included below.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "hcmix.h"
#include "hcmix_common.cuh"
#include "hcmix_reduce.cuh"
#include "hcmix_simt.cuh"
#include "hcmix_tc.cuh"

namespace hcmix {
namespace {

constexpr size_t kAlign = 256;
constexpr int64_t kMaxK = int64_t(1) << 24;
constexpr int64_t kMaxM = (int64_t(1) << 31) - 1;
// AUTO uses the CUDA-core split-K kernel up to this many rows and the
// tensor-core kernel above it.  Measured on GB300 (hc_mix_fused, K = 20480,
// CUDA graphs of 100 calls): the tensor-core path is faster at every M down to
// 1 (14.8 us against 22.8 us at M = 1, 14.7 against 35.9 at M = 64), so AUTO
// always takes it; the CUDA-core kernel stays available by name.
constexpr int64_t kSimtMaxRows = 0;
// Batches up to this many rows are reduced by hcmix_reduce_small_kernel (all
// 32 lanes of a warp fetch one output's slices at once); above it the
// one-lane-per-row kernel, whose loads are coalesced across rows, is used.
constexpr int64_t kReduceSmallMaxM = 16;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Workspace {
  size_t err_off = 0;     // 256-byte header: device error word at byte 0, the tensor-core
                          // kernel's grid-barrier count at byte 64 and generation at byte 128
  size_t part_off = 0;    // fp32 partials [slices][25][Mpad]
  size_t part_bytes = 0;
  size_t total = 0;
  int64_t Mpad = 0;
  int64_t n_slices = 0;
};

Workspace workspace_layout(int64_t M, int64_t K) {
  Workspace w;
  w.n_slices = K / kSlice;
  w.Mpad = (M + 127) / 128 * 128;
  w.err_off = 0;
  w.part_off = kAlign;
  w.part_bytes = align_up((size_t)w.n_slices * kPartStride * (size_t)w.Mpad * 4, kAlign);
  w.total = w.part_off + w.part_bytes;
  return w;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

hcmix_status check_shape(int64_t M, int64_t K, int mix) {
  if (M < 0 || K <= 0) return HCMIX_ERR_INVALID_ARG;
  if (mix != kMix) return HCMIX_ERR_UNSUPPORTED;
  if (K % kSlice != 0 || K > kMaxK || M > kMaxM) return HCMIX_ERR_UNSUPPORTED;
  return HCMIX_OK;
}

hcmix_status check_stats_args(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                              int64_t M, int64_t K, int mix, void* workspace,
                              size_t workspace_bytes) {
  hcmix_status st = check_shape(M, K, mix);
  if (st != HCMIX_OK) return st;
  if (M == 0) return HCMIX_OK;
  if (x == nullptr || W == nullptr || workspace == nullptr) return HCMIX_ERR_INVALID_ARG;
  if (x_stride < K || w_stride < K) return HCMIX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (x_stride * 2) % 16 != 0) return HCMIX_ERR_ALIGNMENT;
  if (!aligned(W, 16) || (w_stride * 4) % 16 != 0) return HCMIX_ERR_ALIGNMENT;
  if (!aligned(workspace, kAlign)) return HCMIX_ERR_ALIGNMENT;
  if (workspace_bytes < workspace_layout(M, K).total) return HCMIX_ERR_WORKSPACE;
  return HCMIX_OK;
}

// Value checks of the epilogue arguments; pointers are checked only when there
// is at least one row (empty tensors may carry null data pointers).
hcmix_status check_epilogue_args(int64_t M, int64_t K, int hc, const float* hc_scale,
                                 const float* hc_base, int iters, const float* pre,
                                 const float* post, const float* comb) {
  if (hc != kHc) return HCMIX_ERR_UNSUPPORTED;
  if (K <= 0 || iters < 0) return HCMIX_ERR_INVALID_ARG;
  if (M > 0 && (hc_scale == nullptr || hc_base == nullptr || pre == nullptr ||
                post == nullptr || comb == nullptr))
    return HCMIX_ERR_INVALID_ARG;
  return HCMIX_OK;
}

hcmix_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? HCMIX_OK : HCMIX_ERR_CUDA;
}

// The CUDA-core kernels stage a whole slice in dynamic shared memory (over
// the 48 KB default).
hcmix_status simt_smem_attributes() {
  if (cudaFuncSetAttribute(hcmix_simt_slice_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSimtSmemBytes) != cudaSuccess ||
      cudaFuncSetAttribute(hcmix_simt_fullk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSimtSmemBytes) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  return HCMIX_OK;
}

bool valid_path(hcmix_path path) {
  return path == HCMIX_PATH_AUTO || path == HCMIX_PATH_SIMT || path == HCMIX_PATH_TC ||
         path == HCMIX_PATH_SIMT_FULLK || path == HCMIX_PATH_TC_TF32X3 ||
         path == HCMIX_PATH_TC_STAGED;
}

hcmix_path resolve_path(hcmix_path path, int64_t M) {
  if (path == HCMIX_PATH_AUTO) return M <= kSimtMaxRows ? HCMIX_PATH_SIMT : HCMIX_PATH_TC;
  return path;
}

bool is_tc(hcmix_path path) { return path == HCMIX_PATH_TC || path == HCMIX_PATH_TC_TF32X3; }

// CUDA-core contraction into the workspace partials (one launch).
hcmix_status launch_simt_contraction(const void* x, int64_t x_stride, const float* W,
                                     int64_t w_stride, int64_t M, int64_t K, void* workspace,
                                     cudaStream_t stream, hcmix_path path) {
  const Workspace ws = workspace_layout(M, K);
  char* base = static_cast<char*>(workspace);
  float* part = reinterpret_cast<float*>(base + ws.part_off);
  if (path == HCMIX_PATH_SIMT) {
    dim3 grid((unsigned)((M + kSimtRows - 1) / kSimtRows), (unsigned)ws.n_slices);
    if (simt_smem_attributes() != HCMIX_OK) return HCMIX_ERR_CUDA;
    hcmix_simt_slice_kernel<<<grid, kSimtThreads, kSimtSmemBytes, stream>>>(
        static_cast<const uint16_t*>(x), x_stride, W, w_stride, (int)M, (int)ws.Mpad, part);
    return launch_status();
  }
  if (path == HCMIX_PATH_SIMT_FULLK) {
    if (simt_smem_attributes() != HCMIX_OK) return HCMIX_ERR_CUDA;
    hcmix_simt_fullk_kernel<<<(unsigned)((M + kSimtRows - 1) / kSimtRows), kSimtThreads,
                              kSimtSmemBytes, stream>>>(static_cast<const uint16_t*>(x), x_stride, W, w_stride,
                                        (int)M, (int)ws.Mpad, (int)ws.n_slices, part);
    return launch_status();
  }
  return HCMIX_ERR_INVALID_ARG;
}

// Ordered reduce of the stored slices (the full-K kernel stores one) and,
// with do_epilogue, the epilogue: the CUDA-core paths' second launch.
hcmix_status launch_reduce(int64_t M, int64_t K, void* workspace, const float* hc_scale,
                           const float* hc_base, int iters, float rms_eps, float hc_eps,
                           float* pre, float* post, float* comb, float* mix_out, float* sq_out,
                           int do_epilogue, cudaStream_t stream, hcmix_path path) {
  const Workspace ws = workspace_layout(M, K);
  const int stored_slices = path == HCMIX_PATH_SIMT_FULLK ? 1 : (int)ws.n_slices;
  const float* part =
      reinterpret_cast<const float*>(static_cast<const char*>(workspace) + ws.part_off);
  const float inv_k = (float)(1.0 / (double)K);
  if (M <= kReduceSmallMaxM && stored_slices <= kReduceSmallMaxSlices) {
    hcmix_reduce_small_kernel<<<(unsigned)((M + kReduceSmallRows - 1) / kReduceSmallRows),
                                kReduceThreads, 0, stream>>>(
        part, stored_slices, (int)ws.Mpad, (int)M, inv_k, hc_scale, hc_base, iters, rms_eps,
        hc_eps, pre, post, comb, mix_out, sq_out, do_epilogue);
    return launch_status();
  }
  dim3 grid((unsigned)((M + kReduceRows - 1) / kReduceRows));
  hcmix_reduce_kernel<<<grid, kReduceThreads, 0, stream>>>(
      part, stored_slices, (int)ws.Mpad, (int)M, inv_k, hc_scale, hc_base, iters, rms_eps,
      hc_eps, pre, post, comb, mix_out, sq_out, do_epilogue);
  return launch_status();
}

// One call on `path`: tail 0 = contraction only (partials), 1 = + mix / sq,
// 2 = + epilogue.  The tensor-core paths run everything in one launch; the
// CUDA-core paths run the contraction and then the reduce kernel.  W null
// with `packed` set: the tensor-core path on limbs packed ahead of time.
hcmix_status run_path(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                      const void* packed, int64_t M, int64_t K, void* workspace, int tail,
                      const float* hc_scale, const float* hc_base, int iters, float rms_eps,
                      float hc_eps, float* pre, float* post, float* comb, float* mix_out,
                      float* sq_out, cudaStream_t stream, hcmix_path path) {
  path = resolve_path(path, M);
  const Workspace ws = workspace_layout(M, K);
  char* base = static_cast<char*>(workspace);
  if (is_tc(path) || path == HCMIX_PATH_TC_STAGED) {
    TcTail t = {tail, (float)(1.0 / (double)K), hc_scale, hc_base, iters, rms_eps, hc_eps, pre,
                post, comb, mix_out, sq_out};
    return tc_launch(static_cast<const uint16_t*>(x), x_stride, W, w_stride, M, K, packed,
                     reinterpret_cast<float*>(base + ws.part_off), (int)ws.Mpad,
                     reinterpret_cast<uint32_t*>(base + ws.err_off), t, stream,
                     path == HCMIX_PATH_TC_TF32X3, path == HCMIX_PATH_TC_STAGED);
  }
  hcmix_status st = launch_simt_contraction(x, x_stride, W, w_stride, M, K, workspace, stream, path);
  if (st != HCMIX_OK || tail == 0) return st;
  return launch_reduce(M, K, workspace, hc_scale, hc_base, iters, rms_eps, hc_eps, pre, post,
                       comb, mix_out, sq_out, tail == 2 ? 1 : 0, stream, path);
}

}  // namespace
}  // namespace hcmix

using namespace hcmix;

extern "C" {

size_t hc_mix_workspace_bytes(int64_t M, int64_t K, int mix) {
  if (check_shape(M, K, mix) != HCMIX_OK) return 0;
  return workspace_layout(M, K).total;
}

hcmix_path hc_mix_auto_path(int64_t M) { return resolve_path(HCMIX_PATH_AUTO, M); }

hcmix_status hc_mix_stats_ex(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                             int64_t M, int64_t K, int mix, float* mix_out, float* sq_out,
                             void* workspace, size_t workspace_bytes, void* stream,
                             hcmix_path path) {
  hcmix_status st = check_stats_args(x, x_stride, W, w_stride, M, K, mix, workspace,
                                     workspace_bytes);
  if (st != HCMIX_OK) return st;
  if (!valid_path(path)) return HCMIX_ERR_INVALID_ARG;
  if (M == 0) return HCMIX_OK;
  if (mix_out == nullptr || sq_out == nullptr) return HCMIX_ERR_INVALID_ARG;
  return run_path(x, x_stride, W, w_stride, nullptr, M, K, workspace, 1, nullptr, nullptr, 0,
                  0.f, 0.f, nullptr, nullptr, nullptr, mix_out, sq_out,
                  static_cast<cudaStream_t>(stream), path);
}

hcmix_status hc_mix_contract_ex(const void* x, int64_t x_stride, const float* W,
                                int64_t w_stride, int64_t M, int64_t K, int mix,
                                void* workspace, size_t workspace_bytes, void* stream,
                                hcmix_path path) {
  hcmix_status st = check_stats_args(x, x_stride, W, w_stride, M, K, mix, workspace,
                                     workspace_bytes);
  if (st != HCMIX_OK) return st;
  if (!valid_path(path)) return HCMIX_ERR_INVALID_ARG;
  if (M == 0) return HCMIX_OK;
  return run_path(x, x_stride, W, w_stride, nullptr, M, K, workspace, 0, nullptr, nullptr, 0,
                  0.f, 0.f, nullptr, nullptr, nullptr, nullptr, nullptr,
                  static_cast<cudaStream_t>(stream), path);
}

hcmix_status hc_mix_stats(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                          int64_t M, int64_t K, int mix, float* mix_out, float* sq_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return hc_mix_stats_ex(x, x_stride, W, w_stride, M, K, mix, mix_out, sq_out, workspace,
                         workspace_bytes, stream, HCMIX_PATH_AUTO);
}

hcmix_status hc_mix_sinkhorn(const float* mix, const float* sq, int64_t M, int64_t K, int mixn,
                             int hc, const float* hc_scale, const float* hc_base,
                             int sinkhorn_iters, float rms_eps, float hc_eps, float* pre,
                             float* post, float* comb, void* stream) {
  if (M < 0) return HCMIX_ERR_INVALID_ARG;
  if (mixn != kMix) return HCMIX_ERR_UNSUPPORTED;
  hcmix_status st =
      check_epilogue_args(M, K, hc, hc_scale, hc_base, sinkhorn_iters, pre, post, comb);
  if (st != HCMIX_OK) return st;
  if (M > kMaxM) return HCMIX_ERR_UNSUPPORTED;
  if (M == 0) return HCMIX_OK;
  if (mix == nullptr || sq == nullptr) return HCMIX_ERR_INVALID_ARG;
  const float inv_k = (float)(1.0 / (double)K);
  hcmix_epilogue_kernel<<<(unsigned)((M + kReduceRows - 1) / kReduceRows), kEpilogueThreads, 0,
                          static_cast<cudaStream_t>(stream)>>>(
      mix, sq, (int)M, inv_k, hc_scale, hc_base, sinkhorn_iters, rms_eps, hc_eps, pre, post, comb);
  return launch_status();
}

hcmix_status hc_mix_fused_ex(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                             int64_t M, int64_t K, int mix, int hc, const float* hc_scale,
                             const float* hc_base, int sinkhorn_iters, float rms_eps,
                             float hc_eps, float* pre, float* post, float* comb, float* mix_out,
                             float* sq_out, void* workspace, size_t workspace_bytes, void* stream,
                             hcmix_path path) {
  hcmix_status st = check_stats_args(x, x_stride, W, w_stride, M, K, mix, workspace,
                                     workspace_bytes);
  if (st != HCMIX_OK) return st;
  st = check_epilogue_args(M, K, hc, hc_scale, hc_base, sinkhorn_iters, pre, post, comb);
  if (st != HCMIX_OK) return st;
  if (!valid_path(path)) return HCMIX_ERR_INVALID_ARG;
  if (M == 0) return HCMIX_OK;
  return run_path(x, x_stride, W, w_stride, nullptr, M, K, workspace, 2, hc_scale, hc_base,
                  sinkhorn_iters, rms_eps, hc_eps, pre, post, comb, mix_out, sq_out,
                  static_cast<cudaStream_t>(stream), path);
}

size_t hc_mix_packed_w_bytes(int64_t K, int mix) {
  if (check_shape(0, K, mix) != HCMIX_OK) return 0;
  return (size_t)4 * kMix * (size_t)K * 2;
}

hcmix_status hc_mix_pack_w(const float* W, int64_t w_stride, int64_t K, int mix, void* packed_w,
                           size_t packed_bytes, void* stream) {
  hcmix_status st = check_shape(0, K, mix);
  if (st != HCMIX_OK) return st;
  if (W == nullptr || packed_w == nullptr || w_stride < K) return HCMIX_ERR_INVALID_ARG;
  if (!aligned(W, 16) || (w_stride * 4) % 16 != 0 || !aligned(packed_w, kAlign))
    return HCMIX_ERR_ALIGNMENT;
  if (packed_bytes < hc_mix_packed_w_bytes(K, mix)) return HCMIX_ERR_WORKSPACE;
  return tc_pack_limbs(W, w_stride, K, static_cast<uint16_t*>(packed_w),
                       static_cast<cudaStream_t>(stream));
}

hcmix_status hc_mix_fused_packed(const void* x, int64_t x_stride, const void* packed_w,
                                 size_t packed_bytes, int64_t M, int64_t K, int mix, int hc,
                                 const float* hc_scale, const float* hc_base, int sinkhorn_iters,
                                 float rms_eps, float hc_eps, float* pre, float* post,
                                 float* comb, float* mix_out, float* sq_out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  hcmix_status st = check_shape(M, K, mix);
  if (st != HCMIX_OK) return st;
  st = check_epilogue_args(M, K, hc, hc_scale, hc_base, sinkhorn_iters, pre, post, comb);
  if (st != HCMIX_OK) return st;
  if (M == 0) return HCMIX_OK;
  if (x == nullptr || packed_w == nullptr || workspace == nullptr || x_stride < K)
    return HCMIX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (x_stride * 2) % 16 != 0 || !aligned(packed_w, kAlign) ||
      !aligned(workspace, kAlign))
    return HCMIX_ERR_ALIGNMENT;
  if (packed_bytes < hc_mix_packed_w_bytes(K, mix) ||
      workspace_bytes < workspace_layout(M, K).total)
    return HCMIX_ERR_WORKSPACE;
  return run_path(x, x_stride, nullptr, 0, packed_w, M, K, workspace, 2, hc_scale, hc_base,
                  sinkhorn_iters, rms_eps, hc_eps, pre, post, comb, mix_out, sq_out,
                  static_cast<cudaStream_t>(stream), HCMIX_PATH_TC);
}

hcmix_status hc_mix_fused(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                          int64_t M, int64_t K, int mix, int hc, const float* hc_scale,
                          const float* hc_base, int sinkhorn_iters, float rms_eps, float hc_eps,
                          float* pre, float* post, float* comb, float* mix_out, float* sq_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return hc_mix_fused_ex(x, x_stride, W, w_stride, M, K, mix, hc, hc_scale, hc_base,
                         sinkhorn_iters, rms_eps, hc_eps, pre, post, comb, mix_out, sq_out,
                         workspace, workspace_bytes, stream, HCMIX_PATH_AUTO);
}

// ---- hc_mix_fused_noalloc: the split-K path with its partials in a fixed
// device array instead of a caller workspace, for callers that may not
// allocate device memory.  The array lives in this file; host code only ever
// uses the device address looked up below, never the array's host-side name.
}  // extern "C"

namespace hcmix {
namespace {

constexpr size_t kStaticScratchBytes = HC_MIX_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_scratch_mutex;
void* g_static_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device, looked up once
// per device (with that device current) and cached.
hcmix_status static_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return HCMIX_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_scratch_mutex);
  if (g_static_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return HCMIX_ERR_CUDA;
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return HCMIX_OK;
}

}  // namespace
}  // namespace hcmix

extern "C" {

hcmix_status hc_mix_fused_noalloc(const void* x, int64_t x_stride, const float* W,
                                  int64_t w_stride, int64_t M, int64_t K, int mix, int hc,
                                  const float* hc_scale, const float* hc_base,
                                  int sinkhorn_iters, float rms_eps, float hc_eps, float* pre,
                                  float* post, float* comb, float* mix_out, float* sq_out,
                                  void* stream) {
  // the static array is the workspace of an ordinary hc_mix_fused call (zero at
  // load, so its header starts as a workspace's must).  The arguments are
  // checked first, before any CUDA call.
  hcmix_status st = check_shape(M, K, mix);
  if (st != HCMIX_OK) return st;
  st = check_epilogue_args(M, K, hc, hc_scale, hc_base, sinkhorn_iters, pre, post, comb);
  if (st != HCMIX_OK) return st;
  if (M == 0) return HCMIX_OK;
  if (x == nullptr || W == nullptr) return HCMIX_ERR_INVALID_ARG;
  if (x_stride < K || w_stride < K) return HCMIX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || (x_stride * 2) % 16 != 0) return HCMIX_ERR_ALIGNMENT;
  if (!aligned(W, 16) || (w_stride * 4) % 16 != 0) return HCMIX_ERR_ALIGNMENT;
  if (workspace_layout(M, K).total > kStaticScratchBytes) return HCMIX_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = static_scratch_address(&scratch);
  if (st != HCMIX_OK) return st;
  return hc_mix_fused_ex(x, x_stride, W, w_stride, M, K, mix, hc, hc_scale, hc_base,
                         sinkhorn_iters, rms_eps, hc_eps, pre, post, comb, mix_out, sq_out,
                         scratch, kStaticScratchBytes, stream, HCMIX_PATH_AUTO);
}

hcmix_status hc_mix_noalloc_device_status(void* stream) {
  void* scratch = nullptr;
  const hcmix_status st = static_scratch_address(&scratch);
  if (st != HCMIX_OK) return st;
  return hc_mix_device_status(scratch, stream);
}

hcmix_status hc_mix_device_status(void* workspace, void* stream) {
  if (workspace == nullptr || !aligned(workspace, kAlign)) return HCMIX_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HCMIX_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return HCMIX_ERR_CUDA;
  if (word != 0) {
    if (cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return HCMIX_ERR_CUDA;
    return HCMIX_ERR_DEVICE;
  }
  return HCMIX_OK;
}

const char* hc_mix_status_string(hcmix_status status) {
  switch (status) {
    case HCMIX_OK: return "HCMIX_OK";
    case HCMIX_ERR_INVALID_ARG: return "HCMIX_ERR_INVALID_ARG: invalid argument";
    case HCMIX_ERR_ALIGNMENT: return "HCMIX_ERR_ALIGNMENT: pointer or row pitch not aligned";
    case HCMIX_ERR_UNSUPPORTED: return "HCMIX_ERR_UNSUPPORTED: shape not supported";
    case HCMIX_ERR_WORKSPACE: return "HCMIX_ERR_WORKSPACE: workspace too small";
    case HCMIX_ERR_CUDA: return "HCMIX_ERR_CUDA: CUDA runtime or launch error";
    case HCMIX_ERR_DEVICE: return "HCMIX_ERR_DEVICE: a kernel recorded an error";
  }
  return "HCMIX: unknown status";
}

}  // extern "C"
