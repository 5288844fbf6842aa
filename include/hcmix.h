/*
 * hcmix.h -- C ABI of libhcmix.so: hyper-connection mix statistics on sm_103a.
 *
 * The operation (hc_fused page, "launcher/docker-images/mia-tp4/adapter/hc_fused.py",
 * module docstring and fused_mix_stats_sinkhorn): for every row m of a bf16
 * activation x[M, K] and an fp32 weight W[mix, K] (mix = 24 = 2*hc + hc*hc, hc = 4)
 *
 *   mix[m, j] = sum over K of x[m, k] * W[j, k], with K walked in slices of 256
 *               columns and each slice in four chunks of 64: every chunk's dot
 *               product is rounded once to fp32, a slice total starts from zero
 *               and adds its chunks in order, and the grand total starts from
 *               zero and adds the slice totals in slice order;
 *   sq[m]     = sum of x[m, k]^2 by the page's fixed tree inside every chunk
 *               (_sq_tree), then the same chunk / slice / total order;
 *   epilogue  : r = 1 / sqrt(sq * (1/K) + rms_eps);
 *               logit[j] = mix[j] * r * hc_scale[g(j)] + hc_base[j],
 *                 g = 0 for j < hc (pre), 1 for hc <= j < 2hc (post), 2 else (comb);
 *               pre  = sigmoid(logit[0:hc]);  post = 2 * sigmoid(logit[hc:2hc]);
 *               comb = sinkhorn_iters rounds of (divide each row by its sum + hc_eps,
 *                      then each column by its sum + hc_eps) of exp(logit[2hc:]),
 *                      viewed row-major as hc x hc.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing and never synchronises the host.  Its only global state
 *     is the fixed scratch array of hc_mix_fused_noalloc and that array's cached
 *     device addresses.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream), so calls may be captured in a CUDA graph.
 *   - Layouts are row-major.  x rows are `x_stride` elements apart (inner stride
 *     1); W rows are `w_stride` elements apart (inner stride 1).
 *   - Arguments are validated on the host before any launch.  A failed check
 *     returns an error status and launches nothing.  Launch failures return
 *     HCMIX_ERR_CUDA.  Kernels never trap: a bounded wait that runs out sets a
 *     device error word in the workspace, read with hc_mix_device_status().
 *   - NaN / Inf inputs propagate per IEEE arithmetic without checks.
 *   - Supported shapes: mix == 24, hc == 4, K a positive multiple of 256 up to
 *     2^24, 0 <= M < 2^31, and for the tensor-core path fewer than 2^31
 *     (128-row tile, 256-column slice) units, ceil(M / 128) * (K / 256)
 *     (HCMIX_ERR_UNSUPPORTED otherwise; x would not fit in device memory long
 *     before that).  Finite |x| < 2^112 and |W| < 2^112 (the exact limb split of
 *     the contraction needs that headroom).
 */
#ifndef HCMIX_H
#define HCMIX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HCMIX_OK = 0,
  HCMIX_ERR_INVALID_ARG = 1, /* negative size, null pointer, stride < K, iters < 0 */
  HCMIX_ERR_ALIGNMENT = 2,   /* x, W or workspace misaligned, or row pitch not 16-byte */
  HCMIX_ERR_UNSUPPORTED = 3, /* mix != 24, hc != 4, K not a multiple of 256, too large */
  HCMIX_ERR_WORKSPACE = 4,   /* workspace smaller than hc_mix_workspace_bytes() */
  HCMIX_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  HCMIX_ERR_DEVICE = 6       /* a kernel recorded an error (see hc_mix_device_status) */
} hcmix_status;

/* Which contraction kernel runs.  AUTO picks by M (hc_mix_auto_path; on
 * GB300 the tensor-core kernel at every M); the others force one path (all
 * give results within the stated tolerance of each other).
 *
 * HCMIX_PATH_SIMT and HCMIX_PATH_SIMT_FULLK are the hc_fused page's two
 * designs on the same CUDA-core arithmetic, kept as an A/B pair: the stock
 * engine's split-K layout (each (slice, row block) pair gets a CTA of its own
 * that writes its slice's totals to the workspace; an ordered reduce follows) against the page's
 * fused kernel (one CTA per row block walks all of K and keeps the running
 * total, so only the total is stored; the page's module docstring).  Their
 * statistics are bit-identical.
 *
 * HCMIX_PATH_TC_TF32X3 is the page's own chunk arithmetic (hc_fused page,
 * module docstring, second bullet; _tf32_rna and the two tl.dot calls of
 * _hc_mix_fullk_kernel) on the tensor-core kernel: W = big + small with
 * big = W rounded to tf32 (nearest, ties away) and small = W - big; every
 * chunk dot is dot(x, small) from zero followed by dot(x, big) on top, as
 * tcgen05 kind::tf32 MMAs.  The tensor core's internal rounding sets the last
 * bits of each chunk dot, so this path is NOT held to the mix tolerance above.
 * Per chunk its error is at most (2^-19 + 2^-21) * sum |x| |W| over the chunk
 * (16 fp32 accumulations and the tf32 truncation of the small part), and its
 * tests hold each output within 2^-18 * sum_k |x[m,k]| |W[j,k]| of the exact
 * result; sq is bit-identical to the other paths.  AUTO never selects it.
 *
 * HCMIX_PATH_TC runs the whole call in one launch: the contraction stores its
 * per-slice totals in the workspace, and the same kernel then adds them in
 * slice order and runs the epilogue after a grid-wide barrier.
 * HCMIX_PATH_TC_STAGED runs the same contraction but leaves the ordered reduce
 * and the epilogue to a second kernel, as the page's stock engine does; its
 * results are bit-identical to HCMIX_PATH_TC's (an A/B of the fused tail). */
typedef enum {
  HCMIX_PATH_AUTO = 0,
  HCMIX_PATH_SIMT = 1,       /* CUDA-core split-K kernel (stock layout) */
  HCMIX_PATH_TC = 2,         /* tcgen05 tensor-core split-K kernel */
  HCMIX_PATH_SIMT_FULLK = 3, /* CUDA-core full-K kernel (the page's fused design) */
  HCMIX_PATH_TC_TF32X3 = 4,  /* tensor-core split-K kernel with the page's tf32x3 chunk dots */
  HCMIX_PATH_TC_STAGED = 5   /* HCMIX_PATH_TC's contraction, then the separate reduce kernel */
} hcmix_path;

/* Bytes of device workspace that hc_mix_stats / hc_mix_fused need for M rows.
 * The workspace must be 256-byte aligned, and its first 256 bytes (the device
 * error word and the grid barrier's counter) zeroed once before its first use;
 * the rest needs no initialising, and every call writes what it reads, so no
 * per-call clearing is needed.  A workspace sized
 * for M rows serves any smaller M.  Calls that share a workspace must not
 * overlap on the GPU (issue them on one stream).  Returns 0 for unsupported
 * (K, mix). */
size_t hc_mix_workspace_bytes(int64_t M, int64_t K, int mix);

/* mix_out[M, mix] (fp32) and sq_out[M] (fp32): the contraction and the sum of
 * squares in the slice order above.
 *   x        bf16 [M, x_stride], 16-byte aligned, x_stride % 8 == 0, x_stride >= K
 *   W        fp32 [mix, w_stride], 16-byte aligned, w_stride % 4 == 0, w_stride >= K
 *   mix_out  fp32 [M, mix] (contiguous), sq_out fp32 [M]
 *   workspace / workspace_bytes: device scratch, see hc_mix_workspace_bytes. */
hcmix_status hc_mix_stats(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                          int64_t M, int64_t K, int mix, float* mix_out, float* sq_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The epilogue alone, from mix[M, mix] and sq[M] (fp32, device, contiguous):
 * writes pre[M, hc], post[M, hc], comb[M, hc, hc] (fp32, contiguous).
 * hc_scale: fp32[3] device; hc_base: fp32[mix] device.  K only sets 1/K. */
hcmix_status hc_mix_sinkhorn(const float* mix, const float* sq, int64_t M, int64_t K, int mixn,
                             int hc, const float* hc_scale, const float* hc_base,
                             int sinkhorn_iters, float rms_eps, float hc_eps,
                             float* pre, float* post, float* comb, void* stream);

/* The whole path: contraction, sum of squares and epilogue.  mix_out / sq_out
 * may be NULL; when given they receive the intermediate statistics. */
hcmix_status hc_mix_fused(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                          int64_t M, int64_t K, int mix, int hc,
                          const float* hc_scale, const float* hc_base, int sinkhorn_iters,
                          float rms_eps, float hc_eps,
                          float* pre, float* post, float* comb,
                          float* mix_out, float* sq_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/* As hc_mix_stats / hc_mix_fused with an explicit kernel path (for tests and
 * benchmarks); HCMIX_PATH_AUTO gives the plain entry points' choice. */
hcmix_status hc_mix_stats_ex(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                             int64_t M, int64_t K, int mix, float* mix_out, float* sq_out,
                             void* workspace, size_t workspace_bytes, void* stream,
                             hcmix_path path);
hcmix_status hc_mix_fused_ex(const void* x, int64_t x_stride, const float* W, int64_t w_stride,
                             int64_t M, int64_t K, int mix, int hc,
                             const float* hc_scale, const float* hc_base, int sinkhorn_iters,
                             float rms_eps, float hc_eps,
                             float* pre, float* post, float* comb,
                             float* mix_out, float* sq_out,
                             void* workspace, size_t workspace_bytes, void* stream,
                             hcmix_path path);

/* The contraction phase alone (the dominant kernel of hc_mix_stats and
 * hc_mix_fused): writes the per-slice partial totals (HCMIX_PATH_SIMT_FULLK:
 * the one running total) into the workspace and nothing else.  Arguments as hc_mix_stats_ex.  For timing and profiling the
 * phase on its own stream position; the partials are not a public format. */
hcmix_status hc_mix_contract_ex(const void* x, int64_t x_stride, const float* W,
                                int64_t w_stride, int64_t M, int64_t K, int mix,
                                void* workspace, size_t workspace_bytes, void* stream,
                                hcmix_path path);

/* W packed once, for callers whose weight does not change between calls (a
 * model layer's W during inference).  The hc_fused page has no counterpart:
 * its kernel reads fp32 W on every call, and so do hc_mix_fused and
 * hc_mix_stats, whose tensor-core path converts W into its MMA operand format
 * each time.  hc_mix_pack_w does that conversion once into a caller buffer
 * (packed_w, 256-byte aligned, hc_mix_packed_w_bytes(K, mix) bytes: the exact
 * bf16 limbs W = w0 + w1 + w2 + w3, an opaque format tied to this library
 * build), and hc_mix_fused_packed runs the tensor-core path (exact limbs) on
 * it.  Its results are bit-identical to hc_mix_fused's tensor-core path on the
 * same W.  Repack after W changes.  Other arguments, validation and error
 * behaviour follow hc_mix_fused (x / workspace) and hc_mix_stats (W). */
size_t hc_mix_packed_w_bytes(int64_t K, int mix);
hcmix_status hc_mix_pack_w(const float* W, int64_t w_stride, int64_t K, int mix, void* packed_w,
                           size_t packed_bytes, void* stream);
hcmix_status hc_mix_fused_packed(const void* x, int64_t x_stride, const void* packed_w,
                                 size_t packed_bytes, int64_t M, int64_t K, int mix, int hc,
                                 const float* hc_scale, const float* hc_base, int sinkhorn_iters,
                                 float rms_eps, float hc_eps, float* pre, float* post,
                                 float* comb, float* mix_out, float* sq_out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* The path HCMIX_PATH_AUTO takes for M rows. */
hcmix_path hc_mix_auto_path(int64_t M);

/* hc_mix_fused without a workspace argument, for callers that cannot hand the
 * library any device memory of their own: for example an engine that reserves
 * its whole device memory budget at start-up and forbids any later
 * cudaMalloc (a late allocation can fail, fragment its pool or synchronise
 * the device), or a plug-in living inside a host framework that owns every
 * device allocation.  The hc_fused page has no counterpart; this is a
 * convenience of this library.
 *
 * Instead of a caller workspace it uses a fixed scratch array of
 * HC_MIX_STATIC_SCRATCH_BYTES (2 MiB) that the library defines in device
 * memory; every GPU that loads libhcmix.so holds that array until the process
 * exits.  It runs hc_mix_fused's default path (HCMIX_PATH_AUTO: the
 * tensor-core kernel on GB300) with that array as its workspace, and
 * allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Limit: hc_mix_workspace_bytes(M, K, mix) must fit the scratch, i.e.
 *     M <= 256 at K = 20480.  Larger problems return HCMIX_ERR_WORKSPACE
 *     before anything is launched.
 *   - The array's header holds the device error word of these calls:
 *     hc_mix_noalloc_device_status reads (and clears) it.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address once and keeps it for later calls; make that
 *     first call before any stream capture starts on that device.  The kept
 *     address belongs to the device's current context: after a context reset
 *     (cudaDeviceReset, or a primary context released and created again) it no
 *     longer points at the array, so do not call this entry point again in a
 *     process that has reset the device.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Every call writes all the scratch it reads, so nothing needs clearing,
 *     but calls whose kernels overlap on the GPU (different streams, or
 *     different host threads on the same device) race on the array: order
 *     them on one stream or serialise them.
 * Other arguments, outputs and error behaviour are those of hc_mix_fused. */
#define HC_MIX_STATIC_SCRATCH_BYTES (2u << 20)
hcmix_status hc_mix_fused_noalloc(const void* x, int64_t x_stride, const float* W,
                                  int64_t w_stride, int64_t M, int64_t K, int mix, int hc,
                                  const float* hc_scale, const float* hc_base,
                                  int sinkhorn_iters, float rms_eps, float hc_eps,
                                  float* pre, float* post, float* comb,
                                  float* mix_out, float* sq_out, void* stream);

/* The device error word of hc_mix_fused_noalloc's calls on the current
 * device (the kernel status of hc_mix_device_status, read from the fixed
 * scratch array): synchronises `stream`, returns HCMIX_OK when clean or the
 * recorded error, and clears it.  HCMIX_ERR_CUDA if the array's address cannot
 * be looked up (see the notes on hc_mix_fused_noalloc). */
hcmix_status hc_mix_noalloc_device_status(void* stream);

/* Synchronises `stream`, then reads and clears the device error word that
 * kernels set in `workspace` when a bounded wait runs out.  HCMIX_OK when clean,
 * HCMIX_ERR_DEVICE when a kernel recorded an error, HCMIX_ERR_CUDA when the
 * stream reports a CUDA error. */
hcmix_status hc_mix_device_status(void* workspace, void* stream);

/* Static, human-readable name of a status. */
const char* hc_mix_status_string(hcmix_status status);

#ifdef __cplusplus
}
#endif

#endif /* HCMIX_H */
