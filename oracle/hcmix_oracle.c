/*
 * CPU oracle for the hyper-connection mix-statistics path.
 *
 * TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / --impl reference legs may load this file's library. The CUDA
 * product path never links, loads or calls it, and it shares no code with it.
 *
 * Source: "launcher/docker-images/mia-tp4/adapter/hc_fused.py" (the hc_fused
 * page), module docstring and _hc_mix_fullk_kernel / _sq_tree /
 * fused_mix_stats_sinkhorn.  Per row m of x[M, K] (bf16) and W[mix, K] (fp32):
 *
 *   K is walked in slices of 256 columns, each slice in four chunks of 64.
 *   mix[m, j]: every chunk's dot product d starts from zero; a slice total acc
 *     starts from zero and adds its four chunk dots in order; the grand total
 *     starts from zero and adds the slice totals in slice order
 *     (docstring bullet 1; kernel loop body and slice-boundary update).
 *   sq[m]: every chunk's x^2 values are summed by a fixed tree: pairs whose
 *     column index differs in bit 4, then bit 3, 2, 1, 0, and finally the two
 *     32-column halves (docstring bullet 3; _sq_tree).  Chunk sums feed slice
 *     totals and slice totals feed the grand total exactly like mix.
 *   epilogue (the page names the reduce+Sinkhorn kernel but its text stops
 *     before that kernel's body, so the formulae are fixed here as the plain
 *     RMS-scaled logits, sigmoids and Sinkhorn): r = 1/sqrt(sq * (1/K) + rms_eps);
 *     logit[j] = mix[j] * r * hc_scale[g(j)] + hc_base[j] with g = 0 for
 *     j < hc, 1 for hc <= j < 2hc, 2 otherwise; pre = sigmoid(logit[0:hc]);
 *     post = 2 sigmoid(logit[hc:2hc]); comb = sinkhorn_iters rounds of
 *     (row normalisation, then column normalisation) of exp(logit[2hc:])
 *     viewed row-major as hc x hc.
 *
 * Readings where the page leaves a step open (each listed in the design notes):
 *   - chunk dot: the page takes it from tensor-core MMAs whose internal order
 *     is not specified.  The oracle uses the plain definition: the 64 products
 *     are exact in double (8-bit x significand times 24-bit W significand), are
 *     summed in double in ascending k, and the sum is rounded once to fp32.
 *   - 1/K is formed in double and rounded to fp32 (the page passes 1.0 / k).
 *   - hc_eps is added to every Sinkhorn row and column sum before dividing.
 *   - sigmoid(z) = 1 / (1 + exp(-z)); libm expf; Sinkhorn sums in index order.
 *
 * Compile with -ffp-contract=off (no fused multiply-add contraction); every
 * float operation below is one IEEE round-to-nearest operation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define CHUNK 64
#define SLICE 256

static float bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Chunk dot of n consecutive columns: double accumulation in ascending k,
 * rounded once to fp32.  Products are exact in double. */
float oracle_chunk_dot(const uint16_t* x, const float* w, int n) {
  double s = 0.0;
  for (int k = 0; k < n; ++k) s += (double)bf16_to_f32(x[k]) * (double)w[k];
  return (float)s;
}

/* The same chunk dot accumulated in fp32, product rounded then sum rounded,
 * ascending k.  Used only to show how far a different in-chunk order drifts. */
float oracle_chunk_dot_seq_f32(const uint16_t* x, const float* w, int n) {
  float s = 0.0f;
  for (int k = 0; k < n; ++k) {
    float p = bf16_to_f32(x[k]) * w[k];
    s = s + p;
  }
  return s;
}

/* The fixed sum-of-squares tree over one 64-column chunk (_sq_tree). */
float oracle_sq_tree(const uint16_t* x) {
  float v[CHUNK];
  for (int k = 0; k < CHUNK; ++k) {
    float f = bf16_to_f32(x[k]);
    v[k] = f * f; /* exact for bf16 inputs */
  }
  /* Combine pairs that differ in bit b, for b = 4, 3, 2, 1, 0.  After the
   * pass for bit b the partial sum for every index with that bit clear sits at
   * that index. */
  static const int bits[5] = {4, 3, 2, 1, 0};
  int done_mask = 0;
  for (int t = 0; t < 5; ++t) {
    int b = 1 << bits[t];
    done_mask |= b;
    for (int i = 0; i < CHUNK; ++i) {
      if (i & done_mask) continue; /* i has every combined bit clear */
      v[i] = v[i] + v[i | b];
    }
  }
  /* v[0] holds the half with k < 32, v[32] the half with k >= 32. */
  return v[0] + v[32];
}

/* mix[row, 0:mix] and sq[row] for rows [row0, row1) with the slice order. */
void oracle_stats(const uint16_t* x, int64_t x_stride, const float* W, int64_t w_stride,
                  int64_t row0, int64_t row1, int64_t K, int mix,
                  float* mix_out, float* sq_out) {
  const int64_t n_slices = K / SLICE;
  for (int64_t m = row0; m < row1; ++m) {
    const uint16_t* xr = x + m * x_stride;
    float tot[64];
    float sqt = 0.0f;
    for (int j = 0; j < mix; ++j) tot[j] = 0.0f;
    for (int64_t s = 0; s < n_slices; ++s) {
      float acc[64];
      float sqs = 0.0f;
      for (int j = 0; j < mix; ++j) acc[j] = 0.0f;
      for (int c = 0; c < SLICE / CHUNK; ++c) {
        int64_t k0 = s * SLICE + (int64_t)c * CHUNK;
        for (int j = 0; j < mix; ++j) {
          float d = oracle_chunk_dot(xr + k0, W + (int64_t)j * w_stride + k0, CHUNK);
          acc[j] = acc[j] + d;
        }
        sqs = sqs + oracle_sq_tree(xr + k0);
      }
      for (int j = 0; j < mix; ++j) tot[j] = tot[j] + acc[j];
      sqt = sqt + sqs;
    }
    for (int j = 0; j < mix; ++j) mix_out[m * mix + j] = tot[j];
    sq_out[m] = sqt;
  }
}

/* As oracle_stats, but with the fp32 ascending in-chunk accumulation. */
void oracle_stats_seq_f32(const uint16_t* x, int64_t x_stride, const float* W, int64_t w_stride,
                          int64_t row0, int64_t row1, int64_t K, int mix, float* mix_out) {
  const int64_t n_slices = K / SLICE;
  for (int64_t m = row0; m < row1; ++m) {
    const uint16_t* xr = x + m * x_stride;
    for (int j = 0; j < mix; ++j) {
      const float* wr = W + (int64_t)j * w_stride;
      float tot = 0.0f;
      for (int64_t s = 0; s < n_slices; ++s) {
        float acc = 0.0f;
        for (int c = 0; c < SLICE / CHUNK; ++c) {
          int64_t k0 = s * SLICE + (int64_t)c * CHUNK;
          acc = acc + oracle_chunk_dot_seq_f32(xr + k0, wr + k0, CHUNK);
        }
        tot = tot + acc;
      }
      mix_out[m * mix + j] = tot;
    }
  }
}

/* The slice structure carried out entirely in double (fp64 twin). */
void oracle_stats_f64(const uint16_t* x, int64_t x_stride, const float* W, int64_t w_stride,
                      int64_t row0, int64_t row1, int64_t K, int mix,
                      double* mix_out, double* sq_out) {
  const int64_t n_slices = K / SLICE;
  for (int64_t m = row0; m < row1; ++m) {
    const uint16_t* xr = x + m * x_stride;
    double sqt = 0.0;
    for (int j = 0; j < mix; ++j) {
      const float* wr = W + (int64_t)j * w_stride;
      double tot = 0.0;
      for (int64_t s = 0; s < n_slices; ++s) {
        double acc = 0.0;
        for (int c = 0; c < SLICE / CHUNK; ++c) {
          int64_t k0 = s * SLICE + (int64_t)c * CHUNK;
          double d = 0.0;
          for (int k = 0; k < CHUNK; ++k) d += (double)bf16_to_f32(xr[k0 + k]) * (double)wr[k0 + k];
          acc += d;
        }
        tot += acc;
      }
      mix_out[m * mix + j] = tot;
    }
    for (int64_t s = 0; s < n_slices; ++s) {
      double sqs = 0.0;
      for (int64_t k = s * SLICE; k < (s + 1) * SLICE; ++k) {
        double f = (double)bf16_to_f32(xr[k]);
        sqs += f * f;
      }
      sqt += sqs;
    }
    sq_out[m] = sqt;
  }
}

/* Plain unsplit sum over all K in double, no slice structure. */
void oracle_mix_unsplit_f64(const uint16_t* x, int64_t x_stride, const float* W, int64_t w_stride,
                            int64_t row0, int64_t row1, int64_t K, int mix, double* mix_out) {
  for (int64_t m = row0; m < row1; ++m) {
    const uint16_t* xr = x + m * x_stride;
    for (int j = 0; j < mix; ++j) {
      const float* wr = W + (int64_t)j * w_stride;
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += (double)bf16_to_f32(xr[k]) * (double)wr[k];
      mix_out[m * mix + j] = s;
    }
  }
}

static int group_of(int j, int hc) { return j < hc ? 0 : (j < 2 * hc ? 1 : 2); }

/* Sinkhorn on one hc x hc block in place (row pass, then column pass). */
void oracle_sinkhorn(float* c, int hc, int iters, float hc_eps) {
  for (int it = 0; it < iters; ++it) {
    for (int i = 0; i < hc; ++i) {
      float s = 0.0f;
      for (int j = 0; j < hc; ++j) s = s + c[i * hc + j];
      float den = s + hc_eps;
      for (int j = 0; j < hc; ++j) c[i * hc + j] = c[i * hc + j] / den;
    }
    for (int j = 0; j < hc; ++j) {
      float s = 0.0f;
      for (int i = 0; i < hc; ++i) s = s + c[i * hc + j];
      float den = s + hc_eps;
      for (int i = 0; i < hc; ++i) c[i * hc + j] = c[i * hc + j] / den;
    }
  }
}

/* Epilogue for rows [row0, row1): pre[M,hc], post[M,hc], comb[M,hc,hc]. */
void oracle_epilogue(const float* mix_in, const float* sq, int64_t row0, int64_t row1, int64_t K,
                     int mix, int hc, const float* hc_scale, const float* hc_base,
                     int iters, float rms_eps, float hc_eps,
                     float* pre, float* post, float* comb) {
  const float inv_k = (float)(1.0 / (double)K);
  for (int64_t m = row0; m < row1; ++m) {
    const float* mx = mix_in + m * mix;
    float v = sq[m] * inv_k;
    v = v + rms_eps;
    float r = 1.0f / sqrtf(v);
    float logit[64];
    for (int j = 0; j < mix; ++j) {
      float t = mx[j] * r;
      t = t * hc_scale[group_of(j, hc)];
      logit[j] = t + hc_base[j];
    }
    for (int i = 0; i < hc; ++i) {
      pre[m * hc + i] = 1.0f / (1.0f + expf(-logit[i]));
      post[m * hc + i] = 2.0f * (1.0f / (1.0f + expf(-logit[hc + i])));
    }
    float* cm = comb + m * hc * hc;
    for (int e = 0; e < hc * hc; ++e) cm[e] = expf(logit[2 * hc + e]);
    oracle_sinkhorn(cm, hc, iters, hc_eps);
  }
}

/* The epilogue carried out in double, for error estimates of the fp32 one. */
void oracle_epilogue_f64(const double* mix_in, const double* sq, int64_t row0, int64_t row1,
                         int64_t K, int mix, int hc, const float* hc_scale, const float* hc_base,
                         int iters, double rms_eps, double hc_eps,
                         double* pre, double* post, double* comb) {
  for (int64_t m = row0; m < row1; ++m) {
    const double* mx = mix_in + m * mix;
    double r = 1.0 / sqrt(sq[m] / (double)K + rms_eps);
    double logit[64];
    for (int j = 0; j < mix; ++j)
      logit[j] = mx[j] * r * (double)hc_scale[group_of(j, hc)] + (double)hc_base[j];
    for (int i = 0; i < hc; ++i) {
      pre[m * hc + i] = 1.0 / (1.0 + exp(-logit[i]));
      post[m * hc + i] = 2.0 / (1.0 + exp(-logit[hc + i]));
    }
    double* cm = comb + m * hc * hc;
    for (int e = 0; e < hc * hc; ++e) cm[e] = exp(logit[2 * hc + e]);
    for (int it = 0; it < iters; ++it) {
      for (int i = 0; i < hc; ++i) {
        double s = 0.0;
        for (int j = 0; j < hc; ++j) s += cm[i * hc + j];
        for (int j = 0; j < hc; ++j) cm[i * hc + j] /= (s + hc_eps);
      }
      for (int j = 0; j < hc; ++j) {
        double s = 0.0;
        for (int i = 0; i < hc; ++i) s += cm[i * hc + j];
        for (int i = 0; i < hc; ++i) cm[i * hc + j] /= (s + hc_eps);
      }
    }
  }
}
