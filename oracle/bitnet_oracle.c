/*
 * bitnet_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU statement of what one W1.58A8 BitLinear projection computes,
 * used by the tests, by __graft_entry__.smoke() and by the CPU-baseline leg of
 * bench.py to check the CUDA library.  It shares no code, header, table or
 * helper with the CUDA path, and the library never calls it.
 *
 * Every function follows one passage of the source pages:
 *   [P1-1]  "BitNet Embeddings GGUF Conversion Implementation", section 1
 *           "Background" (the per-projection chain and the eps of the models)
 *   [P1-3]  same page, section 3, "I2_S Ternary Packing"
 *   [P1-45] same page, section 4.5 "load_tensors" (ggml_rms_norm then ggml_mul
 *           by the projection's norm weight, then ggml_mul_mat)
 *   [P1-64] same page, section 6.4 (int8 x I2_S dot products, vec_dot_i2_i8_s)
 *   [P2-QE] "BitNet Inference Framework", "Quantization and Encoding" and
 *           "Data Layout"
 *   [P2-WA] same page, "Quantization (W1.58A8)" (absmean ternary weights,
 *           per-token absmax 8-bit activations) and "Architectural Details"
 *           (no bias terms)
 *   [P4-R]  "gguf-gemv", "Requirements" (K a multiple of 128 for I2_S) and its
 *           description of I2_S (codes {0,1,2} -> {-1,0,+1}, one f32 scale)
 *   [P1-FF] "BitNet Embeddings GGUF Conversion Implementation", section 4.5,
 *           "FFN per-projection norms" (activation of the gate projection times
 *           the up projection, then the down projection's own norm and matmul),
 *           with the activations of section 1's table: SiLU (Qwen3) and
 *           gelu_pytorch_tanh (Gemma3)
 *
 * Readings where the pages are silent (the same ones the library header states):
 *   - which elements share a byte: byte j of a block holds elements j, 32+j,
 *     64+j, 96+j as c0..c3;
 *   - "round" is round-half-to-even (rint);
 *   - mean(|w|) is summed in double in index order; all-zero -> w_scale 1;
 *   - activation scale 127 / max(max|xn|, 1e-5), codes clamped to [-128, 127];
 *   - RMSNorm sum of squares in double in index order, eps added to the mean,
 *     rstd rounded once to float, then (x * rstd) * g in float;
 *   - y = ((float)acc * (1/a_scale)) * (1/w_scale) in float.
 *   - the down projection's input h = act(gate) * up: the activation evaluated
 *     in double and rounded once to float, then one float multiply by up;
 *     SiLU(x) = x / (1 + e^-x), gelu_pytorch_tanh(x) = x/2 (1 + tanh(sqrt(2/pi)
 *     (x + 0.044715 x^3))).
 * Build with -O2 -ffp-contract=off and no fast-math: every float operation above
 * is a single correctly rounded IEEE operation.
 *
 * Parity pins (tests/test_oracle_pins.py) tie each function to something other
 * than itself: hand-derived byte patterns from the packing passage, the Gaussian
 * zero fraction of absmean quantisation in closed form, torch's rms_norm in
 * float64, numpy integer matmul, brute-force fp64 dot products and quantisation
 * error bounds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- weights --- */

/* [P1-3], [P2-QE]: scale = 1 / mean(|w|) over the whole tensor. */
double oracle_mean_abs(const float* w, int64_t count) {
  double s = 0.0;
  for (int64_t i = 0; i < count; ++i) s += fabs((double)w[i]);
  return s / (double)count;
}

float oracle_weight_scale(const float* w, int64_t count) {
  double mean = oracle_mean_abs(w, count);
  if (mean == 0.0) return 1.0f; /* reading: an all-zero tensor keeps scale 1 */
  return (float)(1.0 / mean);
}

/* [P1-3], [P2-QE]: q = round(w * scale).clamp(-1, 1); one float multiply,
 * rint = round half to even. */
void oracle_quantize_ternary(const float* w, int64_t count, float w_scale, int8_t* q) {
  for (int64_t i = 0; i < count; ++i) {
    float t = w[i] * w_scale;
    float r = rintf(t);
    if (r > 1.0f) r = 1.0f;
    if (r < -1.0f) r = -1.0f;
    q[i] = (int8_t)r;
  }
}

/* [P1-3], [P2-QE]: encode -1 -> 0, 0 -> 1, +1 -> 2; 128 values per 32-byte block,
 * byte = (c0 << 6) | (c1 << 4) | (c2 << 2) | c3 with (reading) c_s taken from
 * element 32*s + j of the block for byte j; the fp32 scale follows the last
 * block.  W is [N, K] row-major, so block b of the flat tensor is row b / (K/128). */
int oracle_encode_i2s(const int8_t* q, int64_t N, int64_t K, float w_scale, uint8_t* packed) {
  if (N < 1 || K < 128 || K % 128 != 0) return 1;
  int64_t nblocks = N * K / 128;
  for (int64_t b = 0; b < nblocks; ++b) {
    const int8_t* v = q + b * 128;
    uint8_t* out = packed + b * 32;
    for (int j = 0; j < 32; ++j) {
      unsigned c0 = (unsigned)(v[j] + 1);
      unsigned c1 = (unsigned)(v[32 + j] + 1);
      unsigned c2 = (unsigned)(v[64 + j] + 1);
      unsigned c3 = (unsigned)(v[96 + j] + 1);
      out[j] = (uint8_t)((c0 << 6) | (c1 << 4) | (c2 << 2) | c3);
    }
  }
  memcpy(packed + N * K / 4, &w_scale, 4); /* little-endian hosts only (x86-64, aarch64) */
  return 0;
}

/* The full conversion of one weight tensor with a given scale. */
int oracle_pack_i2s_with_scale(const float* w, int64_t N, int64_t K, float w_scale,
                               uint8_t* packed) {
  if (N < 1 || K < 128 || K % 128 != 0) return 1;
  int8_t* q = (int8_t*)malloc((size_t)(N * K));
  if (!q) return 2;
  oracle_quantize_ternary(w, N * K, w_scale, q);
  int rc = oracle_encode_i2s(q, N, K, w_scale, packed);
  free(q);
  return rc;
}

int oracle_pack_i2s(const float* w, int64_t N, int64_t K, uint8_t* packed, float* w_scale_out) {
  if (N < 1 || K < 128 || K % 128 != 0) return 1;
  float s = oracle_weight_scale(w, N * K);
  if (w_scale_out) *w_scale_out = s;
  return oracle_pack_i2s_with_scale(w, N, K, s, packed);
}

/* [P2-QE], [P4-R]: decode code -> code - 1.  Code 3 never comes out of the
 * encoder; it decodes to +2 (reading: the plain arithmetic code - 1). */
int oracle_unpack_i2s(const uint8_t* packed, int64_t N, int64_t K, int8_t* q) {
  if (N < 1 || K < 128 || K % 128 != 0) return 1;
  int64_t nblocks = N * K / 128;
  for (int64_t b = 0; b < nblocks; ++b) {
    const uint8_t* in = packed + b * 32;
    int8_t* v = q + b * 128;
    for (int j = 0; j < 32; ++j) {
      v[j] = (int8_t)((int)((in[j] >> 6) & 3) - 1);
      v[32 + j] = (int8_t)((int)((in[j] >> 4) & 3) - 1);
      v[64 + j] = (int8_t)((int)((in[j] >> 2) & 3) - 1);
      v[96 + j] = (int8_t)((int)(in[j] & 3) - 1);
    }
  }
  return 0;
}

/* Number of 2-bit fields holding the invalid code 3. */
int64_t oracle_count_invalid_codes(const uint8_t* packed, int64_t N, int64_t K) {
  int64_t bad = 0;
  for (int64_t i = 0; i < N * K / 4; ++i)
    for (int s = 0; s < 4; ++s)
      if (((packed[i] >> (2 * s)) & 3) == 3) ++bad;
  return bad;
}

/* ------------------------------------------------------------ activations --- */

/* [P1-45], [P1-1]: ggml_rms_norm(x, eps) then ggml_mul by the norm weight. */
void oracle_rmsnorm(const float* x, const float* g, int64_t M, int64_t K, float eps,
                    float* xn, float* rstd_out) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const float* xr = x + m * K;
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) ss += (double)xr[k] * (double)xr[k];
    float rstd = (float)(1.0 / sqrt(ss / (double)K + (double)eps));
    if (rstd_out) rstd_out[m] = rstd;
    for (int64_t k = 0; k < K; ++k) {
      float t = xr[k] * rstd;
      xn[m * K + k] = t * g[k];
    }
  }
}

/* [P1-FF]: the gate activation.  act 1: SiLU, act 2: gelu_pytorch_tanh. */
double oracle_activation(double x, int act) {
  if (act == 1) return x / (1.0 + exp(-x));
  if (act == 2) {
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
  }
  return x;
}

/* [P1-FF]: h = act(gate) * up elementwise, the input of the down projection. */
void oracle_glu(const float* gate, const float* up, int64_t count, int act, float* h) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    float a = (float)oracle_activation((double)gate[i], act);
    h[i] = a * up[i];
  }
}

/* [P2-WA]: per-token absmax quantisation to 8 bits. */
void oracle_quant_a8(const float* xn, int64_t M, int64_t K, int8_t* q, float* a_scale,
                     int32_t* rowsum) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const float* r = xn + m * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float a = fabsf(r[k]);
      if (a > amax) amax = a;
    }
    float s = 127.0f / (amax > 1e-5f ? amax : 1e-5f);
    a_scale[m] = s;
    int32_t sum = 0;
    for (int64_t k = 0; k < K; ++k) {
      float t = r[k] * s;
      float v = rintf(t);
      if (v > 127.0f) v = 127.0f;
      if (v < -128.0f) v = -128.0f;
      q[m * K + k] = (int8_t)v;
      sum += (int32_t)v;
    }
    if (rowsum) rowsum[m] = sum;
  }
}

/* ----------------------------------------------------------- contraction --- */

/* [P1-64], [P1-1]: acc[m, n] = sum_k q[m, k] * t[n, k] with t the decoded
 * ternary weights, exact in 64-bit integers.  No bias ([P2-WA]). */
int oracle_i2s_matmul(const int8_t* q, const uint8_t* packed, int64_t M, int64_t K, int64_t N,
                      int64_t* acc) {
  if (N < 1 || K < 128 || K % 128 != 0) return 1;
  int8_t* t = (int8_t*)malloc((size_t)(N * K));
  if (!t) return 2;
  oracle_unpack_i2s(packed, N, K, t);
  /* every output is one sequential sum of its own; threads share the (m, n)
     pairs, so a single token row still spreads over the host's cores */
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      int64_t s = 0;
      for (int64_t k = 0; k < K; ++k) s += (int64_t)q[m * K + k] * (int64_t)t[n * K + k];
      acc[m * N + n] = s;
    }
  free(t);
  return 0;
}

/* Rescale by the two quantisation scales: the codes stand for xn * a_scale and
 * w * w_scale, so the product is divided by both (as reciprocals, in float). */
void oracle_rescale(const int64_t* acc, const float* a_scale, float w_scale, int64_t M,
                    int64_t N, float* y) {
  float inv_w = 1.0f / w_scale;
  for (int64_t m = 0; m < M; ++m) {
    float inv_a = 1.0f / a_scale[m];
    for (int64_t n = 0; n < N; ++n) {
      float a = (float)acc[m * N + n];
      float t = a * inv_a;
      y[m * N + n] = t * inv_w;
    }
  }
}

/* The whole projection for the rows listed in `rows` (all rows when rows is
 * NULL; then n_rows must equal M).  Intermediates are returned when the
 * corresponding pointer is non-NULL, each laid out [n_rows, ...]. */
int oracle_bitlinear_forward_rows(const float* x, const float* g, const uint8_t* packed,
                                  float w_scale, int64_t M, int64_t K, int64_t N, float eps,
                                  const int64_t* rows, int64_t n_rows, float* y,
                                  float* xn_out, int8_t* q_out, float* a_scale_out,
                                  int64_t* acc_out) {
  if (M < 1 || N < 1 || K < 128 || K % 128 != 0 || n_rows < 1) return 1;
  float* xs = (float*)malloc((size_t)(n_rows * K) * sizeof(float));
  float* xn = (float*)malloc((size_t)(n_rows * K) * sizeof(float));
  int8_t* q = (int8_t*)malloc((size_t)(n_rows * K));
  float* as = (float*)malloc((size_t)n_rows * sizeof(float));
  int64_t* acc = (int64_t*)malloc((size_t)(n_rows * N) * sizeof(int64_t));
  int rc = 0;
  if (!xs || !xn || !q || !as || !acc) {
    rc = 2;
    goto done;
  }
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= M) {
      rc = 1;
      goto done;
    }
    memcpy(xs + i * K, x + r * K, (size_t)K * sizeof(float));
  }
  oracle_rmsnorm(xs, g, n_rows, K, eps, xn, NULL);
  oracle_quant_a8(xn, n_rows, K, q, as, NULL);
  rc = oracle_i2s_matmul(q, packed, n_rows, K, N, acc);
  if (rc) goto done;
  oracle_rescale(acc, as, w_scale, n_rows, N, y);
  if (xn_out) memcpy(xn_out, xn, (size_t)(n_rows * K) * sizeof(float));
  if (q_out) memcpy(q_out, q, (size_t)(n_rows * K));
  if (a_scale_out) memcpy(a_scale_out, as, (size_t)n_rows * sizeof(float));
  if (acc_out) memcpy(acc_out, acc, (size_t)(n_rows * N) * sizeof(int64_t));
done:
  free(xs);
  free(xn);
  free(q);
  free(as);
  free(acc);
  return rc;
}

/* Brute force in double of the same product: sum_k q * t / a_scale / w_scale. */
void oracle_dequant_dot_f64(const int8_t* q, const int8_t* t, const float* a_scale,
                            float w_scale, int64_t M, int64_t K, int64_t N, double* y) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k)
        s += ((double)q[m * K + k] / (double)a_scale[m]) * ((double)t[n * K + k] / (double)w_scale);
      y[m * N + n] = s;
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
