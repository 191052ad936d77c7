// rowquant.cuh -- RMSNorm + per-token absmax int8 quantisation of one row, the
// arithmetic every kernel of this library uses for it, so that all launch paths
// (separate norm kernel, fused decode prologue) round identically.
//
// "BitNet Embeddings GGUF Conversion Implementation", section 1 ("Background")
// and section 4.5 (ggml_rms_norm, then ggml_mul by the projection's norm
// weight); "BitNet Inference Framework", "Quantization (W1.58A8)" (per-token
// absmax 8-bit activations).  Readings: sum of squares and square root in
// double, rstd rounded once to float; xn = (x * rstd) * g; a_scale = 127 /
// max(max|xn|, 1e-5); q = clamp(rint(xn * a_scale), -128, 127); every float
// operation a single correctly rounded one (no FMA contraction).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bitnet {

// Unevaluated sum hi + lo of two floats (about 48 significant bits).
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s = __fadd_rn(a.hi, b.hi);
  float bb = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));  // exact error of s
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  float hi = __fadd_rn(s, e);
  float lo = __fsub_rn(e, __fsub_rn(hi, s));
  return DF{hi, lo};
}

// x*x split exactly into a rounded product and its rounding error.
__device__ __forceinline__ DF df_sq(float x) {
  float p = __fmul_rn(x, x);
  return DF{p, __fmaf_rn(x, x, -p)};
}

// Sum of squares of one row, computed by one full warp.  Lane l owns the float4
// groups at k = 4*l + 128*c (c = 0 .. K/128-1); each of its four components
// accumulates in its own DF over c ascending; the four are combined as
// (0+1)+(2+3); the 32 lanes by an xor butterfly 16, 8, 4, 2, 1.  The result
// (identical in every lane) is accurate to about 2^-44 relative, far inside
// double rounding of the oracle's sequential sum, and bit-identical wherever
// this function is called.  |x| must stay below 1.8e19 (x*x finite in float).
__device__ __forceinline__ double warp_row_sumsq(const float* __restrict__ xrow, int K, int lane) {
  DF a0{0.f, 0.f}, a1{0.f, 0.f}, a2{0.f, 0.f}, a3{0.f, 0.f};
  const int nc = K >> 7;
#pragma unroll 4
  for (int c = 0; c < nc; ++c) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(xrow + 4 * lane + 128 * c));
    a0 = df_add(a0, df_sq(v.x));
    a1 = df_add(a1, df_sq(v.y));
    a2 = df_add(a2, df_sq(v.z));
    a3 = df_add(a3, df_sq(v.w));
  }
  DF t = df_add(df_add(a0, a1), df_add(a2, a3));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    DF o{__shfl_xor_sync(0xffffffffu, t.hi, off), __shfl_xor_sync(0xffffffffu, t.lo, off)};
    // xor partners add in opposite orders; make the pair order canonical so both
    // get bit-identical sums (lower lane's value first).
    t = (lane & off) ? df_add(o, t) : df_add(t, o);
  }
  return static_cast<double>(t.hi) + static_cast<double>(t.lo);
}

__device__ __forceinline__ float rstd_from_sumsq(double ss, int K, float eps) {
  return static_cast<float>(1.0 / sqrt(ss / static_cast<double>(K) + static_cast<double>(eps)));
}

__device__ __forceinline__ float norm_elem(float x, float rstd, float g) {
  return __fmul_rn(__fmul_rn(x, rstd), g);
}

__device__ __forceinline__ float act_scale_from_amax(float amax) {
  return __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
}

__device__ __forceinline__ int quant_elem(float xn, float a_scale) {
  float v = rintf(__fmul_rn(xn, a_scale));
  v = fminf(fmaxf(v, -128.0f), 127.0f);
  return static_cast<int>(v);
}

// y = ((float)acc * (1/a_scale)) * (1/w_scale): the reciprocals are passed in.
__device__ __forceinline__ float rescale_elem(float acc_f, float inv_a, float inv_w) {
  return __fmul_rn(__fmul_rn(acc_f, inv_a), inv_w);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

}  // namespace bitnet
