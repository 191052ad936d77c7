// rowquant.cuh -- RMSNorm + per-token absmax int8 quantisation of one row, the
// arithmetic every kernel of this library uses for it, so that all launch paths
// (separate norm kernel, fused decode prologue) round identically.
//
// "BitNet Embeddings GGUF Conversion Implementation", section 1 ("Background")
// and section 4.5 (ggml_rms_norm, then ggml_mul by the projection's norm
// weight); "BitNet Inference Framework", "Quantization (W1.58A8)" (per-token
// absmax 8-bit activations).  Definition: rstd = 1/sqrt(sum(x^2)/K + eps)
// rounded once to float; xn = (x * rstd) * g; a_scale = 127 / max(max|xn|,
// 1e-5); q = clamp(rint(xn * a_scale), -128, 127); every float operation a
// single correctly rounded one (no FMA contraction).
//
// GB300 has almost no FP64 throughput: the sum of squares is integer arithmetic
// (below, exact up to a per-term truncation under 2^-46 of the largest square)
// and rstd is carried in an fp32 pair (hi + lo) to ~2^-44 before its single
// rounding to float, so it equals the float rounding of the exact value unless
// that value lies within ~2^-43 (relative) of a float rounding boundary.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bitnet {

// Unevaluated sum hi + lo of two floats.
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

// ----------------------------------------------------------- sum of squares
// The sum of squares of a row is an exact integer sum, so it does not depend on
// how a kernel splits the row over lanes, warps or passes: every launch path
// gets the same bits.  With x = m * 2^(e-150) (m the 24-bit significand, e the
// biased exponent, 1 for subnormals) and emax the row's largest e, each square
// contributes the integer m^2 >> (2(emax - e) + 1), i.e. x^2 in units of
// 2^(2 emax - 299) truncated to an integer.  The largest term is below 2^47, so
// 65536 of them fit in 64 bits; each truncation is below 2^-46 of the row's
// largest square.
__device__ __forceinline__ int sq_exp(float x) {
  const unsigned b = __float_as_uint(x) & 0x7fffffffu;
  const int ef = static_cast<int>(b >> 23);
  return ef ? ef : (b ? 1 : 0);
}

__device__ __forceinline__ int sq_exp4(float4 v) {
  return max(max(sq_exp(v.x), sq_exp(v.y)), max(sq_exp(v.z), sq_exp(v.w)));
}

__device__ __forceinline__ unsigned long long sq_term(float x, int emax) {
  const unsigned b = __float_as_uint(x) & 0x7fffffffu;
  const int ef = static_cast<int>(b >> 23);
  const unsigned m = (b & 0x7fffffu) | (ef ? 0x800000u : 0u);
  const int e = ef ? ef : 1;
  const int d = max(2 * (emax - e) + 1, 1);  // >= 1; emax == 0 only for an all-zero row
  const unsigned long long sq = static_cast<unsigned long long>(m) * m;
  return d < 64 ? (sq >> d) : 0ull;
}

__device__ __forceinline__ unsigned long long sq_term4(float4 v, int emax) {
  return (sq_term(v.x, emax) + sq_term(v.y, emax)) + (sq_term(v.z, emax) + sq_term(v.w, emax));
}

// Warp-wide exact sum of per-lane partial sums (the total stays below 2^63):
// three 22-bit limbs, each summed by one redux instruction.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
  const unsigned l0 = static_cast<unsigned>(v) & 0x3fffffu;
  const unsigned l1 = static_cast<unsigned>(v >> 22) & 0x3fffffu;
  const unsigned l2 = static_cast<unsigned>(v >> 44);
  const unsigned long long s0 = __reduce_add_sync(0xffffffffu, l0);
  const unsigned long long s1 = __reduce_add_sync(0xffffffffu, l1);
  const unsigned long long s2 = __reduce_add_sync(0xffffffffu, l2);
  return s0 + (s1 << 22) + (s2 << 44);
}

__device__ __forceinline__ int warp_max_int(int v) {
  return static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<unsigned>(v)));
}

// f * 2^e, exact whenever the result is a normal float (f a small integer).
__device__ __forceinline__ float mul_pow2(float f, int e) {
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int step = e > 127 ? 127 : (e < -126 ? -126 : e);
    f = __fmul_rn(f, __int_as_float((step + 127) << 23));
    e -= step;
  }
  return f;
}

// The fixed-point sum as an fp32 pair (its top 48 bits).
__device__ __forceinline__ DF sq_to_df(unsigned long long acc, int emax) {
  if (acc == 0ull) return DF{0.0f, 0.0f};
  const int p = 63 - __clzll(static_cast<long long>(acc));
  const unsigned long long t = acc << (63 - p);  // leading one at bit 63
  const int base = p - 63 + 2 * emax - 299;      // acc = t * 2^(p-63), one unit = 2^(2 emax - 299)
  const float fh = static_cast<float>(static_cast<unsigned>(t >> 40));                  // exact (< 2^24)
  const float fl = static_cast<float>(static_cast<unsigned>((t >> 16) & 0xffffffull));  // exact (< 2^24)
  const float h = mul_pow2(fh, base + 40);
  const float l = mul_pow2(fl, base + 16);
  const float s = __fadd_rn(h, l);
  return DF{s, __fsub_rn(l, __fsub_rn(s, h))};
}

// Sum of squares of a row read by one full warp (global or shared memory).
template <bool kGlobal>
__device__ __forceinline__ DF warp_row_sumsq(const float* __restrict__ xrow, int K, int lane) {
  const float* p = xrow + 4 * lane;
  const int nc = K >> 7;
  int e = 0;
  for (int c = 0; c < nc; ++c)
    e = max(e, sq_exp4(kGlobal ? __ldg(reinterpret_cast<const float4*>(p + 128 * c))
                               : *reinterpret_cast<const float4*>(p + 128 * c)));
  const int emax = warp_max_int(e);
  unsigned long long acc = 0ull;
  for (int c = 0; c < nc; ++c)
    acc += sq_term4(kGlobal ? __ldg(reinterpret_cast<const float4*>(p + 128 * c))
                            : *reinterpret_cast<const float4*>(p + 128 * c),
                    emax);
  return sq_to_df(warp_sum_u64(acc), emax);
}

// rstd = 1 / sqrt(ss/K + eps), rounded once to float.  ss/K + eps is formed as
// an fp32 pair (quotient by the reciprocal of K; the remainder hi - q*K is
// exact by fma since q is within a few ulp of hi/K and K < 2^23); 1/sqrt by the
// hardware estimate refined with one Newton step whose residual 1 - v*y0^2 is
// evaluated to ~2^-47.
__device__ __forceinline__ float rstd_from_sumsq(DF ss, int K, float eps) {
  const float kf = static_cast<float>(K);  // exact
  const float rk = __frcp_rn(kf);
  const float q = __fmul_rn(ss.hi, rk);
  const float rem = __fmaf_rn(-q, kf, ss.hi);  // exact
  const float ql = __fmul_rn(__fadd_rn(rem, ss.lo), rk);
  DF v = df_add(DF{q, ql}, DF{eps, 0.0f});
  const float y0 = rsqrtf(v.hi);
  const float s_hi = __fmul_rn(y0, y0);
  const float s_lo = __fmaf_rn(y0, y0, -s_hi);  // y0^2 = s_hi + s_lo exactly
  const float t_hi = __fmul_rn(v.hi, s_hi);
  const float t_err = __fmaf_rn(v.hi, s_hi, -t_hi);
  // e = 1 - v*y0^2; 1 - t_hi is exact (t_hi is within a few ulp of 1)
  const float small = __fadd_rn(__fadd_rn(t_err, __fmul_rn(v.hi, s_lo)), __fmul_rn(v.lo, s_hi));
  const float e = __fsub_rn(__fsub_rn(1.0f, t_hi), small);
  const float c = __fmul_rn(__fmul_rn(y0, e), 0.5f);
  return __fadd_rn(y0, c);
}

__device__ __forceinline__ float norm_elem(float x, float rstd, float g) {
  return __fmul_rn(__fmul_rn(x, rstd), g);
}

__device__ __forceinline__ float act_scale_from_amax(float amax) {
  return __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
}

// rint then clamp: cvt.rni rounds half to even exactly like rintf, and the
// product's magnitude never exceeds ~127, far inside the int range.
__device__ __forceinline__ int quant_elem(float xn, float a_scale) {
  return min(max(__float2int_rn(__fmul_rn(xn, a_scale)), -128), 127);
}

// y = ((float)acc * (1/a_scale)) * (1/w_scale): the reciprocals are passed in.
__device__ __forceinline__ float rescale_elem(float acc_f, float inv_a, float inv_w) {
  return __fmul_rn(__fmul_rn(acc_f, inv_a), inv_w);
}

// Max of non-negative floats across the warp (their bit patterns order alike).
__device__ __forceinline__ float warp_max(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

__device__ __forceinline__ int warp_sum_int(int v) {
  return static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(v)));
}

}  // namespace bitnet
