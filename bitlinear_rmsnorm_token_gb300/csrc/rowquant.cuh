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
// GB300 has almost no FP64 throughput, and its integer ALU pipe runs at half
// the rate of the FMA pipe: the sum of squares is a fixed-point integer sum
// (below) whose per-element work is mostly fp32 multiply/add, accurate to
// ~2^-43 of the row's largest square per element and independent of summation
// order, and rstd is carried in an fp32 pair (hi + lo) to ~2^-44 before its
// single rounding to float, so it equals the float rounding of the exact value
// unless that value lies within ~2^-40 (relative) of a float rounding boundary.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 1.5 * 2^23: adding it to a float of magnitude below 2^22 rounds that float to
// an integer (ties to even, like rintf) held in the low mantissa bits.
constexpr float kRoundMagic = 12582912.0f;
constexpr uint32_t kRoundMagicBits = 0x4B400000u;

// ----------------------------------------------------------- sum of squares
// The sum of squares of a row is an integer sum, so it does not depend on how a
// kernel splits the row over lanes, warps or passes: every launch path gets the
// same bits.  The row key is the bit pattern of the row's largest |x|; from its
// exponent the row scale 2^k puts that largest |x| in [2^20, 2^21).  Each
// element contributes, with s = |x| 2^k (exact) split as s = S + r (S = rint(s),
// |r| <= 1/2, both exact):
//     S^2 + rint(u r),  u = fl(2S + r)          ~= s^2 = S^2 + (2S + r) r,
// the first term exact in 64-bit integer arithmetic and the second within 5/8
// of exact (|u r| < 2^21), so the sum is s^2 summed to within
// 5/8 per element in units where the largest square is ~2^41; it is never
// negative and stays below 2^58 for K <= 65536.  ss = sum * 2^(-2k).
__device__ __forceinline__ int sq_key(float x) { return __float_as_int(fabsf(x)); }

__device__ __forceinline__ int sq_key4(float4 v) {
  return __float_as_int(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
}

// k of the row scale.  Rows whose largest |x| is below 2^-106 keep k = 127:
// their sum of squares (< 2^-196) is far below any eps > 0 at float precision.
__device__ __forceinline__ int sq_shift(int key) { return min(147 - (key >> 23), 127); }

__device__ __forceinline__ float sq_scale(int key) { return __int_as_float((sq_shift(key) + 127) << 23); }

// One row's partial sum: `sq` holds the S^2 terms; `cb` the raw bit patterns of
// the rounded sums 1.5 * 2^23 + rint(u r), whose offsets are removed when the
// partial is folded (each rint(u r) is below 2^21 in magnitude, so up to 1023
// elements can be folded at once without leaving the int32 range).
struct SqPartial {
  unsigned long long sq;
  uint32_t cb;
};

__device__ __forceinline__ void sq_add(SqPartial& a, float x, float scale) {
  const float s = __fmul_rn(fabsf(x), scale);  // exact unless it underflows (then S = 0 and rint(u r) = 0)
  const float t = __fadd_rn(s, kRoundMagic);
  const float sf = __fsub_rn(t, kRoundMagic);  // S
  const uint32_t si = __float_as_uint(t) - kRoundMagicBits;
  const float r = __fsub_rn(s, sf);
  const float u = __fmaf_rn(2.0f, sf, r);
  a.cb += __float_as_uint(__fmaf_rn(u, r, kRoundMagic));
  asm("mad.wide.u32 %0, %1, %1, %0;" : "+l"(a.sq) : "r"(si));
}

__device__ __forceinline__ void sq_add4(SqPartial& a, float4 v, float scale) {
  sq_add(a, v.x, scale);
  sq_add(a, v.y, scale);
  sq_add(a, v.z, scale);
  sq_add(a, v.w, scale);
}

// The partial's value after `n` (< 1024) calls of sq_add.
__device__ __forceinline__ unsigned long long sq_fold(const SqPartial& a, int n) {
  const int c = static_cast<int>(a.cb - static_cast<uint32_t>(n) * kRoundMagicBits);
  return a.sq + static_cast<unsigned long long>(static_cast<long long>(c));
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

// rstd = 1 / sqrt(ss/K + eps), rounded once to float, where ss = acc * 2^(-2k)
// is the fixed-point sum of squares of a row with key `key`.
//
// ss spans ~2^-300 .. 2^272, far outside fp32, so both terms are scaled by
// 2^(-e2) first, which leaves every intermediate a normal float, and the result
// by 2^(-e2/2) after (exact for a normal rstd).  e2 is ss's binary exponent
// rounded down to even, which puts ss * 2^-e2 in [1, 4); when ss/K is below
// 2^-59 eps it cannot change the result at the accuracy carried here, is
// dropped, and e2 comes from eps instead.  ss * 2^-e2 is taken as an fp32 pair
// (the top 48 bits of acc), ss/K + eps as an fp32 pair (quotient by the
// reciprocal of K; the remainder hi - q*K is exact by fma since q is within a
// few ulp of hi/K and K < 2^23); 1/sqrt by the hardware estimate refined with
// one Newton step whose residual 1 - v*y0^2 is evaluated to ~2^-47.
__device__ __forceinline__ float rstd_from_fixed(unsigned long long acc, int key, int K, float eps) {
  // eps = em * 2^ee, em in [1, 2)
  float eps_n = eps;
  int ee = -127;
  if ((__float_as_int(eps) >> 23) == 0) {  // subnormal eps
    eps_n = __fmul_rn(eps, 18446744073709551616.0f);  // * 2^64, exact
    ee -= 64;
  }
  ee += __float_as_int(eps_n) >> 23;
  const float em = __int_as_float((__float_as_int(eps_n) & 0x7fffff) | 0x3f800000);
  const int e_eps = ee + (31 - __clz(K)) - 60;
  DF ss = {0.0f, 0.0f};
  int e2 = e_eps;
  if (acc != 0ull) {
    const int p = 63 - __clzll(static_cast<long long>(acc));
    const int lv = p - 2 * sq_shift(key);  // ss in [2^lv, 2^(lv+1))
    if (lv >= e_eps) {
      e2 = lv;
      const int base = lv - (lv & ~1) - 63;            // -63 or -62: ss * 2^-e2 = t * 2^base
      const unsigned long long t = acc << (63 - p);  // leading one at bit 63
      const float h = __fmul_rn(static_cast<float>(static_cast<unsigned>(t >> 40)),
                                __int_as_float((base + 40 + 127) << 23));  // exact, in [1, 4)
      const float l = __fmul_rn(static_cast<float>(static_cast<unsigned>((t >> 16) & 0xffffffull)),
                                __int_as_float((base + 16 + 127) << 23));  // exact
      const float sum = __fadd_rn(h, l);
      ss = DF{sum, __fsub_rn(l, __fsub_rn(sum, h))};
    }
  }
  e2 &= ~1;
  const int es = ee - e2;  // <= 62
  const float eps_s = es >= -126 ? __fmul_rn(em, __int_as_float((es + 127) << 23)) : 0.0f;  // else negligible
  const float kf = static_cast<float>(K);  // exact
  const float rk = __frcp_rn(kf);
  const float q = __fmul_rn(ss.hi, rk);
  const float rem = __fmaf_rn(-q, kf, ss.hi);  // exact
  const float ql = __fmul_rn(__fadd_rn(rem, ss.lo), rk);
  DF v = df_add(DF{q, ql}, DF{eps_s, 0.0f});
  const float y0 = rsqrtf(v.hi);
  const float s_hi = __fmul_rn(y0, y0);
  const float s_lo = __fmaf_rn(y0, y0, -s_hi);  // y0^2 = s_hi + s_lo exactly
  const float t_hi = __fmul_rn(v.hi, s_hi);
  const float t_err = __fmaf_rn(v.hi, s_hi, -t_hi);
  // e = 1 - v*y0^2; 1 - t_hi is exact (t_hi is within a few ulp of 1)
  const float small = __fadd_rn(__fadd_rn(t_err, __fmul_rn(v.hi, s_lo)), __fmul_rn(v.lo, s_hi));
  const float e = __fsub_rn(__fsub_rn(1.0f, t_hi), small);
  const float c = __fmul_rn(__fmul_rn(y0, e), 0.5f);
  const float r = __fadd_rn(y0, c);
  const int j = -(e2 / 2);
  return (j >= -126 && j <= 127) ? __fmul_rn(r, __int_as_float((j + 127) << 23)) : mul_pow2(r, j);
}

// Four consecutive input elements from global memory, widened to fp32 (exact
// for fp32, fp16 and bf16 alike: every such value is an fp32 value).
__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __half* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// An fp32 result rounded once to the output element type (to nearest, ties to
// even; fp16 overflows to infinity past 65504).
template <typename T>
__device__ __forceinline__ T round_out(float v);
template <>
__device__ __forceinline__ float round_out<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half round_out<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 round_out<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// rstd of a row read by one full warp (global memory of any input type, or
// fp32 in shared memory).
template <bool kGlobal, typename InT = float>
__device__ __forceinline__ float warp_row_rstd(const InT* __restrict__ xrow, int K, int lane, float eps) {
  static_assert(kGlobal || sizeof(InT) == 4, "rows in shared memory are fp32");
  const InT* p = xrow + 4 * lane;
  const int nc = K >> 7;
  auto ld = [&](int c) -> float4 {
    if constexpr (kGlobal) return load4(p + 128 * c);
    else return *reinterpret_cast<const float4*>(p + 128 * c);
  };
  int key = 0;
  for (int c = 0; c < nc; ++c) key = max(key, sq_key4(ld(c)));
  key = warp_max_int(key);
  const float scale = sq_scale(key);
  unsigned long long acc = 0ull;
  for (int c0 = 0; c0 < nc; c0 += 128) {  // folds every 512 elements per lane
    SqPartial part = {0ull, 0u};
    const int c1 = min(nc, c0 + 128);
    for (int c = c0; c < c1; ++c) sq_add4(part, ld(c), scale);
    acc += sq_fold(part, 4 * (c1 - c0));
  }
  return rstd_from_fixed(warp_sum_u64(acc), key, K, eps);
}

__device__ __forceinline__ float norm_elem(float x, float rstd, float g) {
  return __fmul_rn(__fmul_rn(x, rstd), g);
}

__device__ __forceinline__ float act_scale_from_amax(float amax) {
  return __fdiv_rn(127.0f, fmaxf(amax, 1e-5f));
}

// q = rint(xn * a_scale).  The definition clamps q to [-128, 127]; for finite
// inputs that clamp never acts: |xn| <= amax and a_scale = fl(127 / max(amax,
// 1e-5)), so |fl(xn * a_scale)| <= fl(127 (1 + 2^-24)) and q lies in [-127, 127].
// Rounding by the 1.5 * 2^23 addition is exact for such products and breaks ties
// to even like rintf.  (Non-finite inputs give unspecified codes.)

// Four codes as int8 bytes (element 0 in the low byte): the low byte of each
// rounded sum is the code in two's complement.
__device__ __forceinline__ uint32_t quant_pack4_i8(float4 n, float a_scale) {
  const uint32_t t0 = __float_as_uint(__fadd_rn(__fmul_rn(n.x, a_scale), kRoundMagic));
  const uint32_t t1 = __float_as_uint(__fadd_rn(__fmul_rn(n.y, a_scale), kRoundMagic));
  const uint32_t t2 = __float_as_uint(__fadd_rn(__fmul_rn(n.z, a_scale), kRoundMagic));
  const uint32_t t3 = __float_as_uint(__fadd_rn(__fmul_rn(n.w, a_scale), kRoundMagic));
  return prmt_b32(prmt_b32(t0, t1, 0x0040u), prmt_b32(t2, t3, 0x0040u), 0x5410u);
}

// Two codes as an fp16 pair (element 0 in the low half).  Adding 1.5 * 2^23 +
// 0x6600 leaves 0x6600 + q, the fp16 pattern of 1536 + q, in the low 16 bits of
// the rounded sum; subtracting 1536 in fp16 is exact.
__device__ __forceinline__ uint32_t quant_pack2_f16(float a, float b, float a_scale) {
  constexpr float kHalfMagic = 12609024.0f;  // 1.5 * 2^23 + 0x6600
  const uint32_t t0 = __float_as_uint(__fadd_rn(__fmul_rn(a, a_scale), kHalfMagic));
  const uint32_t t1 = __float_as_uint(__fadd_rn(__fmul_rn(b, a_scale), kHalfMagic));
  uint32_t h = prmt_b32(t0, t1, 0x5410u);
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __floats2half2_rn(1536.0f, 1536.0f));
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ------------------------------------------------- down-projection input
// h = act(gate) * up, the input of the down projection ("BitNet Embeddings GGUF
// Conversion Implementation", section 4.5, "FFN per-projection norms", with the
// activations of section 1's table): SiLU(x) = x / (1 + e^-x) (Qwen3) and
// gelu_pytorch_tanh(x) = x/2 (1 + tanh(z)), z = sqrt(2/pi) (x + 0.044715 x^3)
// (Gemma3).  Since (1 + tanh z) / 2 = 1 / (1 + e^-2z), both are x / (1 + e^-t)
// with t = x or 2z: evaluated as x * rcp(1 + expf(-t)) (CUDA's expf, a correctly
// rounded reciprocal, every operation rounded on its own), which needs no divide
// and, for very negative x, keeps its relative accuracy where 1 + tanh(z) would
// cancel.  All launch paths use this one function, so they all see the same h.
constexpr int kActSilu = 1;
constexpr int kActGeluTanh = 2;

__device__ __forceinline__ float act_elem(float x, int act) {
  float t = x;
  if (act == kActGeluTanh) {
    const float x3 = __fmul_rn(__fmul_rn(x, x), x);
    t = __fmul_rn(1.5957691216057308f, __fadd_rn(x, __fmul_rn(0.044715f, x3)));  // 2 sqrt(2/pi) (x + 0.044715 x^3)
  }
  return __fmul_rn(x, __frcp_rn(__fadd_rn(1.0f, expf(-t))));
}

__device__ __forceinline__ float4 glu4(float4 g, float4 u, int act) {
  return make_float4(__fmul_rn(act_elem(g.x, act), u.x), __fmul_rn(act_elem(g.y, act), u.y),
                     __fmul_rn(act_elem(g.z, act), u.z), __fmul_rn(act_elem(g.w, act), u.w));
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
