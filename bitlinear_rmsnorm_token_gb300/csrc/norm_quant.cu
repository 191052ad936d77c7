// norm_quant.cu -- fused RMSNorm (per-projection norm weight) + per-token absmax
// int8 quantisation, one warp per token row.
//
// "BitNet Embeddings GGUF Conversion Implementation", sections 1 and 4.5;
// "BitNet Inference Framework", "Quantization (W1.58A8)".  The arithmetic is
// the shared definition in rowquant.cuh.
//
// HBM-bound: it reads x (4 B/elem) once from DRAM and writes 1 B (int8) or 2 B
// (fp16, the tensor-core operand) per element.  The sum of squares, the absmax
// and the quantisation are three sweeps over the row; rows up to K = 3072 are
// held in registers, longer ones are re-read through L1/L2.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

namespace bitnet {
namespace {

constexpr int kNqWarps = 8;

template <typename OutT>
__device__ __forceinline__ void store4(OutT* dst, int q0, int q1, int q2, int q3);

template <>
__device__ __forceinline__ void store4<int8_t>(int8_t* dst, int q0, int q1, int q2, int q3) {
  const uint32_t v = (static_cast<uint32_t>(q0) & 0xFFu) | ((static_cast<uint32_t>(q1) & 0xFFu) << 8) |
                     ((static_cast<uint32_t>(q2) & 0xFFu) << 16) | ((static_cast<uint32_t>(q3) & 0xFFu) << 24);
  *reinterpret_cast<uint32_t*>(dst) = v;
}

template <>
__device__ __forceinline__ void store4<__half>(__half* dst, int q0, int q1, int q2, int q3) {
  // integers in [-128, 127] are exact in fp16
  __half2 a = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
  __half2 b = __halves2half2(__int2half_rn(q2), __int2half_rn(q3));
  uint2 v;
  v.x = *reinterpret_cast<uint32_t*>(&a);
  v.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = v;
}

// kNC > 0: the row (at most kNC float4 groups per lane) is loaded once into
// registers; kNC == 0: any K, the row is read three times (L1/L2 after the first).
template <typename OutT, int kNC>
__global__ void __launch_bounds__(kNqWarps * 32) k_rmsnorm_quant(const float* __restrict__ x, const float* __restrict__ g,
                                                                 int64_t M, int K, float eps, OutT* __restrict__ codes,
                                                                 float* __restrict__ a_scale,
                                                                 int32_t* __restrict__ rowsum,
                                                                 float* __restrict__ xn_out) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNqWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const float* xr = x + row * K + 4 * lane;
  const float* gr = g + 4 * lane;
  const int nc = K >> 7;
  OutT* cr = codes + row * K + 4 * lane;
  float* xo = xn_out ? xn_out + row * K + 4 * lane : nullptr;
  float amax = 0.0f;
  int rs = 0;

  if constexpr (kNC > 0) {
    float4 v[kNC];
#pragma unroll
    for (int c = 0; c < kNC; ++c)
      if (c < nc) v[c] = __ldg(reinterpret_cast<const float4*>(xr + 128 * c));
    int e = 0;
#pragma unroll
    for (int c = 0; c < kNC; ++c)
      if (c < nc) e = max(e, sq_exp4(v[c]));
    const int emax = warp_max_int(e);
    unsigned long long acc = 0ull;
#pragma unroll
    for (int c = 0; c < kNC; ++c)
      if (c < nc) acc += sq_term4(v[c], emax);
    const float rstd = rstd_from_sumsq(sq_to_df(warp_sum_u64(acc), emax), K, eps);
#pragma unroll
    for (int c = 0; c < kNC; ++c) {
      if (c < nc) {
        const float4 gv = __ldg(reinterpret_cast<const float4*>(gr + 128 * c));
        v[c] = make_float4(norm_elem(v[c].x, rstd, gv.x), norm_elem(v[c].y, rstd, gv.y),
                           norm_elem(v[c].z, rstd, gv.z), norm_elem(v[c].w, rstd, gv.w));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[c].x), fabsf(v[c].y)), fmaxf(fabsf(v[c].z), fabsf(v[c].w))));
        if (xo) *reinterpret_cast<float4*>(xo + 128 * c) = v[c];
      }
    }
    const float as = act_scale_from_amax(warp_max(amax));
#pragma unroll
    for (int c = 0; c < kNC; ++c) {
      if (c < nc) {
        const int q0 = quant_elem(v[c].x, as), q1 = quant_elem(v[c].y, as);
        const int q2 = quant_elem(v[c].z, as), q3 = quant_elem(v[c].w, as);
        store4<OutT>(cr + 128 * c, q0, q1, q2, q3);
        rs += q0 + q1 + q2 + q3;
      }
    }
    rs = warp_sum_int(rs);
    if (lane == 0) {
      a_scale[row] = as;
      if (rowsum) rowsum[row] = rs;
    }
  } else {
    const float rstd = rstd_from_sumsq(warp_row_sumsq<true>(x + row * K, K, lane), K, eps);
    for (int c = 0; c < nc; ++c) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(xr + 128 * c));
      const float4 gv = __ldg(reinterpret_cast<const float4*>(gr + 128 * c));
      const float4 n = make_float4(norm_elem(v.x, rstd, gv.x), norm_elem(v.y, rstd, gv.y),
                                   norm_elem(v.z, rstd, gv.z), norm_elem(v.w, rstd, gv.w));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(n.x), fabsf(n.y)), fmaxf(fabsf(n.z), fabsf(n.w))));
      if (xo) *reinterpret_cast<float4*>(xo + 128 * c) = n;
    }
    const float as = act_scale_from_amax(warp_max(amax));
    for (int c = 0; c < nc; ++c) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(xr + 128 * c));
      const float4 gv = __ldg(reinterpret_cast<const float4*>(gr + 128 * c));
      const int q0 = quant_elem(norm_elem(v.x, rstd, gv.x), as), q1 = quant_elem(norm_elem(v.y, rstd, gv.y), as);
      const int q2 = quant_elem(norm_elem(v.z, rstd, gv.z), as), q3 = quant_elem(norm_elem(v.w, rstd, gv.w), as);
      store4<OutT>(cr + 128 * c, q0, q1, q2, q3);
      rs += q0 + q1 + q2 + q3;
    }
    rs = warp_sum_int(rs);
    if (lane == 0) {
      a_scale[row] = as;
      if (rowsum) rowsum[row] = rs;
    }
  }
}

__global__ void __launch_bounds__(256) k_codes_to_f16(const int8_t* __restrict__ in, __half* __restrict__ out,
                                                      int64_t n4) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n4) return;
  const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(in) + t);
  store4<__half>(out + 4 * t, static_cast<int8_t>(v & 0xFF), static_cast<int8_t>((v >> 8) & 0xFF),
                 static_cast<int8_t>((v >> 16) & 0xFF), static_cast<int8_t>(v >> 24));
}

template <typename OutT, int kNC>
cudaError_t launch_nq(const float* x, const float* g, int64_t M, int K, float eps, OutT* codes, float* a_scale,
                      int32_t* rowsum, float* xn_out, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((M + kNqWarps - 1) / kNqWarps));
  cfg.blockDim = dim3(kNqWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_rmsnorm_quant<OutT, kNC>, x, g, M, K, eps, codes, a_scale, rowsum, xn_out);
}

template <typename OutT>
cudaError_t launch_nq_k(const float* x, const float* g, int64_t M, int K, float eps, OutT* codes, float* a_scale,
                        int32_t* rowsum, float* xn_out, bool pdl, cudaStream_t s) {
  const int nc = K >> 7;
  if (nc <= 8) return launch_nq<OutT, 8>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
  if (nc <= 24) return launch_nq<OutT, 24>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
  return launch_nq<OutT, 0>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const float* x, const float* g, int64_t M, int K, float eps, int8_t* codes_i8,
                                 __half* codes_f16, float* a_scale, int32_t* rowsum, float* xn_out, bool pdl,
                                 cudaStream_t s) {
  if (codes_f16) return launch_nq_k<__half>(x, g, M, K, eps, codes_f16, a_scale, rowsum, xn_out, pdl, s);
  return launch_nq_k<int8_t>(x, g, M, K, eps, codes_i8, a_scale, rowsum, xn_out, pdl, s);
}

cudaError_t launch_codes_to_f16(const int8_t* codes, __half* out, int64_t count, cudaStream_t s) {
  const int64_t n4 = count / 4;
  const int64_t blocks = (n4 + 255) / 256;
  k_codes_to_f16<<<static_cast<unsigned>(blocks), 256, 0, s>>>(codes, out, n4);
  return cudaGetLastError();
}

}  // namespace bitnet
