// norm_quant.cu -- fused RMSNorm (per-projection norm weight) + per-token absmax
// int8 quantisation, one warp per token row.
//
// "BitNet Embeddings GGUF Conversion Implementation", sections 1 and 4.5;
// "BitNet Inference Framework", "Quantization (W1.58A8)".  The arithmetic is
// the shared definition in rowquant.cuh.
//
// HBM-bound: it reads x (4 B/elem) once from DRAM and writes 1 B (int8) or 2 B
// (fp16, the tensor-core operand) per element.  The sum of squares, the absmax
// and the quantisation are three sweeps over the row; when the row fits
// (K <= 32*4*kRegVec) it is held in registers, otherwise the second and third
// sweeps re-read it through L1/L2.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

namespace bitnet {
namespace {

constexpr int kNqWarps = 8;
constexpr int kRegVec = 8;  // float4 groups per lane held in registers (K <= 1024)

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

template <typename OutT, bool kRegs>
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
  const float* xr = x + row * K;
  const int nc = K >> 7;

  const double ss = warp_row_sumsq(xr, K, lane);
  const float rstd = rstd_from_sumsq(ss, K, eps);

  float4 xv[kRegs ? kRegVec : 1];
  float amax = 0.0f;
  if (kRegs) {
#pragma unroll
    for (int c = 0; c < kRegVec; ++c) {
      if (c < nc) {
        const int k = 4 * lane + 128 * c;
        const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
        const float4 gv = __ldg(reinterpret_cast<const float4*>(g + k));
        const float4 n = make_float4(norm_elem(v.x, rstd, gv.x), norm_elem(v.y, rstd, gv.y),
                                     norm_elem(v.z, rstd, gv.z), norm_elem(v.w, rstd, gv.w));
        xv[c] = n;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(n.x), fabsf(n.y)), fmaxf(fabsf(n.z), fabsf(n.w))));
        if (xn_out) *reinterpret_cast<float4*>(xn_out + row * K + k) = n;
      }
    }
  } else {
    for (int c = 0; c < nc; ++c) {
      const int k = 4 * lane + 128 * c;
      const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
      const float4 gv = __ldg(reinterpret_cast<const float4*>(g + k));
      const float4 n = make_float4(norm_elem(v.x, rstd, gv.x), norm_elem(v.y, rstd, gv.y),
                                   norm_elem(v.z, rstd, gv.z), norm_elem(v.w, rstd, gv.w));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(n.x), fabsf(n.y)), fmaxf(fabsf(n.z), fabsf(n.w))));
      if (xn_out) *reinterpret_cast<float4*>(xn_out + row * K + k) = n;
    }
  }
  amax = warp_max(amax);
  const float as = act_scale_from_amax(amax);

  int rs = 0;
  OutT* cr = codes + row * K;
  if (kRegs) {
#pragma unroll
    for (int c = 0; c < kRegVec; ++c) {
      if (c < nc) {
        const int k = 4 * lane + 128 * c;
        const int q0 = quant_elem(xv[c].x, as), q1 = quant_elem(xv[c].y, as);
        const int q2 = quant_elem(xv[c].z, as), q3 = quant_elem(xv[c].w, as);
        store4<OutT>(cr + k, q0, q1, q2, q3);
        rs += q0 + q1 + q2 + q3;
      }
    }
  } else {
    for (int c = 0; c < nc; ++c) {
      const int k = 4 * lane + 128 * c;
      const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
      const float4 gv = __ldg(reinterpret_cast<const float4*>(g + k));
      const int q0 = quant_elem(norm_elem(v.x, rstd, gv.x), as), q1 = quant_elem(norm_elem(v.y, rstd, gv.y), as);
      const int q2 = quant_elem(norm_elem(v.z, rstd, gv.z), as), q3 = quant_elem(norm_elem(v.w, rstd, gv.w), as);
      store4<OutT>(cr + k, q0, q1, q2, q3);
      rs += q0 + q1 + q2 + q3;
    }
  }
  rs = warp_sum_int(rs);
  if (lane == 0) {
    a_scale[row] = as;
    if (rowsum) rowsum[row] = rs;
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

template <typename OutT, bool kRegs>
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
  return cudaLaunchKernelEx(&cfg, k_rmsnorm_quant<OutT, kRegs>, x, g, M, K, eps, codes, a_scale, rowsum, xn_out);
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const float* x, const float* g, int64_t M, int K, float eps, int8_t* codes_i8,
                                 __half* codes_f16, float* a_scale, int32_t* rowsum, float* xn_out, bool pdl,
                                 cudaStream_t s) {
  const bool regs = K <= 128 * kRegVec;
  if (codes_f16) {
    return regs ? launch_nq<__half, true>(x, g, M, K, eps, codes_f16, a_scale, rowsum, xn_out, pdl, s)
                : launch_nq<__half, false>(x, g, M, K, eps, codes_f16, a_scale, rowsum, xn_out, pdl, s);
  }
  return regs ? launch_nq<int8_t, true>(x, g, M, K, eps, codes_i8, a_scale, rowsum, xn_out, pdl, s)
              : launch_nq<int8_t, false>(x, g, M, K, eps, codes_i8, a_scale, rowsum, xn_out, pdl, s);
}

cudaError_t launch_codes_to_f16(const int8_t* codes, __half* out, int64_t count, cudaStream_t s) {
  const int64_t n4 = count / 4;
  const int64_t blocks = (n4 + 255) / 256;
  k_codes_to_f16<<<static_cast<unsigned>(blocks), 256, 0, s>>>(codes, out, n4);
  return cudaGetLastError();
}

}  // namespace bitnet
