// norm_quant.cu -- fused RMSNorm (per-projection norm weight) + per-token absmax
// int8 quantisation, one warp per token row.
//
// "BitNet Embeddings GGUF Conversion Implementation", sections 1 and 4.5;
// "BitNet Inference Framework", "Quantization (W1.58A8)".  The arithmetic is
// the shared definition in rowquant.cuh.
//
// x is fp32, or fp16 / bf16 (InT: widened to fp32 as it is loaded, exactly, so
// everything after the load is the fp32 definition).
// HBM-bound: it reads x (4 or 2 B/elem) once from DRAM and writes 1 B (int8) or 2 B
// (fp16, the tensor-core operand) per element.  The sum of squares, the absmax
// and the quantisation are three sweeps over the row; rows up to K = 3072 are
// held in registers, longer ones are re-read through L1/L2.
#include "common.cuh"
#include "internal.h"
#include "planes.cuh"
#include "rowquant.cuh"

namespace bitnet {
namespace {

constexpr int kNqWarps = 8;

// Quantises four normalised values and stores their codes; the int8 form also
// adds them to the running row sum (dp4a of the packed bytes with ones).
template <typename OutT>
__device__ __forceinline__ void store_codes4(OutT* dst, float4 n, float a_scale, int& rs);

template <>
__device__ __forceinline__ void store_codes4<int8_t>(int8_t* dst, float4 n, float a_scale, int& rs) {
  const uint32_t p = quant_pack4_i8(n, a_scale);
  *reinterpret_cast<uint32_t*>(dst) = p;
  rs = __dp4a(static_cast<int>(p), 0x01010101, rs);
}

template <>
__device__ __forceinline__ void store_codes4<__half>(__half* dst, float4 n, float a_scale, int&) {
  uint2 v;
  v.x = quant_pack2_f16(n.x, n.y, a_scale);
  v.y = quant_pack2_f16(n.z, n.w, a_scale);
  *reinterpret_cast<uint2*>(dst) = v;
}

// The codes as the two e4m3 planes of the 9..63-token contraction (planes.cuh),
// in the footprint of fp16 codes; the int8 codes' arithmetic, and their row sum.
struct PlaneCode {
  uint16_t bits;
};
template <>
__device__ __forceinline__ void store_codes4<PlaneCode>(PlaneCode* dst, float4 n, float a_scale, int& rs) {
  const uint32_t p = quant_pack4_i8(n, a_scale);
  rs = __dp4a(static_cast<int>(p), 0x01010101, rs);
  uint32_t hi, lo;
  plane_words4(p, hi, lo);
  store_planes4(dst, hi, lo);
}

// kNC > 0: the row (at most kNC float4 groups per lane; exactly kNC when kExact,
// which spares the predicated-off groups) is loaded once into registers;
// kNC == 0: any K, the row is read three times (L1/L2 after the first).
// kGlu (kNC > 0 only): the row is act(x) * up, computed as it is loaded.
// At most 128 registers (two CTAs per SM): a CTA normalises 8 rows and exits,
// so a second resident CTA overlaps one's reductions with the other's loads
// (the K = 2048 form took 168 registers, one CTA per SM and 53% of DRAM
// bandwidth); every form, rows of up to 24 float4 per lane included, fits.
template <typename InT, typename OutT, int kNC, bool kExact, bool kGlu = false>
__global__ void __launch_bounds__(kNqWarps * 32, 2) k_rmsnorm_quant(const InT* __restrict__ x, const float* __restrict__ g,
                                                                 int64_t M, int K, float eps, OutT* __restrict__ codes,
                                                                 float* __restrict__ a_scale,
                                                                 int32_t* __restrict__ rowsum,
                                                                 float* __restrict__ xn_out,
                                                                 const float* __restrict__ up = nullptr,
                                                                 int act = 0) {
  static_assert(!kGlu || kNC > 0, "the activation is applied to rows held in registers");
  static_assert(!kGlu || sizeof(InT) == 4, "the activation form reads fp32 gate and up rows");
  // dependents may start only once the kernels before this one have completed
  // (they may then read any input this kernel does not write before their own
  // wait)
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNqWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const InT* xr = x + row * K + 4 * lane;
  const float* gr = g + 4 * lane;
  const int nc = kExact ? kNC : (K >> 7);
  OutT* cr = codes + row * K + 4 * lane;
  float* xo = xn_out ? xn_out + row * K + 4 * lane : nullptr;
  float amax = 0.0f;
  int rs = 0;

  if constexpr (kNC > 0) {
    float4 v[kNC];
#pragma unroll
    for (int c = 0; c < kNC; ++c) {
      if (c < nc) {
        v[c] = load4(xr + 128 * c);
        if constexpr (kGlu) v[c] = glu4(v[c], __ldg(reinterpret_cast<const float4*>(up + row * K + 4 * lane + 128 * c)), act);
      }
    }
    int key = 0;
#pragma unroll
    for (int c = 0; c < kNC; ++c)
      if (c < nc) key = max(key, sq_key4(v[c]));
    key = warp_max_int(key);
    const float scale = sq_scale(key);
    SqPartial part = {0ull, 0u};
#pragma unroll
    for (int c = 0; c < kNC; ++c)
      if (c < nc) sq_add4(part, v[c], scale);
    const unsigned long long acc = sq_fold(part, 4 * min(nc, kNC));
    const float rstd = rstd_from_fixed(warp_sum_u64(acc), key, K, eps);
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
      if (c < nc) store_codes4<OutT>(cr + 128 * c, v[c], as, rs);
    }
    if (rowsum) rs = warp_sum_int(rs);
    if (lane == 0) {
      a_scale[row] = as;
      if (rowsum) rowsum[row] = rs;
    }
  } else {
    const float rstd = warp_row_rstd<true, InT>(x + row * K, K, lane, eps);
    for (int c = 0; c < nc; ++c) {
      const float4 v = load4(xr + 128 * c);
      const float4 gv = __ldg(reinterpret_cast<const float4*>(gr + 128 * c));
      const float4 n = make_float4(norm_elem(v.x, rstd, gv.x), norm_elem(v.y, rstd, gv.y),
                                   norm_elem(v.z, rstd, gv.z), norm_elem(v.w, rstd, gv.w));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(n.x), fabsf(n.y)), fmaxf(fabsf(n.z), fabsf(n.w))));
      if (xo) *reinterpret_cast<float4*>(xo + 128 * c) = n;
    }
    const float as = act_scale_from_amax(warp_max(amax));
    for (int c = 0; c < nc; ++c) {
      const float4 v = load4(xr + 128 * c);
      const float4 gv = __ldg(reinterpret_cast<const float4*>(gr + 128 * c));
      const float4 n = make_float4(norm_elem(v.x, rstd, gv.x), norm_elem(v.y, rstd, gv.y),
                                   norm_elem(v.z, rstd, gv.z), norm_elem(v.w, rstd, gv.w));
      store_codes4<OutT>(cr + 128 * c, n, as, rs);
    }
    if (rowsum) rs = warp_sum_int(rs);
    if (lane == 0) {
      a_scale[row] = as;
      if (rowsum) rowsum[row] = rs;
    }
  }
}

// Long rows (K a multiple of 2048 above 3072): one CTA per row, block-wide
// reductions through shared-memory atomics (integer and max: order-free).
// kRegs: K <= 16384, K/16 threads each holding 16 elements in registers
// (float4 groups t, t+T, t+2T, t+3T of the row: every load instruction of a
// warp is coalesced).  Otherwise 1024 threads loop over the row's float4 groups
// with the same stride and read the row again from L2 in every pass.
template <typename InT, typename OutT, bool kRegs>
__global__ void __launch_bounds__(1024) k_rmsnorm_quant_rows(const InT* __restrict__ x,
                                                             const float* __restrict__ g, int K, float eps,
                                                             OutT* __restrict__ codes, float* __restrict__ a_scale,
                                                             int32_t* __restrict__ rowsum,
                                                             float* __restrict__ xn_out) {
  constexpr int kV = 4;  // float4 groups per thread held in registers (kRegs)
  __shared__ int s_key;
  __shared__ unsigned long long s_ss;
  __shared__ unsigned s_amax;
  __shared__ int s_rs;
  pdl_wait();
  pdl_launch_dependents();
  const int T = blockDim.x;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int64_t row = blockIdx.x;
  // float4 groups of this thread: tid + T i for i < nv (exactly kV when kRegs)
  const int nv = kRegs ? kV : ((K >> 2) - tid + T - 1) / T;
  if (tid == 0) {
    s_key = 0;
    s_ss = 0ull;
    s_amax = 0u;
    s_rs = 0;
  }
  const InT* xr = x + row * K;
  const float4* gr = reinterpret_cast<const float4*>(g);
  float4 v[kV];
  if (kRegs) {
#pragma unroll
    for (int i = 0; i < kV; ++i) v[i] = load4(xr + 4 * (tid + T * i));
  }
  auto xv = [&](int i) { return kRegs ? v[i] : load4(xr + 4 * (tid + T * i)); };
  __syncthreads();
  int key = 0;
#pragma unroll 4
  for (int i = 0; i < nv; ++i) key = max(key, sq_key4(xv(i)));
  key = warp_max_int(key);
  if (lane == 0 && key) atomicMax(&s_key, key);
  __syncthreads();
  key = s_key;
  const float scale = sq_scale(key);
  SqPartial part = {0ull, 0u};
#pragma unroll 4
  for (int i = 0; i < nv; ++i) sq_add4(part, xv(i), scale);
  const unsigned long long w = warp_sum_u64(sq_fold(part, 4 * nv));
  if (lane == 0 && w) atomicAdd(&s_ss, w);
  __syncthreads();
  const float rstd = rstd_from_fixed(s_ss, key, K, eps);
  auto norm4 = [&](float4 a, float4 gv) {
    return make_float4(norm_elem(a.x, rstd, gv.x), norm_elem(a.y, rstd, gv.y), norm_elem(a.z, rstd, gv.z),
                       norm_elem(a.w, rstd, gv.w));
  };
  float amax = 0.0f;
#pragma unroll 4
  for (int i = 0; i < nv; ++i) {
    const float4 n = norm4(xv(i), __ldg(gr + tid + T * i));
    if (kRegs) v[i] = n;
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(n.x), fabsf(n.y)), fmaxf(fabsf(n.z), fabsf(n.w))));
    if (xn_out) reinterpret_cast<float4*>(xn_out + row * K)[tid + T * i] = n;
  }
  amax = warp_max(amax);
  if (lane == 0) atomicMax(&s_amax, __float_as_uint(amax));
  __syncthreads();
  const float as = act_scale_from_amax(__uint_as_float(s_amax));
  int rs = 0;
#pragma unroll 4
  for (int i = 0; i < nv; ++i) {
    const float4 n = kRegs ? v[i] : norm4(load4(xr + 4 * (tid + T * i)), __ldg(gr + tid + T * i));
    store_codes4<OutT>(codes + row * K + 4 * (tid + T * i), n, as, rs);
  }
  if (rowsum) {
    rs = warp_sum_int(rs);
    if (lane == 0 && rs) atomicAdd(&s_rs, rs);
    __syncthreads();
  }
  if (tid == 0) {
    a_scale[row] = as;
    if (rowsum) rowsum[row] = s_rs;
  }
}

__global__ void __launch_bounds__(256) k_codes_to_f16(const int8_t* __restrict__ in, __half* __restrict__ out,
                                                      int64_t n4) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n4) return;
  const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(in) + t);
  // integers in [-128, 127] are exact in fp16
  const __half2 a = __halves2half2(__int2half_rn(static_cast<int8_t>(v & 0xFFu)),
                                   __int2half_rn(static_cast<int8_t>((v >> 8) & 0xFFu)));
  const __half2 b = __halves2half2(__int2half_rn(static_cast<int8_t>((v >> 16) & 0xFFu)),
                                   __int2half_rn(static_cast<int8_t>(v >> 24)));
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&a);
  o.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(out + 4 * t) = o;
}

template <typename InT, typename OutT, int kNC, bool kExact = false, bool kGlu = false>
cudaError_t launch_nq(const InT* x, const float* g, int64_t M, int K, float eps, OutT* codes, float* a_scale,
                      int32_t* rowsum, float* xn_out, bool pdl, cudaStream_t s, const float* up = nullptr,
                      int act = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((M + kNqWarps - 1) / kNqWarps));
  cfg.blockDim = dim3(kNqWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_rmsnorm_quant<InT, OutT, kNC, kExact, kGlu>, x, g, M, K, eps, codes, a_scale, rowsum,
                            xn_out, up, act);
}

template <typename InT, typename OutT>
cudaError_t launch_nq_rows(const InT* x, const float* g, int64_t M, int K, float eps, OutT* codes, float* a_scale,
                           int32_t* rowsum, float* xn_out, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  const bool regs = K <= 16384;
  cfg.gridDim = dim3(static_cast<unsigned>(M));
  cfg.blockDim = dim3(static_cast<unsigned>(regs ? K / 16 : 1024));
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (regs)
    return cudaLaunchKernelEx(&cfg, k_rmsnorm_quant_rows<InT, OutT, true>, x, g, K, eps, codes, a_scale, rowsum, xn_out);
  return cudaLaunchKernelEx(&cfg, k_rmsnorm_quant_rows<InT, OutT, false>, x, g, K, eps, codes, a_scale, rowsum, xn_out);
}

template <typename InT, typename OutT>
cudaError_t launch_nq_k(const InT* x, const float* g, int64_t M, int K, float eps, OutT* codes, float* a_scale,
                        int32_t* rowsum, float* xn_out, bool pdl, cudaStream_t s) {
  const int nc = K >> 7;
  if (nc > 24 && K % 2048 == 0 && M < (int64_t(1) << 31))  // keep in step with rmsnorm_quant_ctas
    return launch_nq_rows<InT, OutT>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
  switch (nc) {  // the model widths of the prefill shapes: K = 640, 1024, 2048, 3072
    case 5: return launch_nq<InT, OutT, 5, true>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
    case 8: return launch_nq<InT, OutT, 8, true>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
    case 16: return launch_nq<InT, OutT, 16, true>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
    case 24: return launch_nq<InT, OutT, 24, true>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
    default: break;
  }
  if (nc <= 8) return launch_nq<InT, OutT, 8>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
  if (nc <= 24) return launch_nq<InT, OutT, 24>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
  return launch_nq<InT, OutT, 0>(x, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s);
}

template <typename OutT>
cudaError_t launch_nq_glu_k(const float* gate, const float* up, int act, const float* g, int64_t M, int K, float eps,
                            OutT* codes, float* a_scale, int32_t* rowsum, float* xn_out, bool pdl, cudaStream_t s) {
  switch (K >> 7) {  // the down-projection widths: 2048 (Gemma3), 3072 (Qwen3)
    case 16:
      return launch_nq<float, OutT, 16, true, true>(gate, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s, up,
                                                    act);
    case 24:
      return launch_nq<float, OutT, 24, true, true>(gate, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s, up,
                                                    act);
    default:
      break;
  }
  if ((K >> 7) <= 8)
    return launch_nq<float, OutT, 8, false, true>(gate, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s, up,
                                                  act);
  return launch_nq<float, OutT, 24, false, true>(gate, g, M, K, eps, codes, a_scale, rowsum, xn_out, pdl, s, up, act);
}

__global__ void __launch_bounds__(256) k_glu(const float* __restrict__ gate, const float* __restrict__ up, int act,
                                             int64_t n4, float* __restrict__ h) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n4) return;
  reinterpret_cast<float4*>(h)[t] = glu4(__ldg(reinterpret_cast<const float4*>(gate) + t),
                                         __ldg(reinterpret_cast<const float4*>(up) + t), act);
}

// Head norm of projection outputs: one warp per (token, head) row of hd
// values (a multiple of 128), out = (y * rstd) * w with the row arithmetic of
// the input norm.  out may be y (each element is read by the thread that
// writes it, after the row's reductions), hence no __restrict__.
__global__ void __launch_bounds__(kNqWarps * 32) k_head_rmsnorm(const float* y, int64_t rows, int hd,
                                                                const float* __restrict__ w, float eps, float* out) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kNqWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* yr = y + row * hd;
  const float rstd = warp_row_rstd<true>(yr, hd, lane, eps);
  for (int c = 0; c < (hd >> 7); ++c) {
    const float4 v = load4(yr + 128 * c + 4 * lane);
    const float4 g = __ldg(reinterpret_cast<const float4*>(w + 128 * c + 4 * lane));
    *reinterpret_cast<float4*>(out + row * hd + 128 * c + 4 * lane) =
        make_float4(norm_elem(v.x, rstd, g.x), norm_elem(v.y, rstd, g.y), norm_elem(v.z, rstd, g.z),
                    norm_elem(v.w, rstd, g.w));
  }
}

}  // namespace

cudaError_t launch_head_rmsnorm(const float* y, int64_t rows, int hd, const float* w, float eps, float* out, bool pdl,
                                cudaStream_t s) {
  if (rows < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + kNqWarps - 1) / kNqWarps));
  cfg.blockDim = dim3(kNqWarps * 32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_head_rmsnorm, y, rows, hd, w, eps, out);
}

bool rmsnorm_quant_glu_fused_supported(int K) { return K >= 128 && K % 128 == 0 && (K >> 7) <= 24; }

cudaError_t launch_rmsnorm_quant_glu(const float* gate, const float* up, int act, const float* g, int64_t M, int K,
                                     float eps, int8_t* codes_i8, __half* codes_f16, float* a_scale, int32_t* rowsum,
                                     float* xn_out, bool pdl, cudaStream_t s) {
  if (!rmsnorm_quant_glu_fused_supported(K)) return cudaErrorInvalidValue;
  if (codes_f16) {
    if (rowsum) return cudaErrorInvalidValue;
    return launch_nq_glu_k<__half>(gate, up, act, g, M, K, eps, codes_f16, a_scale, nullptr, xn_out, pdl, s);
  }
  return launch_nq_glu_k<int8_t>(gate, up, act, g, M, K, eps, codes_i8, a_scale, rowsum, xn_out, pdl, s);
}

cudaError_t launch_glu(const float* gate, const float* up, int act, int64_t count, float* h, cudaStream_t s) {
  const int64_t n4 = count / 4;
  if (n4 < 1) return cudaSuccess;
  k_glu<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, s>>>(gate, up, act, n4, h);
  return cudaGetLastError();
}

int64_t rmsnorm_quant_ctas(int64_t M, int K) {
  const int nc = K >> 7;
  if (nc > 24 && K % 2048 == 0) return M;  // one CTA per row
  return (M + kNqWarps - 1) / kNqWarps;
}

cudaError_t launch_rmsnorm_quant(const float* x, const float* g, int64_t M, int K, float eps, int8_t* codes_i8,
                                 __half* codes_f16, float* a_scale, int32_t* rowsum, float* xn_out, bool pdl,
                                 cudaStream_t s) {
  if (codes_f16) {
    if (rowsum) return cudaErrorInvalidValue;  // row sums are produced with int8 codes only
    return launch_nq_k<float, __half>(x, g, M, K, eps, codes_f16, a_scale, nullptr, xn_out, pdl, s);
  }
  return launch_nq_k<float, int8_t>(x, g, M, K, eps, codes_i8, a_scale, rowsum, xn_out, pdl, s);
}

cudaError_t launch_rmsnorm_quant_f16_in(const void* x, int x_dtype, const float* g, int64_t M, int K, float eps,
                                        __half* codes_f16, float* a_scale, bool pdl, cudaStream_t s) {
  switch (x_dtype) {
    case BITNET_DTYPE_F32:
      return launch_nq_k<float, __half>(static_cast<const float*>(x), g, M, K, eps, codes_f16, a_scale, nullptr,
                                        nullptr, pdl, s);
    case BITNET_DTYPE_F16:
      return launch_nq_k<__half, __half>(static_cast<const __half*>(x), g, M, K, eps, codes_f16, a_scale, nullptr,
                                         nullptr, pdl, s);
    case BITNET_DTYPE_BF16:
      return launch_nq_k<__nv_bfloat16, __half>(static_cast<const __nv_bfloat16*>(x), g, M, K, eps, codes_f16, a_scale,
                                                nullptr, nullptr, pdl, s);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rmsnorm_quant_planes(const void* x, int x_dtype, const float* g, int64_t M, int K, float eps,
                                       void* planes, float* a_scale, int32_t* rowsum, bool pdl, cudaStream_t s) {
  PlaneCode* out = static_cast<PlaneCode*>(planes);
  switch (x_dtype) {
    case BITNET_DTYPE_F32:
      return launch_nq_k<float, PlaneCode>(static_cast<const float*>(x), g, M, K, eps, out, a_scale, rowsum, nullptr,
                                           pdl, s);
    case BITNET_DTYPE_F16:
      return launch_nq_k<__half, PlaneCode>(static_cast<const __half*>(x), g, M, K, eps, out, a_scale, rowsum,
                                            nullptr, pdl, s);
    case BITNET_DTYPE_BF16:
      return launch_nq_k<__nv_bfloat16, PlaneCode>(static_cast<const __nv_bfloat16*>(x), g, M, K, eps, out, a_scale,
                                                   rowsum, nullptr, pdl, s);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rmsnorm_quant_glu_planes(const float* gate, const float* up, int act, const float* g, int64_t M,
                                           int K, float eps, void* planes, float* a_scale, int32_t* rowsum, bool pdl,
                                           cudaStream_t s) {
  if (!rmsnorm_quant_glu_fused_supported(K)) return cudaErrorInvalidValue;
  return launch_nq_glu_k<PlaneCode>(gate, up, act, g, M, K, eps, static_cast<PlaneCode*>(planes), a_scale, rowsum,
                                    nullptr, pdl, s);
}

cudaError_t launch_codes_to_f16(const int8_t* codes, __half* out, int64_t count, cudaStream_t s) {
  const int64_t n4 = count / 4;
  const int64_t blocks = (n4 + 255) / 256;
  k_codes_to_f16<<<static_cast<unsigned>(blocks), 256, 0, s>>>(codes, out, n4);
  return cudaGetLastError();
}

}  // namespace bitnet
