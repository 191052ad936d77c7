// convert.cu -- element-wise conversion between fp32 and the 16-bit I/O types
// (fp16, bf16) of the typed projection entry point.  Widening is exact (every
// fp16 and bf16 value is an fp32 value); narrowing rounds once to nearest,
// ties to even.  Used where a path reads or writes fp32 only: the few-token
// kernels and an fp16 norm weight.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

namespace bitnet {
namespace {

template <typename T>
__device__ __forceinline__ float widen(T v);
template <>
__device__ __forceinline__ float widen<float>(float v) { return v; }
template <>
__device__ __forceinline__ float widen<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float widen<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename In, typename Out>
__global__ void __launch_bounds__(256) k_convert(const In* __restrict__ in, Out* __restrict__ out, int64_t count) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride)
    out[i] = round_out<Out>(widen<In>(in[i]));
}

template <typename In, typename Out>
cudaError_t launch_k(const void* in, void* out, int64_t count, cudaStream_t s) {
  const int64_t blocks = (count + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks < 4096 ? blocks : 4096);
  k_convert<In, Out><<<grid, 256, 0, s>>>(static_cast<const In*>(in), static_cast<Out*>(out), count);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_convert(const void* in, int in_dtype, void* out, int out_dtype, int64_t count, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  if (in_dtype == BITNET_DTYPE_F32 && out_dtype == BITNET_DTYPE_F16) return launch_k<float, __half>(in, out, count, s);
  if (in_dtype == BITNET_DTYPE_F32 && out_dtype == BITNET_DTYPE_BF16)
    return launch_k<float, __nv_bfloat16>(in, out, count, s);
  if (in_dtype == BITNET_DTYPE_F16 && out_dtype == BITNET_DTYPE_F32) return launch_k<__half, float>(in, out, count, s);
  if (in_dtype == BITNET_DTYPE_BF16 && out_dtype == BITNET_DTYPE_F32)
    return launch_k<__nv_bfloat16, float>(in, out, count, s);
  return cudaErrorInvalidValue;
}

}  // namespace bitnet
