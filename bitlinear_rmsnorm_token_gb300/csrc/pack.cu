// pack.cu -- I2_S absmean ternary packing and unpacking on the GPU.
//
// "BitNet Embeddings GGUF Conversion Implementation", section 3 ("I2_S Ternary
// Packing") and "BitNet Inference Framework" ("Quantization and Encoding",
// "Data Layout"): w_scale = 1 / mean|w|, q = clamp(round(w * w_scale), -1, 1),
// code = q + 1, 128 values per 32-byte block, byte = c0<<6 | c1<<4 | c2<<2 | c3,
// one fp32 scale after the last block.  The element-to-byte map (byte j <-
// elements j, 32+j, 64+j, 96+j) is the library's own (bitnet.h).
//
// mean|w| is reduced in double in a fixed order that depends only on the
// element count (fixed grid and tree), so a tensor always packs to the same
// bytes on any GPU.  This is off the hot path: weights are packed once.
#include "common.cuh"
#include "internal.h"

namespace bitnet {
namespace {

constexpr int kAbsThreads = 256;

// Partial sums of |w| in double.  Block b handles a contiguous span; thread t
// of it sums every 256th element of the span; the block then adds its 256
// thread sums with a fixed tree.
__global__ void __launch_bounds__(kAbsThreads) k_abs_partial(const float* __restrict__ w, int64_t count,
                                                             int64_t span, double* __restrict__ partials) {
  __shared__ double red[kAbsThreads];
  const int64_t begin = static_cast<int64_t>(blockIdx.x) * span;
  const int64_t end = begin + span < count ? begin + span : count;
  double s = 0.0;
  for (int64_t i = begin + threadIdx.x; i < end; i += kAbsThreads) s += fabs(static_cast<double>(__ldg(w + i)));
  red[threadIdx.x] = s;
  __syncthreads();
  for (int h = kAbsThreads / 2; h > 0; h >>= 1) {
    if (threadIdx.x < h) red[threadIdx.x] = red[threadIdx.x] + red[threadIdx.x + h];
    __syncthreads();
  }
  if (threadIdx.x == 0) partials[blockIdx.x] = red[0];
}

// Adds the partials in index order and stores w_scale (1 / mean, or 1 when the
// tensor is all zero) at the end of the packed buffer.
__global__ void k_abs_final(const double* __restrict__ partials, int n, int64_t count, float* __restrict__ scale_out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += partials[i];
  const double mean = s / static_cast<double>(count);
  *scale_out = mean == 0.0 ? 1.0f : static_cast<float>(1.0 / mean);
}

__device__ __forceinline__ unsigned ternary_code(float w, float scale) {
  float r = rintf(__fmul_rn(w, scale));
  r = fminf(fmaxf(r, -1.0f), 1.0f);
  return static_cast<unsigned>(static_cast<int>(r) + 1);
}

// One thread -> one 32-bit word = bytes 4i..4i+3 of block b, i.e. elements
// 4i..4i+3 of each of the block's four 32-element slots.
__global__ void __launch_bounds__(256) k_pack(const float* __restrict__ w, int64_t nwords,
                                              const float* __restrict__ scale_ptr, uint32_t* __restrict__ out) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nwords) return;
  const float scale = *scale_ptr;
  const int64_t b = t >> 3;
  const int i = static_cast<int>(t & 7);
  const float* blk = w + b * 128 + 4 * i;
  unsigned c[4][4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(blk + 32 * s));
    c[s][0] = ternary_code(v.x, scale);
    c[s][1] = ternary_code(v.y, scale);
    c[s][2] = ternary_code(v.z, scale);
    c[s][3] = ternary_code(v.w, scale);
  }
  uint32_t word = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t byte = (c[0][e] << 6) | (c[1][e] << 4) | (c[2][e] << 2) | c[3][e];
    word |= byte << (8 * e);  // byte 4i+e sits at the lower address
  }
  out[t] = word;
}

// One thread -> one 32-bit word of codes -> 16 ternary int8 values.
__global__ void __launch_bounds__(256) k_unpack(const uint32_t* __restrict__ in, int64_t nwords,
                                                int8_t* __restrict__ out) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nwords) return;
  const uint32_t word = __ldg(in + t);
  const int64_t b = t >> 3;
  const int i = static_cast<int>(t & 7);
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const uint32_t codes = (word >> (6 - 2 * s)) & 0x03030303u;
    // code - 1 per byte: bytes are 0..3, subtracting 0x01010101 borrows nothing
    // for codes >= 1; code 0 -> 0xFF = -1.  Computed per byte to stay exact.
    uint32_t v = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int q = static_cast<int>((codes >> (8 * e)) & 0xFFu) - 1;
      v |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * e);
    }
    *reinterpret_cast<uint32_t*>(out + b * 128 + 32 * s + 4 * i) = v;
  }
}

}  // namespace

int pack_num_partials(int64_t count) {
  // depends on the element count only, so the reduction order is fixed
  int64_t n = (count + (1 << 16) - 1) >> 16;  // about 64 Ki elements per block
  if (n < 1) n = 1;
  if (n > 4096) n = 4096;
  return static_cast<int>(n);
}

cudaError_t launch_pack_i2s(const DeviceContext* ctx, const float* w, int64_t N, int64_t K, uint8_t* packed,
                            double* partials, int num_partials, cudaStream_t s) {
  (void)ctx;
  const int64_t count = N * K;
  const int64_t span = (count + num_partials - 1) / num_partials;
  float* scale_out = reinterpret_cast<float*>(packed + count / 4);
  k_abs_partial<<<num_partials, kAbsThreads, 0, s>>>(w, count, span, partials);
  k_abs_final<<<1, 32, 0, s>>>(partials, num_partials, count, scale_out);
  const int64_t nwords = count / 16;
  const int64_t blocks = (nwords + 255) / 256;
  k_pack<<<static_cast<unsigned>(blocks), 256, 0, s>>>(w, nwords, scale_out, reinterpret_cast<uint32_t*>(packed));
  return cudaGetLastError();
}

cudaError_t launch_unpack_i2s(const uint8_t* packed, int64_t N, int64_t K, int8_t* out, cudaStream_t s) {
  const int64_t nwords = N * K / 16;
  const int64_t blocks = (nwords + 255) / 256;
  k_unpack<<<static_cast<unsigned>(blocks), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(packed), nwords, out);
  return cudaGetLastError();
}

}  // namespace bitnet
