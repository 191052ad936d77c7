// unpack_f16.cuh -- I2_S packed bytes to fp16 tensor-core operand rows.
//
// I2_S ("BitNet Embeddings GGUF Conversion Implementation", I2_S packing): a
// 128-value block is 32 bytes; byte j holds the 2-bit codes of elements j,
// 32+j, 64+j and 96+j in bits 7:6, 5:4, 3:2 and 1:0; the weight is code - 1.
// The rows written here are K-major with the 128-byte swizzle of tcgen05
// shared-memory operands: a 64-value (128-byte) slab per row, 16-byte chunk c
// of row r stored at chunk c ^ (r & 7).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace bitnet {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four 2-bit codes (one per byte, values 0..2) -> two half2 words holding code-1.
__device__ __forceinline__ void codes_to_h2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  const uint32_t kMagic = 0x64646464u;     // high byte of fp16 1024.0
  const uint32_t kBias = 0x64016401u;      // half2(1025, 1025)
  uint32_t a = prmt(v, kMagic, 0x4140u);   // {1024 + c0, 1024 + c1}
  uint32_t b = prmt(v, kMagic, 0x4342u);   // {1024 + c2, 1024 + c3}
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<const __half2*>(&kBias));
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), *reinterpret_cast<const __half2*>(&kBias));
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// Chunks c0 .. c0+kChunks-1 (16 bytes = 8 values each) of one weight row's
// 64-value slab (slots 2*hf and 2*hf+1 of its I2_S block) as fp16 into the
// swizzled K-major row `dst` (row r of an 8-row atom: sw = r & 7).
template <int kChunks>
__device__ __forceinline__ void unpack_row_slab(const uint32_t (&wd)[8], int hf, int c0, uint8_t* dst, int sw) {
#pragma unroll
  for (int ci = 0; ci < kChunks; ++ci) {
    const int c = c0 + ci;
    const int sl = 2 * hf + (c >> 2);  // slot of the block: elements 32*sl + j
    const int jw = 2 * (c & 3);        // words jw, jw+1 = bytes j = 8*(c&3) .. +7
    const int sh = 6 - 2 * sl;
    const uint32_t v0 = (wd[jw] >> sh) & 0x03030303u;
    const uint32_t v1 = (wd[jw + 1] >> sh) & 0x03030303u;
    uint4 out;
    codes_to_h2(v0, out.x, out.y);
    codes_to_h2(v1, out.z, out.w);
    *reinterpret_cast<uint4*>(dst + ((c ^ sw) << 4)) = out;
  }
}

}  // namespace bitnet
