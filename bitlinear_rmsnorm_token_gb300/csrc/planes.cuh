// planes.cuh -- the token operand of the 9..63-token tensor-core contraction:
// each int8 activation code q written as q = 16 hi + lo, hi = floor(q / 16) in
// [-8, 7] and lo = q mod 16 in [0, 15], both exact e4m3 values.  Layout over a
// row-major [M, K] array of 2-byte slots (the footprint of fp16 codes, K a
// multiple of 128, the array 256-byte aligned): each 128-value block of a row
// (256 bytes) holds its 128 hi bytes, then its 128 lo bytes.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace bitnet {

// e4m3 byte of a small integer (exact for -8 .. 15)
__device__ __forceinline__ uint32_t e4m3_int_byte(int v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(static_cast<float>(v), __NV_SATFINITE, __NV_E4M3));
}

// hi- and lo-plane words of four codes packed as int8 bytes (first code in the
// lowest byte, as quant_pack4_i8 packs them)
__device__ __forceinline__ void plane_words4(uint32_t packed, uint32_t& hi, uint32_t& lo) {
  hi = 0;
  lo = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = static_cast<int8_t>((packed >> (8 * i)) & 0xFF);
    const int l = q & 15;
    lo |= e4m3_int_byte(l) << (8 * i);
    hi |= e4m3_int_byte((q - l) / 16) << (8 * i);
  }
}

// Stores the planes of the four codes of elements k .. k + 3 of a row (k a
// multiple of 4) given the address the fp16 code of element k has in the
// array: the block's 256 bytes start at that address rounded down to 256, and
// element k sits at byte k mod 128 of each half.
__device__ __forceinline__ void store_planes4(void* fp16_slot, uint32_t hi, uint32_t lo) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(fp16_slot);
  uint8_t* blk = reinterpret_cast<uint8_t*>(a & ~uintptr_t(255));
  const unsigned e = static_cast<unsigned>(a & 255u) >> 1;
  *reinterpret_cast<uint32_t*>(blk + e) = hi;
  *reinterpret_cast<uint32_t*>(blk + 128 + e) = lo;
}

}  // namespace bitnet
