// noalloc.cu -- bitnet_bitlinear_forward_noalloc: the whole projection without
// any device-memory allocation by the library.
//
// Who needs it: callers that may not allocate device memory once they are
// running -- for example a serving process that reserved all of HBM for its own
// caching allocator at start-up (so a cudaMalloc from a library would fail or
// fragment), or a latency-critical loop where an allocation's cost or possible
// failure is not acceptable.  They still pass their own inputs and outputs.
//
// How: most shapes need temporary space for the activation codes, the per-token
// scales and, where K is split over CTAs, fp32 partial sums.  Here that space is
// one file-scope device array of fixed size.  CUDA loads this file's module
// (and with it the array) on a device the first time its address is asked for,
// so the first call on each device does that for every shape, including the
// fused few-token shapes that never touch the array; from then on the device
// keeps the array until the process exits.  The array's name in host code is
// only a host-side stand-in and must never be handed to a kernel: the device
// address comes from cudaGetSymbolAddress, once per device.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace bitnet {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[BITNET_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_np_mu;
void* g_np_scratch[kMaxDev];
bool g_np_ready[kMaxDev];

// Device address of this device's copy of the scratch array (looked up once
// per device, with that device current).
int scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return BITNET_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_np_mu);
  if (!g_np_ready[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return BITNET_ERR_CUDA;
    }
    g_np_scratch[dev] = p;
    g_np_ready[dev] = true;
  }
  *out = g_np_scratch[dev];
  return BITNET_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace bitnet

using namespace bitnet;

extern "C" int bitnet_bitlinear_forward_noalloc(const float* x, const float* norm_w, const uint8_t* packed_w,
                                                float w_scale, int64_t M, int64_t K, int64_t N, float eps,
                                                float* y, bitnet_stream_t stream) {
  if (!x || !norm_w || !packed_w || !y) return BITNET_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || !(w_scale > 0.0f) || w_scale == INFINITY) return BITNET_ERR_INVALID_ARG;
  if (M < 1 || N < 1) return BITNET_ERR_INVALID_ARG;
  if (K < BITNET_I2S_BLOCK || K % BITNET_I2S_BLOCK != 0 || K > BITNET_MAX_K) return BITNET_ERR_UNSUPPORTED_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1) return BITNET_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(packed_w) || !aligned16(y)) return BITNET_ERR_MISALIGNED;
  const bool fused = decode_fused_supported(M, K) && !decode_split_preferred(M, K);
  const bool decode = decode_supported(M, K);
  // scratch layout: codes [M, K] (int8 for the decode kernel, fp16 for the
  // tensor-core kernel), then fp32 scales [M], 256-byte aligned
  const size_t code_bytes =
      (static_cast<size_t>(M) * static_cast<size_t>(K) * (decode ? 1 : 2) + 255) & ~size_t(255);
  if (!fused && code_bytes + static_cast<size_t>(M) * 4 > static_cast<size_t>(BITNET_NOALLOC_SCRATCH_BYTES))
    return BITNET_ERR_SCRATCH_LIMIT;

  DeviceContext* ctx;
  int rc = device_context_nopool(&ctx);
  if (rc) return rc;
  // looked up on every route, so that the first call on a device does all of
  // the one-time set-up whichever shape it has
  void* scratch = nullptr;
  if ((rc = scratch_for_current_device(&scratch))) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (fused) {
    DecodeJob j = {};
    j.x = x;
    j.g = norm_w;
    j.w = packed_w;
    j.w_scale = w_scale;
    j.K = static_cast<int>(K);
    j.N = static_cast<int>(N);
    j.y = y;
    return launch_decode(ctx, &j, 1, static_cast<int>(M), eps, true, false, s) == cudaSuccess ? BITNET_OK
                                                                                          : BITNET_ERR_CUDA;
  }
  float* as = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + code_bytes);
  // every element of the used scratch region is written by the norm launch
  // before the contraction reads it, so nothing has to be cleared first
  if (decode) {
    int8_t* codes = static_cast<int8_t*>(scratch);
    // the norm kernel lets the decode kernel start only after the kernels
    // before it have completed, so the weights may be streamed early
    cudaError_t e = launch_rmsnorm_quant(x, norm_w, M, static_cast<int>(K), eps, codes, nullptr, as, nullptr,
                                         nullptr, true, s);
    if (e == cudaSuccess) {
      DecodeJob j = {};
      j.codes = codes;
      j.a_scale = as;
      j.w = packed_w;
      j.w_scale = w_scale;
      j.K = static_cast<int>(K);
      j.N = static_cast<int>(N);
      j.y = y;
      e = launch_decode(ctx, &j, 1, static_cast<int>(M), eps, false, true, s,
                        static_cast<int>(rmsnorm_quant_ctas(M, static_cast<int>(K))));
    }
    return e == cudaSuccess ? BITNET_OK : BITNET_ERR_CUDA;
  }
  __half* f16 = static_cast<__half*>(scratch);
  // 9..63 tokens: the split-K contraction, when its workspace also fits; the
  // tokens-as-M contraction splits K too when its workspace fits.  When the
  // workspace does not fit, the tokens-as-M contraction runs without a K split
  // (the same y: every plan sums the same integers exactly).
  const size_t scale_bytes = (static_cast<size_t>(M) * 4 + 255) & ~size_t(255);
  const bool sk_shape = gemm_skinny_supported(M, K, N);
  const size_t gws_bytes = sk_shape ? gemm_skinny_workspace(ctx, M, K, N) : gemm_tc_workspace(ctx, M, K, N);
  const bool fits = code_bytes + scale_bytes + gws_bytes <= static_cast<size_t>(BITNET_NOALLOC_SCRATCH_BYTES);
  const bool skinny = sk_shape && fits;
  uint8_t* gws = static_cast<uint8_t*>(scratch) + code_bytes + scale_bytes;
  void* tc_ws = (!sk_shape && fits && gws_bytes) ? static_cast<void*>(gws) : nullptr;
  const size_t zero_bytes = skinny ? gemm_skinny_zeroed_bytes(ctx, M, K, N) : gws_bytes;
  cudaError_t e = (fits && zero_bytes) ? cudaMemsetAsync(gws, 0, zero_bytes, s) : cudaSuccess;
  // 9..63 tokens: the norm launch writes the contraction's planes, and their
  // row sums into the workspace (the array is 256-byte aligned)
  int32_t* rs = skinny ? gemm_skinny_rowsum_area(ctx, gws, M, K, N) : nullptr;
  if (e == cudaSuccess)
    e = rs ? launch_rmsnorm_quant_planes(x, BITNET_DTYPE_F32, norm_w, M, static_cast<int>(K), eps, f16, as, rs, true,
                                         s)
           : launch_rmsnorm_quant(x, norm_w, M, static_cast<int>(K), eps, nullptr, f16, as, nullptr, nullptr, true, s);
  int st = BITNET_OK;
  if (e == cudaSuccess)
    e = skinny ? launch_gemm_skinny(ctx, f16, rs, as, packed_w, w_scale, M, K, N, y, nullptr, gws, true, true, s, &st)
               : launch_gemm_tc(ctx, f16, as, packed_w, w_scale, M, K, N, y, BITNET_DTYPE_F32, nullptr, tc_ws, true, true, s, &st);
  if (st != BITNET_OK) return st;
  return e == cudaSuccess ? BITNET_OK : BITNET_ERR_CUDA;
}
