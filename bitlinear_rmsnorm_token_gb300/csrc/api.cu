// api.cu -- the C ABI declared in include/bitnet.h: argument checks, dispatch
// between the decode and tensor-core paths, per-device state.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace bitnet {

// Per-device record of device-side failures (bitnet_last_device_status).
__device__ unsigned g_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceContext g_ctx[kMaxDevices];
bool g_ready[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_shape(int64_t M, int64_t K, int64_t N) {
  if (M < 1 || N < 1) return BITNET_ERR_INVALID_ARG;
  if (K < BITNET_I2S_BLOCK || K % BITNET_I2S_BLOCK != 0 || K > BITNET_MAX_K) return BITNET_ERR_UNSUPPORTED_SHAPE;
  if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1) return BITNET_ERR_UNSUPPORTED_SHAPE;
  return BITNET_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? BITNET_OK : BITNET_ERR_CUDA; }

}  // namespace

int device_context(DeviceContext** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return BITNET_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return BITNET_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return BITNET_ERR_NO_DEVICE;  // built for sm_103a only
    DeviceContext c;
    c.device = dev;
    c.num_sms = prop.multiProcessorCount;
    void* ew = nullptr;
    if (cudaGetSymbolAddress(&ew, g_error_word) != cudaSuccess) return BITNET_ERR_CUDA;
    // the word starts at zero when the module loads; it is not cleared here, so
    // a timeout an earlier call recorded (the no-alloc entry point's, say) stays
    // until bitnet_last_device_status reports it
    c.err_word = static_cast<unsigned*>(ew);
    cudaMemPoolProps pp = {};
    pp.allocType = cudaMemAllocationTypePinned;
    pp.handleTypes = cudaMemHandleTypeNone;
    pp.location.type = cudaMemLocationTypeDevice;
    pp.location.id = dev;
    if (cudaMemPoolCreate(&c.pool, &pp) != cudaSuccess) return BITNET_ERR_CUDA;
    uint64_t keep = UINT64_MAX;  // keep freed blocks cached in the pool
    cudaMemPoolSetAttribute(c.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    g_ctx[dev] = c;
    g_ready[dev] = true;
  }
  *out = &g_ctx[dev];
  return BITNET_OK;
}

namespace {
DeviceContext g_ctx_np[kMaxDevices];
bool g_ready_np[kMaxDevices];
}  // namespace

int device_context_nopool(DeviceContext** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return BITNET_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready_np[dev]) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return BITNET_ERR_NO_DEVICE;
    if (prop.major != 10 || prop.minor != 3) return BITNET_ERR_NO_DEVICE;
    DeviceContext c;
    c.device = dev;
    c.num_sms = prop.multiProcessorCount;
    void* ew = nullptr;
    if (cudaGetSymbolAddress(&ew, g_error_word) != cudaSuccess) return BITNET_ERR_CUDA;
    c.err_word = static_cast<unsigned*>(ew);
    g_ctx_np[dev] = c;
    g_ready_np[dev] = true;
  }
  *out = &g_ctx_np[dev];
  return BITNET_OK;
}

int pool_alloc(DeviceContext* ctx, void** p, size_t bytes, cudaStream_t stream) {
  if (cudaMallocFromPoolAsync(p, bytes, ctx->pool, stream) != cudaSuccess) {
    cudaGetLastError();
    return BITNET_ERR_CUDA;
  }
  return BITNET_OK;
}

void pool_free(void* p, cudaStream_t stream) {
  if (p) cudaFreeAsync(p, stream);
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

}  // namespace bitnet

using namespace bitnet;

extern "C" {

size_t bitnet_i2s_packed_bytes(int64_t N, int64_t K) {
  if (N < 1 || K < BITNET_I2S_BLOCK || K % BITNET_I2S_BLOCK != 0) return 0;
  return static_cast<size_t>(N) * static_cast<size_t>(K) / 4 + 4;
}

const char* bitnet_status_string(int status) {
  switch (status) {
    case BITNET_OK: return "ok";
    case BITNET_ERR_INVALID_ARG: return "invalid argument";
    case BITNET_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (K must be a positive multiple of 128, <= 65536)";
    case BITNET_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case BITNET_ERR_CUDA: return "CUDA error";
    case BITNET_ERR_TIMEOUT: return "device-side wait timed out";
    case BITNET_ERR_NO_DEVICE: return "no sm_103 CUDA device";
    case BITNET_ERR_SCRATCH_LIMIT:
      return "problem needs more than the 16 MiB no-alloc scratch (2*M*K + 4*M bytes); use bitnet_bitlinear_forward";
    default: return "unknown status";
  }
}

int bitnet_pack_i2s(const float* w, int64_t N, int64_t K, uint8_t* packed, float* w_scale_out,
                    bitnet_stream_t stream) {
  if (!w || !packed) return BITNET_ERR_INVALID_ARG;
  int rc = check_shape(1, K, N);
  if (rc) return rc;
  if (!aligned16(w) || !aligned16(packed)) return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  if ((rc = device_context(&ctx))) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int np = pack_num_partials(N * K);
  double* partials = nullptr;
  if ((rc = pool_alloc(ctx, reinterpret_cast<void**>(&partials), np * sizeof(double), s))) return rc;
  cudaError_t e = launch_pack_i2s(ctx, w, N, K, packed, partials, np, s);
  pool_free(partials, s);
  if (e != cudaSuccess) return BITNET_ERR_CUDA;
  if (w_scale_out) {
    e = cudaMemcpyAsync(w_scale_out, packed + N * K / 4, sizeof(float), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return BITNET_ERR_CUDA;
  }
  return BITNET_OK;
}

int bitnet_unpack_i2s(const uint8_t* packed, int64_t N, int64_t K, int8_t* w_ternary, bitnet_stream_t stream) {
  if (!packed || !w_ternary) return BITNET_ERR_INVALID_ARG;
  int rc = check_shape(1, K, N);
  if (rc) return rc;
  if (!aligned16(packed) || !aligned16(w_ternary)) return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  if ((rc = device_context(&ctx))) return rc;
  return cuda_status(launch_unpack_i2s(packed, N, K, w_ternary, reinterpret_cast<cudaStream_t>(stream)));
}

int bitnet_rmsnorm_quant_a8(const float* x, const float* norm_w, int64_t M, int64_t K, float eps, int8_t* a_codes,
                            float* a_scale, int32_t* a_rowsum, float* xn_out, bitnet_stream_t stream) {
  if (!x || !norm_w || !a_codes || !a_scale) return BITNET_ERR_INVALID_ARG;
  if (!(eps > 0.0f)) return BITNET_ERR_INVALID_ARG;
  int rc = check_shape(M, K, 1);
  if (rc) return rc;
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(a_codes) || !aligned4(a_scale) ||
      (a_rowsum && !aligned4(a_rowsum)) || (xn_out && !aligned16(xn_out)))
    return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  if ((rc = device_context(&ctx))) return rc;
  return cuda_status(launch_rmsnorm_quant(x, norm_w, M, static_cast<int>(K), eps, a_codes, nullptr, a_scale,
                                          a_rowsum, xn_out, false, reinterpret_cast<cudaStream_t>(stream)));
}

int bitnet_i2s_gemm(const int8_t* a_codes, const float* a_scale, const uint8_t* packed_w, float w_scale, int64_t M,
                    int64_t K, int64_t N, float* y, int32_t* acc_out, bitnet_stream_t stream) {
  if (!a_codes || !a_scale || !packed_w || !y) return BITNET_ERR_INVALID_ARG;
  if (!(w_scale > 0.0f) || w_scale == INFINITY) return BITNET_ERR_INVALID_ARG;
  int rc = check_shape(M, K, N);
  if (rc) return rc;
  if (!aligned16(a_codes) || !aligned4(a_scale) || !aligned16(packed_w) || !aligned16(y) ||
      (acc_out && !aligned16(acc_out)))
    return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  if ((rc = device_context(&ctx))) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (decode_supported(M, K)) {
    DecodeJob j = {};
    j.codes = a_codes;
    j.a_scale = a_scale;
    j.w = packed_w;
    j.w_scale = w_scale;
    j.K = static_cast<int>(K);
    j.N = static_cast<int>(N);
    j.y = y;
    j.acc_out = acc_out;
    return cuda_status(launch_decode(ctx, &j, 1, static_cast<int>(M), 0.0f, false, false, s));
  }
  const bool skinny = gemm_skinny_supported(M, K, N);
  const size_t code_bytes = (static_cast<size_t>(M * K) * 2 + 255) & ~size_t(255);
  const size_t gws_bytes = skinny ? gemm_skinny_workspace(ctx, M, K, N) : gemm_tc_workspace(ctx, M, K, N);
  uint8_t* buf = nullptr;
  if ((rc = pool_alloc(ctx, reinterpret_cast<void**>(&buf), code_bytes + gws_bytes, s))) return rc;
  __half* f16 = reinterpret_cast<__half*>(buf);
  void* gws = gws_bytes ? static_cast<void*>(buf + code_bytes) : nullptr;
  cudaError_t e = launch_codes_to_f16(a_codes, f16, M * K, s);
  int st = BITNET_OK;
  if (e == cudaSuccess)
    e = skinny ? launch_gemm_skinny(ctx, f16, nullptr, a_scale, packed_w, w_scale, M, K, N, y, acc_out, gws, false,
                                    true, s, &st)
               : launch_gemm_tc(ctx, f16, a_scale, packed_w, w_scale, M, K, N, y, BITNET_DTYPE_F32, acc_out, gws, false, true, s, &st);
  pool_free(buf, s);
  if (st != BITNET_OK) return st;
  return cuda_status(e);
}

}  // extern "C"

namespace {

// The norm + quant launch of a forward: x directly (act == 0), or the down
// projection's input act(x) * up -- computed as the rows are loaded when they
// fit registers (K <= 3072), else written to h_buf (M*K floats) first.
cudaError_t launch_norm_any(const float* x, const float* up, int act, const float* g, int64_t M, int K, float eps,
                            int8_t* codes_i8, __half* codes_f16, float* a_scale, float* h_buf, bool pdl,
                            cudaStream_t s) {
  if (act == 0)
    return launch_rmsnorm_quant(x, g, M, K, eps, codes_i8, codes_f16, a_scale, nullptr, nullptr, pdl, s);
  if (rmsnorm_quant_glu_fused_supported(K))
    return launch_rmsnorm_quant_glu(x, up, act, g, M, K, eps, codes_i8, codes_f16, a_scale, nullptr, nullptr, pdl,
                                    s);
  cudaError_t e = launch_glu(x, up, act, M * K, h_buf, s);
  if (e != cudaSuccess) return e;
  return launch_rmsnorm_quant(h_buf, g, M, K, eps, codes_i8, codes_f16, a_scale, nullptr, nullptr, pdl, s);
}

// The same for the 9..63-token contraction: the codes as its two e4m3 planes
// (`planes` 256-byte aligned) and their row sums.
cudaError_t launch_norm_planes_any(const float* x, const float* up, int act, const float* g, int64_t M, int K,
                                   float eps, void* planes, float* a_scale, int32_t* rowsum, float* h_buf, bool pdl,
                                   cudaStream_t s) {
  if (act == 0)
    return launch_rmsnorm_quant_planes(x, BITNET_DTYPE_F32, g, M, K, eps, planes, a_scale, rowsum, pdl, s);
  if (rmsnorm_quant_glu_fused_supported(K))
    return launch_rmsnorm_quant_glu_planes(x, up, act, g, M, K, eps, planes, a_scale, rowsum, pdl, s);
  cudaError_t e = launch_glu(x, up, act, M * K, h_buf, s);
  if (e != cudaSuccess) return e;
  return launch_rmsnorm_quant_planes(h_buf, BITNET_DTYPE_F32, g, M, K, eps, planes, a_scale, rowsum, pdl, s);
}

bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

size_t glu_buffer_bytes(int act, int64_t M, int64_t K) {
  return (act != 0 && !rmsnorm_quant_glu_fused_supported(static_cast<int>(K)))
             ? ((static_cast<size_t>(M * K) * 4 + 255) & ~size_t(255))
             : 0;
}

// bitnet_bitlinear_forward (act == 0) and bitnet_bitlinear_forward_glu: x is the
// input, or the gate projection's output when act != 0 (the row is act(x) * up).
// head_w / head_dim / head_fused: the QK head norm, applied in the tensor-core
// epilogue when that route is taken and its plan allows (*head_fused then true).
int forward_impl(const float* x, const float* up, int act, const float* norm_w, const uint8_t* packed_w,
                 float w_scale, int64_t M, int64_t K, int64_t N, float eps, float* y, bitnet_stream_t stream,
                 const float* head_w = nullptr, int head_dim = 0, bool* head_fused = nullptr) {
  if (head_fused) *head_fused = false;
  if (!x || !norm_w || !packed_w || !y || (act != 0 && !up)) return BITNET_ERR_INVALID_ARG;
  if (act != 0 && act != BITNET_ACT_SILU && act != BITNET_ACT_GELU_TANH) return BITNET_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || !(w_scale > 0.0f) || w_scale == INFINITY) return BITNET_ERR_INVALID_ARG;
  int rc = check_shape(M, K, N);
  if (rc) return rc;
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(packed_w) || !aligned16(y) || (up && !aligned16(up)))
    return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  if ((rc = device_context(&ctx))) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool fused = act != 0 ? decode_fused_glu_supported(M, K)
                              : (decode_fused_supported(M, K) && !decode_split_preferred(M, K));
  if (fused) {
    DecodeJob j = {};
    j.x = x;
    j.up = up;
    j.act = act;
    j.g = norm_w;
    j.w = packed_w;
    j.w_scale = w_scale;
    j.K = static_cast<int>(K);
    j.N = static_cast<int>(N);
    j.y = y;
    return cuda_status(launch_decode(ctx, &j, 1, static_cast<int>(M), eps, true, false, s));
  }
  const size_t h_bytes = glu_buffer_bytes(act, M, K);
  if (decode_supported(M, K)) {
    // few tokens but long rows: int8 codes through the pool, then the decode
    // kernel.  The norm kernel lets its dependent start only after the kernels
    // before it have completed, and it writes no weights, so the decode kernel
    // may stream its weights before its own dependency wait, overlapping the
    // norm kernel.
    const size_t code_bytes = (static_cast<size_t>(M * K) + 255) & ~size_t(255);
    const size_t scale_bytes = (static_cast<size_t>(M) * 4 + 255) & ~size_t(255);
    uint8_t* ws = nullptr;
    if ((rc = pool_alloc(ctx, reinterpret_cast<void**>(&ws), code_bytes + scale_bytes + h_bytes, s))) return rc;
    int8_t* codes = reinterpret_cast<int8_t*>(ws);
    float* as = reinterpret_cast<float*>(ws + code_bytes);
    float* h = h_bytes ? reinterpret_cast<float*>(ws + code_bytes + scale_bytes) : nullptr;
    cudaError_t e = launch_norm_any(x, up, act, norm_w, M, static_cast<int>(K), eps, codes, nullptr, as, h, true, s);
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
    pool_free(ws, s);
    return cuda_status(e);
  }
  // norm + quant to fp16 codes, then the tensor-core contraction (the split-K
  // form for up to 128 tokens, its workspace zeroed ahead of the norm launch so
  // that the two kernels stay chained by programmatic dependent launch)
  const bool skinny = gemm_skinny_supported(M, K, N);
  const size_t code_bytes = (static_cast<size_t>(M * K) * 2 + 255) & ~size_t(255);
  const size_t scale_bytes = (static_cast<size_t>(M) * 4 + 255) & ~size_t(255);
  // rounded up: the workspace ends with 4-byte tile tickets, and h (16-byte
  // accesses) follows it
  const size_t gws_raw = skinny ? gemm_skinny_workspace(ctx, M, K, N) : gemm_tc_workspace(ctx, M, K, N);
  const size_t gws_bytes = (gws_raw + 255) & ~size_t(255);
  const size_t rs_bytes = skinny ? (static_cast<size_t>(M) * 4 + 255) & ~size_t(255) : 0;
  uint8_t* ws = nullptr;
  if ((rc = pool_alloc(ctx, reinterpret_cast<void**>(&ws),
                       code_bytes + scale_bytes + gws_bytes + h_bytes + rs_bytes, s)))
    return rc;
  __half* f16 = reinterpret_cast<__half*>(ws);
  float* as = reinterpret_cast<float*>(ws + code_bytes);
  uint8_t* gws = ws + code_bytes + scale_bytes;
  float* h = h_bytes ? reinterpret_cast<float*>(ws + code_bytes + scale_bytes + gws_bytes) : nullptr;
  // 9..63 tokens: the norm launch writes the contraction's planes and row sums
  // directly (its block layout needs a 256-byte aligned array)
  int32_t* rs = skinny && aligned256(f16)
                    ? reinterpret_cast<int32_t*>(ws + code_bytes + scale_bytes + gws_bytes + h_bytes)
                    : nullptr;
  const size_t zero_bytes = skinny ? gemm_skinny_zeroed_bytes(ctx, M, K, N) : gws_bytes;
  cudaError_t e = zero_bytes ? cudaMemsetAsync(gws, 0, zero_bytes, s) : cudaSuccess;
  if (e == cudaSuccess)
    e = rs ? launch_norm_planes_any(x, up, act, norm_w, M, static_cast<int>(K), eps, f16, as, rs, h, true, s)
           : launch_norm_any(x, up, act, norm_w, M, static_cast<int>(K), eps, nullptr, f16, as, h, true, s);
  int st = BITNET_OK;
  if (e == cudaSuccess)
    e = skinny ? launch_gemm_skinny(ctx, f16, rs, as, packed_w, w_scale, M, K, N, y, nullptr, gws, true, true, s, &st)
               : launch_gemm_tc(ctx, f16, as, packed_w, w_scale, M, K, N, y, BITNET_DTYPE_F32, nullptr, gws_bytes ? gws : nullptr, true,
                                true, s, &st, head_w, head_dim, eps, head_fused);
  pool_free(ws, s);
  if (st != BITNET_OK) return st;
  return cuda_status(e);
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// The projection with 16-bit x / y and an fp16 norm weight: inputs widened to
// fp32 exactly, the fp32 path's arithmetic, y rounded once to its type.
int forward_typed(const void* x, int x_dtype, const void* norm_w, int g_dtype, const uint8_t* packed_w,
                  float w_scale, int64_t M, int64_t K, int64_t N, float eps, void* y, int y_dtype,
                  bitnet_stream_t stream) {
  auto io_type = [](int t) { return t == BITNET_DTYPE_F32 || t == BITNET_DTYPE_F16 || t == BITNET_DTYPE_BF16; };
  if (!x || !norm_w || !packed_w || !y) return BITNET_ERR_INVALID_ARG;
  if (!io_type(x_dtype) || !io_type(y_dtype) || (g_dtype != BITNET_DTYPE_F32 && g_dtype != BITNET_DTYPE_F16))
    return BITNET_ERR_INVALID_ARG;
  if (x_dtype == BITNET_DTYPE_F32 && g_dtype == BITNET_DTYPE_F32 && y_dtype == BITNET_DTYPE_F32)
    return forward_impl(static_cast<const float*>(x), nullptr, 0, static_cast<const float*>(norm_w), packed_w,
                        w_scale, M, K, N, eps, static_cast<float*>(y), stream);
  if (!(eps > 0.0f) || !(w_scale > 0.0f) || w_scale == INFINITY) return BITNET_ERR_INVALID_ARG;
  int rc = check_shape(M, K, N);
  if (rc) return rc;
  if (!aligned16(x) || !aligned16(norm_w) || !aligned16(packed_w) || !aligned16(y)) return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  if ((rc = device_context(&ctx))) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // few tokens (the weight-streaming kernels read and write fp32): the fp32
  // path on converted copies; otherwise the norm launch reads x as it is
  const bool few = M <= kDecodeMaxM;
  const bool skinny = !few && gemm_skinny_supported(M, K, N);
  const bool x_copy = few && x_dtype != BITNET_DTYPE_F32;
  const bool y_copy = (few || skinny) && y_dtype != BITNET_DTYPE_F32;
  const size_t g_bytes = g_dtype != BITNET_DTYPE_F32 ? round256(static_cast<size_t>(K) * 4) : 0;
  const size_t x_bytes = x_copy ? round256(static_cast<size_t>(M * K) * 4) : 0;
  const size_t y_bytes = y_copy ? round256(static_cast<size_t>(M * N) * 4) : 0;
  const size_t code_bytes = few ? 0 : round256(static_cast<size_t>(M * K) * 2);
  const size_t scale_bytes = few ? 0 : round256(static_cast<size_t>(M) * 4);
  const size_t gws_bytes =
      few ? 0 : round256(skinny ? gemm_skinny_workspace(ctx, M, K, N) : gemm_tc_workspace(ctx, M, K, N));
  const size_t rs_bytes = skinny ? round256(static_cast<size_t>(M) * 4) : 0;
  const size_t total = g_bytes + x_bytes + y_bytes + code_bytes + scale_bytes + gws_bytes + rs_bytes;
  uint8_t* pool = nullptr;
  if (total && (rc = pool_alloc(ctx, reinterpret_cast<void**>(&pool), total, s))) return rc;
  uint8_t* at = pool;
  auto take = [&](size_t b) {
    uint8_t* p = b ? at : nullptr;
    at += b;
    return p;
  };
  float* g32 = reinterpret_cast<float*>(take(g_bytes));
  float* x32 = reinterpret_cast<float*>(take(x_bytes));
  float* y32 = reinterpret_cast<float*>(take(y_bytes));
  __half* f16 = reinterpret_cast<__half*>(take(code_bytes));
  float* as = reinterpret_cast<float*>(take(scale_bytes));
  uint8_t* gws = take(gws_bytes);
  int32_t* rs = reinterpret_cast<int32_t*>(take(rs_bytes));
  if (rs && !aligned256(f16)) rs = nullptr;  // the planes' block layout needs a 256-byte aligned array
  const float* g = g32 ? g32 : static_cast<const float*>(norm_w);
  cudaError_t e = cudaSuccess;
  if (g32) e = launch_convert(norm_w, g_dtype, g32, BITNET_DTYPE_F32, K, s);
  int st = BITNET_OK;
  if (few) {
    if (e == cudaSuccess && x32) e = launch_convert(x, x_dtype, x32, BITNET_DTYPE_F32, M * K, s);
    if (e == cudaSuccess) {
      st = forward_impl(x32 ? x32 : static_cast<const float*>(x), nullptr, 0, g, packed_w, w_scale, M, K, N, eps,
                        y32 ? y32 : static_cast<float*>(y), stream);
      if (st != BITNET_OK) e = cudaErrorUnknown;
    }
  } else {
    const size_t zero_bytes = skinny ? gemm_skinny_zeroed_bytes(ctx, M, K, N) : gws_bytes;
    if (e == cudaSuccess && zero_bytes) e = cudaMemsetAsync(gws, 0, zero_bytes, s);
    if (e == cudaSuccess)
      e = rs ? launch_rmsnorm_quant_planes(x, x_dtype, g, M, static_cast<int>(K), eps, f16, as, rs, true, s)
             : launch_rmsnorm_quant_f16_in(x, x_dtype, g, M, static_cast<int>(K), eps, f16, as, true, s);
    if (e == cudaSuccess)
      e = skinny ? launch_gemm_skinny(ctx, f16, rs, as, packed_w, w_scale, M, K, N,
                                      y32 ? y32 : static_cast<float*>(y), nullptr, gws, true, true, s, &st)
                 : launch_gemm_tc(ctx, f16, as, packed_w, w_scale, M, K, N, y, y_dtype, nullptr,
                                  gws_bytes ? gws : nullptr, true, true, s, &st);
  }
  if (e == cudaSuccess && st == BITNET_OK && y32) e = launch_convert(y32, BITNET_DTYPE_F32, y, y_dtype, M * N, s);
  if (pool) pool_free(pool, s);
  if (st != BITNET_OK) return st;
  return cuda_status(e);
}

}  // namespace

extern "C" {

int bitnet_head_rmsnorm(const float* y, int64_t M, int64_t N, int64_t head_dim, const float* head_w, float eps,
                        float* out, bitnet_stream_t stream) {
  if (!y || !head_w || !out || M < 1 || N < 1 || !(eps > 0.0f)) return BITNET_ERR_INVALID_ARG;
  if (head_dim < 128 || head_dim % 128 != 0 || head_dim > BITNET_MAX_K || N % head_dim != 0)
    return BITNET_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(y) || !aligned16(head_w) || !aligned16(out)) return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  int rc = device_context(&ctx);
  if (rc) return rc;
  return cuda_status(launch_head_rmsnorm(y, M * (N / head_dim), static_cast<int>(head_dim), head_w, eps, out, false,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int bitnet_bitlinear_forward_qk(const float* x, const float* norm_w, const uint8_t* packed_w, float w_scale, int64_t M,
                                int64_t K, int64_t N, float eps, int64_t head_dim, const float* head_w, float* y,
                                bitnet_stream_t stream) {
  if (!head_w) return BITNET_ERR_INVALID_ARG;
  if (head_dim < 128 || head_dim % 128 != 0 || head_dim > BITNET_MAX_K || N < 1 || N % head_dim != 0)
    return BITNET_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(head_w)) return BITNET_ERR_MISALIGNED;
  bool fused = false;
  int rc = forward_impl(x, nullptr, 0, norm_w, packed_w, w_scale, M, K, N, eps, y, stream, head_w,
                        static_cast<int>(head_dim), &fused);
  if (rc || fused) return rc;
  // otherwise one more launch, chained to the projection's last: the head norm
  // waits for it on the device
  return cuda_status(launch_head_rmsnorm(y, M * (N / head_dim), static_cast<int>(head_dim), head_w, eps, y, true,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int bitnet_bitlinear_forward_typed(const void* x, int x_dtype, const void* norm_w, int norm_w_dtype,
                                   const uint8_t* packed_w, float w_scale, int64_t M, int64_t K, int64_t N, float eps,
                                   void* y, int y_dtype, bitnet_stream_t stream) {
  return forward_typed(x, x_dtype, norm_w, norm_w_dtype, packed_w, w_scale, M, K, N, eps, y, y_dtype, stream);
}

int bitnet_bitlinear_forward(const float* x, const float* norm_w, const uint8_t* packed_w, float w_scale, int64_t M,
                             int64_t K, int64_t N, float eps, float* y, bitnet_stream_t stream) {
  return forward_impl(x, nullptr, 0, norm_w, packed_w, w_scale, M, K, N, eps, y, stream);
}

int bitnet_bitlinear_forward_glu(const float* gate, const float* up, int act, const float* norm_w,
                                 const uint8_t* packed_w, float w_scale, int64_t M, int64_t K, int64_t N, float eps,
                                 float* y, bitnet_stream_t stream) {
  if (act == 0) return BITNET_ERR_INVALID_ARG;
  return forward_impl(gate, up, act, norm_w, packed_w, w_scale, M, K, N, eps, y, stream);
}

int bitnet_glu(const float* gate, const float* up, int act, int64_t count, float* h, bitnet_stream_t stream) {
  if (!gate || !up || !h || count < 4 || count % 4 != 0) return BITNET_ERR_INVALID_ARG;
  if (act != BITNET_ACT_SILU && act != BITNET_ACT_GELU_TANH) return BITNET_ERR_INVALID_ARG;
  if (!aligned16(gate) || !aligned16(up) || !aligned16(h)) return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  int rc = device_context(&ctx);
  if (rc) return rc;
  return cuda_status(launch_glu(gate, up, act, count, h, reinterpret_cast<cudaStream_t>(stream)));
}

int bitnet_glu_rmsnorm_quant_a8(const float* gate, const float* up, int act, const float* norm_w, int64_t M,
                                int64_t K, float eps, int8_t* a_codes, float* a_scale, int32_t* a_rowsum,
                                float* xn_out, bitnet_stream_t stream) {
  if (!gate || !up || !norm_w || !a_codes || !a_scale) return BITNET_ERR_INVALID_ARG;
  if (act != BITNET_ACT_SILU && act != BITNET_ACT_GELU_TANH) return BITNET_ERR_INVALID_ARG;
  if (!(eps > 0.0f)) return BITNET_ERR_INVALID_ARG;
  int rc = check_shape(M, K, 1);
  if (rc) return rc;
  if (!rmsnorm_quant_glu_fused_supported(static_cast<int>(K))) return BITNET_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(gate) || !aligned16(up) || !aligned16(norm_w) || !aligned16(a_codes) || !aligned4(a_scale) ||
      (a_rowsum && !aligned4(a_rowsum)) || (xn_out && !aligned16(xn_out)))
    return BITNET_ERR_MISALIGNED;
  DeviceContext* ctx;
  if ((rc = device_context(&ctx))) return rc;
  return cuda_status(launch_rmsnorm_quant_glu(gate, up, act, norm_w, M, static_cast<int>(K), eps, a_codes, nullptr,
                                              a_scale, a_rowsum, xn_out, false,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int bitnet_bitlinear_forward_group(const bitnet_projection* projs, int32_t count, int64_t M, float eps,
                                   uint32_t flags, bitnet_stream_t stream) {
  if (!projs || count < 1 || count > BITNET_MAX_GROUP) return BITNET_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || (flags & ~BITNET_FLAG_WEIGHTS_STATIC)) return BITNET_ERR_INVALID_ARG;
  if (M < 1) return BITNET_ERR_INVALID_ARG;
  DecodeJob jobs[BITNET_MAX_GROUP];
  for (int i = 0; i < count; ++i) {
    const bitnet_projection& p = projs[i];
    if (!p.x || !p.norm_w || !p.packed_w || !p.y) return BITNET_ERR_INVALID_ARG;
    if (!(p.w_scale > 0.0f) || p.w_scale == INFINITY) return BITNET_ERR_INVALID_ARG;
    int rc = check_shape(M, p.K, p.N);
    if (rc) return rc;
    if (!aligned16(p.x) || !aligned16(p.norm_w) || !aligned16(p.packed_w) || !aligned16(p.y))
      return BITNET_ERR_MISALIGNED;
    if (!decode_fused_supported(M, p.K)) return BITNET_ERR_UNSUPPORTED_SHAPE;
    DecodeJob j = {};
    j.x = p.x;
    j.g = p.norm_w;
    j.w = p.packed_w;
    j.w_scale = p.w_scale;
    j.K = static_cast<int>(p.K);
    j.N = static_cast<int>(p.N);
    j.y = p.y;
    jobs[i] = j;
  }
  DeviceContext* ctx;
  int rc = device_context(&ctx);
  if (rc) return rc;
  return cuda_status(launch_decode(ctx, jobs, count, static_cast<int>(M), eps, true,
                                   (flags & BITNET_FLAG_WEIGHTS_STATIC) != 0,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace bitnet {
namespace {

// One lane per warp waits on a barrier that nothing ever completes, through the
// same bounded wait as every pipeline of this library; the shared abort flag
// stops the other waiters as soon as the first one gives up.
__global__ void k_bounded_wait_selftest(unsigned* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) mbar_wait(&bar, 0, err, &abort_flag);
  __syncthreads();
}

}  // namespace
}  // namespace bitnet

extern "C" {

int bitnet_selftest_bounded_wait(bitnet_stream_t stream) {
  DeviceContext* ctx;
  int rc = device_context(&ctx);
  if (rc) return rc;
  k_bounded_wait_selftest<<<1, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ctx->err_word);
  return cuda_status(cudaGetLastError());
}

int bitnet_last_device_status(bitnet_stream_t stream) {
  DeviceContext* ctx;
  int rc = device_context(&ctx);
  if (rc) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return BITNET_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, ctx->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return BITNET_ERR_CUDA;
  if (word == 0) return BITNET_OK;
  if (cudaMemset(ctx->err_word, 0, sizeof(unsigned)) != cudaSuccess) return BITNET_ERR_CUDA;
  return BITNET_ERR_TIMEOUT;
}

}  // extern "C"
