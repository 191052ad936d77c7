// internal.h -- host-side interfaces between the translation units of the
// library (launchers, per-device context).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bitnet.h"

namespace bitnet {

struct DeviceContext {
  int device = -1;
  int num_sms = 0;
  unsigned* err_word = nullptr;  // device address of this device's error word
  cudaMemPool_t pool = nullptr;  // stream-ordered pool for temporary buffers
};

// Returns BITNET_OK and fills *ctx for the current device (lazily initialised,
// thread safe), or BITNET_ERR_NO_DEVICE / BITNET_ERR_CUDA.
int device_context(DeviceContext** ctx);

// Same as device_context but never creates the memory pool (ctx->pool stays
// null): for entry points that must not allocate.
int device_context_nopool(DeviceContext** ctx);

// Temporary device memory ordered on `stream` (freed with pool_free on the
// same stream after its last use has been enqueued).
int pool_alloc(DeviceContext* ctx, void** p, size_t bytes, cudaStream_t stream);
void pool_free(void* p, cudaStream_t stream);

// cuTensorMapEncodeTiled fetched through the runtime (no link to libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// ---------------------------------------------------------------- launchers
// All launchers return cudaError_t of the launch (cudaSuccess when fine).

// I2_S packing: absmean (two deterministic reduction launches) + pack.
cudaError_t launch_pack_i2s(const DeviceContext* ctx, const float* w, int64_t N, int64_t K, uint8_t* packed,
                            double* partials, int num_partials, cudaStream_t s);
int pack_num_partials(int64_t count);
cudaError_t launch_unpack_i2s(const uint8_t* packed, int64_t N, int64_t K, int8_t* out, cudaStream_t s);

// RMSNorm + absmax int8 quantisation, one warp per row.  Exactly one of
// codes_i8 / codes_f16 is non-null.
// CTAs of the norm + quant launch for M rows of K.
int64_t rmsnorm_quant_ctas(int64_t M, int K);
cudaError_t launch_rmsnorm_quant(const float* x, const float* g, int64_t M, int K, float eps, int8_t* codes_i8,
                                 __half* codes_f16, float* a_scale, int32_t* rowsum, float* xn_out,
                                 bool pdl, cudaStream_t s);
// The same norm/quant to fp16 codes with x in x_dtype (BITNET_DTYPE_F32, _F16
// or _BF16), widened to fp32 as it is loaded.
cudaError_t launch_rmsnorm_quant_f16_in(const void* x, int x_dtype, const float* g, int64_t M, int K, float eps,
                                        __half* codes_f16, float* a_scale, bool pdl, cudaStream_t s);
// Head norm of projection outputs: rows of hd values (a multiple of 128),
// out = (y * rstd(row)) * w, the input norm's row arithmetic; out may be y.
cudaError_t launch_head_rmsnorm(const float* y, int64_t rows, int hd, const float* w, float eps, float* out, bool pdl,
                                cudaStream_t s);
// Element-wise conversion of `count` values between BITNET_DTYPE_* types:
// widening is exact, narrowing rounds to nearest, ties to even.
cudaError_t launch_convert(const void* in, int in_dtype, void* out, int out_dtype, int64_t count, cudaStream_t s);

// The down projection's input h = act(gate) * up (act 1: SiLU, 2: tanh GELU):
// fused into the norm launch for K <= 3072, or elementwise into h (count a
// multiple of 4).
bool rmsnorm_quant_glu_fused_supported(int K);
cudaError_t launch_rmsnorm_quant_glu(const float* gate, const float* up, int act, const float* g, int64_t M, int K,
                                     float eps, int8_t* codes_i8, __half* codes_f16, float* a_scale, int32_t* rowsum,
                                     float* xn_out, bool pdl, cudaStream_t s);
cudaError_t launch_glu(const float* gate, const float* up, int act, int64_t count, float* h, cudaStream_t s);

// The norm/quant writing the codes as the 9..63-token contraction's two e4m3
// planes (planes.cuh; `planes` 256-byte aligned, 2*M*K bytes) and their row
// sums (rowsum[M], required): x in x_dtype, or the down projection's
// act(gate) * up for K <= 3072.
cudaError_t launch_rmsnorm_quant_planes(const void* x, int x_dtype, const float* g, int64_t M, int K, float eps,
                                       void* planes, float* a_scale, int32_t* rowsum, bool pdl, cudaStream_t s);
cudaError_t launch_rmsnorm_quant_glu_planes(const float* gate, const float* up, int act, const float* g, int64_t M,
                                           int K, float eps, void* planes, float* a_scale, int32_t* rowsum, bool pdl,
                                           cudaStream_t s);

// int8 codes -> fp16 codes (for the tensor-core path of the int8 API).
cudaError_t launch_codes_to_f16(const int8_t* codes, __half* out, int64_t count, cudaStream_t s);

// Decode (small M) weight-streaming kernels.
constexpr int kDecodeMaxM = 8;
constexpr int64_t kDecodeMaxCodeBytes = 65536;  // M * K bytes of codes held in shared memory
// fused launch: x (4 B) and codes (1 B) per element plus the norm weight (4 B
// per feature) staged in shared memory next to the 72 KB weight ring
constexpr int64_t kDecodeFusedMaxStageBytes = 144 * 1024;

struct DecodeJob {
  const float* x;          // fused: activations [M, K] (act != 0: the gate projection's output)
  const float* up;         // fused, act != 0: the up projection's output [M, K]
  int act;                 // 0, or the activation of the down-projection input act(x) * up
  const float* g;          // fused: norm weight [K]
  const int8_t* codes;     // unfused: int8 codes [M, K]
  const float* a_scale;    // unfused: activation scales [M]
  const uint8_t* w;        // I2_S codes [N, K/4]
  float w_scale;
  int K;
  int N;
  float* y;                // [M, N]
  int32_t* acc_out;        // [M, N] or null
};
bool decode_supported(int64_t M, int64_t K);        // codes given (int8 in global memory)
bool decode_fused_supported(int64_t M, int64_t K);  // norm + quant in the same launch
bool decode_fused_glu_supported(int64_t M, int64_t K);  // the same, with the down-projection input
// Few tokens with long rows (K >= 8192, a multiple of 2048): a separate norm
// kernel with one CTA per row, then the decode kernel streaming weights
// during it, beats every CTA normalising the whole row in its prologue.
bool decode_split_preferred(int64_t M, int64_t K);
// One token, K = 4096, 8192 or 16384, fused norm + quant: the row kernel
// (activation codes in registers, 32 KB weight stages); launch_decode sends
// such single-projection launches there.
bool gemv_row1_supported(int64_t M, int64_t K);
cudaError_t launch_gemv_row1(const DeviceContext* ctx, const DecodeJob& job, float eps, bool weights_static,
                             cudaStream_t s);
// reserve_sms: SMs left to the kernel this launch follows (its CTAs still
// running when the decode CTAs start), so that every decode CTA is resident at
// once.
cudaError_t launch_decode(const DeviceContext* ctx, const DecodeJob* jobs, int njobs, int M, float eps, bool fused,
                          bool weights_static, cudaStream_t s, int reserve_sms = 0);

// Tensor-core (tcgen05) contraction on fp16 codes, tokens as the MMA's M side.
// When its output tiles would leave SMs idle it splits K: it then needs
// gemm_tc_workspace() bytes of device memory, zero on entry (zeroed here on the
// stream unless workspace_zeroed); with a null workspace it does not split.
size_t gemm_tc_workspace(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N);
// y is y_dtype (BITNET_DTYPE_F32, _F16 or _BF16): the fp32 result rounded once.
// With head_w / head_dim / head_fused given, the QK head norm is applied in the
// epilogue when the plan allows it (*head_fused says whether it was).
cudaError_t launch_gemm_tc(const DeviceContext* ctx, const __half* codes_f16, const float* a_scale,
                           const uint8_t* packed_w, float w_scale, int64_t M, int64_t K, int64_t N, void* y,
                           int y_dtype, int32_t* acc_out, void* workspace, bool workspace_zeroed, bool pdl,
                           cudaStream_t s, int* status, const float* head_w = nullptr, int head_dim = 0,
                           float eps = 0.0f, bool* head_fused = nullptr);

// Tensor-core contraction for 9..63 tokens (8-bit operands, weights as the
// MMA's M side, K split across CTAs where that pays).  `codes` holds either the
// fp16 codes (scratch of the caller; rowsum null), rewritten in place here as
// the operand's two e4m3 planes, or the planes already (launch_rmsnorm_quant_
// planes) with their row sums in rowsum.  Needs gemm_skinny_workspace() bytes
// of device memory, of which the first gemm_skinny_zeroed_bytes() (0 when K
// is not split) must be zero on entry: zeroed here on the stream unless
// workspace_zeroed.
bool gemm_skinny_supported(int64_t M, int64_t K, int64_t N);
size_t gemm_skinny_workspace(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N);
size_t gemm_skinny_zeroed_bytes(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N);
// M ints inside that workspace (not zeroed) where a norm launch that writes
// the planes may put their row sums.
int32_t* gemm_skinny_rowsum_area(const DeviceContext* ctx, void* workspace, int64_t M, int64_t K, int64_t N);
cudaError_t launch_gemm_skinny(const DeviceContext* ctx, void* codes, const int32_t* rowsum, const float* a_scale,
                               const uint8_t* packed_w, float w_scale, int64_t M, int64_t K, int64_t N, float* y,
                               int32_t* acc_out, void* workspace, bool workspace_zeroed, bool pdl, cudaStream_t s,
                               int* status);

}  // namespace bitnet
