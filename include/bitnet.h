/*
 * bitnet.h -- C ABI of the GB300 (sm_103a) W1.58A8 BitLinear library.
 *
 * One BitLinear projection, as the "BitNet Embeddings GGUF Conversion
 * Implementation" page describes it (section 1, "Background"), is
 *
 *     x -> RMSNorm(x, norm.weight) -> 8-bit activation quant -> matmul with
 *          ternary weights -> fp32 output
 *
 * with the per-projection norm weight applied after ggml_rms_norm (section 4.5,
 * "load_tensors", graph code) and eps = 1e-6 (section 1, model table).  The
 * "BitNet Inference Framework" page, "Quantization (W1.58A8)", fixes absmean
 * ternary weights and per-token absmax 8-bit activations; it also states that
 * neither linear nor norm layers carry a bias ("Architectural Details").
 *
 * Weight storage is I2_S ("I2_S Ternary Packing" in section 3 of the first page;
 * "Quantization and Encoding" and "Data Layout" on the second page):
 *   - w_scale = 1 / mean(|w|) over the whole tensor,
 *     q = clamp(round(w * w_scale), -1, 1), code = q + 1 (-1 -> 0, 0 -> 1, +1 -> 2);
 *   - 128 consecutive values of the flattened tensor form a block of 32 bytes;
 *     every byte holds four codes as (c0 << 6) | (c1 << 4) | (c2 << 2) | c3;
 *   - one float32 scale is appended after the last block.
 * The pages leave open which four elements share a byte.  This library fixes it:
 * byte j (0..31) of a block holds the block's elements j, 32+j, 64+j and 96+j as
 * c0, c1, c2 and c3.  A weight matrix W is [N, K] (N outputs, K inputs, K
 * contiguous), so with K % 128 == 0 ("gguf-gemv" page, "Requirements") no block
 * straddles two rows: row n, block kb lives at byte offset 32 * (n*K/128 + kb),
 * and the scale at byte offset N*K/4 (little endian).
 *
 * Readings taken where the pages are silent:
 *   - "round" is round-half-to-even (rint) for weights and activations;
 *   - mean(|w|) is accumulated in double; an all-zero tensor gets w_scale = 1;
 *   - activations: a_scale = 127 / max(max|xn|, 1e-5), q = clamp(rint(xn * a_scale),
 *     -128, 127), both multiplies in fp32 without FMA contraction;
 *   - RMSNorm: rstd = (float)(1 / sqrt(sum(x^2)/K + eps)) with the sum and the
 *     square root in double; xn = (x * rstd) * norm_w, two fp32 multiplies;
 *   - output: y = ((float)acc * (1/a_scale)) * (1/w_scale), fp32, each reciprocal
 *     and product correctly rounded, where acc = sum_k q_x[k] * q_w[k] exactly.
 *
 * Conventions shared by every entry point:
 *   - all tensor pointers are DEVICE pointers to contiguous row-major buffers owned
 *     by the caller; the library never frees or retains them;
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream); every call
 *     is asynchronous on it unless its comment says otherwise;
 *   - the return value is a bitnet_status; argument errors are detected on the
 *     host before anything is launched and leave every output untouched;
 *   - a device-side failure (a bounded wait that expired) is recorded in a
 *     per-device error word that bitnet_last_device_status() reads and clears;
 *     no kernel of this library traps or aborts;
 *   - K must be a positive multiple of 128 and at most BITNET_MAX_K; M and N at
 *     least 1; x, y and packed weights 16-byte aligned.
 *   - temporary device memory (where a call needs it) comes from a stream-ordered
 *     pool that the library owns per device; it is reused across calls and never
 *     returned to the caller.
 */
#ifndef BITNET_GB300_H
#define BITNET_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define BITNET_API __attribute__((visibility("default")))
#else
#define BITNET_API
#endif

#define BITNET_I2S_BLOCK 128       /* values per I2_S block                         */
#define BITNET_I2S_BLOCK_BYTES 32  /* bytes per I2_S block                          */
#define BITNET_GGML_TYPE_I2_S 36   /* GGML type id ("gguf-py: I2_S Type", first page) */
#define BITNET_MAX_K 65536         /* keeps every partial sum below 2^24 (exact in fp32) */
#define BITNET_MAX_GROUP 16        /* projections per bitnet_bitlinear_forward_group  */

/* Flag for bitnet_bitlinear_forward_group: the packed weights and norm weights
 * were written by work that finished before the previous kernel on `stream`
 * began, so the kernel may start streaming them before that kernel has finished
 * (programmatic dependent launch).  Activations are always read, and outputs
 * written, after the previous kernel. */
#define BITNET_FLAG_WEIGHTS_STATIC 1u

typedef enum {
  BITNET_OK = 0,
  BITNET_ERR_INVALID_ARG = 1,       /* null pointer, M/N < 1, eps <= 0, count out of range */
  BITNET_ERR_UNSUPPORTED_SHAPE = 2, /* K not a positive multiple of 128, or K > BITNET_MAX_K */
  BITNET_ERR_MISALIGNED = 3,        /* a pointer that must be 16-byte aligned is not       */
  BITNET_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed                */
  BITNET_ERR_TIMEOUT = 5,           /* a device-side bounded wait expired (see last_device_status) */
  BITNET_ERR_NO_DEVICE = 6,         /* no CUDA device, or it is not sm_103                 */
  BITNET_ERR_SCRATCH_LIMIT = 7      /* too large for bitnet_bitlinear_forward_noalloc      */
} bitnet_status;

typedef struct CUstream_st* bitnet_stream_t; /* == cudaStream_t */

/* Bytes of an I2_S buffer for an [N, K] matrix: N*K/4 code bytes plus the 4-byte
 * scale.  Returns 0 for an invalid shape (N < 1, K not a positive multiple of 128). */
BITNET_API size_t bitnet_i2s_packed_bytes(int64_t N, int64_t K);

/* Absmean ternary quantisation and I2_S packing of w[N, K] (fp32) into
 * packed[bitnet_i2s_packed_bytes(N, K)] ("I2_S Ternary Packing", first page
 * section 3; "Quantization and Encoding" / "Data Layout", second page).
 * The scale is written to the buffer's last 4 bytes; if w_scale_out (a HOST
 * pointer) is non-NULL the call synchronises `stream` and stores it there too.
 * mean(|w|) is reduced in double in a fixed order, so repeated calls give
 * identical bytes.  packed must be 16-byte aligned. */
BITNET_API int bitnet_pack_i2s(const float* w, int64_t N, int64_t K, uint8_t* packed,
                    float* w_scale_out, bitnet_stream_t stream);

/* Decode an I2_S buffer into ternary int8 values w_ternary[N, K] = code - 1.
 * A (malformed) code 3 decodes to +2, the same value every kernel here uses. */
BITNET_API int bitnet_unpack_i2s(const uint8_t* packed, int64_t N, int64_t K, int8_t* w_ternary,
                      bitnet_stream_t stream);

/* RMSNorm with the projection's norm weight followed by per-token absmax int8
 * quantisation ("Background" and "load_tensors" on the first page; "Quantization
 * (W1.58A8)" on the second).  x[M, K] fp32, norm_w[K] fp32 ->
 *   a_codes[M, K] int8, a_scale[M] fp32 (= 127 / max(max|xn|, 1e-5)),
 *   a_rowsum[M] int32 (sum of the row's codes; may be NULL),
 *   xn_out[M, K] fp32 (the normalised row before quantisation; may be NULL).
 * eps > 0 (the pages' models use 1e-6). */
BITNET_API int bitnet_rmsnorm_quant_a8(const float* x, const float* norm_w, int64_t M, int64_t K,
                            float eps, int8_t* a_codes, float* a_scale, int32_t* a_rowsum,
                            float* xn_out, bitnet_stream_t stream);

/* I2_S x int8 contraction and fp32 rescale (the int8 x ternary dot products of
 * ggml_vec_dot_i2_i8_s named in section 6.4 of the first page, plus the two
 * scales): for every m < M, n < N
 *   acc[m, n] = sum_k a_codes[m, k] * (code(n, k) - 1)          (exact integer)
 *   y[m, n]   = ((float)acc * (1 / a_scale[m])) * (1 / w_scale)
 * a_codes[M, K] int8, a_scale[M] fp32, packed_w in I2_S layout (its trailing
 * scale is ignored: w_scale is the argument), y[M, N] fp32; acc_out[M, N] int32
 * receives acc when non-NULL.  M <= 8 runs a dp4a weight-streaming kernel,
 * larger M the tcgen05 tensor-core kernel (pool memory: 2*M*K bytes). */
BITNET_API int bitnet_i2s_gemm(const int8_t* a_codes, const float* a_scale, const uint8_t* packed_w,
                    float w_scale, int64_t M, int64_t K, int64_t N, float* y,
                    int32_t* acc_out, bitnet_stream_t stream);

/* The whole projection: y[M, N] = BitLinear(x[M, K]) with norm weight norm_w[K],
 * weights packed_w (I2_S, [N, K]) and their scale w_scale.  Bit-for-bit the
 * composition of bitnet_rmsnorm_quant_a8 and bitnet_i2s_gemm.  Small M runs
 * one fused launch; larger M a norm/quant launch (pool memory: 2*M*K + 4*M
 * bytes) followed by the tensor-core launch. */
BITNET_API int bitnet_bitlinear_forward(const float* x, const float* norm_w, const uint8_t* packed_w,
                             float w_scale, int64_t M, int64_t K, int64_t N, float eps,
                             float* y, bitnet_stream_t stream);

/* One projection of a group (all pointers device pointers, as above). */
typedef struct {
  const float* x;          /* [M, K] fp32 */
  const float* norm_w;     /* [K] fp32 */
  const uint8_t* packed_w; /* I2_S [N, K] */
  float w_scale;           /* the weights' I2_S scale */
  int64_t K;
  int64_t N;
  float* y;                /* [M, N] fp32 */
} bitnet_projection;

/* Several independent projections with the same token count M in ONE launch
 * (e.g. the seven projections of a layer at decode, each with its own input
 * and norm weight).  Each output equals bitnet_bitlinear_forward of that
 * projection, bit for bit.  `projs` is a HOST array of `count` descriptors
 * (1..BITNET_MAX_GROUP), read before the call returns.  Supported for
 * M <= 8 with, for every projection, either 5*M*K + 4*K <= 147456
 * (activations, codes and norm weight staged in shared memory) or K a multiple
 * of 2048 in [4096, 16384] with M*K <= 65536 (activations and norm weight held
 * in registers, codes in shared memory); other shapes return
 * BITNET_ERR_UNSUPPORTED_SHAPE.
 * flags: 0 or BITNET_FLAG_WEIGHTS_STATIC. */
BITNET_API int bitnet_bitlinear_forward_group(const bitnet_projection* projs, int32_t count, int64_t M,
                                   float eps, uint32_t flags, bitnet_stream_t stream);

/* Size of the fixed device array bitnet_bitlinear_forward_noalloc works in. */
#define BITNET_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB per GPU */

/* bitnet_bitlinear_forward without any device-memory allocation.  The pages have
 * no counterpart: this exists for callers that may not allocate once running --
 * e.g. a server that reserved all device memory for its own allocator at start-up,
 * or a latency-critical loop where an allocation's cost or failure is not
 * acceptable.  Same arguments and the same y as bitnet_bitlinear_forward.
 *   - Temporary data lives in one fixed 16 MiB device array that every GPU
 *     using the library keeps until the process exits: the activation codes
 *     (int8 for M <= 8, fp16 otherwise: M*K or 2*M*K bytes) and per-token
 *     scales (4*M bytes), each rounded up to 256 bytes, then the fp32 partial
 *     sums of a K split (up to 4*M*N bytes plus 4 bytes per output tile) where
 *     the contraction splits K, and for 9..63 tokens the sums of the codes per
 *     2048-value chunk (4*M*ceil(K/2048) bytes; the fp16 codes are rewritten
 *     in place there as the contraction's 8-bit operand).  Problems whose
 *     codes and scales do not fit
 *     return BITNET_ERR_SCRATCH_LIMIT without launching anything.  When the
 *     codes and scales fit but the partial sums do not, the contraction runs
 *     without the K split (the same y; a slower plan than
 *     bitnet_bitlinear_forward's for those shapes).  Only M <= 8 with the fused
 *     norm prologue (bitnet_bitlinear_forward_group's shapes, except K > 16384
 *     with K a multiple of 2048, which take a separate norm launch) leave the
 *     array untouched.
 *   - The first call on each device, whatever its shape, does the one-time
 *     set-up: device properties, and loading the array onto the device to look
 *     up its address.  Make that first call before reserving the rest of device
 *     memory for other use and before any stream capture.
 *   - All calls on a device share the one array, and it keeps whatever the last
 *     call left (every byte a call reads it first writes, and partial sums are
 *     zeroed on the stream before use).  Calls whose work can overlap on the
 *     GPU -- different streams without ordering between them, or several host
 *     threads -- race on it and must be serialised by the caller. */
BITNET_API int bitnet_bitlinear_forward_noalloc(const float* x, const float* norm_w,
                                                const uint8_t* packed_w, float w_scale, int64_t M,
                                                int64_t K, int64_t N, float eps, float* y,
                                                bitnet_stream_t stream);

/* Activations of the down projection's input (the gate projection's activation;
 * "BitNet Embeddings GGUF Conversion Implementation", section 1's table). */
#define BITNET_ACT_SILU 1      /* x / (1 + e^-x)                                  (Qwen3)  */
#define BITNET_ACT_GELU_TANH 2 /* x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))   (Gemma3) */

/* The down projection's input ("BitNet Embeddings GGUF Conversion
 * Implementation", section 4.5, "FFN per-projection norms": the gate
 * projection's output through the activation, times the up projection's):
 *   h[i] = act(gate[i]) * up[i]   for i < count
 * in float, both activations as x * (1 / (1 + e^-t)) with t = x (SiLU) or
 * t = 2 sqrt(2/pi) (x + 0.044715 x^3) (tanh GELU: (1 + tanh z) / 2 = 1 / (1 + e^-2z)),
 * CUDA's expf and a correctly rounded reciprocal, every operation rounded on its
 * own -- the arithmetic every fused path below uses, so they all see the same h.
 * gate, up, h: device pointers, 16-byte aligned, count a positive multiple of 4;
 * h may alias gate or up (elementwise).  act: BITNET_ACT_SILU or
 * BITNET_ACT_GELU_TANH, else BITNET_ERR_INVALID_ARG. */
BITNET_API int bitnet_glu(const float* gate, const float* up, int act, int64_t count, float* h,
                          bitnet_stream_t stream);

/* bitnet_rmsnorm_quant_a8 of the rows h = act(gate) * up (gate, up [M, K] fp32)
 * without writing h: bit for bit bitnet_rmsnorm_quant_a8 applied to the output
 * of bitnet_glu.  The rows are held in registers: K <= 3072, else
 * BITNET_ERR_UNSUPPORTED_SHAPE.  Other arguments as bitnet_rmsnorm_quant_a8. */
BITNET_API int bitnet_glu_rmsnorm_quant_a8(const float* gate, const float* up, int act, const float* norm_w,
                                           int64_t M, int64_t K, float eps, int8_t* a_codes, float* a_scale,
                                           int32_t* a_rowsum, float* xn_out, bitnet_stream_t stream);

/* The down projection y[M, N] = BitLinear(act(gate) * up): bit for bit
 * bitnet_bitlinear_forward applied to the output of bitnet_glu, without writing
 * h where it can be avoided -- one fused launch for M <= 8 when the rows fit
 * registers (M = 1 with K <= 3840, or K a multiple of 2048 in [4096, 16384]
 * with M*K <= 65536); otherwise the norm launch computes h as it loads the rows
 * (K <= 3072) or h goes through pool memory first (4*M*K bytes more).  gate
 * and up are [M, K] fp32, 16-byte aligned; the other arguments as
 * bitnet_bitlinear_forward.  act must be BITNET_ACT_SILU or
 * BITNET_ACT_GELU_TANH. */
BITNET_API int bitnet_bitlinear_forward_glu(const float* gate, const float* up, int act, const float* norm_w,
                                            const uint8_t* packed_w, float w_scale, int64_t M, int64_t K,
                                            int64_t N, float eps, float* y, bitnet_stream_t stream);

/* Element types of bitnet_bitlinear_forward_typed. */
#define BITNET_DTYPE_F32 0
#define BITNET_DTYPE_F16 1  /* IEEE binary16                                       */
#define BITNET_DTYPE_BF16 2 /* bfloat16: the upper 16 bits of an fp32              */

/* The projection of bitnet_bitlinear_forward with 16-bit input and output
 * tensors: x[M, K] in x_dtype (F32, F16 or BF16; "gguf-gemv", "Requirements":
 * f32 or bf16 activations, the output in the input's type), norm_w[K] in
 * norm_w_dtype (F32 or F16: the conversion stores norm weights as float16,
 * "BitNet Embeddings GGUF Conversion Implementation", section 6.1) and y[M, N]
 * in y_dtype (F32, F16 or BF16).
 * Every input value is widened to fp32 (exact), the projection is computed as
 * bitnet_bitlinear_forward computes it on the widened values, and y is that
 * fp32 result rounded once to y_dtype (to nearest, ties to even; fp16 results
 * beyond 65504 become infinities).  So y equals bitnet_bitlinear_forward of
 * the widened inputs, rounded.
 * Layout, alignment (16 bytes), ownership and pool memory as for
 * bitnet_bitlinear_forward.  From 9 tokens on, the norm launch reads 16-bit x
 * itself and the tensor-core launch of 64 or more tokens writes 16-bit y
 * itself; otherwise x and y pass through fp32 copies in pool memory
 * (M * K * 4 and M * N * 4 bytes), converted by extra launches, as does an
 * fp16 norm weight (K * 4 bytes).
 * Errors: BITNET_ERR_INVALID_ARG for an unknown dtype or BF16 norm weights,
 * otherwise as bitnet_bitlinear_forward. */
BITNET_API int bitnet_bitlinear_forward_typed(const void* x, int x_dtype, const void* norm_w, int norm_w_dtype,
                                              const uint8_t* packed_w, float w_scale, int64_t M, int64_t K,
                                              int64_t N, float eps, void* y, int y_dtype, bitnet_stream_t stream);

/* QK head norm of a projection's output ("BitNet Embeddings GGUF Conversion
 * Implementation", section 4.5, "Attention per-projection norms": after the q
 * and k matmuls, an RMSNorm with the attention eps times attn_q_norm /
 * attn_k_norm, the "QK head norms" of the model table).  Read per head: y[M, N]
 * holds N / head_dim heads of head_dim consecutive values per token, and for
 * every (token, head) row r of head_dim values
 *   out[r] = (r * rstd) * head_w,  rstd = 1 / sqrt(sum(r^2) / head_dim + eps),
 * with the same arithmetic as the input norm of bitnet_rmsnorm_quant_a8 (rstd
 * the float rounding of the exact value, two float multiplies).
 * head_w[head_dim] fp32; out may be y (in place).  head_dim a multiple of 128
 * (Qwen3 128, Gemma3 256) dividing N.  Errors: BITNET_ERR_INVALID_ARG (NULL,
 * M or N < 1, eps <= 0), BITNET_ERR_UNSUPPORTED_SHAPE, BITNET_ERR_MISALIGNED
 * (16 bytes), BITNET_ERR_CUDA. */
BITNET_API int bitnet_head_rmsnorm(const float* y, int64_t M, int64_t N, int64_t head_dim, const float* head_w,
                                   float eps, float* out, bitnet_stream_t stream);

/* The q or k projection followed by its head norm: y = head_rmsnorm(
 * bitnet_bitlinear_forward(x, ...)), eps used by both norms, bit for bit.  On
 * the tensor-core route (64 tokens and more) the head norm runs in the
 * contraction's epilogue when a weight tile holds whole heads and K is not
 * split; otherwise one more launch, chained to the projection's, normalises y
 * in place.  Arguments and errors as bitnet_bitlinear_forward and
 * bitnet_head_rmsnorm. */
BITNET_API int bitnet_bitlinear_forward_qk(const float* x, const float* norm_w, const uint8_t* packed_w, float w_scale,
                                           int64_t M, int64_t K, int64_t N, float eps, int64_t head_dim,
                                           const float* head_w, float* y, bitnet_stream_t stream);

/* Static description of a status code (never NULL). */
BITNET_API const char* bitnet_status_string(int status);

/* Synchronises `stream`, then returns BITNET_ERR_TIMEOUT if a kernel of this
 * library on the current device gave up a bounded wait since the last call
 * (and clears that record), BITNET_ERR_CUDA if the synchronisation failed, and
 * BITNET_OK otherwise. */
BITNET_API int bitnet_last_device_status(bitnet_stream_t stream);

/* Diagnostic, with no counterpart in the method: launches one small kernel on
 * `stream` whose waits target a barrier that nothing ever completes, through
 * the bounded wait every pipeline of this library uses.  The waits give up
 * after their time limit (about one second), record the failure in the error
 * word and return; the kernel exits normally and the context stays usable.
 * A following bitnet_last_device_status(stream) returns BITNET_ERR_TIMEOUT.
 * Returns BITNET_OK if the launch succeeded, BITNET_ERR_NO_DEVICE without a
 * GB300, BITNET_ERR_CUDA on a launch failure. */
BITNET_API int bitnet_selftest_bounded_wait(bitnet_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BITNET_GB300_H */
