// gemv.cu -- small-M (decode) BitLinear: the I2_S weight stream is the whole cost.
//
// The contraction is the int8 x ternary dot product of ggml_vec_dot_i2_i8_s
// ("BitNet Embeddings GGUF Conversion Implementation", section 6.4); the
// "gguf-gemv" page ("Performance") notes that decode at M=1 is bound by the
// packed-block byte stream, and the "BitNet Inference Kernel" page (gpu/README,
// "dp4a Instruction") uses dp4a for the same 2-bit x 8-bit products.
//
// Design (sm_103a):
//  * one CTA owns a contiguous range of weight rows of one projection; a
//    producer warp streams that range through a ring of shared-memory stages
//    with 1-D bulk async copies (cp.async.bulk + mbarrier transaction counts),
//    so tens of KB per SM are in flight without per-thread loads;
//  * the activation codes of all M tokens sit in shared memory: either
//    computed in the prologue (RMSNorm + absmax quant, the shared rowquant.cuh
//    arithmetic) or copied from a codes buffer;
//  * decoding needs no shifts: with byte j holding elements j, 32+j, 64+j, 96+j
//    as 2-bit fields, (word & (0xC0C0C0C0 >> 2s)) is 4 codes of slot s, each
//    times 4^(3-s), next to 4 consecutive activation codes of that slot;
//    dp4a.u32.s32 accumulates them per slot, and the slot sums are shifted
//    back at the end (exact: every term is a multiple of 4^(3-s)).  The codes
//    are c = q + 1, so sum(c * x) - sum(x) = sum(q * x) (acc - rowsum);
//  * several projections can share one launch (descriptor table, CTAs
//    apportioned by weight bytes): one launch per decoder layer.
//  * With weights declared static, the producer starts streaming before the
//    programmatic-dependent-launch wait, overlapping the previous kernel's tail.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

namespace bitnet {
namespace {

constexpr int kDecWarps = 8;                       // compute warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one producer warp
constexpr int kDecStageBytes = 16384;
constexpr int kDecStages = 6;

struct DecodeProj {
  const float* x;
  const float* g;
  const int8_t* codes;
  const float* a_scale;
  const uint8_t* w;
  float inv_w;
  int K;
  int N;
  float* y;
  int32_t* acc_out;
  int cta_begin;
  int rows_per_cta;
};

struct DecodeParams {
  DecodeProj p[BITNET_MAX_GROUP];
  int nproj;
  int M;
  float eps;
  int weights_static;
};

struct DecodeSmemTail {
  uint64_t full[kDecStages];
  uint64_t empty[kDecStages];
  float rstd[kDecodeMaxM];
  float amax_part[kDecWarps][kDecodeMaxM];
  int rs_part[kDecWarps][kDecodeMaxM];
  float inv_a[kDecodeMaxM];
  int rowsum[kDecodeMaxM];
  int abort_flag;
};

__device__ __forceinline__ void compute_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
}

template <int MT, bool kFused>
__global__ void __launch_bounds__(kDecThreads) k_decode(const __grid_constant__ DecodeParams P, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  int8_t* xq = reinterpret_cast<int8_t*>(smem + kDecStages * kDecStageBytes);

  // which projection this CTA serves
  int pi = 0;
#pragma unroll 1
  for (int i = 1; i < P.nproj; ++i)
    if (static_cast<int>(blockIdx.x) >= P.p[i].cta_begin) pi = i;
  const DecodeProj& pr = P.p[pi];
  const int K = pr.K;
  const int N = pr.N;
  const int row_bytes = K >> 2;
  const int r0 = (static_cast<int>(blockIdx.x) - pr.cta_begin) * pr.rows_per_cta;
  const int r1 = min(N, r0 + pr.rows_per_cta);
  const int rps = kDecStageBytes / row_bytes;  // rows per stage (K <= 65536 keeps it >= 1)
  const int nst = (r1 - r0 + rps - 1) / rps;

  DecodeSmemTail* tail =
      reinterpret_cast<DecodeSmemTail*>(smem + kDecStages * kDecStageBytes + ((MT * K + 127) & ~127));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], kDecWarps);
    }
    tail->abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kDecWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      if (!P.weights_static) pdl_wait();
      const uint8_t* src = pr.w + static_cast<int64_t>(r0) * row_bytes;
      int issued = 0;
      for (int st = 0; st < nst; ++st) {
        const int s = st % kDecStages;
        if (st >= kDecStages &&
            !mbar_wait(&tail->empty[s], ((st / kDecStages) - 1) & 1, err, &tail->abort_flag))
          break;
        const int rows = min(rps, r1 - r0 - st * rps);
        const unsigned bytes = static_cast<unsigned>(rows * row_bytes);
        mbar_arrive_expect_tx(&tail->full[s], bytes);
        bulk_load(ring + s * kDecStageBytes, src + static_cast<int64_t>(st) * rps * row_bytes, bytes,
                  &tail->full[s]);
        issued = st + 1;
      }
      // leave no copy in flight when the CTA retires
      for (int st = max(0, issued - kDecStages); st < issued; ++st)
        mbar_wait(&tail->full[st % kDecStages], (st / kDecStages) & 1, err, nullptr);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  pdl_wait();
  const int tid = threadIdx.x;  // 0 .. kDecWarps*32-1
  const int M = P.M;
  if (kFused) {
    // sum of squares: one warp per token row (the shared canonical reduction)
    if (warp < M) {
      const double ss = warp_row_sumsq(pr.x + static_cast<int64_t>(warp) * K, K, lane);
      if (lane == 0) tail->rstd[warp] = rstd_from_sumsq(ss, K, P.eps);
    }
    compute_bar();
    // absmax of the normalised rows
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < M) {
        const float* xr = pr.x + static_cast<int64_t>(m) * K;
        const float rstd = tail->rstd[m];
        float amax = 0.0f;
        for (int k = 4 * tid; k < K; k += 4 * kDecWarps * 32) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
          const float4 gv = __ldg(reinterpret_cast<const float4*>(pr.g + k));
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(norm_elem(v.x, rstd, gv.x)), fabsf(norm_elem(v.y, rstd, gv.y))),
                                   fmaxf(fabsf(norm_elem(v.z, rstd, gv.z)), fabsf(norm_elem(v.w, rstd, gv.w)))));
        }
        amax = warp_max(amax);
        if (lane == 0) tail->amax_part[warp][m] = amax;
      }
    }
    compute_bar();
    // quantise into shared memory
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < M) {
        float amax = 0.0f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) amax = fmaxf(amax, tail->amax_part[w][m]);
        const float as = act_scale_from_amax(amax);
        const float* xr = pr.x + static_cast<int64_t>(m) * K;
        const float rstd = tail->rstd[m];
        int rs = 0;
        for (int k = 4 * tid; k < K; k += 4 * kDecWarps * 32) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(xr + k));
          const float4 gv = __ldg(reinterpret_cast<const float4*>(pr.g + k));
          const int q0 = quant_elem(norm_elem(v.x, rstd, gv.x), as);
          const int q1 = quant_elem(norm_elem(v.y, rstd, gv.y), as);
          const int q2 = quant_elem(norm_elem(v.z, rstd, gv.z), as);
          const int q3 = quant_elem(norm_elem(v.w, rstd, gv.w), as);
          rs += q0 + q1 + q2 + q3;
          *reinterpret_cast<uint32_t*>(xq + m * K + k) =
              (static_cast<uint32_t>(q0) & 0xFFu) | ((static_cast<uint32_t>(q1) & 0xFFu) << 8) |
              ((static_cast<uint32_t>(q2) & 0xFFu) << 16) | ((static_cast<uint32_t>(q3) & 0xFFu) << 24);
        }
        rs = warp_sum_int(rs);
        if (lane == 0) tail->rs_part[warp][m] = rs;
        if (tid == 0) tail->inv_a[m] = __fdiv_rn(1.0f, as);
      }
    }
  } else {
    // codes computed elsewhere: copy them in and sum them
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < M) {
        const int8_t* src = pr.codes + static_cast<int64_t>(m) * K;
        int rs = 0;
        for (int k = 16 * tid; k < K; k += 16 * kDecWarps * 32) {
          const int4 v = __ldg(reinterpret_cast<const int4*>(src + k));
          *reinterpret_cast<int4*>(xq + m * K + k) = v;
          const int vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) rs = __dp4a(vv[e], 0x01010101, rs);
        }
        rs = warp_sum_int(rs);
        if (lane == 0) tail->rs_part[warp][m] = rs;
        if (tid == 0) tail->inv_a[m] = __fdiv_rn(1.0f, __ldg(pr.a_scale + m));
      }
    }
  }
  compute_bar();
  if (tid < M) {
    int rs = 0;
    for (int w = 0; w < kDecWarps; ++w) rs += tail->rs_part[w][tid];
    tail->rowsum[tid] = rs;
  }
  compute_bar();

  // ------------------------------------------------------------ main loop
  const int cpr = K >> 6;  // 16-byte chunks per row
  int lpr = 32;            // lanes per row: largest power of two <= 32 dividing cpr
  while (cpr % lpr) lpr >>= 1;
  const int rpp = 32 / lpr;  // rows per warp pass
  const int sub = lane & (lpr - 1);
  int rowsum[MT];
  float inv_a[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    rowsum[m] = m < M ? tail->rowsum[m] : 0;
    inv_a[m] = m < M ? tail->inv_a[m] : 0.0f;
  }
  const float inv_w = pr.inv_w;

  for (int st = 0; st < nst; ++st) {
    const int s = st % kDecStages;
    if (!mbar_wait(&tail->full[s], (st / kDecStages) & 1, err, &tail->abort_flag)) break;
    const uint8_t* stage = ring + s * kDecStageBytes;
    const int rows = min(rps, r1 - r0 - st * rps);
    for (int base = warp * rpp; base < rows; base += kDecWarps * rpp) {
      const int r = base + lane / lpr;
      const bool valid = r < rows;
      int acc[MT][4];
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[m][q] = 0;
      if (valid) {
        const uint8_t* wrow = stage + r * row_bytes;
        for (int c = sub; c < cpr; c += lpr) {
          const uint4 wv = *reinterpret_cast<const uint4*>(wrow + c * 16);
          const unsigned wd[4] = {wv.x, wv.y, wv.z, wv.w};
          const int8_t* xb = xq + (c >> 1) * 128 + 16 * (c & 1);
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            const unsigned mask = 0xC0C0C0C0u >> (2 * sl);
            const unsigned m0 = wd[0] & mask, m1 = wd[1] & mask, m2 = wd[2] & mask, m3 = wd[3] & mask;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              if (m < M) {
                const int4 xv = *reinterpret_cast<const int4*>(xb + m * K + 32 * sl);
                int a = acc[m][sl];
                a = dp4a_us(m0, xv.x, a);
                a = dp4a_us(m1, xv.y, a);
                a = dp4a_us(m2, xv.z, a);
                a = dp4a_us(m3, xv.w, a);
                acc[m][sl] = a;
              }
            }
          }
        }
      }
      const int n = r0 + st * rps + r;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        int t = (acc[m][0] >> 6) + (acc[m][1] >> 4) + (acc[m][2] >> 2) + acc[m][3];
        for (int off = lpr >> 1; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (valid && sub == 0 && m < M) {
          const int a = t - rowsum[m];
          pr.y[static_cast<int64_t>(m) * N + n] = rescale_elem(__int2float_rn(a), inv_a[m], inv_w);
          if (pr.acc_out) pr.acc_out[static_cast<int64_t>(m) * N + n] = a;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);
  }
}

size_t decode_smem_bytes(int M, int K) {
  return static_cast<size_t>(kDecStages) * kDecStageBytes + ((static_cast<size_t>(M) * K + 127) & ~size_t(127)) +
         sizeof(DecodeSmemTail);
}

template <int MT, bool kFused>
cudaError_t launch_decode_t(const DecodeParams& P, int grid, size_t smem, bool pdl, unsigned* err, cudaStream_t s) {
  auto kern = k_decode<MT, kFused>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P, err);
}

template <bool kFused>
cudaError_t dispatch_m(int M, const DecodeParams& P, int grid, size_t smem, bool pdl, unsigned* err,
                       cudaStream_t s) {
  switch (M) {
    case 1: return launch_decode_t<1, kFused>(P, grid, smem, pdl, err, s);
    case 2: return launch_decode_t<2, kFused>(P, grid, smem, pdl, err, s);
    case 3:
    case 4: return launch_decode_t<4, kFused>(P, grid, smem, pdl, err, s);
    default: return launch_decode_t<8, kFused>(P, grid, smem, pdl, err, s);
  }
}

}  // namespace

bool decode_supported(int64_t M, int64_t K) {
  return M >= 1 && M <= kDecodeMaxM && M * K <= kDecodeMaxCodeBytes;
}

cudaError_t launch_decode(const DeviceContext* ctx, const DecodeJob* jobs, int njobs, int M, float eps, bool fused,
                          bool weights_static, cudaStream_t s) {
  DecodeParams P = {};
  P.nproj = njobs;
  P.M = M;
  P.eps = eps;
  P.weights_static = weights_static ? 1 : 0;
  double total = 0.0;
  int maxK = 0;
  for (int i = 0; i < njobs; ++i) {
    total += static_cast<double>(jobs[i].N) * jobs[i].K / 4.0;
    maxK = jobs[i].K > maxK ? jobs[i].K : maxK;
  }
  const int target = 2 * ctx->num_sms;  // about two resident CTAs per SM
  int cta = 0;
  for (int i = 0; i < njobs; ++i) {
    const DecodeJob& j = jobs[i];
    const double bytes = static_cast<double>(j.N) * j.K / 4.0;
    int want = static_cast<int>(target * bytes / total + 0.5);
    if (want < 1) want = 1;
    if (want > j.N) want = j.N;
    const int rpc = (j.N + want - 1) / want;
    const int n_ctas = (j.N + rpc - 1) / rpc;
    DecodeProj& p = P.p[i];
    p.x = j.x;
    p.g = j.g;
    p.codes = j.codes;
    p.a_scale = j.a_scale;
    p.w = j.w;
    p.inv_w = 1.0f / j.w_scale;  // IEEE division, as in the oracle
    p.K = j.K;
    p.N = j.N;
    p.y = j.y;
    p.acc_out = j.acc_out;
    p.cta_begin = cta;
    p.rows_per_cta = rpc;
    cta += n_ctas;
  }
  int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
  const size_t smem = decode_smem_bytes(mt, maxK);
  const bool pdl = true;  // without BITNET_FLAG_WEIGHTS_STATIC every thread waits before reading
  return fused ? dispatch_m<true>(M, P, cta, smem, pdl, ctx->err_word, s)
               : dispatch_m<false>(M, P, cta, smem, pdl, ctx->err_word, s);
}

}  // namespace bitnet
