// gemv_row.cu -- BitLinear for one token with long rows (M = 1, K = 4096, 8192
// or 16384): the whole cost is the I2_S weight stream ("gguf-gemv",
// "Performance": decode at M = 1 is bound by the packed-block bytes).
//
// The arithmetic is the fused decode path's: RMSNorm + absmax int8 quant of the
// row (rowquant.cuh, "BitNet Inference Framework", "Quantization (W1.58A8)"),
// the int8 x ternary dot products of ggml_vec_dot_i2_i8_s ("BitNet Embeddings
// GGUF Conversion Implementation", section 6.4) with dp4a, and the rescale
// y = ((float)acc * (1/a_scale)) * (1/w_scale).  Every sum is an integer, so y
// is bit for bit the one every other route of the library computes.
//
// Layout of the work (one CTA per SM: 16 consumer warps and one stream warp):
//  * thread t owns two 16-byte chunks, c and c + K/128 with c = t mod (K/128),
//    of every weight row it reads (chunk c: block c/2, bytes 16 (c&1) .. +15,
//    elements 128 (c/2) + 32 s + 16 (c&1) + j of slot s), so the activation
//    codes it multiplies are the same 128 bytes for every row: they stay in 32
//    registers for the whole stream, and its only shared-memory reads are the
//    weight bytes themselves (consecutive threads read consecutive 16 bytes:
//    no bank conflicts);
//  * K/128 threads share a row (row group); 512/(K/128) groups take the rows of
//    a stage in turn, four rows per group per 64 KB stage at every supported K;
//  * a consumer warp reduces its part of a row with one redux, stores it in the
//    stage's table of per-warp partial sums and, after its rows of a stage,
//    arrives on the stage's barrier; consumers never wait for one another;
//  * the stream warp issues the weight copies, and when the 16 consumers have
//    passed a stage it adds up each row's partial sums, rescales the rows,
//    writes y and refills the slot with the stage one lap later;
//  * weights stream through a ring of three 64 KB stages (1-D bulk copies with
//    an L2 evict-first policy).  The ring's first fill is prefetched into the L2
//    before the grid-dependency wait (a prefetch changes no value any load
//    returns, so this holds whatever earlier work on the stream writes); the
//    copies themselves are issued once this CTA's share of x is loaded: issued
//    earlier, they queue the prologue's loads of x (L2 hits) behind the weight
//    misses (measured: ~1.6 us later prologue at K = 16384).  With the copies,
//    the next two stages are prefetched into the L2, so that the HBM stream
//    keeps going through the rest of the prologue (K = N = 16384: 14.8 ->
//    13.6 us; deeper prefetching, or prefetching before x, measured slower).
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

namespace bitnet {
namespace {

constexpr int kR1Threads = 512;             // consumers
constexpr int kR1Warps = kR1Threads / 32;
constexpr int kR1Block = kR1Threads + 32;    // + the stream warp
constexpr int kR1StageBytes = 65536;
constexpr int kR1Stages = 3;
constexpr int kR1RowsPerGroup = 4;               // rows of a stage per row group
constexpr int kR1MaxRows = kR1StageBytes / 1024;  // rows per stage at K = 4096
constexpr int kR1MaxParts = 4;                    // consumer warps per row at K = 16384
constexpr int kR1MaxGroups = 8;                   // float4 groups of x per thread: 16384 / 4 / 512
constexpr int kR1PrefetchAhead = 2;               // stages past the ring prefetched into L2 once x is in

struct Row1Params {
  const float* x;
  const float* g;
  const uint8_t* w;
  float inv_w;
  int K;
  int N;
  float* y;
  int32_t* acc_out;
  float eps;
  int weights_static;  // the norm weight may be read before the dependency wait
  int rows_per_cta;
};

struct Row1Tail {
  uint64_t full[kR1Stages];  // the stage's bulk copy has landed
  uint64_t done[kR1Stages];  // every consumer warp has added its part of the stage's rows
  int part[kR1Stages][kR1MaxRows][kR1MaxParts];  // per-warp partial sums of code * q
  int last_issued[kR1Stages];                     // last stage copied into the slot, -1 for none
  int red_key[kR1Warps];
  unsigned long long red_ss[kR1Warps];
  unsigned red_amax[kR1Warps];
  int red_rs[kR1Warps];
  int abort_flag;
};

constexpr size_t row1_smem_bytes(int K) {
  return static_cast<size_t>(kR1Stages) * kR1StageBytes + static_cast<size_t>(K) + sizeof(Row1Tail);
}

// Offset of activation element k (k % 4 == 0) in the slot-major code layout:
// chunk c's 16 codes of slot s sit at ((s * cpr + c) * 16).
__device__ __forceinline__ int r1_slot_major(int k, int cpr) {
  const int b = k >> 7, e = k & 127;
  const int sl = e >> 5, j = e & 31;
  return ((sl * cpr + 2 * b + (j >> 4)) << 4) + (j & 15);
}

// Adds chunk `wv`'s four slots (times the activation codes xc) into a[slot].
__device__ __forceinline__ void r1_chunk(const uint4& wv, const int4 (&xc)[4], int (&a)[4]) {
#pragma unroll
  for (int sl = 0; sl < 4; ++sl) {
    const unsigned m = 0xC0C0C0C0u >> (2 * sl);
    int t = dp4a_us(wv.x & m, xc[sl].x, a[sl]);
    t = dp4a_us(wv.y & m, xc[sl].y, t);
    t = dp4a_us(wv.z & m, xc[sl].z, t);
    a[sl] = dp4a_us(wv.w & m, xc[sl].w, t);
  }
}

__global__ void __launch_bounds__(kR1Block, 1) k_gemv_row1(const __grid_constant__ Row1Params P, unsigned* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int K = P.K;
  const int row_bytes = K >> 2;
  const int rps = kR1StageBytes / row_bytes;  // rows per stage
  const int r0 = static_cast<int>(blockIdx.x) * P.rows_per_cta;
  const int r1 = min(P.N, r0 + P.rows_per_cta);
  const int nst = (r1 - r0 + rps - 1) / rps;
  uint8_t* ring = smem;
  int8_t* xq = reinterpret_cast<int8_t*>(smem + kR1Stages * kR1StageBytes);
  Row1Tail* tail = reinterpret_cast<Row1Tail*>(smem + kR1Stages * kR1StageBytes + K);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool streamer = warp == kR1Warps;

  if (tid == 0) {
    for (int s = 0; s < kR1Stages; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->done[s], kR1Warps);
      tail->last_issued[s] = -1;
    }
    tail->abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  const uint8_t* wsrc = P.w + static_cast<int64_t>(r0) * row_bytes;
  const int cta_bytes = (r1 - r0) * row_bytes;
  const uint64_t wpol = l2_policy_evict_first();
  auto stage_len = [&](int st) { return min(kR1StageBytes, cta_bytes - st * kR1StageBytes); };
  auto issue = [&](int st) {  // one thread of the stream warp
    const int s = st % kR1Stages;
    const unsigned b = static_cast<unsigned>(stage_len(st));
    mbar_arrive_expect_tx(&tail->full[s], b);
    bulk_load_hint(ring + s * kR1StageBytes, wsrc + static_cast<int64_t>(st) * kR1StageBytes, b, &tail->full[s],
                   wpol);
    tail->last_issued[s] = st;
  };
  const int first = min(kR1Stages, nst);
  if (streamer && lane == 0)
    for (int st = 0; st < first; ++st)
      bulk_prefetch_l2(wsrc + static_cast<int64_t>(st) * kR1StageBytes, static_cast<unsigned>(stage_len(st)));

  // ------------------------------------------------------------- prologue
  // RMSNorm + absmax quant of the row by the 512 consumer threads: thread tid
  // holds the float4 groups (tid + 512 i + rot) mod G, rot depending on the CTA
  // so that the CTAs' simultaneous requests for the same x and norm weight
  // spread over the L2.  The stream warp only passes the barriers.
  const int G = K >> 2;
  const int cpr = K >> 6;
  const float4* x4 = reinterpret_cast<const float4*>(P.x);
  const float4* g4 = reinterpret_cast<const float4*>(P.g);
  const int rot = (static_cast<int>(blockIdx.x) * 64) % G;
  const int nv = streamer ? 0 : (G - tid + kR1Threads - 1) / kR1Threads;
  auto gidx = [&](int i) {
    const int j = tid + kR1Threads * i + rot;
    return j < G ? j : j - G;
  };
  float4 gv[kR1MaxGroups], v[kR1MaxGroups];
  auto load_g = [&]() {
#pragma unroll
    for (int i = 0; i < kR1MaxGroups; ++i) gv[i] = i < nv ? __ldg(g4 + gidx(i)) : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  if (P.weights_static) load_g();
  pdl_wait();  // x (and y) belong to the previous kernel's stream order
  if (!P.weights_static) load_g();
  int key = 0;
#pragma unroll
  for (int i = 0; i < kR1MaxGroups; ++i) {
    v[i] = i < nv ? __ldg(x4 + gidx(i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    key = max(key, sq_key4(v[i]));
  }
  key = warp_max_int(key);
  if (lane == 0 && !streamer) tail->red_key[warp] = key;
  __syncthreads();
  if (streamer && lane == 0) {
    for (int st = 0; st < first; ++st) issue(st);
    // the HBM stream keeps going through the rest of the prologue
    for (int st = first; st < min(nst, first + kR1PrefetchAhead); ++st)
      bulk_prefetch_l2(wsrc + static_cast<int64_t>(st) * kR1StageBytes, static_cast<unsigned>(stage_len(st)));
  }
  key = warp_max_int(lane < kR1Warps ? tail->red_key[lane] : 0);
  {
    const float scale = sq_scale(key);
    SqPartial part = {0ull, 0u};
#pragma unroll
    for (int i = 0; i < kR1MaxGroups; ++i)
      if (i < nv) sq_add4(part, v[i], scale);
    const unsigned long long wsum = warp_sum_u64(sq_fold(part, 4 * nv));
    if (lane == 0 && !streamer) tail->red_ss[warp] = wsum;
  }
  __syncthreads();
  const float rstd = rstd_from_fixed(warp_sum_u64(lane < kR1Warps ? tail->red_ss[lane] : 0ull), key, K, P.eps);
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kR1MaxGroups; ++i) {
    if (i < nv) {
      v[i] = make_float4(norm_elem(v[i].x, rstd, gv[i].x), norm_elem(v[i].y, rstd, gv[i].y),
                         norm_elem(v[i].z, rstd, gv[i].z), norm_elem(v[i].w, rstd, gv[i].w));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
  }
  amax = warp_max(amax);
  if (lane == 0 && !streamer) tail->red_amax[warp] = __float_as_uint(amax);
  __syncthreads();
  const float as = act_scale_from_amax(
      __uint_as_float(__reduce_max_sync(0xffffffffu, lane < kR1Warps ? tail->red_amax[lane] : 0u)));
  {
    int rs = 0;
#pragma unroll
    for (int i = 0; i < kR1MaxGroups; ++i) {
      if (i < nv) {
        const uint32_t pk = quant_pack4_i8(v[i], as);
        *reinterpret_cast<uint32_t*>(xq + r1_slot_major(4 * gidx(i), cpr)) = pk;
        rs = __dp4a(static_cast<int>(pk), 0x01010101, rs);
      }
    }
    rs = warp_sum_int(rs);
    if (lane == 0 && !streamer) tail->red_rs[warp] = rs;
  }
  __syncthreads();
  const int rowsum = warp_sum_int(lane < kR1Warps ? tail->red_rs[lane] : 0);
  const float inv_a = __frcp_rn(as);
  const float inv_w = P.inv_w;
  const int L = cpr >> 1;  // threads per row: 32, 64 or 128
  const int WPR = L >> 5;  // warps per row: 1, 2 or 4

  if (streamer) {
    // ------------------------------------------------------ stream warp
    for (int st = 0; st < nst; ++st) {
      const int s = st % kR1Stages;
      if (!mbar_wait(&tail->done[s], (st / kR1Stages) & 1, err, &tail->abort_flag)) break;
      const int rows = min(rps, r1 - r0 - st * rps);
      for (int r = lane; r < rows; r += 32) {
        int sum = 0;
        for (int w = 0; w < WPR; ++w) sum += tail->part[s][r][w];
        const int acc = sum - rowsum;  // sum of (code - 1) * q
        const int n = r0 + st * rps + r;
        P.y[n] = rescale_elem(__int2float_rn(acc), inv_a, inv_w);
        if (P.acc_out) P.acc_out[n] = acc;
      }
      __syncwarp();
      if (lane == 0 && st + kR1Stages < nst) issue(st + kR1Stages);
    }
  } else {
    // --------------------------------------------------------- dot products
    const int RG = kR1Threads / L;  // row groups: 16, 8 or 4
    const int grp = tid / L;
    const int c = tid - grp * L;    // this thread's chunks: c and c + L
    const int wi = c >> 5;          // this warp's index among the row's warps
    int4 xc[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int s = 0; s < 4; ++s) xc[h][s] = *reinterpret_cast<const int4*>(xq + ((s * cpr + c + h * L) << 4));

    for (int st = 0; st < nst; ++st) {
      const int s = st % kR1Stages;
      if (!mbar_wait(&tail->full[s], (st / kR1Stages) & 1, err, &tail->abort_flag)) break;
      const uint8_t* stage = ring + s * kR1StageBytes;
      const int rows = min(rps, r1 - r0 - st * rps);
      // rps = 4 RG at every supported K: four rows per group per full stage
      uint4 wv[kR1RowsPerGroup][2];
#pragma unroll
      for (int q = 0; q < kR1RowsPerGroup; ++q) {
        const int r = grp + q * RG;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          wv[q][h] = r < rows ? *reinterpret_cast<const uint4*>(stage + r * row_bytes + (c + h * L) * 16)
                              : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < kR1RowsPerGroup; ++q) {
        int a[4] = {0, 0, 0, 0};
        r1_chunk(wv[q][0], xc[0], a);
        r1_chunk(wv[q][1], xc[1], a);
        // slot s's sum carries the factor 4^(3-s) of its bit position (exact)
        const int sum = warp_sum_int((a[0] >> 6) + (a[1] >> 4) + (a[2] >> 2) + a[3]);
        const int r = grp + q * RG;
        if (lane == 0 && r < rows) tail->part[s][r][wi] = sum;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->done[s]);
    }
  }
  // leave no copy in flight when the CTA retires (every issued copy has
  // normally been consumed already)
  __syncthreads();
  if (streamer && lane == 0) {
    for (int s = 0; s < kR1Stages; ++s) {
      const int st = tail->last_issued[s];
      if (st >= 0) mbar_wait(&tail->full[s], (st / kR1Stages) & 1, err, nullptr);
    }
  }
}

}  // namespace

bool gemv_row1_supported(int64_t M, int64_t K) { return M == 1 && (K == 4096 || K == 8192 || K == 16384); }

cudaError_t launch_gemv_row1(const DeviceContext* ctx, const DecodeJob& j, float eps, bool weights_static,
                             cudaStream_t s) {
  Row1Params P = {};
  P.x = j.x;
  P.g = j.g;
  P.w = j.w;
  P.inv_w = 1.0f / j.w_scale;  // IEEE division, as in the oracle
  P.K = j.K;
  P.N = j.N;
  P.y = j.y;
  P.acc_out = j.acc_out;
  P.eps = eps;
  P.weights_static = weights_static ? 1 : 0;
  const int ctas_want = ctx->num_sms < j.N ? ctx->num_sms : j.N;
  P.rows_per_cta = (j.N + ctas_want - 1) / ctas_want;
  const int grid = (j.N + P.rows_per_cta - 1) / P.rows_per_cta;
  const size_t smem = row1_smem_bytes(j.K);
  cudaError_t e = cudaFuncSetAttribute(k_gemv_row1, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kR1Block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_row1, P, ctx->err_word);
}

}  // namespace bitnet
