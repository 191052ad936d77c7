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

constexpr int kDecWarps = 15;                      // compute warps (16 warps in all: 128 registers per thread)
constexpr int kDecThreads = (kDecWarps + 1) * 32;  // + one producer warp
constexpr int kDecStageBytes = 24576;
constexpr int kDecMaxStages = 6;  // ring depth is chosen per launch (3 or 6)
// Long rows (K >= 4096, K a multiple of 2048): small stages of whole rows, each
// consumed by one warp, up to kDecMaxSlots of them in the ring, filled by bulk
// copies of about kDecLongCopyBytes (one copy per group of consecutive slots:
// a bulk copy carries a fixed cost, and 4 KB copies reach only about half the
// streaming rate of 16 KB ones).
constexpr int kDecLongStageBytes = 8192;
constexpr int kDecLongCopyBytes = 16384;
constexpr int kDecMaxSlots = 64;

struct DecodeProj {
  const float* x;   // activations, or the gate projection's output when act != 0
  const float* up;  // act != 0: the up projection's output (the row is act(x) * up)
  int act;
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
  int stages;      // weight ring depth in 24 KB stages (short rows, <= kDecMaxStages)
  int ring_bytes;  // weight ring size (long rows use it as kDecLongStageBytes-sized slots)
};

struct DecodeSmemTail {
  uint64_t full[kDecMaxSlots];
  uint64_t empty[kDecMaxSlots];
  uint64_t in_full;  // activations (and norm weight) staged; register prologue: loaded into registers
  // per-row reductions, combined across warps with shared-memory atomics
  // (integer or max: the result does not depend on the order)
  unsigned long long ss[kDecodeMaxM];
  int sq_key[kDecodeMaxM];  // bit pattern of the row's largest |x|
  unsigned amax_bits[kDecodeMaxM];
  int rowsum[kDecodeMaxM];
  float rstd[kDecodeMaxM];
  float inv_a[kDecodeMaxM];
  // register prologue: per-warp partials of the current row (written without
  // atomics, combined by every thread after the barrier) and per-warp row sums
  int red_key[kDecWarps];
  unsigned long long red_ss[kDecWarps];
  unsigned red_amax[kDecWarps];
  int red_rs[kDecodeMaxM][kDecWarps];
  int abort_flag;
};

// Fused norm with x and the norm weight held in registers (every compute
// thread holds at most kDecRegGroups float4 groups of each) instead of staged
// in shared memory: long rows up to K = 16384, and single-token rows up to
// K = 3840 (two groups per thread, within the register budget of the
// two-CTAs-per-SM kernels).
__host__ __device__ inline bool register_prologue_long(int K) { return K >= 4096 && K % 2048 == 0 && K <= 16384; }
__host__ __device__ inline bool register_prologue(bool fused, int K, int M) {
  return fused && (register_prologue_long(K) || (M == 1 && K <= 3840));
}
constexpr int kDecRegGroups = 9;  // float4 groups per thread: 16384 / 4 <= 9 * 480

// Shared-memory carve-up for one CTA: weight ring | x fp32 [M,K] (fused and
// staged) or the incoming int8 codes [M,K] (unfused) | g fp32 [K] (fused and
// staged) | codes int8 [M,K] in slot-major order | tail.
//
// Slot-major codes: the 16-byte chunk c of a weight row (block c/2, bytes
// 16(c&1)..+15) pairs, for slot s, with activation elements
// 128(c/2) + 32s + 16(c&1) + 0..15.  They are stored at ((s*cpr + c) * 16),
// cpr = K/64 chunks per row, so lanes reading consecutive chunks of one slot
// read consecutive 16-byte words (no bank conflicts).
struct DecodeLayout {
  int xs, gs, xq, tail, total;
  __host__ __device__ DecodeLayout(int M, int K, bool fused, int ring_bytes) {
    const bool staged = fused && !register_prologue(fused, K, M);
    xs = ring_bytes;
    gs = xs + (staged ? M * K * 4 : (fused ? 0 : ((M * K + 127) & ~127)));
    xq = gs + (staged ? K * 4 : 0);
    tail = xq + ((M * K + 127) & ~127);
    total = tail + static_cast<int>(sizeof(DecodeSmemTail));
  }
};

// Offset of activation element k (k % 4 == 0: the 4 elements k..k+3 stay
// together) in the slot-major layout.
__device__ __forceinline__ int slot_major(int k, int cpr) {
  const int b = k >> 7, e = k & 127;
  const int sl = e >> 5, j = e & 31;
  return ((sl * cpr + 2 * b + (j >> 4)) << 4) + (j & 15);
}

__device__ __forceinline__ void compute_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(kDecWarps * 32) : "memory");
}

// Short rows and few tokens: registers for two CTAs per SM, so that the next
// dependent launch can become resident while this one drains.  Long rows and
// more tokens: one CTA per SM with up to 128 registers per thread.
// kGlu: some projection's row is act(x) * up (the down projection's input),
// computed as the rows are loaded (register prologue only).
template <int MT, bool kFused, bool kLong, bool kGlu>
__global__ void __launch_bounds__(kDecThreads, (kLong || MT >= 4) ? 1 : 2) k_decode(const __grid_constant__ DecodeParams P, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];

  // which projection this CTA serves
  int pi = 0;
#pragma unroll 1
  for (int i = 1; i < P.nproj; ++i)
    if (static_cast<int>(blockIdx.x) >= P.p[i].cta_begin) pi = i;
  const DecodeProj& pr = P.p[pi];
  const int K = pr.K;
  const int N = pr.N;
  const int M = P.M;
  const int row_bytes = K >> 2;
  const int r0 = (static_cast<int>(blockIdx.x) - pr.cta_begin) * pr.rows_per_cta;
  const int r1 = min(N, r0 + pr.rows_per_cta);
  // lpr lanes share a weight row (each taking cpr/lpr of its 16-byte chunks);
  // at least 4 where the row allows it (two rows of a shared-memory phase then
  // touch different banks) and chosen to shorten the busiest warp's chain: each
  // further pass over rows costs a whole dot-product latency, each chunk of a
  // lane a few issue cycles and each lane-halving a shuffle.  A stage holds a
  // whole number of passes.
  const int cpr = K >> 6;
  int lpr = (cpr & 3) ? 2 : 4;
  {
    const int R = max(r1 - r0, 1);
    int best = 1 << 30;
    for (int l = lpr; l <= 32 && cpr % l == 0; l *= 2) {
      const int passes = (R + kDecWarps * (32 / l) - 1) / (kDecWarps * (32 / l));
      const int cost = passes * ((cpr / l) * 40 + (31 - __clz(l)) * 30 + 120);
      if (cost < best) {
        best = cost;
        lpr = l;
      }
    }
  }
  const int rpp = 32 / lpr;  // rows per warp pass
  // Long rows (cpr a multiple of 32, >= 64): stages of whole rows, about 4 KB,
  // one warp per stage.  Otherwise whole warps take rows and a 24 KB stage
  // holds whole passes of all warps.
  const bool lng = kLong && cpr >= 64 && (cpr & 31) == 0;
  int rps, sbytes, nslots, grp;  // grp: consecutive slots filled by one copy
  if (lng) {
    rps = max(1, kDecLongStageBytes / row_bytes);
    sbytes = rps * row_bytes;
    grp = max(1, kDecLongCopyBytes / sbytes);
    nslots = min(kDecMaxSlots, P.ring_bytes / sbytes);
    grp = min(grp, nslots);
    nslots -= nslots % grp;
  } else {
    rps = kDecStageBytes / row_bytes;  // rows per stage (K <= 65536 keeps it >= 1)
    if (rps >= kDecWarps * rpp) rps -= rps % (kDecWarps * rpp);
    sbytes = kDecStageBytes;
    nslots = P.stages;
    grp = 1;
  }
  const int nst = (r1 - r0 + rps - 1) / rps;
  const bool regp = register_prologue(kFused, K, M);
  // Long rows, register prologue, weights not requested before the grid
  // dependency wait: the weight stream starts only once every compute warp
  // holds its x and norm weight, which otherwise arrive far later (each CTA
  // brings in the whole row, up to 128 KB, next to its weight ring).
  const bool gate_weights = regp && lng && !P.weights_static;

  const DecodeLayout lay(M, K, kFused, P.ring_bytes);
  uint8_t* ring = smem;
  float* xs = reinterpret_cast<float*>(smem + lay.xs);
  float* gs = reinterpret_cast<float*>(smem + lay.gs);
  int8_t* xq = reinterpret_cast<int8_t*>(smem + lay.xq);
  DecodeSmemTail* tail = reinterpret_cast<DecodeSmemTail*>(smem + lay.tail);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nslots; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], lng ? 1 : kDecWarps);
    }
    mbar_init(&tail->in_full, gate_weights ? kDecWarps : 1);
    for (int m = 0; m < kDecodeMaxM; ++m) {
      tail->ss[m] = 0ull;
      tail->sq_key[m] = 0;
      tail->amax_bits[m] = 0u;
      tail->rowsum[m] = 0;
    }
    tail->abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kDecWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint8_t* src = pr.w + static_cast<int64_t>(r0) * row_bytes;
      const unsigned in_bytes = kFused ? static_cast<unsigned>((M + 1) * K * 4) : static_cast<unsigned>(M * K);
      if (!regp) mbar_arrive_expect_tx(&tail->in_full, in_bytes);
      // Copy c fills stages c*grp .. c*grp + grp - 1 (slots of one group of the
      // ring, completion counted on the group's first full barrier); it is
      // issued once every slot of the group is free again.
      const int ncopy = (nst + grp - 1) / grp;
      const int first = min(ncopy, nslots / grp);
      // the weights are read once per call: evict them first from the L2
      const uint64_t wpol = l2_policy_evict_first();
      auto issue = [&](int c) {
        const int st0 = c * grp;
        const int s = st0 % nslots;
        const int rows = min(grp * rps, r1 - r0 - st0 * rps);
        const unsigned bytes = static_cast<unsigned>(rows * row_bytes);
        mbar_arrive_expect_tx(&tail->full[s], bytes);
        bulk_load_hint(ring + s * sbytes, src + static_cast<int64_t>(st0) * rps * row_bytes, bytes, &tail->full[s],
                       wpol);
      };
      // parameters (packed weights, norm weight) may be requested before the
      // previous kernel has finished when they are known not to be written by
      // it; the activations always after the wait, and ahead of the weights
      // when those wait too, so that the prologue starts as early as possible
      if (P.weights_static) {
        if (kFused && !regp) bulk_load(gs, pr.g, static_cast<unsigned>(K * 4), &tail->in_full);
        for (int c = 0; c < first; ++c) issue(c);
      }
      pdl_wait();
      if (gate_weights && !mbar_wait(&tail->in_full, 0, err, &tail->abort_flag)) return;
      if (kFused) {
        if (!regp) {
          if (!P.weights_static) bulk_load(gs, pr.g, static_cast<unsigned>(K * 4), &tail->in_full);
          bulk_load(xs, pr.x, static_cast<unsigned>(M * K * 4), &tail->in_full);
        }
      } else {
        bulk_load(xs, pr.codes, static_cast<unsigned>(M * K), &tail->in_full);
      }
      if (!P.weights_static)
        for (int c = 0; c < first; ++c) issue(c);
      int issued = first;
      for (int c = first; c < ncopy; ++c) {
        bool ok = true;
        for (int j = 0; j < grp && ok; ++j) {
          const int st = c * grp + j - nslots;  // the stage this slot held one lap earlier
          ok = mbar_wait(&tail->empty[st % nslots], (st / nslots) & 1, err, &tail->abort_flag);
        }
        if (!ok) break;
        issue(c);
        issued = c + 1;
      }
      // leave no copy in flight when the CTA retires
      if (!regp) mbar_wait(&tail->in_full, 0, err, nullptr);
      for (int c = max(0, issued - nslots / grp); c < issued; ++c)
        mbar_wait(&tail->full[(c * grp) % nslots], ((c * grp) / nslots) & 1, err, nullptr);
    }
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int tid = threadIdx.x;  // 0 .. kDecWarps*32-1
  constexpr int kThr = kDecWarps * 32;
  // (row, float4 group) of this thread's first element in the flat prologue
  // loops, worked out while the inputs are still in flight
  const int G = K >> 2;      // float4 groups per row
  const int total = M * G;
  const int m_start = tid / G;
  const int g_start = tid - m_start * G;
  if (kFused && regp) {
    // register prologue: row by row, x and the norm weight straight from
    // global memory into registers, the same order-free reductions as below
    // through shared-memory atomics.  Thread tid holds the float4 groups
    // (tid + 480 i + rot) mod G: every CTA reads the same x and norm weight,
    // and the CTA-dependent rotation spreads their simultaneous requests over
    // the L2 instead of sending all of them to the same lines at once.
    const float4* g4 = reinterpret_cast<const float4*>(pr.g);
    const int rot = (static_cast<int>(blockIdx.x) * 32) % G;
    auto gidx = [&](int i) {
      const int j = tid + kThr * i + rot;
      return j < G ? j : j - G;  // valid when tid + 480 i < G
    };
    // groups of this thread (at most kRG: 9 for long rows, 2 for one short row)
    constexpr int kRG = kLong ? kDecRegGroups : 2;
    const int nv = (G - tid + kThr - 1) / kThr;
    float4 gv[kRG];
    auto load_g = [&]() {
#pragma unroll
      for (int i = 0; i < kRG; ++i)
        gv[i] = i < nv ? __ldg(g4 + gidx(i)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    };
    if (P.weights_static) load_g();
    pdl_wait();  // x (and y) belong to the previous kernel's stream order
    if (!P.weights_static) load_g();
#pragma unroll 1
    for (int m = 0; m < M; ++m) {
      const float4* x4 = reinterpret_cast<const float4*>(pr.x) + static_cast<int64_t>(m) * G;
      float4 v[kRG];
      int key = 0;
      const float4* u4 = reinterpret_cast<const float4*>(pr.up) + static_cast<int64_t>(m) * G;
#pragma unroll
      for (int i = 0; i < kRG; ++i) {
        v[i] = i < nv ? __ldg(x4 + gidx(i)) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (kGlu && pr.act != 0 && i < nv) v[i] = glu4(v[i], __ldg(u4 + gidx(i)), pr.act);  // down projection input
        key = max(key, sq_key4(v[i]));
      }
      key = warp_max_int(key);
      if (lane == 0) tail->red_key[warp] = key;
      if (gate_weights && m == 0 && lane == 0) mbar_arrive(&tail->in_full);  // this warp's x and g are in
      compute_bar();
      // cross-warp combines: lane w reads warp w's partial, one warp reduction
      key = warp_max_int(lane < kDecWarps ? tail->red_key[lane] : 0);
      const float scale = sq_scale(key);
      SqPartial part = {0ull, 0u};
#pragma unroll
      for (int i = 0; i < kRG; ++i)
        if (i < nv) sq_add4(part, v[i], scale);
      const unsigned long long wsum = warp_sum_u64(sq_fold(part, 4 * nv));
      if (lane == 0) tail->red_ss[warp] = wsum;
      compute_bar();
      const unsigned long long ss = warp_sum_u64(lane < kDecWarps ? tail->red_ss[lane] : 0ull);
      const float rstd = rstd_from_fixed(ss, key, K, P.eps);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < kRG; ++i) {
        if (i < nv) {
          v[i] = make_float4(norm_elem(v[i].x, rstd, gv[i].x), norm_elem(v[i].y, rstd, gv[i].y),
                             norm_elem(v[i].z, rstd, gv[i].z), norm_elem(v[i].w, rstd, gv[i].w));
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
        }
      }
      amax = warp_max(amax);
      if (lane == 0) tail->red_amax[warp] = __float_as_uint(amax);
      compute_bar();
      const unsigned amax_bits = __reduce_max_sync(0xffffffffu, lane < kDecWarps ? tail->red_amax[lane] : 0u);
      const float as = act_scale_from_amax(__uint_as_float(amax_bits));
      int rs = 0;
#pragma unroll
      for (int i = 0; i < kRG; ++i) {
        if (i < nv) {
          const uint32_t pk = quant_pack4_i8(v[i], as);
          *reinterpret_cast<uint32_t*>(xq + m * K + slot_major(4 * gidx(i), cpr)) = pk;
          rs = __dp4a(static_cast<int>(pk), 0x01010101, rs);
        }
      }
      rs = warp_sum_int(rs);
      if (lane == 0) tail->red_rs[m][warp] = rs;
      if (tid == 0) tail->inv_a[m] = __frcp_rn(as);
    }
  } else {
  if (!mbar_wait(&tail->in_full, 0, err, &tail->abort_flag)) return;
  // Prologue loops run over all (row, float4 group) pairs of the M x K block in
  // one flat, non-unrolled loop; K/4 is a multiple of 32, so the 32 lanes of a
  // warp always hold groups of the same row and one warp reduction plus one
  // shared atomic per warp combines them (integer sums and maxima: order-free).
  // Per-row reductions accumulate in registers while a thread's elements stay
  // in one row and are flushed (one warp reduction, one shared atomic per warp)
  // when the row changes: a warp's lanes always share the row, so flushes are
  // warp-uniform.
  if (kFused) {
    {
      int e = 0, cur = m_start;
#pragma unroll 1
      for (int i = tid, m = m_start, gi = g_start; i < total; i += kThr, gi += kThr) {
        while (gi >= G) { gi -= G; ++m; }
        if (m != cur) {
          const int w = warp_max_int(e);
          if (lane == 0 && w) atomicMax(&tail->sq_key[cur], w);
          e = 0;
          cur = m;
        }
        e = max(e, sq_key4(*reinterpret_cast<const float4*>(xs + 4 * i)));
      }
      if (cur < M) {
        const int w = warp_max_int(e);
        if (lane == 0 && w) atomicMax(&tail->sq_key[cur], w);
      }
    }
    compute_bar();
    {
      unsigned long long acc = 0ull;
      int cur = m_start;
      float scale = sq_scale(cur < M ? tail->sq_key[cur] : 0);
#pragma unroll 1
      for (int i = tid, m = m_start, gi = g_start; i < total; i += kThr, gi += kThr) {
        while (gi >= G) { gi -= G; ++m; }
        if (m != cur) {
          const unsigned long long w = warp_sum_u64(acc);
          if (lane == 0 && w) atomicAdd(&tail->ss[cur], w);
          acc = 0ull;
          cur = m;
          scale = sq_scale(tail->sq_key[cur]);
        }
        SqPartial part = {0ull, 0u};
        sq_add4(part, *reinterpret_cast<const float4*>(xs + 4 * i), scale);
        acc += sq_fold(part, 4);
      }
      if (cur < M) {
        const unsigned long long w = warp_sum_u64(acc);
        if (lane == 0 && w) atomicAdd(&tail->ss[cur], w);
      }
    }
    compute_bar();
    if (tid < M) tail->rstd[tid] = rstd_from_fixed(tail->ss[tid], tail->sq_key[tid], K, P.eps);
    compute_bar();
    // normalise in place and take the absmax
    {
      float amax = 0.0f;
      int cur = m_start;
      float rstd = cur < M ? tail->rstd[cur] : 0.0f;
#pragma unroll 1
      for (int i = tid, m = m_start, gi = g_start; i < total; i += kThr, gi += kThr) {
        while (gi >= G) { gi -= G; ++m; }
        if (m != cur) {
          const float w = warp_max(amax);
          if (lane == 0) atomicMax(&tail->amax_bits[cur], __float_as_uint(w));
          amax = 0.0f;
          cur = m;
          rstd = tail->rstd[cur];
        }
        const int k = 4 * gi;
        const float4 v = *reinterpret_cast<const float4*>(xs + 4 * i);
        const float4 gv = *reinterpret_cast<const float4*>(gs + k);
        const float4 n = make_float4(norm_elem(v.x, rstd, gv.x), norm_elem(v.y, rstd, gv.y),
                                     norm_elem(v.z, rstd, gv.z), norm_elem(v.w, rstd, gv.w));
        *reinterpret_cast<float4*>(xs + 4 * i) = n;
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(n.x), fabsf(n.y)), fmaxf(fabsf(n.z), fabsf(n.w))));
      }
      if (cur < M) {
        const float w = warp_max(amax);
        if (lane == 0) atomicMax(&tail->amax_bits[cur], __float_as_uint(w));
      }
    }
    compute_bar();
    // quantise into the slot-major code layout; lane m of every warp computes
    // row m's scale and passes it round
    const float my_as = act_scale_from_amax(lane < M ? __uint_as_float(tail->amax_bits[lane]) : 1.0f);
    {
      int rs = 0, cur = m_start;
#pragma unroll 1
      for (int i = tid, m = m_start, gi = g_start; i < total; i += kThr, gi += kThr) {
        while (gi >= G) { gi -= G; ++m; }
        if (m != cur) {
          const int w = warp_sum_int(rs);
          if (lane == 0 && w) atomicAdd(&tail->rowsum[cur], w);
          rs = 0;
          cur = m;
        }
        const int k = 4 * gi;
        const float as = __shfl_sync(0xffffffffu, my_as, m);
        const uint32_t pk = quant_pack4_i8(*reinterpret_cast<const float4*>(xs + 4 * i), as);
        *reinterpret_cast<uint32_t*>(xq + m * K + slot_major(k, cpr)) = pk;
        rs = __dp4a(static_cast<int>(pk), 0x01010101, rs);
      }
      if (cur < M) {
        const int w = warp_sum_int(rs);
        if (lane == 0 && w) atomicAdd(&tail->rowsum[cur], w);
      }
    }
    if (tid < M) tail->inv_a[tid] = __frcp_rn(my_as);
  } else {
    // codes computed elsewhere (staged in natural order): reorder to slot-major
    // 16 bytes at a time, sum them, fetch the scales
    pdl_wait();
    const int8_t* stg = reinterpret_cast<const int8_t*>(xs);
    const int upr = K >> 4;  // 16-byte units per row (a multiple of 8)
#pragma unroll 1
    for (int i = tid, m = tid / upr, u = tid - (tid / upr) * upr; i < M * upr; i += kThr, u += kThr) {
      while (u >= upr) { u -= upr; ++m; }
      const int4 v = *reinterpret_cast<const int4*>(stg + 16 * i);
      const int b = u >> 3, r = u & 7;
      *reinterpret_cast<int4*>(xq + m * K + (((r >> 1) * cpr + 2 * b + (r & 1)) << 4)) = v;
      int rs = __dp4a(v.x, 0x01010101, 0);
      rs = __dp4a(v.y, 0x01010101, rs);
      rs = __dp4a(v.z, 0x01010101, rs);
      rs = __dp4a(v.w, 0x01010101, rs);
      // a warp's 32 units may span two rows when K/16 is not a multiple of 32
      if (upr % 32 == 0) {
        rs = warp_sum_int(rs);
        if (lane == 0 && rs) atomicAdd(&tail->rowsum[m], rs);
      } else if (rs) {
        atomicAdd(&tail->rowsum[m], rs);
      }
    }
    if (tid < M) tail->inv_a[tid] = __frcp_rn(__ldg(pr.a_scale + tid));
  }
  }
  compute_bar();
  // Writing y needs the previous kernel finished: on the unfused path this
  // thread waited above; on the fused path the activations arrived by a copy the
  // producer issued only after its own wait returned.

  // ------------------------------------------------------------ main loop
  // Odd rows start lpr chunks further on, so with 4 lanes per row the 8 lanes of
  // a shared-memory phase (two rows) touch 8 different 16-byte bank groups for
  // weights and codes alike.
  const int cpl = cpr / lpr;
  const int sub = lane & (lpr - 1);
  const int rot = lpr * ((lane / lpr) & 1);
  int rowsum[MT];
  float inv_a[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    int rsum = 0;
    if (m < M) {
      if (kFused && regp) {
        rsum = warp_sum_int(lane < kDecWarps ? tail->red_rs[m][lane] : 0);
      } else {
        rsum = tail->rowsum[m];
      }
    }
    rowsum[m] = rsum;
    inv_a[m] = m < M ? tail->inv_a[m] : 0.0f;
  }
  const float inv_w = pr.inv_w;
  const int slot_stride = cpr << 4;

  if (kLong && lng) {
    // Long rows: warp w takes the stages in ring slots w, w + 15, ...; lane l takes the 16-byte
    // chunks l, l + 32, ... of each row, so a warp reads 512 consecutive bytes
    // of weights and of each slot's activation codes per step (no bank
    // conflicts), and one redux per row and token finishes the dot product.
    // With one token the codes of the first 128 chunk positions stay in
    // registers for the whole stream.
    const int npos = cpr >> 5;
    int4 xr[4][4];
    if (MT == 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
          xr[i][sl] = i < npos ? *reinterpret_cast<const int4*>(xq + ((lane + 32 * i) << 4) + sl * slot_stride)
                               : make_int4(0, 0, 0, 0);
    }
    // Slot s belongs to warp s % 15, which consumes every use of it in order:
    // a parity wait must never be posted for a phase two ahead of the slot's.
    for (int st = warp < nslots ? warp : nst; st < nst; st += (st % nslots) + kDecWarps < nslots ? kDecWarps
                                                                           : nslots - (st % nslots) + warp) {
      const int s = st % nslots;
      if (!mbar_wait(&tail->full[s - s % grp], (st / nslots) & 1, err, &tail->abort_flag)) break;
      const uint8_t* stage = ring + s * sbytes;
      const int rows = min(rps, r1 - r0 - st * rps);
      int r = 0;
      if (MT == 1) {
        // One token: two rows per pass.  A chunk position's activation codes
        // are read (or held) once for both rows, and the two dot products are
        // independent work for the warp.
        for (; r + 1 < rows; r += 2) {
          const uint8_t* w0 = stage + r * row_bytes;
          const uint8_t* w1 = w0 + row_bytes;
          int a0[4] = {0, 0, 0, 0}, a1[4] = {0, 0, 0, 0};
          auto chunk2 = [&](int c, const int4(&xv)[4]) {
            const uint4 u = *reinterpret_cast<const uint4*>(w0 + c * 16);
            const uint4 v = *reinterpret_cast<const uint4*>(w1 + c * 16);
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
              const unsigned mask = 0xC0C0C0C0u >> (2 * sl);
              int p = a0[sl], q = a1[sl];
              p = dp4a_us(u.x & mask, xv[sl].x, p);
              q = dp4a_us(v.x & mask, xv[sl].x, q);
              p = dp4a_us(u.y & mask, xv[sl].y, p);
              q = dp4a_us(v.y & mask, xv[sl].y, q);
              p = dp4a_us(u.z & mask, xv[sl].z, p);
              q = dp4a_us(v.z & mask, xv[sl].z, q);
              p = dp4a_us(u.w & mask, xv[sl].w, p);
              q = dp4a_us(v.w & mask, xv[sl].w, q);
              a0[sl] = p;
              a1[sl] = q;
            }
          };
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < npos) chunk2(lane + 32 * i, xr[i]);
#pragma unroll 1
          for (int i = 4; i < npos; ++i) {
            const int c = lane + 32 * i;
            int4 xs[4];
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) xs[sl] = *reinterpret_cast<const int4*>(xq + (c << 4) + sl * slot_stride);
            chunk2(c, xs);
          }
          const int t0 = warp_sum_int((a0[0] >> 6) + (a0[1] >> 4) + (a0[2] >> 2) + a0[3]);
          const int t1 = warp_sum_int((a1[0] >> 6) + (a1[1] >> 4) + (a1[2] >> 2) + a1[3]);
          if (lane == 0) {
            const int n = r0 + st * rps + r;
            const int e0 = t0 - rowsum[0], e1 = t1 - rowsum[0];
            pr.y[n] = rescale_elem(__int2float_rn(e0), inv_a[0], inv_w);
            pr.y[n + 1] = rescale_elem(__int2float_rn(e1), inv_a[0], inv_w);
            if (pr.acc_out) {
              pr.acc_out[n] = e0;
              pr.acc_out[n + 1] = e1;
            }
          }
        }
      }
      for (; r < rows; ++r) {
        const uint8_t* wrow = stage + r * row_bytes;
        int acc[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[m][q] = 0;
        auto chunk = [&](int c, const int4(&xreg)[4], bool from_regs) {
          const uint4 wv = *reinterpret_cast<const uint4*>(wrow + c * 16);
          const unsigned wd[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            const unsigned mask = 0xC0C0C0C0u >> (2 * sl);
            const unsigned m0 = wd[0] & mask, m1 = wd[1] & mask, m2 = wd[2] & mask, m3 = wd[3] & mask;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              if (m < M) {
                const int4 xv =
                    from_regs ? xreg[sl] : *reinterpret_cast<const int4*>(xq + (c << 4) + m * K + sl * slot_stride);
                int a = acc[m][sl];
                a = dp4a_us(m0, xv.x, a);
                a = dp4a_us(m1, xv.y, a);
                a = dp4a_us(m2, xv.z, a);
                a = dp4a_us(m3, xv.w, a);
                acc[m][sl] = a;
              }
            }
          }
        };
        if (MT == 1) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (i < npos) chunk(lane + 32 * i, xr[i], true);
#pragma unroll 1
          for (int i = 4; i < npos; ++i) chunk(lane + 32 * i, xr[0], false);
        } else {
#pragma unroll 1
          for (int i = 0; i < npos; ++i) chunk(lane + 32 * i, xr[0], false);
        }
        const int n = r0 + st * rps + r;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < M) {
            const int t = warp_sum_int((acc[m][0] >> 6) + (acc[m][1] >> 4) + (acc[m][2] >> 2) + acc[m][3]);
            if (lane == 0) {
              const int a = t - rowsum[m];
              pr.y[static_cast<int64_t>(m) * N + n] = rescale_elem(__int2float_rn(a), inv_a[m], inv_w);
              if (pr.acc_out) pr.acc_out[static_cast<int64_t>(m) * N + n] = a;
            }
          }
        }
      }
      // the stage's loads are complete (their values fed the dot products);
      // order them before the producer's next bulk copy into the slot
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->empty[s]);
    }
    return;
  }

  // One pass of lpr lanes per row over rpp rows: chunk loop, lane reduction,
  // rescale and store (every lane takes part in the shuffles).
  auto row_pass = [&](const uint8_t* wrow, bool valid, int n) {
    int acc[MT][4];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[m][q] = 0;
    if (valid) {
      int c = sub + rot;
      if (c >= cpr) c -= cpr;
#pragma unroll 2
      for (int i = 0; i < cpl; ++i) {
        const uint4 wv = *reinterpret_cast<const uint4*>(wrow + c * 16);
        const unsigned wd[4] = {wv.x, wv.y, wv.z, wv.w};
        const int8_t* xb = xq + (c << 4);
#pragma unroll
        for (int sl = 0; sl < 4; ++sl) {
          const unsigned mask = 0xC0C0C0C0u >> (2 * sl);
          const unsigned m0 = wd[0] & mask, m1 = wd[1] & mask, m2 = wd[2] & mask, m3 = wd[3] & mask;
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            if (m < M) {
              const int4 xv = *reinterpret_cast<const int4*>(xb + m * K + sl * slot_stride);
              int a = acc[m][sl];
              a = dp4a_us(m0, xv.x, a);
              a = dp4a_us(m1, xv.y, a);
              a = dp4a_us(m2, xv.z, a);
              a = dp4a_us(m3, xv.w, a);
              acc[m][sl] = a;
            }
          }
        }
        c += lpr;
        if (c >= cpr) c -= cpr;
      }
    }
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
  };

  if (nst <= nslots) {
    // Every stage of this CTA is in the ring at once (no slot is reused): wait
    // for all of them, then share the CTA's rows among the warps as one list,
    // with no per-stage hand-back.
    for (int st = 0; st < nst; ++st)
      if (!mbar_wait(&tail->full[st], 0, err, &tail->abort_flag)) return;
    const int R = r1 - r0;
    for (int base = warp * rpp; base < R; base += kDecWarps * rpp) {
      const int r = base + lane / lpr;
      const int st = r / rps;
      row_pass(ring + st * sbytes + (r - st * rps) * row_bytes, r < R, r0 + r);
    }
    return;
  }

  for (int st = 0; st < nst; ++st) {
    const int s = st % nslots;
    if (!mbar_wait(&tail->full[s], (st / nslots) & 1, err, &tail->abort_flag)) break;
    const uint8_t* stage = ring + s * sbytes;
    const int rows = min(rps, r1 - r0 - st * rps);
    for (int base = warp * rpp; base < rows; base += kDecWarps * rpp) {
      const int r = base + lane / lpr;
      row_pass(stage + r * row_bytes, r < rows, r0 + st * rps + r);
    }
    // the stage's loads are complete (their values fed the dot products);
    // order them before the producer's next bulk copy into the stage
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[s]);
  }
}

template <int MT, bool kFused, bool kLong, bool kGlu>
cudaError_t launch_decode_t(const DecodeParams& P, int grid, size_t smem, bool pdl, unsigned* err, cudaStream_t s) {
  auto kern = k_decode<MT, kFused, kLong, kGlu>;
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

template <bool kFused, bool kLong, bool kGlu = false>
cudaError_t dispatch_m(int mt, const DecodeParams& P, int grid, size_t smem, bool pdl, unsigned* err,
                       cudaStream_t s) {
  switch (mt) {
    case 1: return launch_decode_t<1, kFused, kLong, kGlu>(P, grid, smem, pdl, err, s);
    case 2: return launch_decode_t<2, kFused, kLong, kGlu>(P, grid, smem, pdl, err, s);
    case 4: return launch_decode_t<4, kFused, kLong, kGlu>(P, grid, smem, pdl, err, s);
    default: return launch_decode_t<8, kFused, kLong, kGlu>(P, grid, smem, pdl, err, s);
  }
}

}  // namespace

bool decode_supported(int64_t M, int64_t K) {
  return M >= 1 && M <= kDecodeMaxM && M * K <= kDecodeMaxCodeBytes;
}

bool decode_split_preferred(int64_t M, int64_t K) {
  return decode_supported(M, K) && K > 16384 && K % 2048 == 0;
}

bool decode_fused_glu_supported(int64_t M, int64_t K) {
  return M >= 1 && M <= kDecodeMaxM && K <= 16384 && !decode_split_preferred(M, K) &&
         register_prologue(true, static_cast<int>(K), static_cast<int>(M)) && decode_supported(M, K);
}

bool decode_fused_supported(int64_t M, int64_t K) {
  if (M < 1 || M > kDecodeMaxM) return false;
  if (K <= 16384 && register_prologue(true, static_cast<int>(K), static_cast<int>(M))) return decode_supported(M, K);
  return 5 * M * K + 4 * K <= kDecodeFusedMaxStageBytes;
}

cudaError_t launch_decode(const DeviceContext* ctx, const DecodeJob* jobs_in, int njobs, int M, float eps, bool fused,
                          bool weights_static, cudaStream_t s, int reserve_sms) {
  if (njobs < 1 || njobs > BITNET_MAX_GROUP) return cudaErrorInvalidValue;
  if (njobs == 1 && fused && jobs_in[0].act == 0 && gemv_row1_supported(M, jobs_in[0].K))
    return launch_gemv_row1(ctx, jobs_in[0], eps, weights_static, s);
  // Projections with the longest rows (the longest prologues) take the lowest
  // CTA indices: the CTAs dispatched last start latest, and the launch ends
  // with its slowest CTA.  Each projection's outputs do not depend on the order.
  DecodeJob jobs[BITNET_MAX_GROUP];
  for (int i = 0; i < njobs; ++i) jobs[i] = jobs_in[i];
  for (int i = 1; i < njobs; ++i)
    for (int j = i; j > 0 && jobs[j].K > jobs[j - 1].K; --j) {
      const DecodeJob t = jobs[j];
      jobs[j] = jobs[j - 1];
      jobs[j - 1] = t;
    }
  DecodeParams P = {};
  P.nproj = njobs;
  P.M = M;
  P.eps = eps;
  P.weights_static = weights_static ? 1 : 0;
  double total = 0.0;
  int maxK = 0;
  for (int i = 0; i < njobs; ++i) {
    total += static_cast<double>(jobs[i].N) * jobs[i].K;
    maxK = jobs[i].K > maxK ? jobs[i].K : maxK;
  }
  // One CTA per SM in total (never a second wave, and room for the next
  // dependent launch to become resident early), apportioned to the
  // projections by weight bytes with the largest-remainder rule.
  const int avail = ctx->num_sms - reserve_sms;
  int target = avail > njobs ? avail : njobs;
  int want[BITNET_MAX_GROUP];
  double frac[BITNET_MAX_GROUP];
  int used = 0;
  for (int i = 0; i < njobs; ++i) {
    const double q = target * (static_cast<double>(jobs[i].N) * jobs[i].K) / total;
    want[i] = static_cast<int>(q);
    if (want[i] < 1) want[i] = 1;
    frac[i] = q - static_cast<int>(q);
    used += want[i];
  }
  while (used < target) {
    int best = -1;
    for (int i = 0; i < njobs; ++i)
      if (want[i] < jobs[i].N && (best < 0 || frac[i] > frac[best])) best = i;
    if (best < 0) break;
    ++want[best];
    frac[best] = -1.0;
    ++used;
  }
  int cta = 0;
  for (int i = 0; i < njobs; ++i) {
    const DecodeJob& j = jobs[i];
    int w = want[i] > j.N ? j.N : want[i];
    const int rpc = (j.N + w - 1) / w;
    const int n_ctas = (j.N + rpc - 1) / rpc;
    DecodeProj& p = P.p[i];
    p.x = j.x;
    p.up = j.up;
    p.act = j.act;
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
  const int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;
  // Short rows: three 24 KB stages when no CTA streams more than three of them
  // (the latency-bound case: small enough for two CTAs per SM, so the next
  // dependent launch can become resident early), six for long streams (more
  // bytes in flight per SM) when shared memory allows.  Long rows: all the
  // shared memory left after the activations, as 4 KB (or one-row) slots.
  bool lng = false;
  int max_stages = 1;
  for (int i = 0; i < njobs; ++i) {
    const int cpr = jobs[i].K / 64;
    if (cpr >= 64 && cpr % 32 == 0) lng = true;
    const int rps = kDecStageBytes / (jobs[i].K / 4);
    const int nst = (P.p[i].rows_per_cta + rps - 1) / rps;
    max_stages = nst > max_stages ? nst : max_stages;
  }
  constexpr int kSmemMax = 227 * 1024;
  // the projections' layouts differ (staged or register prologue): size for the largest
  auto layout_total = [&](int ring) {
    int t = 0;
    for (int i = 0; i < njobs; ++i) {
      const int v = DecodeLayout(M, jobs[i].K, fused, ring).total;
      t = v > t ? v : t;
    }
    return t;
  };
  P.stages = 3;
  if (max_stages > 3 && layout_total(kDecMaxStages * kDecStageBytes) <= kSmemMax) P.stages = kDecMaxStages;
  P.ring_bytes = P.stages * kDecStageBytes;
  if (lng) {
    const int other = layout_total(0);
    int ring = (kSmemMax - other) & ~1023;
    ring = ring < kDecMaxSlots * kDecLongStageBytes ? ring : kDecMaxSlots * kDecLongStageBytes;
    // never smaller than the short-row ring of the same launch, and room for
    // at least two slots of the longest row
    const int min_ring = maxK / 4 * 2 > P.ring_bytes ? maxK / 4 * 2 : P.ring_bytes;
    P.ring_bytes = ring > min_ring ? ring : min_ring;
  }
  const size_t smem = static_cast<size_t>(layout_total(P.ring_bytes));
  if (smem > static_cast<size_t>(kSmemMax)) return cudaErrorInvalidConfiguration;  // unreachable with the dispatch limits
  const bool pdl = true;  // without prefetch permission every read waits for the previous kernel
  bool glu = false;
  for (int i = 0; i < njobs; ++i) glu = glu || jobs[i].act != 0;
  if (glu && !fused) return cudaErrorInvalidValue;  // the activation runs in the fused prologue only
  if (lng) {
    if (glu) return dispatch_m<true, true, true>(mt, P, cta, smem, pdl, ctx->err_word, s);
    return fused ? dispatch_m<true, true>(mt, P, cta, smem, pdl, ctx->err_word, s)
                 : dispatch_m<false, true>(mt, P, cta, smem, pdl, ctx->err_word, s);
  }
  if (glu) return dispatch_m<true, false, true>(mt, P, cta, smem, pdl, ctx->err_word, s);
  return fused ? dispatch_m<true, false>(mt, P, cta, smem, pdl, ctx->err_word, s)
               : dispatch_m<false, false>(mt, P, cta, smem, pdl, ctx->err_word, s);
}

}  // namespace bitnet
