// gemm_skinny.cu -- BitLinear contraction for a few tens of tokens (9..64) on
// the 5th-generation tensor cores, with the K dimension split across CTAs.
//
// acc[m, n] = sum_k q[m, k] * (code(n, k) - 1) (int8 activations x ternary
// weights, the product of ggml_vec_dot_i2_i8_s named in section 6.4 of "BitNet
// Embeddings GGUF Conversion Implementation"), then y = (acc / a_scale[m]) /
// w_scale in fp32 ("BitNet Inference Framework", "Quantization (W1.58A8)").
//
// With few tokens the weight stream is the cost, so the weights are the MMA's
// M side (128 rows per tile) and the tokens its N side (BN = 16, 32 or 64
// columns, all tokens in one tile): the MMA work is proportional to the real
// token count.  A weight matrix has only N/128 tiles, so the K dimension of
// each tile is split into S ranges of whole I2_S blocks; (tile, range) units
// are spread over one persistent CTA per SM.
//
// Exactness: operands are integers exact in fp16, every partial sum is an
// integer of magnitude <= 127 * K < 2^24, so the fp32 TMEM accumulator and the
// fp32 atomic additions that combine the S partial sums of a tile are exact,
// whatever their order.  The split that completes a tile (a per-tile ticket)
// rescales it: y = ((float)acc * (1/a_scale)) * (1/w_scale).
//
// One stage = one I2_S block column (128 values of K) of the tile:
//   warp 20    TMA producer: the tokens' fp16 codes of TG consecutive stages
//              (2 TG 64-wide slabs of BN rows, 128-byte swizzle) in one copy, a
//              3-D view of the [M, K] codes (64 values, token, 64-value slab),
//              into a 96 KB ring of their own: a TMA copy has a fixed cost of
//              its own (measured on sm_103a: 2 KB boxes of 16 rows from L2
//              arrive at ~25 GB/s per SM, 16 KB boxes at ~94), which with one
//              copy per 2 KB slab set the stage rate; the tile's packed bytes
//              arrive in groups of 4 block columns (128 rows x 128 contiguous
//              bytes, 128-byte swizzle, so that 8 consecutive rows read their
//              columns from 8 different bank groups) into a ring of 6 slots
//              (96 KB in flight per SM keeps the HBM stream busy); K is split
//              in whole groups
//   two stage pipelines, j = 0, 1, take the stages of even and odd running
//   index (over the CTA's units) in turn, each with
//     8 unpack warps (warps 8j .. 8j+7): warp w holds weight rows 32 (w % 4)
//              .. + 31 (the TMEM lanes it may write) and half (w % 8) / 4 of
//              each block's bytes, and turns them into the MMA's A operand
//              directly in tensor memory (fp16 pairs, one tcgen05.st of 32
//              columns per thread and stage): the weights never pass through
//              shared memory as fp16, which is 16x the bytes of their packed
//              form
//     1 MMA warp (warp 21 + j): one lane issues tcgen05.mma (M=128, N=BN,
//              K=16, A from TMEM), 8 per stage, into the pipeline's own
//              accumulator, from its own two A stages of 64 TMEM columns
//   A stage is a chain of dependent steps (shared-memory load, unpack, wait
//   for a free A stage, tensor-memory store and its wait, fences, arrival,
//   the MMA thread's wait, MMAs, commit) that leaves the SM's pipes mostly
//   idle (measured on sm_103a: ~1200 cycles per stage for one pipeline, ALU
//   pipe 39% busy); two pipelines overlap two such chains.  Warp 21 also
//   allocates all 512 TMEM columns (4 accumulators, then the A stages).
//   warps 16-19 epilogue: warp q reads TMEM lanes 32q..32q+31 = 32 weight rows
//              of both pipelines' accumulators and adds them (integers below
//              2^24: exact); each thread owns one weight row, so for every
//              token the warp writes (or atomically adds) 32 consecutive
//              outputs
// The eight MMAs of a stage take the block's K values in the order (slot s,
// half h) = (t mod 4, t / 4), t = 0..7: A stage columns 32 h + 8 s .. + 7 hold
// elements 32 s + 16 h + 0..15 (so each unpack thread writes 32 consecutive
// columns), and the token operand of step t starts at element 32 s + 16 h.
// Every wait is bounded; an expired wait sets the device error word and the CTA
// unwinds without trapping.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"
#include "unpack_f16.cuh"

namespace bitnet {
namespace {

constexpr int kSkPipes = 2;                                  // stage pipelines (running stage index mod 2)
constexpr int kSkPipeWarps = 8;                              // unpack warps per pipeline
constexpr int kSkUnpackWarps = kSkPipes * kSkPipeWarps;      // warps 0 .. 15
constexpr int kSkEpiWarp0 = kSkUnpackWarps;                  // warps 16 .. 19
constexpr int kSkProducerWarp = kSkEpiWarp0 + 4;             // warp 20
constexpr int kSkMmaWarp0 = kSkProducerWarp + 1;             // warps 21, 22
constexpr int kSkThreads = (kSkMmaWarp0 + kSkPipes) * 32;
constexpr int kSkBM = 128;  // weight rows per tile (MMA M)
constexpr int kSkAPerPipe = 2;                    // A operand stages in TMEM per pipeline
constexpr int kSkAStages = kSkPipes * kSkAPerPipe;
constexpr int kSkAStageCols = 64;  // TMEM columns per stage: 128 K values as fp16 pairs
constexpr int kSkTmemCols = 512;   // accumulator of buffer a, pipeline j at columns (2 a + j) BN; A stages from kSkACol0
constexpr int kSkACol0 = 256;

constexpr int kSkPkGroup = 4;  // block columns per packed-weight load: 128 bytes per row

template <int BN>
struct SkLayout {
  static constexpr int kPkSlots = 6;
  static constexpr int kPk = kSkBM * 32 * kSkPkGroup;  // packed bytes of a slot: 128 rows x 128 B
  static constexpr int kB = 2 * BN * 64 * 2;           // a stage's two 64-wide fp16 slabs of the tokens
  static constexpr int kTG = BN == 64 ? 2 : 4;         // stages per token copy (a divisor of kSkPkGroup)
  static constexpr int kTSlot = kTG * kB;              // bytes of a token slot
  static constexpr int kTSlots = (96 * 1024) / kTSlot; // token slots
  static constexpr int offB = 0;                           // [token slots][kTG stages][kB]
  static constexpr int offPk = offB + kTSlots * kTSlot;    // [packed slots][kPk]
  static constexpr int offInv = offPk + kPkSlots * kPk;    // [BN] float: 1 / a_scale
  static constexpr int kNumBars = 2 * kSkAStages + 2 * kTSlots + 2 * kPkSlots + 4;
  static constexpr int offBar = offInv + BN * 4;
  static constexpr int offMisc = offBar + kNumBars * 8;  // tmem base, abort flag, last flag
  static constexpr int kBytes = offMisc + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kTSlots >= 3 && kSkPkGroup % kTG == 0, "token ring too shallow");
  static_assert(kB % 1024 == 0 && kPk % 1024 == 0, "swizzled operands need 1 KB alignment");
  static_assert(kAlloc <= 232448, "over the 227 KB of shared memory a CTA may use");
  static_assert(2 * kSkPipes * BN <= kSkACol0 && kSkACol0 + kSkAStages * kSkAStageCols <= kSkTmemCols,
                "TMEM columns");
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Unit u = (weight tile, K range): the tile's I2_S blocks [kb0, kb1), whole
// groups of kSkPkGroup blocks (the last one cut at K).  The i-th block a unit
// processes is kb0 + (i + rot) mod (kb1 - kb0), rot a whole number of groups
// that depends on the tile: the CTAs working on one K range at the same time
// then read its token codes in different orders, instead of all requesting
// the same L2 lines at once (the sums are order-free integers).
struct SkUnit {
  int wt, kb0, kb1, rot;
  __device__ __forceinline__ int len() const { return kb1 - kb0; }
  __device__ __forceinline__ int kb(int i) const {
    const int j = i + rot;
    return kb0 + (j < len() ? j : j - len());
  }
};
__device__ __forceinline__ SkUnit sk_unit(int u, int S, int nkb) {
  const int ngrp = (nkb + kSkPkGroup - 1) / kSkPkGroup;
  SkUnit r;
  r.wt = u / S;
  const int ks = u - r.wt * S;
  r.kb0 = kSkPkGroup * static_cast<int>((static_cast<int64_t>(ngrp) * ks) / S);
  r.kb1 = min(nkb, kSkPkGroup * static_cast<int>((static_cast<int64_t>(ngrp) * (ks + 1)) / S));
  const int len = r.kb1 - r.kb0;
  r.rot = len % kSkPkGroup == 0 ? kSkPkGroup * (r.wt % (len / kSkPkGroup)) : 0;
  return r;
}

template <int BN>
__global__ void __launch_bounds__(kSkThreads, 1)
    k_gemm_skinny(const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_w,
                  const float* __restrict__ a_scale, float inv_w, int M, int N, int K, int S,
                  float* __restrict__ y, int32_t* __restrict__ acc_out, float* __restrict__ ws,
                  int* __restrict__ tickets, unsigned* err) {
  using L = SkLayout<BN>;
  constexpr int kTS = L::kTSlots;
  constexpr int kTG = L::kTG;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sB = smem + L::offB;
  uint8_t* sPk = smem + L::offPk;
  float* sInv = reinterpret_cast<float*>(smem + L::offInv);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
  uint64_t* afull = bars;                  // A stage written to TMEM (and the stage's tokens landed)
  uint64_t* aempty = bars + kSkAStages;    // MMAs reading the A stage done
  uint64_t* tfull = bars + 2 * kSkAStages; // token slabs of a slot landed
  uint64_t* tempty = tfull + kTS;          // MMAs of every stage of the token slot done
  uint64_t* pk_full = tempty + kTS;        // packed group landed
  uint64_t* pk_empty = pk_full + L::kPkSlots;
  uint64_t* acc_full = pk_empty + L::kPkSlots;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = K >> 7;
  const int n_wt = (N + kSkBM - 1) / kSkBM;
  const int units = n_wt * S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kSkAStages; ++i) {
      mbar_init(&afull[i], kSkPipeWarps);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < kTS; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kTG);
    }
    for (int i = 0; i < L::kPkSlots; ++i) {
      mbar_init(&pk_full[i], 1);
      mbar_init(&pk_empty[i], kSkUnpackWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], kSkPipes);
      mbar_init(&acc_empty[i], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kSkMmaWarp0) {
    tmem_alloc(tmem_slot, kSkTmemCols);
    tmem_relinquish();
  }
  if (warp == kSkProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_tok);
    prefetch_tensormap(&tm_w);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // everything below reads what the previous kernel on the stream produced
  pdl_wait();

  if (warp == kSkProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0, ph = 0, p = 0, pph = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const SkUnit w = sk_unit(u, S, nkb);
        for (int i = 0; i < w.len(); ++i) {
          const int kb = w.kb(i);
          if (i % kSkPkGroup == 0) {
            // the next group of packed block columns (columns past K read as 0)
            if (!mbar_wait(&pk_empty[p], pph ^ 1, err, abort_flag)) goto producer_done;
            mbar_arrive_expect_tx(&pk_full[p], static_cast<unsigned>(L::kPk));
            tma_load_2d(sPk + p * L::kPk, &tm_w, kb * 32, w.wt * kSkBM, &pk_full[p]);
            if (++p == L::kPkSlots) { p = 0; pph ^= 1; }
          }
          if (i % kTG == 0) {
            // slabs 2 kb .. 2 (kb + kTG) - 1: the stages of a token slot have
            // consecutive block columns (rotations are whole packed groups);
            // slabs past K read as 0
            if (!mbar_wait(&tempty[s], ph ^ 1, err, abort_flag)) goto producer_done;
            mbar_arrive_expect_tx(&tfull[s], static_cast<unsigned>(L::kTSlot));
            tma_load_3d(sB + s * L::kTSlot, &tm_tok, 0, 0, 2 * kb, &tfull[s]);
            if (++s == kTS) { s = 0; ph ^= 1; }
          }
        }
      }
    producer_done:;
    }
  } else if (warp >= kSkMmaWarp0) {
    // -------------------------------------------------------- MMA issuers
    // pipeline j issues the stages of running index g = j mod 2; it walks
    // every stage to keep its place in the token ring
    if (lane == 0) {
      const int j = warp - kSkMmaWarp0;
      constexpr uint32_t idesc = idesc_f16_f32(kSkBM, BN);
      int n = 0, b = 0, g = 0, tl = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x, ++tl) {
        const SkUnit w = sk_unit(u, S, nkb);
        const int a = tl & 1;
        // also keeps a pipeline without stages in this unit from arriving on
        // acc_full ahead of the epilogue
        if (!mbar_wait(&acc_empty[a], ((tl >> 1) & 1) ^ 1, err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((kSkPipes * a + j) * BN);
        bool ok = true, any = false;
        for (int i = 0; i < w.len(); ++i, ++g) {
          if ((g & 1) == j) {
            const int s = kSkAPerPipe * j + n % kSkAPerPipe;
            if (!mbar_wait(&afull[s], (n / kSkAPerPipe) & 1, err, abort_flag)) {  // also covers the token slot
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(kSkACol0 + s * kSkAStageCols);
            const uint8_t* btok = sB + b * L::kTSlot + (i % kTG) * L::kB;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const int sl = t & 3, hh = t >> 2;
              const uint64_t bdesc = sw128_kmajor_desc(smem_u32(btok + (sl >> 1) * (L::kB / 2))) +
                                     static_cast<uint64_t>(2 * (2 * (sl & 1) + hh));
              tc_mma_f16_ta(d_tmem, a_tmem + static_cast<uint32_t>(8 * t), bdesc, idesc, (any || t) ? 1u : 0u);
            }
            any = true;
            tc_commit(&aempty[s]);
            tc_commit(&tempty[b]);
            // a unit's last token slot may hold fewer than kTG of its stages:
            // arrive for the missing ones (the slot is released once the
            // commits of the stages it does hold have arrived as well)
            if (i == w.len() - 1)
              for (int r = i % kTG + 1; r < kTG; ++r) mbar_arrive(&tempty[b]);
            ++n;
          }
          if (i % kTG == kTG - 1 || i == w.len() - 1)
            if (++b == kTS) b = 0;
        }
        if (!ok) break;
        if (any) tc_commit(&acc_full[a]);
        else mbar_arrive(&acc_full[a]);
      }
    }
  } else if (warp < kSkUnpackWarps) {
    // --------------------------------------------------------------- unpack
    const int pj = warp / kSkPipeWarps;  // pipeline: stages of running index pj mod 2
    const int q = warp & 3;              // TMEM lane quadrant: weight rows 32q .. 32q + 31
    const int hf = (warp & 7) >> 2;      // half of each block's 32 bytes
    const int row = 32 * q + lane;       // weight row of the tile
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                        static_cast<uint32_t>(kSkACol0 + 32 * hf);
    int n = 0, p = 0, pph = 0, b = 0, bph = 0, g = 0;
    bool pk_ready = false;  // the current packed group has been waited for
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const SkUnit w = sk_unit(u, S, nkb);
      for (int i = 0; i < w.len(); ++i, ++g) {
        const int gi = i % kSkPkGroup;  // column within the packed group (groups stay whole)
        if ((g & 1) == pj) {
          if (!pk_ready && !mbar_wait(&pk_full[p], pph, err, abort_flag)) goto unpack_done;
          pk_ready = true;
          // chunk 2 gi + hf of the row (stored at chunk c ^ (row & 7))
          const uint4 u4 = *reinterpret_cast<const uint4*>(sPk + p * L::kPk + row * 128 +
                                                             (((2 * gi + hf) ^ (row & 7)) << 4));
          uint32_t cols[32];
          unpack_half_block_cols(u4, cols);
          const int s = kSkAPerPipe * pj + n % kSkAPerPipe;
          // the MMAs of the A stage's previous use must be done with it
          if (!mbar_wait(&aempty[s], ((n / kSkAPerPipe) & 1) ^ 1, err, abort_flag)) goto unpack_done;
          tc_fence_after();
          __syncwarp();
          tmem_st_32x32b_x32(tq + static_cast<uint32_t>(s * kSkAStageCols), cols);
          tmem_st_wait();
          tc_fence_before();
          // the packed bytes are consumed: order the reads before the next TMA
          // into the slot
          fence_proxy_async_smem();
          // afull also tells the MMA thread that the stage's token slabs have
          // landed: it then waits on one barrier per stage instead of two
          if (!mbar_wait(&tfull[b], bph, err, abort_flag)) goto unpack_done;
          __syncwarp();
          if (lane == 0) mbar_arrive(&afull[s]);
          ++n;
        }
        if (i % kTG == kTG - 1 || i == w.len() - 1)
          if (++b == kTS) { b = 0; bph ^= 1; }
        // every unpack warp of both pipelines releases the packed group once
        // it is past the group's last stage
        if (gi == kSkPkGroup - 1 || i == w.len() - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&pk_empty[p]);
          if (++p == L::kPkSlots) { p = 0; pph ^= 1; }
          pk_ready = false;
        }
      }
    }
  unpack_done:;
  } else {
    // ------------------------------------------------------------- epilogue
    const int et = threadIdx.x - kSkEpiWarp0 * 32;  // 0..127
    const int q = warp & 3;            // TMEM lane quadrant this warp may access
    for (int j = et; j < BN; j += 128) sInv[j] = j < M ? __frcp_rn(__ldg(a_scale + j)) : 0.0f;
    epi_bar();
    int tl = 0, g0 = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++tl) {
      const SkUnit w = sk_unit(u, S, nkb);
      const int a = tl & 1;
      const int n = w.wt * kSkBM + q * 32 + lane;  // this thread's weight row
      const bool n_ok = n < N;
      // pipelines with a stage in this unit (running indices g0 .. g0 + len - 1)
      const bool act0 = w.len() >= 2 || (g0 & 1) == 0;
      const bool act1 = w.len() >= 2 || (g0 & 1) == 1;
      g0 += w.len();
      if (!mbar_wait_idle(&acc_full[a], (tl >> 1) & 1, err, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(kSkPipes * a * BN);
      // 16 tokens at a time: y (one split) or the partial sum (several splits;
      // exact fp32 atomic additions)
#pragma unroll 1
      for (int j0 = 0; j0 < BN && j0 < M; j0 += 16) {
        // the sum of the pipelines' accumulators (integers below 2^24: exact)
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll 1
        for (int pj = 0; pj < kSkPipes; ++pj) {
          if (!(pj == 0 ? act0 : act1)) continue;
          uint32_t r[16];
          tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(pj * BN + j0), r);
          tmem_ld_wait();
          tmem_reg_fence16(r);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(r[i]);
        }
        if (n_ok) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int j = j0 + i;
            if (j < M) {
              const float accf = acc[i];
              if (S == 1) {
                y[static_cast<int64_t>(j) * N + n] = rescale_elem(accf, sInv[j], inv_w);
                if (acc_out) acc_out[static_cast<int64_t>(j) * N + n] = __float2int_rn(accf);
              } else {
                red_add_f32(ws + static_cast<int64_t>(j) * N + n, accf);
              }
            }
          }
        }
      }
      // the accumulator has been read: release it to the MMAs of a later unit
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
      if (S == 1) continue;
      // the split that brings the tile's ticket to S writes the tile
      __threadfence();
      epi_bar();
      if (et == 0) *last_flag = atomicAdd(&tickets[w.wt], 1) == S - 1;
      epi_bar();
      if (*last_flag) {
        __threadfence();
        if (n_ok) {
          for (int j = 0; j < M && j < BN; ++j) {
            const float accf = __ldcg(ws + static_cast<int64_t>(j) * N + n);
            y[static_cast<int64_t>(j) * N + n] = rescale_elem(accf, sInv[j], inv_w);
            if (acc_out) acc_out[static_cast<int64_t>(j) * N + n] = __float2int_rn(accf);
          }
        }
      }
      epi_bar();  // last_flag is rewritten by the next unit
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSkMmaWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kSkTmemCols);
  }
}

// Number of K splits: the one with the least estimated time, which is the
// busiest CTA's stages plus, with a split, the epilogues' fp32 atomic
// additions (M N S of them, a throughput the whole GPU shares) and the per-unit
// ticket and read-back.  Fitted to GB300 timings of this kernel with forced
// split counts: ~0.5 us per stage, ~85 atomic additions per ns, ~1 us per
// split unit (M = 63, K = N = 16384: 70 us unsplit, 89 / 121 / 182 us with
// S = 2 / 4 / 8, where a count of stages alone picks 8).  Ties go to fewer
// splits.
int choose_splits(int64_t M, int n_wt, int nkb, int64_t N, int ctas) {
  constexpr double kStageNs = 500.0, kAtomicsPerNs = 85.0, kSplitUnitNs = 1000.0;
  const int ngrp = (nkb + kSkPkGroup - 1) / kSkPkGroup;
  int best = 1;
  double best_cost = 0.0;
  const int max_s = ngrp < 64 ? ngrp : 64;
  for (int S = 1; S <= max_s; ++S) {
    const int64_t units = static_cast<int64_t>(n_wt) * S;
    const int64_t per_cta = (units + ctas - 1) / ctas;
    double cost = static_cast<double>(per_cta) * kSkPkGroup * ((ngrp + S - 1) / S) * kStageNs;
    if (S > 1)
      cost += static_cast<double>(M) * static_cast<double>(N) * S / kAtomicsPerNs +
              static_cast<double>(per_cta) * kSplitUnitNs;
    if (S == 1 || cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

template <int BN>
cudaError_t launch_bn(const DeviceContext* ctx, EncodeTiledFn encode, const __half* codes_f16, const float* a_scale,
                      const uint8_t* packed_w, float inv_w, int M, int K, int N, int S, float* y, int32_t* acc_out,
                      float* ws, int* tickets, bool pdl, cudaStream_t s, int* status) {
  using L = SkLayout<BN>;
  CUtensorMap tm_tok, tm_w;
  {
    // tokens: fp16 [M, K] viewed as (64 values, token, 64-value slab): boxes of
    // 64 values x BN tokens x 2 kTG slabs, each slab a swizzled BN x 128 B
    // block (tokens >= M and slabs past K read as 0)
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BN), static_cast<cuuint32_t>(2 * L::kTG)};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = encode(&tm_tok, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(codes_f16), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *status = BITNET_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  {
    // packed weights: bytes [N, K/4]; boxes of 4 block columns (128 B) x 128 rows
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 4), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 4)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(32 * kSkPkGroup), static_cast<cuuint32_t>(kSkBM)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed_w), dims, strides, box,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *status = BITNET_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  auto kern = k_gemm_skinny<BN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int units = ((N + kSkBM - 1) / kSkBM) * S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units < ctx->num_sms ? units : ctx->num_sms);
  cfg.blockDim = dim3(kSkThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_tok, tm_w, a_scale, inv_w, M, N, K, S, y, acc_out, ws, tickets,
                            ctx->err_word);
}

}  // namespace

// Used for 9..63 tokens when the weight stream is long enough to pay for the
// split's extra work (zeroing the partial sums, a final pass per tile); below
// that (K <= 2048 and N <= 8192, a few us) the tokens-as-M kernel is faster.
// From 64 tokens on the tokens-as-M kernel is used: its tiles hold 128 tokens,
// so its time hardly depends on the count.  Measured on GB300 at
// K = N = 16384: 67 / 69 / 70 us for 16 / 32 / 63 tokens here against 78-79 us
// there.
bool gemm_skinny_supported(int64_t M, int64_t K, int64_t N) {
  return M > kDecodeMaxM && M < 64 && K >= 128 && K % 128 == 0 && N >= 1 && (K >= 4096 || N >= 16384);
}

size_t gemm_skinny_workspace(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N) {
  const int n_wt = static_cast<int>((N + kSkBM - 1) / kSkBM);
  const int S = choose_splits(M, n_wt, static_cast<int>(K >> 7), N, ctx->num_sms);
  if (S == 1) return 0;
  return ((static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~size_t(255)) +
         static_cast<size_t>(n_wt) * 4;
}

cudaError_t launch_gemm_skinny(const DeviceContext* ctx, const __half* codes_f16, const float* a_scale,
                               const uint8_t* packed_w, float w_scale, int64_t M, int64_t K, int64_t N, float* y,
                               int32_t* acc_out, void* workspace, bool workspace_zeroed, bool pdl, cudaStream_t s,
                               int* status) {
  *status = BITNET_OK;
  EncodeTiledFn encode = encode_tiled_fn();
  if (!encode) {
    *status = BITNET_ERR_CUDA;
    return cudaErrorNotSupported;
  }
  const float inv_w = 1.0f / w_scale;  // IEEE division, as in the oracle
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const int n_wt = (n + kSkBM - 1) / kSkBM;
  const int S = choose_splits(M, n_wt, k >> 7, N, ctx->num_sms);
  float* ws = nullptr;
  int* tickets = nullptr;
  if (S > 1) {
    // the partial sums are added into a zeroed fp32 [M, N] array
    const size_t ws_bytes = (static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~size_t(255);
    ws = static_cast<float*>(workspace);
    tickets = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + ws_bytes);
    if (!workspace_zeroed) {
      cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes + static_cast<size_t>(n_wt) * 4, s);
      if (e != cudaSuccess) return e;
    }
  }
  const int bn = m <= 16 ? 16 : m <= 32 ? 32 : 64;
  switch (bn) {
    case 16:
      return launch_bn<16>(ctx, encode, codes_f16, a_scale, packed_w, inv_w, m, k, n, S, y, acc_out, ws, tickets,
                           pdl, s, status);
    case 32:
      return launch_bn<32>(ctx, encode, codes_f16, a_scale, packed_w, inv_w, m, k, n, S, y, acc_out, ws, tickets,
                           pdl, s, status);
    default:
      return launch_bn<64>(ctx, encode, codes_f16, a_scale, packed_w, inv_w, m, k, n, S, y, acc_out, ws, tickets,
                           pdl, s, status);
  }
}

}  // namespace bitnet
