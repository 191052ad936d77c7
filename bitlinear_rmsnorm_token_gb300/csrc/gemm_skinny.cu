// gemm_skinny.cu -- BitLinear contraction for a few tens of tokens (9..63) on
// the 5th-generation tensor cores with 8-bit operands, the K dimension split
// across CTAs where that pays.
//
// acc[m, n] = sum_k q[m, k] * (code(n, k) - 1) (int8 activations x ternary
// weights, the product of ggml_vec_dot_i2_i8_s named in section 6.4 of "BitNet
// Embeddings GGUF Conversion Implementation"), then y = (acc / a_scale[m]) /
// w_scale in fp32 ("BitNet Inference Framework", "Quantization (W1.58A8)").
//
// With few tokens the weight stream is the cost, so the weights are the MMA's
// M side (128 rows per tile) and the tokens its N side (all tokens in one
// tile): the MMA work is proportional to the real token count.  A weight
// matrix has only N/128 tiles, so the K dimension of each tile may be split
// into S ranges of whole I2_S blocks; (tile, range) units are spread over one
// persistent CTA per SM.
//
// Operands (tcgen05 kind::f8f6f4, e4m3 x e4m3, fp32 accumulation):
//   weights: the 2-bit code c in {0, 1, 2} itself as an e4m3 byte, the
//     subnormal c * 2^-9 (a shift and an AND per four weights);
//   tokens: each int8 code written as q = 16 hi + lo with hi = floor(q / 16)
//     in [-8, 7] and lo = q mod 16 in [0, 15], both exact e4m3 integers, in
//     two operand rows per token (row 2t: hi, row 2t + 1: lo).
// A token's two accumulator columns then hold D_hi = 2^-9 sum c hi and D_lo =
// 2^-9 sum c lo: multiples of 2^-9 below 2^12 in magnitude (K <= 65536), held
// exactly by the fp32 accumulator whatever the order of the additions
// (checked on GB300 with e4m3 subnormal operands and sums to 2^21 units), and
//     acc = 512 (16 D_hi + D_lo) - sum_k q[m, k]
// in exact integer arithmetic, the last term (the row sum of the codes)
// removing the +1 offset of the weight codes.  Partial sums of split tiles are
// integers below 2^24, combined with exact fp32 atomic additions.
//
// The planes (layout in planes.cuh) and the row sums come from the norm
// launch, or, for int8 codes given by the caller, from k_token_planes, which
// rewrites their fp16 copy in place (each 128-value block of a row, 256 bytes
// as fp16, becomes its 128 hi bytes then its 128 lo bytes) and sums the codes
// per 2048-value chunk.
//
// One stage = one I2_S block column (128 values of K) of the tile:
//   producer warp: the token planes of TG consecutive stages in one 4-D TMA
//              copy (128 bytes, plane, token, block) into a 96 KB ring (a TMA
//              copy has a fixed cost: measured on sm_103a, 2 KB boxes from L2
//              arrive at ~25 GB/s per SM, 16 KB boxes at ~94); the tile's
//              packed bytes in groups of 4 block columns (128 rows x 128
//              contiguous bytes, 128-byte swizzle: 8 consecutive rows read 8
//              different bank groups) into a ring of 6 slots (96 KB in flight
//              per SM keeps the HBM stream busy); K is split in whole groups
//   P stage pipelines (4; 3 for 48-token and 2 for 64-token tiles, whose
//   accumulators take more of the tensor memory) take the stages of running
//   index j mod P (over the CTA's units), each with
//     4 unpack warps: warp q holds weight rows 32q .. 32q + 31 (the TMEM lanes
//              it may write); each thread turns its row's 32 packed bytes into
//              the 32 TMEM columns of the A stage (column 8 s + c: the four
//              weights of slot s in bytes 4c .. 4c + 3, elements 32 s + 4c ..
//              + 3) with one tcgen05.st
//     1 MMA warp: one lane issues the stage's 4 MMAs (M = 128, N = 2 x token
//              tile, K = 32, A from TMEM; MMA s covers slot s) into the
//              pipeline's own accumulator
//   A stage is a chain of dependent steps (loads, unpack, tensor-memory store,
//   fences, barrier hand-offs, MMAs, commit) that leaves the SM's pipes idle
//   most of the time (one pipeline: ~1200 cycles per stage measured on
//   sm_103a), so several pipelines overlap their chains; each of these warps
//   visits only its own stages, ring positions following from running counts.
//   4 epilogue warps: warp q reads TMEM lanes 32q..32q+31 = 32 weight rows of
//              every pipeline's accumulator and adds them (exact integers);
//              each thread owns one weight row, so for every token the warp
//              writes (or atomically adds) 32 consecutive outputs
// Every wait is bounded; an expired wait sets the device error word and the CTA
// unwinds without trapping.
#include "common.cuh"
#include "internal.h"
#include "planes.cuh"
#include "rowquant.cuh"

namespace bitnet {
namespace {

constexpr int kSkBM = 128;         // weight rows per tile (MMA M)
constexpr int kSkAStageCols = 32;  // TMEM columns per A stage: 128 K values of one byte
constexpr int kSkTmemCols = 512;
constexpr int kSkPkGroup = 4;      // block columns per packed-weight load: 128 bytes per row

// BN: token tile (16, 32, 48 or 64 tokens); the MMA's N is 2 BN (two planes).
template <int BN>
struct SkLayout {
  static constexpr int kN2 = 2 * BN;                     // MMA N
  static constexpr int kPipes = BN == 64 ? 2 : BN == 48 ? 3 : 4;
  static constexpr int kUnpackWarps = 4 * kPipes;        // warps 0 .. 4P - 1
  static constexpr int kEpiWarp0 = kUnpackWarps;         // 4 warps
  static constexpr int kProducerWarp = kEpiWarp0 + 4;
  static constexpr int kMmaWarp0 = kProducerWarp + 1;    // P warps
  static constexpr int kThreads = (kMmaWarp0 + kPipes) * 32;
  // TMEM: accumulator of buffer a, pipeline j at columns (a P + j) 2 BN, then
  // the A stages
  static constexpr int kAccBufs = 2 * kPipes * kN2 <= 256 ? 2 : 1;
  static constexpr int kACol0 = kAccBufs * kPipes * kN2;
  static constexpr int kAStages = (kSkTmemCols - kACol0) / kSkAStageCols;
  static constexpr int kAPerPipe = kAStages / kPipes;
  static constexpr int kPkSlots = 6;
  static constexpr int kPk = kSkBM * 32 * kSkPkGroup;  // packed bytes of a slot: 128 rows x 128 B
  static constexpr int kB = kN2 * 128;                 // a stage's token rows (2 per token) of 128 B
  static constexpr int kTG = BN >= 48 ? 2 : 4;         // stages per token copy (a divisor of kSkPkGroup)
  static constexpr int kTSlot = kTG * kB;              // bytes of a token slot
  static constexpr int kTSlots = (96 * 1024) / kTSlot; // token slots
  static constexpr int offB = 0;                           // [token slots][kTG stages][kB]
  static constexpr int offPk = offB + kTSlots * kTSlot;    // [packed slots][kPk]
  static constexpr int offInv = offPk + kPkSlots * kPk;    // [BN] float: 1 / a_scale
  static constexpr int offRs = offInv + BN * 4;            // [BN] int: row sums of the codes
  static constexpr int kNumBars = 2 * kAStages + 2 * kTSlots + 2 * kPkSlots + 2 * kAccBufs;
  static constexpr int offBar = offRs + BN * 4;
  static constexpr int offMisc = offBar + kNumBars * 8;  // tmem base, abort flag, last flag
  static constexpr int kBytes = offMisc + 32;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kTSlots >= 3 && kSkPkGroup % kTG == 0, "token ring too shallow");
  static_assert(kB % 1024 == 0 && kPk % 1024 == 0, "swizzled operands need 1 KB alignment");
  static_assert(kAlloc <= 232448, "over the 227 KB of shared memory a CTA may use");
  static_assert(kAPerPipe >= 2 && kACol0 + kAStages * kSkAStageCols <= kSkTmemCols, "TMEM columns");
  static_assert(kThreads <= 1024, "block size");
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// One CTA per (token row, 2048-value chunk): the chunk's fp16 codes rewritten
// in place as the two e4m3 planes, block by block (a warp reads its two
// 256-byte blocks, both loads in flight, before writing them back), and the
// chunk's code sum in rowsum_part[m][chunk] (the epilogue adds a row's
// partials: integers, order-free).
constexpr int kPlaneThreads = 256;
constexpr int kPlaneChunk = 2048;  // values per CTA: 8 warps x 2 blocks of 128
__global__ void __launch_bounds__(kPlaneThreads) k_token_planes(__half* codes, int K, int* __restrict__ rowsum_part) {
  __shared__ int red[kPlaneThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* row = reinterpret_cast<uint8_t*>(codes) + static_cast<int64_t>(blockIdx.y) * K * 2;
  const int nkb = K >> 7;
  const int kb0 = blockIdx.x * (kPlaneChunk / 128) + 2 * warp;
  uint2 v[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    v[h] = kb0 + h < nkb ? *reinterpret_cast<const uint2*>(row + (kb0 + h) * 256 + lane * 8) : make_uint2(0u, 0u);
  __syncwarp();  // both blocks are read before any lane writes into them
  int sum = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (kb0 + h >= nkb) break;
    const __half2 h01 = *reinterpret_cast<const __half2*>(&v[h].x);
    const __half2 h23 = *reinterpret_cast<const __half2*>(&v[h].y);
    const int q[4] = {static_cast<int>(__low2float(h01)), static_cast<int>(__high2float(h01)),
                      static_cast<int>(__low2float(h23)), static_cast<int>(__high2float(h23))};
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      packed |= (static_cast<uint32_t>(q[i]) & 0xFFu) << (8 * i);
      sum += q[i];
    }
    uint32_t hi, lo;
    plane_words4(packed, hi, lo);
    uint8_t* blk = row + (kb0 + h) * 256;
    *reinterpret_cast<uint32_t*>(blk + lane * 4) = hi;
    *reinterpret_cast<uint32_t*>(blk + 128 + lane * 4) = lo;
  }
  sum = warp_sum_int(sum);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  if (warp == 0) {
    sum = warp_sum_int(lane < kPlaneThreads / 32 ? red[lane] : 0);
    if (lane == 0) rowsum_part[blockIdx.y * gridDim.x + blockIdx.x] = sum;
  }
}

__host__ __device__ constexpr int plane_chunks(int K) { return (K + kPlaneChunk - 1) / kPlaneChunk; }

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
__global__ void __launch_bounds__(SkLayout<BN>::kThreads, 1)
    k_gemm_skinny(const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_w,
                  const float* __restrict__ a_scale, const int* __restrict__ rowsum_part, int nparts, float inv_w,
                  int M, int N, int K, int S, float* __restrict__ y, int32_t* __restrict__ acc_out,
                  float* __restrict__ ws,
                  int* __restrict__ tickets, unsigned* err) {
  using L = SkLayout<BN>;
  constexpr int kP = L::kPipes;
  constexpr int kTS = L::kTSlots;
  constexpr int kTG = L::kTG;
  constexpr int kAS = L::kAStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* sB = smem + L::offB;
  uint8_t* sPk = smem + L::offPk;
  float* sInv = reinterpret_cast<float*>(smem + L::offInv);
  int* sRs = reinterpret_cast<int*>(smem + L::offRs);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
  uint64_t* afull = bars;                  // A stage written to TMEM (and the stage's tokens landed)
  uint64_t* aempty = bars + kAS;           // MMAs reading the A stage done
  uint64_t* tfull = bars + 2 * kAS;        // token planes of a slot landed
  uint64_t* tempty = tfull + kTS;          // MMAs of every stage of the token slot done
  uint64_t* pk_full = tempty + kTS;        // packed group landed
  uint64_t* pk_empty = pk_full + L::kPkSlots;
  uint64_t* acc_full = pk_empty + L::kPkSlots;  // every pipeline done with the unit
  uint64_t* acc_empty = acc_full + L::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = K >> 7;
  const int n_wt = (N + kSkBM - 1) / kSkBM;
  const int units = n_wt * S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAS; ++i) {
      mbar_init(&afull[i], 4);
      mbar_init(&aempty[i], 1);
    }
    for (int i = 0; i < kTS; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kTG);
    }
    for (int i = 0; i < L::kPkSlots; ++i) {
      mbar_init(&pk_full[i], 1);
      mbar_init(&pk_empty[i], L::kUnpackWarps);
    }
    for (int i = 0; i < L::kAccBufs; ++i) {
      mbar_init(&acc_full[i], kP);
      mbar_init(&acc_empty[i], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == L::kMmaWarp0) {
    tmem_alloc(tmem_slot, kSkTmemCols);
    tmem_relinquish();
  }
  if (warp == L::kProducerWarp && lane == 0) {
    prefetch_tensormap(&tm_tok);
    prefetch_tensormap(&tm_w);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // everything below reads what the previous kernels on the stream produced
  pdl_wait();

  if (warp == L::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0, ph = 0, p = 0, pph = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const SkUnit w = sk_unit(u, S, nkb);
        // the stages of a packed group (and of a token slot) have consecutive
        // block columns: rotations are whole groups
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
            // blocks kb .. kb + kTG - 1 of every token's two planes (tokens >=
            // M and blocks past K read as 0)
            if (!mbar_wait(&tempty[s], ph ^ 1, err, abort_flag)) goto producer_done;
            mbar_arrive_expect_tx(&tfull[s], static_cast<unsigned>(L::kTSlot));
            tma_load_4d(sB + s * L::kTSlot, &tm_tok, 0, 0, 0, kb, &tfull[s]);
            if (++s == kTS) { s = 0; ph ^= 1; }
          }
        }
      }
    producer_done:;
    }
  } else if (warp >= L::kMmaWarp0) {
    // -------------------------------------------------------- MMA issuers
    // pipeline j issues the stages of running index g = j mod P (over the
    // CTA's units); ring positions follow from the running counts of stages,
    // packed groups and token slots, so the loop visits its own stages only
    // (walking every stage put ~1000 cycles of loop overhead between two of a
    // warp's stages)
    if (lane == 0) {
      const int j = warp - L::kMmaWarp0;
      constexpr uint32_t idesc = idesc_e4m3_f32(kSkBM, L::kN2);
      int n = 0, g0 = 0, tg0 = 0, tl = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x, ++tl) {
        const SkUnit w = sk_unit(u, S, nkb);
        const int len = w.len();
        const int a = L::kAccBufs == 2 ? (tl & 1) : 0;
        const int use = L::kAccBufs == 2 ? (tl >> 1) : tl;  // earlier uses of buffer a
        // also keeps a pipeline without stages in this unit from arriving on
        // acc_full ahead of the epilogue
        if (!mbar_wait(&acc_empty[a], (use & 1) ^ 1, err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>((kP * a + j) * L::kN2);
        bool ok = true, any = false;
        for (int i = ((j - g0) % kP + kP) % kP; i < len; i += kP) {
          const int s = L::kAPerPipe * j + n % L::kAPerPipe;
          if (!mbar_wait(&afull[s], (n / L::kAPerPipe) & 1, err, abort_flag)) {  // also covers the tokens
            ok = false;
            break;
          }
          tc_fence_after();
          const int b = (tg0 + i / kTG) % kTS;
          const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(L::kACol0 + s * kSkAStageCols);
          const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + b * L::kTSlot + (i % kTG) * L::kB));
#pragma unroll
          for (int t = 0; t < 4; ++t)
            tc_mma_f8_ta(d_tmem, a_tmem + static_cast<uint32_t>(8 * t), bdesc + static_cast<uint64_t>(2 * t), idesc,
                         (any || t) ? 1u : 0u);
          any = true;
          tc_commit(&aempty[s]);
          tc_commit(&tempty[b]);
          // a unit's last token slot may hold fewer than kTG of its stages:
          // arrive for the missing ones (the slot is released once the
          // commits of the stages it does hold have arrived as well)
          if (i == len - 1)
            for (int r = i % kTG + 1; r < kTG; ++r) mbar_arrive(&tempty[b]);
          ++n;
        }
        if (!ok) break;
        if (any) tc_commit(&acc_full[a]);
        else mbar_arrive(&acc_full[a]);
        g0 += len;
        tg0 += (len + kTG - 1) / kTG;
      }
    }
  } else if (warp < L::kUnpackWarps) {
    // --------------------------------------------------------------- unpack
    // pipeline pj's stages, group by group; every unpack warp releases each
    // packed group once, after its own stages in it (a full group of 4 stages
    // holds 1 or 2 of every pipeline; a unit's short last group may hold none)
    const int pj = warp >> 2;            // pipeline: stages of running index pj mod P
    const int q = warp & 3;              // TMEM lane quadrant: weight rows 32q .. 32q + 31
    const int row = 32 * q + lane;       // weight row of the tile
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(L::kACol0);
    int n = 0, g0 = 0, pg0 = 0, tg0 = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const SkUnit w = sk_unit(u, S, nkb);
      const int len = w.len();
      const int ngroups = (len + kSkPkGroup - 1) / kSkPkGroup;
      int i = ((pj - g0) % kP + kP) % kP;  // this pipeline's first stage of the unit
      for (int G = 0; G < ngroups; ++G) {
        const int pidx = pg0 + G;
        const int p = pidx % L::kPkSlots;
        const int gend = min(kSkPkGroup * (G + 1), len);
        if (i < gend) {
          if (!mbar_wait(&pk_full[p], (pidx / L::kPkSlots) & 1, err, abort_flag)) goto unpack_done;
          for (; i < gend; i += kP) {
            const int gi = i - kSkPkGroup * G;  // column within the packed group
            // the row's 32 bytes of block column gi: chunks 2 gi, 2 gi + 1,
            // stored at chunk c ^ (row & 7)
            const uint8_t* src = sPk + p * L::kPk + row * 128;
            const uint4 c0 = *reinterpret_cast<const uint4*>(src + (((2 * gi) ^ (row & 7)) << 4));
            const uint4 c1 = *reinterpret_cast<const uint4*>(src + (((2 * gi + 1) ^ (row & 7)) << 4));
            const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            uint32_t cols[32];
#pragma unroll
            for (int c = 0; c < 8; ++c)
#pragma unroll
              for (int sl = 0; sl < 4; ++sl) cols[8 * sl + c] = (wd[c] >> (6 - 2 * sl)) & 0x03030303u;
            const int s = L::kAPerPipe * pj + n % L::kAPerPipe;
            // the MMAs of the A stage's previous use must be done with it
            if (!mbar_wait(&aempty[s], ((n / L::kAPerPipe) & 1) ^ 1, err, abort_flag)) goto unpack_done;
            tc_fence_after();
            __syncwarp();
            tmem_st_32x32b_x32(tq + static_cast<uint32_t>(s * kSkAStageCols), cols);
            tmem_st_wait();
            tc_fence_before();
            // the packed bytes are consumed: order the reads before the next
            // TMA into the slot
            fence_proxy_async_smem();
            // afull also tells the MMA thread that the stage's token planes
            // have landed: it then waits on one barrier per stage, not two
            const int tidx = tg0 + i / kTG;
            if (!mbar_wait(&tfull[tidx % kTS], (tidx / kTS) & 1, err, abort_flag)) goto unpack_done;
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[s]);
            ++n;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pk_empty[p]);
      }
      g0 += len;
      pg0 += ngroups;
      tg0 += (len + kTG - 1) / kTG;
    }
  unpack_done:;
  } else {
    // ------------------------------------------------------------- epilogue
    const int et = threadIdx.x - L::kEpiWarp0 * 32;  // 0..127
    const int q = warp & 3;                           // TMEM lane quadrant this warp may access
    for (int t = et; t < BN; t += 128) {
      sInv[t] = t < M ? __frcp_rn(__ldg(a_scale + t)) : 0.0f;
      int rs = 0;
      if (t < M)
        for (int c = 0; c < nparts; ++c) rs += __ldg(rowsum_part + t * nparts + c);
      sRs[t] = rs;
    }
    epi_bar();
    int tl = 0, g0 = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++tl) {
      const SkUnit w = sk_unit(u, S, nkb);
      const int a = L::kAccBufs == 2 ? (tl & 1) : 0;
      const int use = L::kAccBufs == 2 ? (tl >> 1) : tl;
      const int n = w.wt * kSkBM + q * 32 + lane;  // this thread's weight row
      const bool n_ok = n < N;
      const int len = w.len(), r0 = g0 % kP;  // pipelines with a stage: those of running indices g0 ..
      g0 += len;
      if (!mbar_wait_idle(&acc_full[a], use & 1, err, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(kP * a * L::kN2);
      // 8 tokens (16 columns: hi, lo) at a time: y (one split) or the partial
      // sum (several splits; exact fp32 atomic additions)
#pragma unroll 1
      for (int c0 = 0; c0 < L::kN2 && (c0 >> 1) < M; c0 += 16) {
        int acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0;
#pragma unroll 1
        for (int pj = 0; pj < kP; ++pj) {
          if (len < kP && (pj - r0 + kP) % kP >= len) continue;  // no stage of this unit
          uint32_t r[16];
          tmem_ld_32x32b_x16(tbase + static_cast<uint32_t>(pj * L::kN2 + c0), r);
          tmem_ld_wait();
          tmem_reg_fence16(r);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] += __float2int_rn(__fmul_rn(__uint_as_float(r[i]), 512.0f));
        }
        if (n_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int t = (c0 >> 1) + i;
            if (t < M) {
              const int v = 16 * acc[2 * i] + acc[2 * i + 1];  // sum c q over the unit's blocks
              if (S == 1) {
                const int full = v - sRs[t];
                y[static_cast<int64_t>(t) * N + n] = rescale_elem(static_cast<float>(full), sInv[t], inv_w);
                if (acc_out) acc_out[static_cast<int64_t>(t) * N + n] = full;
              } else {
                red_add_f32(ws + static_cast<int64_t>(t) * N + n, static_cast<float>(v));
              }
            }
          }
        }
      }
      // the accumulators have been read: release them to a later unit's MMAs
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
          // 16 tokens' sums loaded before any is used: one L2 round trip per
          // 16 tokens instead of one per token
#pragma unroll 1
          for (int t0 = 0; t0 < M && t0 < BN; t0 += 16) {
            float part[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              part[i] = t0 + i < M ? __ldcg(ws + static_cast<int64_t>(t0 + i) * N + n) : 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int t = t0 + i;
              if (t < M) {
                // both exact integers below 2^24: the difference is exact
                const float accf = __fsub_rn(part[i], static_cast<float>(sRs[t]));
                y[static_cast<int64_t>(t) * N + n] = rescale_elem(accf, sInv[t], inv_w);
                if (acc_out) acc_out[static_cast<int64_t>(t) * N + n] = __float2int_rn(accf);
              }
            }
          }
        }
      }
      epi_bar();  // last_flag is rewritten by the next unit
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::kMmaWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kSkTmemCols);
  }
}

// Token tile of the contraction for M tokens (16, 32, 48 or 64).
int skinny_tile(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 48 ? 48 : 64; }

// Number of K splits: the one with the least estimated time, which is the
// busiest CTA's stages plus, with a split, a fixed cost (the partial sums'
// zeroing, the tickets, the last split's read-back) and the epilogues' fp32
// atomic additions (M N S of them, a throughput the whole GPU shares).  Fitted
// to GB300 timings of 12 shapes (9..63 tokens, K = 4096..65536, N =
// 1024..16384) at forced split counts, within ~1 us rms: per stage ~185 /
// 210 / 235 / 400 ns for tiles of 16 / 32 / 48 / 64 tokens, ~1.9 us fixed and
// ~128 atomic additions per ns.  Ties go to fewer splits.
int choose_splits(int64_t M, int n_wt, int nkb, int64_t N, int ctas) {
  constexpr double kSplitNs = 1900.0, kAtomicsPerNs = 128.0;
  const int bn = skinny_tile(M);
  const double stage_ns = bn == 16 ? 185.0 : bn == 32 ? 210.0 : bn == 48 ? 235.0 : 400.0;
  const int ngrp = (nkb + kSkPkGroup - 1) / kSkPkGroup;
  int best = 1;
  double best_cost = 0.0;
  const int max_s = ngrp < 64 ? ngrp : 64;
  for (int S = 1; S <= max_s; ++S) {
    const int64_t units = static_cast<int64_t>(n_wt) * S;
    const int64_t per_cta = (units + ctas - 1) / ctas;
    double cost = static_cast<double>(per_cta) * kSkPkGroup * ((ngrp + S - 1) / S) * stage_ns;
    if (S > 1) cost += kSplitNs + static_cast<double>(M) * static_cast<double>(N) * S / kAtomicsPerNs;
    if (S == 1 || cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

template <int BN>
cudaError_t launch_bn(const DeviceContext* ctx, EncodeTiledFn encode, const uint8_t* planes, const float* a_scale,
                      const int* rowsum_part, int nparts, const uint8_t* packed_w, float inv_w, int M, int K, int N, int S, float* y,
                      int32_t* acc_out, float* ws, int* tickets, cudaStream_t s, int* status) {
  using L = SkLayout<BN>;
  CUtensorMap tm_tok, tm_w;
  {
    // token planes: bytes [M][K/128][2][128] viewed as (byte, plane, token,
    // block); boxes of 128 bytes x 2 planes x BN tokens x TG blocks land as TG
    // stages of 2 BN swizzled rows of 128 bytes, row 2 t + plane (tokens >= M
    // and blocks past K read as 0)
    cuuint64_t dims[4] = {128, 2, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 128)};
    cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(K) * 2, 256};
    cuuint32_t box[4] = {128, 2, static_cast<cuuint32_t>(BN), static_cast<cuuint32_t>(L::kTG)};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = encode(&tm_tok, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(planes), dims, strides, box,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;  // behind the plane conversion
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_tok, tm_w, a_scale, rowsum_part, nparts, inv_w, M, N, K, S, y, acc_out,
                            ws, tickets, ctx->err_word);
}

// Workspace: [fp32 partial sums M x N, tile tickets] (split K only; zero on
// entry) then the chunk sums of the codes (M x plane_chunks(K) ints).
struct SkWorkspace {
  int S;
  size_t zeroed;  // bytes that must be zero on entry
  size_t total;
};
SkWorkspace skinny_workspace(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N) {
  SkWorkspace w;
  const int n_wt = static_cast<int>((N + kSkBM - 1) / kSkBM);
  w.S = choose_splits(M, n_wt, static_cast<int>(K >> 7), N, ctx->num_sms);
  w.zeroed = w.S == 1 ? 0
                      : ((static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~size_t(255)) +
                            static_cast<size_t>(n_wt) * 4;
  w.total = ((w.zeroed + 255) & ~size_t(255)) +
            ((static_cast<size_t>(M) * plane_chunks(static_cast<int>(K)) * 4 + 255) & ~size_t(255));
  return w;
}

}  // namespace

// Used for 9..63 tokens when the weight stream is long enough to pay for the
// split's extra work (zeroing the partial sums, a final pass per tile); below
// that (K <= 2048 and N <= 8192, a few us) the tokens-as-M kernel is faster.
// From 64 tokens on the tokens-as-M kernel is used: its tiles hold 128 tokens,
// so its time hardly depends on the count.  Measured on GB300 at
// K = N = 16384: 37 / 40 / 45 / 50 us for 16 / 32 / 48 / 63 tokens here against
// 78-79 us there.
bool gemm_skinny_supported(int64_t M, int64_t K, int64_t N) {
  return M > kDecodeMaxM && M < 64 && K >= 128 && K % 128 == 0 && N >= 1 && (K >= 4096 || N >= 16384);
}

size_t gemm_skinny_workspace(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N) {
  return skinny_workspace(ctx, M, K, N).total;
}

size_t gemm_skinny_zeroed_bytes(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N) {
  return skinny_workspace(ctx, M, K, N).zeroed;
}

int32_t* gemm_skinny_rowsum_area(const DeviceContext* ctx, void* workspace, int64_t M, int64_t K, int64_t N) {
  const SkWorkspace w = skinny_workspace(ctx, M, K, N);
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + ((w.zeroed + 255) & ~size_t(255)));
}

cudaError_t launch_gemm_skinny(const DeviceContext* ctx, void* codes, const int32_t* rowsum, const float* a_scale,
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
  const SkWorkspace wl = skinny_workspace(ctx, M, K, N);
  const int S = wl.S;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  float* ws = nullptr;
  int* tickets = nullptr;
  if (S > 1) {
    // the partial sums are added into a zeroed fp32 [M, N] array
    const size_t ws_bytes = (static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~size_t(255);
    ws = reinterpret_cast<float*>(wsb);
    tickets = reinterpret_cast<int*>(wsb + ws_bytes);
    if (!workspace_zeroed) {
      cudaError_t e = cudaMemsetAsync(workspace, 0, wl.zeroed, s);
      if (e != cudaSuccess) return e;
    }
  }
  const int* rowsum_part = rowsum;
  int nparts = 1;
  if (!rowsum) {
    int* parts = reinterpret_cast<int*>(wsb + ((wl.zeroed + 255) & ~size_t(255)));
    rowsum_part = parts;
    nparts = plane_chunks(k);
    // the codes as the two e4m3 planes, in place, and their chunk sums
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plane_chunks(k)), static_cast<unsigned>(m));
    cfg.blockDim = dim3(kPlaneThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_token_planes, static_cast<__half*>(codes), k, parts);
    if (e != cudaSuccess) return e;
  }
  const uint8_t* planes = static_cast<const uint8_t*>(codes);
  switch (skinny_tile(M)) {
    case 16:
      return launch_bn<16>(ctx, encode, planes, a_scale, rowsum_part, nparts, packed_w, inv_w, m, k, n, S, y, acc_out, ws,
                           tickets, s, status);
    case 32:
      return launch_bn<32>(ctx, encode, planes, a_scale, rowsum_part, nparts, packed_w, inv_w, m, k, n, S, y, acc_out, ws,
                           tickets, s, status);
    case 48:
      return launch_bn<48>(ctx, encode, planes, a_scale, rowsum_part, nparts, packed_w, inv_w, m, k, n, S, y, acc_out,
                           ws, tickets, s, status);
    default:
      return launch_bn<64>(ctx, encode, planes, a_scale, rowsum_part, nparts, packed_w, inv_w, m, k, n, S, y, acc_out, ws,
                           tickets, s, status);
  }
}

}  // namespace bitnet
