// gemm_tc.cu -- prefill BitLinear contraction on the 5th-generation tensor cores.
//
// acc[m, n] = sum_k q[m, k] * (code(n, k) - 1)   (int8 activations x ternary
// weights, the product of ggml_vec_dot_i2_i8_s named in section 6.4 of "BitNet
// Embeddings GGUF Conversion Implementation"), then y = (acc / a_scale[m]) /
// w_scale in fp32 ("BitNet Inference Framework", "Quantization (W1.58A8)").
//
// sm_103a has no integer tcgen05 MMA, so the contraction runs as kind::f16 with
// fp16 operands that hold integers: activation codes in [-128, 127] and
// ternary weights are exact in fp16, every product is exact, and every partial
// sum is an integer of magnitude <= 127 * K < 2^24 (K <= 65536), so the fp32
// TMEM accumulator holds the exact integer.
//
// One CTA per SM, persistent over output tiles of 128 tokens x BW weights:
//   warp 12    TMA producer: token codes (fp16, 64-wide K slabs, 128B swizzle;
//              the MMA's A operand) and the tile's raw I2_S bytes (one
//              128-value block per weight row, 32 bytes)
//   warps 0-7  unpack: decode the BW weight rows of each slab from their packed
//              bytes into fp16 (magic-number conversion: 0x6400|c is 1024+c,
//              minus 1025) straight into the 128B-swizzled K-major layout of
//              the MMA's B operand; each packed block feeds two 64-wide slabs
//   warp 13    allocates TMEM (2 x BW columns: two accumulators) and one lane
//              issues tcgen05.mma (M=128 tokens, N=BW weights, K=16)
//   warps 8-11 epilogue: warp q reads TMEM lanes 32q..32q+31 = 32 tokens; each
//              thread owns one token (one activation scale per tile).  The
//              warp loads 32 accumulator columns at a time (the next load in
//              flight while the current columns are written), rescales them
//              into two 64B-swizzled 32-token x 16-column blocks in shared
//              memory, and one lane writes each block to y with a TMA store
//              (whole rows per transaction, no per-thread global stores); the
//              two blocks alternate so that one store reads shared memory
//              while the other block is filled.  This overlaps the next
//              tile's MMAs (double-buffered accumulator).  Without a usable
//              tensor map for y (row pitch not a multiple of 16 bytes) or with
//              the accumulator test output, threads store directly.
//              y is fp32, or fp16 / bf16 (YT: the fp32 result rounded once;
//              a 16-bit block holds 32 columns in the same 64-byte rows).
//              With a QK head norm (hd > 0, hd dividing BW, no K split) each
//              thread normalises its token's heads of hd columns itself: three
//              passes over the head in TMEM (largest |y|, the fixed-point sum
//              of squares, the output), the row arithmetic of the input norm.
// Split K: when the output tiles are too few to give every SM work (a few
// hundred tokens, long rows), the K blocks of each tile are split into S
// ranges and the CTAs iterate over (tile, range) units.  A unit's epilogue adds
// its partial sums to a zeroed fp32 workspace with red.global.add (exact: the
// partial sums are integers below 2^24, so the order of the additions does not
// matter); a per-tile ticket lets the unit that completes the tile read the
// sums back, rescale them and write y.
// Every wait is bounded; an expired wait sets the device error word and the
// CTA unwinds without trapping.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"
#include "unpack_f16.cuh"

#include <type_traits>

namespace bitnet {
namespace {

constexpr int kBT = 128;                   // tokens per tile (MMA M)
constexpr int kBK = 64;                    // K per sub-slab: one 128-byte swizzle row of fp16
constexpr int kPkSlots = 2;                // packed-weight slots (one I2_S block column each)
constexpr int kUnpackWarps = 8;
constexpr int kThreads = 448;  // warps 0-7 unpack, 8-11 epilogue, 12 producer, 13 MMA
constexpr int kAStageBytes = kBT * kBK * 2;  // 16 KB of token codes

__device__ __forceinline__ void epi_bar_tc() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__device__ __forceinline__ void red_add_global_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// A stage holds kSub 64-wide K sub-slabs of both operands, and the MMA thread
// waits once per stage.  A wait of the issuing thread behind MMAs still in
// flight costs a few hundred cycles (measured on sm_103a: ~240 cycles, with
// ~45 more per issued instruction), so a stage must carry enough MMA work to
// hide it: 4 MMAs of N=256 (512 cycles) do; narrower tiles take 128-wide
// stages (8 MMAs per wait).
template <int BW>
struct TcLayout {
  static constexpr int kSub = BW == 256 ? 1 : 2;         // 64-wide sub-slabs per stage
  static constexpr int kStages = BW == 128 ? 3 : 4;      // ~192 KB of operand stages
  static constexpr int kSubBBytes = BW * kBK * 2;        // one sub-slab of weights (fp16)
  static constexpr int kAStage = kSub * kAStageBytes;
  static constexpr int kBStage = kSub * kSubBBytes;
  static constexpr int kPkSlotBytes = BW * 32;
  static constexpr int offA = 0;
  static constexpr int offB = offA + kStages * kAStage;
  static constexpr int offP = offB + kStages * kBStage;
  static constexpr int offStg = offP + kPkSlots * kPkSlotBytes;  // 1 KB aligned: all sizes above are
  static constexpr int kStgBytes = 4 * 2 * 32 * 16 * 4;          // two 32 x 16 fp32 blocks per epilogue warp
  static constexpr int offBar = offStg + kStgBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kPkSlots + 4;
  static constexpr int offMisc = offBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kBytes = offMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1 KB
  static_assert(offStg % 1024 == 0, "swizzled staging blocks need 1 KB alignment");
  static_assert(kAlloc <= 232448, "over the 227 KB of shared memory a CTA may use");
};

// Two results rounded to a 16-bit type, packed low half first.
template <typename YT>
__device__ __forceinline__ uint32_t pack2_out(float a, float b) {
  const YT lo = round_out<YT>(a), hi = round_out<YT>(b);
  return static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&lo)) |
         (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
}

template <int BW, typename YT>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_y, int y_by_tma, const float* __restrict__ a_scale,
              float inv_w, int M, int N, int K, int S, YT* __restrict__ y, int32_t* __restrict__ acc_out,
              float* __restrict__ ws, int* __restrict__ tickets, const float* __restrict__ head_w, int hd,
              float eps, unsigned* err) {
  using L = TcLayout<BW>;
  constexpr int kTpr = kUnpackWarps * 32 / BW;  // unpack threads per weight row (1, 2 or 4)
  constexpr int kCpt = 8 / kTpr;                 // 16-byte chunks of a slab row per thread
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

  uint8_t* sA = smem + L::offA;
  uint8_t* sB = smem + L::offB;
  uint8_t* sP = smem + L::offP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::offBar);
  // full[s]: the token slabs have landed (producer's expect-tx arrival plus the
  // bytes) and every unpack warp has written its weight rows; one wait per stage
  uint64_t* full = bars;
  uint64_t* st_empty = bars + L::kStages;
  uint64_t* pk_full = bars + 2 * L::kStages;
  uint64_t* pk_empty = pk_full + kPkSlots;
  uint64_t* acc_full = pk_empty + kPkSlots;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_wt = (N + BW - 1) / BW;
  const int n_mt = (M + kBT - 1) / kBT;
  const int num_tiles = n_wt * n_mt;
  const int nkb = K >> 7;
  const int num_units = num_tiles * S;
  // unit u: tile u / S, I2_S block columns [kb_lo, kb_hi) of range u % S
  auto kb_lo = [&](int u) { return static_cast<int>((static_cast<int64_t>(nkb) * (u % S)) / S); };
  auto kb_hi = [&](int u) { return static_cast<int>((static_cast<int64_t>(nkb) * (u % S + 1)) / S); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < L::kStages; ++i) {
      mbar_init(&full[i], 1 + kUnpackWarps);
      mbar_init(&st_empty[i], 1);
    }
    for (int i = 0; i < kPkSlots; ++i) {
      mbar_init(&pk_full[i], 1);
      mbar_init(&pk_empty[i], kUnpackWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 2 * BW);
    tmem_relinquish();
  }
  if (warp == 12 && lane == 0) {
    prefetch_tensormap(&tm_tok);
    prefetch_tensormap(&tm_w);
    if (y_by_tma) prefetch_tensormap(&tm_y);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // everything below reads what the previous kernel on the stream produced
  pdl_wait();

  if (warp == 12) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0, sph = 0, p = 0, pph = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        const int tile = u / S;
        const int n0 = (tile % n_wt) * BW;
        const int m0 = (tile / n_wt) * kBT;
        for (int kb = kb_lo(u); kb < kb_hi(u); ++kb) {
          if (!mbar_wait(&pk_empty[p], pph ^ 1, err, abort_flag)) goto producer_done;
          mbar_arrive_expect_tx(&pk_full[p], L::kPkSlotBytes);
          tma_load_2d(sP + p * L::kPkSlotBytes, &tm_w, kb * 32, n0, &pk_full[p]);
          if (++p == kPkSlots) { p = 0; pph ^= 1; }
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const int h = hf % L::kSub;
            if (h == 0) {
              if (!mbar_wait(&st_empty[s], sph ^ 1, err, abort_flag)) goto producer_done;
              mbar_arrive_expect_tx(&full[s], L::kAStage);
            }
            tma_load_2d(sA + s * L::kAStage + h * kAStageBytes, &tm_tok, kb * 128 + hf * kBK, m0, &full[s]);
            if (h == L::kSub - 1 && ++s == L::kStages) { s = 0; sph ^= 1; }
          }
        }
      }
    producer_done:;
    }
  } else if (warp == 13) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kBT, BW);
      int s = 0, sph = 0, tl = 0;
      for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++tl) {
        const int a = tl & 1;
        if (!mbar_wait(&acc_empty[a], ((tl >> 1) & 1) ^ 1, err, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * BW);
        bool ok = true;
        const int nstages = 2 * (kb_hi(u) - kb_lo(u)) / L::kSub;
        for (int ks = 0; ks < nstages; ++ks) {
          if (!mbar_wait(&full[s], sph, err, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < L::kSub; ++h) {
            const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + s * L::kAStage + h * kAStageBytes));
            const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + s * L::kBStage + h * L::kSubBBytes));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              tc_mma_f16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (ks | h | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&st_empty[s]);
          if (++s == L::kStages) { s = 0; sph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&acc_full[a]);
      }
    }
  } else if (warp < kUnpackWarps) {
    // --------------------------------------------------------------- unpack
    // kTpr threads share a weight row of the tile; each writes kCpt of its 8
    // chunks per slab (all of them need the row's 8 packed words)
    const int t = threadIdx.x;
    const int row = t / kTpr;
    const int c0 = (t % kTpr) * kCpt;
    uint8_t* const brow = sB + (row >> 3) * 1024 + (row & 7) * 128;
    int s = 0, sph = 0, p = 0, pph = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      for (int kb = kb_lo(u); kb < kb_hi(u); ++kb) {
        if (!mbar_wait(&pk_full[p], pph, err, abort_flag)) goto unpack_done;
        uint32_t wd[8];
        {
          const uint4* src = reinterpret_cast<const uint4*>(sP + p * L::kPkSlotBytes + row * 32);
          const uint4 lo4 = src[0];
          const uint4 hi4 = src[1];
          wd[0] = lo4.x; wd[1] = lo4.y; wd[2] = lo4.z; wd[3] = lo4.w;
          wd[4] = hi4.x; wd[5] = hi4.y; wd[6] = hi4.z; wd[7] = hi4.w;
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int h = hf % L::kSub;
          if (h == 0 && !mbar_wait(&st_empty[s], sph ^ 1, err, abort_flag)) goto unpack_done;
          unpack_row_slab<kCpt>(wd, hf, c0, brow + s * L::kBStage + h * L::kSubBBytes, row & 7);
          if (h == L::kSub - 1) {
            // orders this thread's shared-memory accesses (the packed-slot
            // reads and the slab writes) before later async-proxy accesses:
            // the MMA reading the slab, the next TMA overwriting the packed slot
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&full[s]);
              // the slot's words have been used by now (every chunk needs all
              // eight), so its loads are complete: it may be refilled
              if (hf == L::kSub - 1) mbar_arrive(&pk_empty[p]);
            }
            if (++s == L::kStages) { s = 0; sph ^= 1; }
          }
        }
        if (++p == kPkSlots) { p = 0; pph ^= 1; }
      }
    }
  unpack_done:;
  } else {
    // ------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    uint8_t* const stg = smem + L::offStg + q * 4096;  // this warp's two 32 x 16 fp32 staging blocks
    const int swz = (lane >> 1) & 3;                  // 64B swizzle of this thread's staging row
    int tl = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++tl) {
      const int tile = u / S;
      const int a = tl & 1;
      const int n0 = (tile % n_wt) * BW;
      const int m0 = (tile / n_wt) * kBT;
      const int m = m0 + q * 32 + lane;  // this thread's token
      const bool m_ok = m < M;
      const bool rows_ok = m0 + q * 32 < M;  // warp-uniform: any of the warp's tokens exist
      // rcp.rn == 1.0f / a_scale in IEEE arithmetic
      const float inv_a = m_ok ? __frcp_rn(__ldg(a_scale + m)) : 0.0f;
      // with split K the four epilogue warps meet at named barriers for every
      // unit, so they leave the loop together: a failed wait only skips the
      // unit's work and the abort flag is read after the unit's last barrier
      const bool got = mbar_wait_idle(&acc_full[a], (tl >> 1) & 1, err, abort_flag);
      if (!got && S == 1) break;
      if (got) tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(a * BW);
      if (S > 1) {
        // One range of the tile: add the partial sums to the workspace.  Each
        // 32 x 32 block (this warp's 32 tokens x 32 columns) is transposed
        // through the warp's staging buffer (XOR-swizzled: conflict-free both
        // ways) so that every atomic instruction covers 32 consecutive outputs
        // of one token.
        float* const blk = reinterpret_cast<float*>(stg);
        if (got && rows_ok) {
#pragma unroll 1
          for (int j0 = 0; j0 < BW; j0 += 32) {
            const int nb = n0 + j0;
            if (nb >= N) break;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(j0), r);
            tmem_ld_wait();
            tmem_reg_fence(r);
#pragma unroll
            for (int c = 0; c < 32; ++c) blk[lane * 32 + (c ^ lane)] = __uint_as_float(r[c]);
            __syncwarp();
            const int col = nb + lane;
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
              const int mi = m0 + q * 32 + i;
              if (mi < M && col < N) red_add_global_f32(ws + static_cast<int64_t>(mi) * N + col, blk[i * 32 + (lane ^ i)]);
            }
            __syncwarp();
          }
        }
        // the accumulator has been read: release it to the MMAs of a later unit
        if (got) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[a]);
        }
        // the range that brings the tile's ticket to S writes the tile
        __threadfence();
        epi_bar_tc();
        if (warp == 8 && lane == 0) *last_flag = !*abort_flag && atomicAdd(&tickets[tile], 1) == S - 1;
        epi_bar_tc();
        if (*last_flag && rows_ok) {
          __threadfence();
          // 32 columns at a time, lane = column: each load and each store
          // instruction covers 32 consecutive sums or outputs of one token
          // (32 loads in flight per lane).  Lane = token would make every load
          // touch 32 rows: ~11k cycles per 32-column block instead of ~1k.
#pragma unroll 1
          for (int j0 = 0; j0 < BW; j0 += 32) {
            const int nb = n0 + j0;
            if (nb >= N) break;
            const int col = nb + lane;
            const int nrow = min(32, M - (m0 + q * 32));  // tokens of this warp (>= 1)
            const int64_t base = static_cast<int64_t>(m0 + q * 32) * N + col;
            const float* wcol = ws + base;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = (i < nrow && col < N) ? __ldcg(wcol + i * N) : 0.0f;
            YT* ycol = y + base;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float inv_ai = __shfl_sync(0xffffffffu, inv_a, i);
              if (i < nrow && col < N) {
                ycol[i * N] = round_out<YT>(rescale_elem(v[i], inv_ai, inv_w));
                if (acc_out) acc_out[base + i * N] = __float2int_rn(v[i]);
              }
            }
          }
        }
        epi_bar_tc();  // last_flag is rewritten by the next unit
        if (*abort_flag) break;
        continue;
      }
      if (BW >= 128 && hd > 0) {  // (heads of 128 or 256 values never fit 64-wide tiles)
        if (rows_ok) {
          // 32 values of this thread's token, columns c .. c + 31 of the tile
          auto load32 = [&](int c, uint32_t(&r)[32]) {
            tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(c), r);
            tmem_ld_wait();
            tmem_reg_fence(r);
          };
          auto y4 = [&](const uint32_t(&r)[32], int v) {
            return make_float4(rescale_elem(__uint_as_float(r[4 * v + 0]), inv_a, inv_w),
                               rescale_elem(__uint_as_float(r[4 * v + 1]), inv_a, inv_w),
                               rescale_elem(__uint_as_float(r[4 * v + 2]), inv_a, inv_w),
                               rescale_elem(__uint_as_float(r[4 * v + 3]), inv_a, inv_w));
          };
          int blk = 0;  // staging blocks written so far (they alternate between two buffers)
          const int ncols = min(BW, N - n0);  // whole heads: hd divides N and BW
          for (int h0 = 0; h0 < ncols; h0 += hd) {
            uint32_t r[32];
            int key = 0;
            for (int c = h0; c < h0 + hd; c += 32) {
              load32(c, r);
#pragma unroll
              for (int v = 0; v < 8; ++v) key = max(key, sq_key4(y4(r, v)));
            }
            const float scale = sq_scale(key);
            SqPartial part = {0ull, 0u};
            for (int c = h0; c < h0 + hd; c += 32) {
              load32(c, r);
#pragma unroll
              for (int v = 0; v < 8; ++v) sq_add4(part, y4(r, v), scale);
            }
            const float rstd = rstd_from_fixed(sq_fold(part, hd), key, hd, eps);
            for (int c = h0; c < h0 + hd; c += 32) {
              load32(c, r);
              const float* hw = head_w + (c - h0);
#pragma unroll
              for (int v = 0; v < 8; ++v) {
                const float4 yv = y4(r, v);
                const float4 g = __ldg(reinterpret_cast<const float4*>(hw + 4 * v));
                r[4 * v + 0] = __float_as_uint(norm_elem(yv.x, rstd, g.x));
                r[4 * v + 1] = __float_as_uint(norm_elem(yv.y, rstd, g.y));
                r[4 * v + 2] = __float_as_uint(norm_elem(yv.z, rstd, g.z));
                r[4 * v + 3] = __float_as_uint(norm_elem(yv.w, rstd, g.w));
              }
              const int col = n0 + c;
              if (y_by_tma) {
                constexpr int kPer = sizeof(YT) == 2 ? 32 : 16;  // columns per 64-byte staging row
#pragma unroll
                for (int b = 0; b < 32 / kPer; ++b) {
                  if (lane == 0) bulk_wait_group_read<1>();
                  __syncwarp();
                  uint8_t* const buf = stg + (blk & 1) * 2048;
#pragma unroll
                  for (int v = 0; v < 4; ++v) {
                    uint4 o;
                    if constexpr (sizeof(YT) == 2) {
                      o.x = pack2_out<YT>(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                      o.y = pack2_out<YT>(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                      o.z = pack2_out<YT>(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                      o.w = pack2_out<YT>(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                    } else {
                      o = make_uint4(r[16 * b + 4 * v + 0], r[16 * b + 4 * v + 1], r[16 * b + 4 * v + 2],
                                     r[16 * b + 4 * v + 3]);
                    }
                    *reinterpret_cast<uint4*>(buf + lane * 64 + ((v ^ swz) << 4)) = o;
                  }
                  fence_proxy_async_smem();
                  __syncwarp();
                  if (lane == 0) {
                    tma_store_2d(&tm_y, buf, col + kPer * b, m0 + q * 32);
                    bulk_commit_group();
                  }
                  ++blk;
                }
              } else if (m_ok) {
                YT* yrow = y + static_cast<int64_t>(m) * N + col;
#pragma unroll
                for (int j = 0; j < 32; ++j) yrow[j] = round_out<YT>(__uint_as_float(r[j]));
              }
            }
          }
        }
      } else if (y_by_tma && rows_ok) {
        const int nch = (min(BW, N - n0) + 31) >> 5;  // 32-column chunks holding outputs
        // rescale the chunk in r (columns n0 + 32 ch ..) and store it as two
        // fp32 blocks, or as one block of 16-bit values
        auto emit = [&](const uint32_t(&r)[32], int ch) {
          if constexpr (sizeof(YT) == 2) {
            // the store issued two chunks ago, from this buffer, must have read it
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            uint8_t* const buf = stg + (ch & 1) * 2048;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 o;
              o.x = pack2_out<YT>(rescale_elem(__uint_as_float(r[8 * v + 0]), inv_a, inv_w),
                                  rescale_elem(__uint_as_float(r[8 * v + 1]), inv_a, inv_w));
              o.y = pack2_out<YT>(rescale_elem(__uint_as_float(r[8 * v + 2]), inv_a, inv_w),
                                  rescale_elem(__uint_as_float(r[8 * v + 3]), inv_a, inv_w));
              o.z = pack2_out<YT>(rescale_elem(__uint_as_float(r[8 * v + 4]), inv_a, inv_w),
                                  rescale_elem(__uint_as_float(r[8 * v + 5]), inv_a, inv_w));
              o.w = pack2_out<YT>(rescale_elem(__uint_as_float(r[8 * v + 6]), inv_a, inv_w),
                                  rescale_elem(__uint_as_float(r[8 * v + 7]), inv_a, inv_w));
              *reinterpret_cast<uint4*>(buf + lane * 64 + ((v ^ swz) << 4)) = o;
            }
            fence_proxy_async_smem();
            __syncwarp();
            // rows >= M and columns >= N of the block are clipped by the copy
            if (lane == 0) {
              tma_store_2d(&tm_y, buf, n0 + 32 * ch, m0 + q * 32);
              bulk_commit_group();
            }
            return;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = n0 + 32 * ch + 16 * h;
            if (col >= N) break;
            // the store issued two blocks ago, from this buffer, must have read it
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            uint8_t* const buf = stg + h * 2048;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float4 o;
              o.x = rescale_elem(__uint_as_float(r[16 * h + 4 * v + 0]), inv_a, inv_w);
              o.y = rescale_elem(__uint_as_float(r[16 * h + 4 * v + 1]), inv_a, inv_w);
              o.z = rescale_elem(__uint_as_float(r[16 * h + 4 * v + 2]), inv_a, inv_w);
              o.w = rescale_elem(__uint_as_float(r[16 * h + 4 * v + 3]), inv_a, inv_w);
              *reinterpret_cast<float4*>(buf + lane * 64 + ((v ^ swz) << 4)) = o;
            }
            fence_proxy_async_smem();
            __syncwarp();
            // rows >= M and columns >= N of the block are clipped by the copy
            if (lane == 0) {
              tma_store_2d(&tm_y, buf, col, m0 + q * 32);
              bulk_commit_group();
            }
          }
        };
        uint32_t ra[32], rb[32];
        tmem_ld_32x32b_x32(tbase, ra);
        tmem_ld_wait();
        tmem_reg_fence(ra);
        for (int ch = 0;; ch += 2) {
          const bool more = ch + 1 < nch;
          if (more) tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(32 * (ch + 1)), rb);
          emit(ra, ch);
          if (!more) break;
          tmem_ld_wait();
          tmem_reg_fence(rb);
          const bool more2 = ch + 2 < nch;
          if (more2) tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(32 * (ch + 2)), ra);
          emit(rb, ch + 1);
          if (!more2) break;
          tmem_ld_wait();
          tmem_reg_fence(ra);
        }
      } else if (!y_by_tma && rows_ok) {
        YT* yrow = y + static_cast<int64_t>(m) * N;
#pragma unroll 1
        for (int j0 = 0; j0 < BW; j0 += 32) {
          const int nb = n0 + j0;
          if (nb >= N) break;
          uint32_t r[32];
          tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(j0), r);
          tmem_ld_wait();
          tmem_reg_fence(r);
          if (!m_ok) continue;
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            if (nb + jj < N) {
              const float accf = __uint_as_float(r[jj]);
              yrow[nb + jj] = round_out<YT>(rescale_elem(accf, inv_a, inv_w));
              if (acc_out) acc_out[static_cast<int64_t>(m) * N + nb + jj] = __float2int_rn(accf);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
    }
    // stores still in flight read this CTA's shared memory: finish them first
    if (y_by_tma && lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * BW);
  }
}

template <int BW, typename YT>
cudaError_t launch_bw(const DeviceContext* ctx, EncodeTiledFn encode, const __half* codes_f16, const float* a_scale,
                      const uint8_t* packed_w, float inv_w, int M, int N, int K, int S, YT* y, int32_t* acc_out,
                      float* ws, int* tickets, const float* head_w, int hd, float eps, bool pdl, cudaStream_t s,
                      int* status) {
  using L = TcLayout<BW>;
  CUtensorMap tm_tok, tm_w;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBT)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&tm_tok, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(codes_f16), dims, strides,
                        box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *status = BITNET_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 4), static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 4)};
    cuuint32_t box[2] = {32, static_cast<cuuint32_t>(BW)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed_w), dims, strides, box,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *status = BITNET_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  // y through TMA stores: [M, N], 32-row boxes of 64-byte rows (16 fp32 or 32
  // 16-bit columns), 64B swizzle (the row pitch must be a multiple of 16 bytes)
  constexpr int kYBytes = static_cast<int>(sizeof(YT));
  CUtensorMap tm_y = tm_tok;  // placeholder, never read unless y_by_tma
  const int y_by_tma = ((static_cast<int64_t>(N) * kYBytes) % 16 == 0 && acc_out == nullptr && S == 1) ? 1 : 0;
  if (y_by_tma) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * kYBytes};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / kYBytes), 32};
    cuuint32_t es[2] = {1, 1};
    const CUtensorMapDataType yt = kYBytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : (std::is_same<YT, __half>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    CUresult r = encode(&tm_y, yt, 2, y, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      *status = BITNET_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  auto kern = k_gemm_tc<BW, YT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const int units = ((N + BW - 1) / BW) * ((M + kBT - 1) / kBT) * S;
  const int grid = units < ctx->num_sms ? units : ctx->num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_tok, tm_w, tm_y, y_by_tma, a_scale, inv_w, M, N, K, S, y, acc_out, ws,
                            tickets, head_w, hd, eps, ctx->err_word);
}

// Weight-tile width and number of K ranges.  Wide tiles re-read the tokens
// least; when they leave SMs idle, K is split.  The cost of the busiest CTA is
// counted in units of 10 ns, measured on GB300 with one unit per CTA: an I2_S
// block column (128 values of K) costs 48 / 53 / 86 at BW = 64 / 128 / 256,
// and a split unit's atomic additions, ticket and read-back 250 + 9 BW; the
// cheapest option wins, ties to wider tiles and fewer ranges.
struct TcPlan {
  int bw, S;
};
TcPlan tc_plan(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N, bool can_split) {
  const int64_t m_tiles = (M + kBT - 1) / kBT;
  const int nkb = static_cast<int>(K >> 7);
  TcPlan best = {256, 1};
  int64_t best_cost = INT64_MAX;
  for (int bw = 256; bw >= 64; bw >>= 1) {
    const int64_t tiles = m_tiles * ((N + bw - 1) / bw);
    const int max_s = can_split ? (nkb < 64 ? nkb : 64) : 1;
    for (int S = 1; S <= max_s; ++S) {
      const int64_t units = tiles * S;
      const int64_t per_cta = (units + ctx->num_sms - 1) / ctx->num_sms;
      const int64_t per_kb = bw == 256 ? 86 : (bw == 128 ? 53 : 48);
      const int64_t cost = per_cta * (((nkb + S - 1) / S) * per_kb + (S > 1 ? 250 + 9 * bw : 0));
      if (cost < best_cost) {
        best_cost = cost;
        best = {bw, S};
      }
    }
  }
  return best;
}

}  // namespace

size_t gemm_tc_workspace(const DeviceContext* ctx, int64_t M, int64_t K, int64_t N) {
  const TcPlan pl = tc_plan(ctx, M, K, N, true);
  if (pl.S == 1) return 0;
  const int64_t tiles = ((M + kBT - 1) / kBT) * ((N + pl.bw - 1) / pl.bw);
  return ((static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~size_t(255)) +
         static_cast<size_t>(tiles) * 4;
}

cudaError_t launch_gemm_tc(const DeviceContext* ctx, const __half* codes_f16, const float* a_scale,
                           const uint8_t* packed_w, float w_scale, int64_t M, int64_t K, int64_t N, void* y,
                           int y_dtype, int32_t* acc_out, void* workspace, bool workspace_zeroed, bool pdl,
                           cudaStream_t s, int* status, const float* head_w, int head_dim, float eps,
                           bool* head_fused) {
  *status = BITNET_OK;
  if (head_fused) *head_fused = false;
  EncodeTiledFn encode = encode_tiled_fn();
  if (!encode) {
    *status = BITNET_ERR_CUDA;
    return cudaErrorNotSupported;
  }
  const float inv_w = 1.0f / w_scale;  // IEEE division, as in the oracle
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  // the same plan gemm_tc_workspace sized the workspace for; none: no split
  const TcPlan pl = tc_plan(ctx, M, K, N, workspace != nullptr);
  float* ws = nullptr;
  int* tickets = nullptr;
  if (pl.S > 1) {
    const int64_t tiles = ((M + kBT - 1) / kBT) * ((N + pl.bw - 1) / pl.bw);
    const size_t part = (static_cast<size_t>(M) * static_cast<size_t>(N) * 4 + 255) & ~size_t(255);
    ws = static_cast<float*>(workspace);
    tickets = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + part);
    if (!workspace_zeroed) {
      cudaError_t e = cudaMemsetAsync(workspace, 0, part + static_cast<size_t>(tiles) * 4, s);
      if (e != cudaSuccess) return e;
    }
  }
  // the head norm rides in the epilogue when a tile holds whole heads and K is not split
  const bool fuse = head_w && head_dim > 0 && head_fused && pl.S == 1 && pl.bw % head_dim == 0 && acc_out == nullptr;
  if (fuse) *head_fused = true;
  const float* hw = fuse ? head_w : nullptr;
  const int hd = fuse ? head_dim : 0;
  auto go = [&](auto* yt) {
    using YT = std::remove_pointer_t<decltype(yt)>;
    switch (pl.bw) {
      case 64:
        return launch_bw<64, YT>(ctx, encode, codes_f16, a_scale, packed_w, inv_w, m, n, k, pl.S, yt, acc_out, ws,
                                 tickets, hw, hd, eps, pdl, s, status);
      case 128:
        return launch_bw<128, YT>(ctx, encode, codes_f16, a_scale, packed_w, inv_w, m, n, k, pl.S, yt, acc_out, ws,
                                  tickets, hw, hd, eps, pdl, s, status);
      default:
        return launch_bw<256, YT>(ctx, encode, codes_f16, a_scale, packed_w, inv_w, m, n, k, pl.S, yt, acc_out, ws,
                                  tickets, hw, hd, eps, pdl, s, status);
    }
  };
  switch (y_dtype) {
    case BITNET_DTYPE_F32: return go(static_cast<float*>(y));
    case BITNET_DTYPE_F16: return go(static_cast<__half*>(y));
    case BITNET_DTYPE_BF16: return go(static_cast<__nv_bfloat16*>(y));
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bitnet
