// Planning arithmetic shared by the host planner, the device plan kernel and
// the GEMM kernels' schedulers: rounded counts, the two plan ratios in a fixed
// IEEE order, and the token-tile selector's cost model.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define MG_HD __host__ __device__ __forceinline__
#else
#define MG_HD inline
#endif

namespace mg {

MG_HD int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
// The same for 0 <= a < 2^32, 0 < b < 2^32 in 32-bit arithmetic: a kernel's
// prologue runs these once per expert and candidate, and on the GPU a 64-bit
// division is a long instruction sequence (the prologue's schedule took
// ~19000 cycles, measured with clock64 stamps, mostly in such loops).
MG_HD uint32_t cdiv_u32(uint32_t a, uint32_t b) { return a / b + (a % b != 0u ? 1u : 0u); }
// cdiv64 with a 32-bit path when both fit.
MG_HD int64_t cdiv_fast(int64_t a, int64_t b) {
  return (a >= 0 && a <= 0xffffffffll && b > 0 && b <= 0xffffffffll) ? (int64_t)cdiv_u32((uint32_t)a, (uint32_t)b)
                                                                     : cdiv64(a, b);
}
MG_HD int32_t round_up16(int32_t x) { return (x + 15) & ~15; }
MG_HD int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

MG_HD double i64_to_f64(int64_t x) {
#ifdef __CUDA_ARCH__
  return __ll2double_rn(x);
#else
  return static_cast<double>(x);
#endif
}
MG_HD double f64_div(double a, double b) {
#ifdef __CUDA_ARCH__
  return __ddiv_rn(a, b);
#else
  return a / b;
#endif
}
MG_HD double f64_mul(double a, double b) {
#ifdef __CUDA_ARCH__
  return __dmul_rn(a, b);
#else
  return a * b;
#endif
}

// (P-U)/P ("MoE GroupGEMM padding under expert skew", "Calculate padded token
// columns"); 0 for an empty layer.
MG_HD double plan_pad_frac(int64_t P, int64_t U) {
  return P == 0 ? 0.0 : f64_div(i64_to_f64(P - U), i64_to_f64(P));
}
// U^2 / sum t^2 ("Summarize skew without losing the histogram"); 0 if no
// expert has tokens.
MG_HD double plan_eff_experts(int64_t U, int64_t sumsq) {
  if (sumsq == 0) return 0.0;
  const double u = i64_to_f64(U);
  return f64_div(f64_mul(u, u), i64_to_f64(sumsq));
}

// ------------------------------------------------------------- selector
// Token-tile candidates.  The fp8 path caps the tile at 240 so two fp32
// accumulators plus the block-scale columns fit in the 512 TMEM columns.
constexpr int kNumTileCand = 4;
MG_HD int tile_candidate(bool fp8, int i) {
  return i == 0 ? 32 : i == 1 ? 64 : i == 2 ? 128 : (fp8 ? 240 : 256);
}

// Cost of one tile on one SM, in SM cycles, for KB K-blocks of 128 bytes:
// w_blocks 128-row weight blocks against q token columns, of which the SM
// stages b_rows token rows itself.  Per K-block and weight block the tensor
// core needs about 2.1q cycles for bf16 (128 x q x 64 multiply-adds) and
// 2.7q for block-scaled e4m3 (128 x q x 128), but never less than a floor
// that narrow tiles do not go below (about 350 and 600 cycles measured on
// GB300); the operands (128 w_blocks + b_rows rows of 128 bytes) must stream
// into shared memory; whichever is slower sets the pace, plus a fixed cost
// per tile for the pipeline fill and the accumulator hand-off.  These are the
// three kernel-side terms of "MoE GroupGEMM padding under expert skew",
// "Padding is not the whole cost model" (padded MMA work, weight/activation
// traffic, scheduling overhead).
constexpr int64_t kSelMmaSlopeX10Bf16 = 21, kSelMmaSlopeX10Fp8 = 27;  // cycles x10 per token column
constexpr int64_t kSelMmaFloorBf16 = 350, kSelMmaFloorFp8 = 600;      // cycles per K-block and block
constexpr int64_t kSelLoadNum = 8, kSelLoadDen = 5;  // cycles per 128-byte row (1.6)
constexpr int64_t kSelTileOverhead = 2500;        // per tile
// Round trip of a stage's loads when every SM streams weights from DRAM
// (masked decode batches), in SM cycles: a ring of S stages cannot turn a
// stage over faster than this over S.  Fitted to in-kernel clock stamps of
// the 16-expert decode with E2M1 weights (five 40 KB stages at ~814
// cycles, a third of them waiting for data).
constexpr int64_t kSelLoadRoundTrip = 4000;

// stage_floor: a lower bound on the cycles of one stage (0: none).
MG_HD int64_t tile_cost_cycles(bool fp8, int q, int64_t KB, int w_blocks, int b_rows, int64_t stage_floor = 0) {
  const int64_t per_block = fp8 ? max64(kSelMmaSlopeX10Fp8 * q / 10, kSelMmaFloorFp8)
                                : max64(kSelMmaSlopeX10Bf16 * q / 10, kSelMmaFloorBf16);
  const int64_t mma = per_block * w_blocks;
  const int64_t load = (128 * (int64_t)w_blocks + b_rows) * kSelLoadNum / kSelLoadDen;
  return KB * max64(max64(mma, load), stage_floor) + kSelTileOverhead;
}

// Number of 128-byte K blocks of one operand row: the unit tile_cost_cycles
// is expressed in (64 bf16 or 128 e4m3 elements).
MG_HD int64_t sel_kblocks(bool fp8, int64_t K) { return K * (fp8 ? 1 : 2) / 128; }

// Kernel families of the contiguous and masked forms: weight rows per tile
// and whether two SMs share each MMA (cta_group::2).
enum FwdVariant : int {
  kFwdSingle = 0,    // one CTA: 128 weight rows x q tokens
  kFwdDual = 1,      // one CTA: 256 weight rows x q tokens (N % 256 == 0)
  kFwdPair = 2,      // CTA pair: 256 weight rows x q tokens, q/2 staged per SM (N % 256 == 0)
  kFwdPairDual = 3,  // CTA pair: 512 weight rows x q tokens, q/2 staged per SM (N % 512 == 0)
  kFwdTokM = 4,      // one CTA, tokens on the MMA's M: 128 tokens x 256 weight rows (N % 256 == 0)
};
MG_HD int fwd_tile_rows(int variant) {
  return variant == kFwdSingle ? 128 : variant == kFwdPairDual ? 512 : 256;
}

// (The candidate loops here stay rolled: they run once per launch in the
// GEMM prologue, whose instructions come from DRAM when the L2 holds no
// code, and unrolled they cost the 16-expert decode ~2 % of its time in
// instruction fetch, measured with the L2 flushed before every launch.)
//
// Picks the token tile from the per-candidate token-tile counts
// sum_e ceil(t_e/q).  The kernel's makespan is priced as whole waves of
// tiles over the workers (CTAs, or CTA pairs) times the cost of one tile on
// one SM; ties go to the larger tile.
MG_HD int pick_tile(bool fp8, const int64_t (&token_tiles)[kNumTileCand], int variant, int64_t N,
                    int64_t KB, int num_sms) {
  // tokens on M: the MMA computes 128 token rows whatever the tile
  if (variant == kFwdTokM) return 128;
  const bool pair = variant == kFwdPair || variant == kFwdPairDual;
  const int64_t NB = N / fwd_tile_rows(variant);
  const int workers = pair ? (num_sms >= 2 ? num_sms / 2 : 1) : num_sms;
  const int w_blocks = (variant == kFwdDual || variant == kFwdPairDual) ? 2 : 1;  // per SM
  int best_q = tile_candidate(fp8, kNumTileCand - 1);
  int64_t best = -1;
#pragma unroll 1
  for (int i = 0; i < kNumTileCand; ++i) {
    const int q = tile_candidate(fp8, i);
    const int64_t T = token_tiles[i] * NB;
    const int64_t waves = cdiv_fast(T, workers);
    const int64_t cost = waves * tile_cost_cycles(fp8, q, KB, w_blocks, pair ? q / 2 : q);
    if (best < 0 || cost <= best) {
      best = cost;
      best_q = q;
    }
  }
  return best_q;
}

// Masked form on the single-SM two-block kernel: the token tile and the
// weight blocks per tile (one or two 128-row blocks) chosen together, every
// (q, blocks) candidate priced as pick_tile prices a tile size: whole waves
// of tiles over the SMs times the cost of one tile.  (Choosing q for
// two-block tiles first and switching to one block when two-block tiles
// would not fill two waves came out 7 % above the fastest candidate on the
// tuning sweeps of the decode table, against 1.7 % for the joint choice.)
// E2M1 weights (w4) fill 16 KB of shared memory per block and stage for 8 KB
// of DRAM data, so the ring holds half the weight bytes in flight and the
// decode waits on loads: their launches take two-block tiles only, and a
// stage costs at least the load round trip over the stages the ring holds
// (ring_bytes / (128-byte rows of both blocks and the tile, plus sf_bytes of
// scale data per stage)).  Replayed on the measured tactic sweeps of the
// decode table's 68 held-out histograms with E2M1 weights, this rule lands
// at 1.012 of the fastest tactic against 1.043 for the joint rule (the
// 16-expert decode: 64 x 2 tiles, 0.092 ms, rather than 128 x 1, 0.104).
// With E4M3 weights the floor made the choice worse (measured 1.038 ->
// 1.076), so it stays off there.
// Ties go to the larger tile, then to two blocks.
MG_HD void pick_tile_blocks(bool fp8, bool w4, const int64_t (&token_tiles)[kNumTileCand], int64_t N, int64_t KB,
                            int num_sms, int64_t ring_bytes, int64_t sf_bytes, int max_stages, int* q_out,
                            int* blocks_out) {
  int64_t best = -1;
  int bq = tile_candidate(fp8, kNumTileCand - 1), bb = 2;
#pragma unroll 1
  for (int i = 0; i < kNumTileCand; ++i) {
    const int q = tile_candidate(fp8, i);
#pragma unroll 1
    for (int nb = w4 ? 2 : 1; nb <= 2; ++nb) {
      const int64_t T = token_tiles[i] * (N / (128 * nb));
      const int64_t stage = 128 * (128 * (int64_t)nb + q) + sf_bytes;
      const int64_t S = (w4 && ring_bytes > 0) ? max64(1, ring_bytes / stage) : 0;
      const int64_t floor = S > 0 ? kSelLoadRoundTrip / (S < max_stages ? S : max_stages) : 0;
      const int64_t cost = cdiv_fast(T, num_sms > 0 ? num_sms : 1) * tile_cost_cycles(fp8, q, KB, nb, q, floor);
      if (best < 0 || cost <= best) {
        best = cost;
        bq = q;
        bb = nb;
      }
    }
  }
  *q_out = bq;
  *blocks_out = bb;
}

#ifdef __CUDACC__
// pick_tile_blocks with one candidate per lane (lane 2i + nb - 1 prices tile
// candidate i with nb blocks) and a warp reduction to the cheapest, ties to
// the higher lane, i.e. the same order of preference as the loop above.
// Called by all 32 lanes of a warp; every lane gets the choice.  (In a GEMM
// prologue whose instructions come from DRAM, eight candidates priced one
// after another cost the 16-expert decode ~1.6 us.)
__device__ __forceinline__ void pick_tile_blocks_warp(bool fp8, bool w4, const int64_t (&token_tiles)[kNumTileCand],
                                                      int64_t N, int64_t KB, int num_sms, int64_t ring_bytes,
                                                      int64_t sf_bytes, int max_stages, int* q_out, int* blocks_out) {
  const int lane = (int)(threadIdx.x & 31u);
  const int i = (lane >> 1) & (kNumTileCand - 1), nb = (lane & 1) + 1;
  const bool valid = lane < 2 * kNumTileCand && (!w4 || nb == 2);
  const int q = tile_candidate(fp8, i);
  const int64_t tiles = i == 0 ? token_tiles[0] : i == 1 ? token_tiles[1] : i == 2 ? token_tiles[2] : token_tiles[3];
  const int64_t T = tiles * (N / (128 * nb));
  const int64_t stage = 128 * (128 * (int64_t)nb + q) + sf_bytes;
  const int64_t S = (w4 && ring_bytes > 0) ? max64(1, ring_bytes / stage) : 0;
  const int64_t floor = S > 0 ? kSelLoadRoundTrip / (S < max_stages ? S : max_stages) : 0;
  int64_t cost = valid ? cdiv_fast(T, num_sms > 0 ? num_sms : 1) * tile_cost_cycles(fp8, q, KB, nb, q, floor)
                       : INT64_MAX;
  int best = lane;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const int64_t oc = __shfl_xor_sync(0xffffffffu, cost, o);
    const int ol = __shfl_xor_sync(0xffffffffu, best, o);
    if (oc < cost || (oc == cost && ol > best)) {
      cost = oc;
      best = ol;
    }
  }
  *q_out = tile_candidate(fp8, (best >> 1) & (kNumTileCand - 1));
  *blocks_out = (best & 1) + 1;
}
#endif

}  // namespace mg
