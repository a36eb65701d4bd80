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

// Cost of one 128-weight-row x q-token tile, in SM cycles, for KB K-blocks
// of 128 bytes.  Per K-block the tensor core needs about 2q cycles (128 x q x
// 64 bf16 or 128 x q x 128 e4m3 multiply-adds) and the tile's operands
// (128 + q rows of 128 bytes) must stream in from L2; whichever is slower
// sets the pace, plus a fixed cost per tile for the pipeline fill and the
// accumulator hand-off.  These are the three kernel-side terms of "MoE
// GroupGEMM padding under expert skew", "Padding is not the whole cost model"
// (padded MMA work, weight/activation traffic, scheduling overhead).
constexpr int64_t kSelMmaCyclesPerTok = 2;        // per K-block, per token column
constexpr int64_t kSelLoadNum = 8, kSelLoadDen = 5;  // cycles per 128-byte row (1.6)
constexpr int64_t kSelTileOverhead = 2500;        // per tile

MG_HD int64_t tile_cost_cycles(int q, int64_t KB, int b_rows_per_sm) {
  const int64_t mma = kSelMmaCyclesPerTok * q;
  const int64_t load = (128 + b_rows_per_sm) * kSelLoadNum / kSelLoadDen;
  return KB * max64(mma, load) + kSelTileOverhead;
}

// Number of 128-byte K blocks of one operand row: the unit tile_cost_cycles
// is expressed in (64 bf16 or 128 e4m3 elements).
MG_HD int64_t sel_kblocks(bool fp8, int64_t K) { return K * (fp8 ? 1 : 2) / 128; }

// Picks the token tile from the per-candidate token-tile counts
// sum_e ceil(t_e/q).  The kernel's makespan is priced as whole waves of
// tiles over the SMs times the cost of one tile; ties go to the larger tile.
MG_HD int pick_tile(bool fp8, const int64_t (&token_tiles)[kNumTileCand], int64_t NB,
                    int64_t KB, int num_sms) {
  int best_q = tile_candidate(fp8, kNumTileCand - 1);
  int64_t best = -1;
  for (int i = 0; i < kNumTileCand; ++i) {
    const int q = tile_candidate(fp8, i);
    const int64_t T = token_tiles[i] * NB;
    const int64_t waves = cdiv64(T, num_sms);
    const int64_t cost = waves * tile_cost_cycles(q, KB, q);
    if (best < 0 || cost <= best) {
      best = cost;
      best_q = q;
    }
  }
  return best_q;
}

// Same choice for the CTA-pair kernel: a pair tile covers 256 weight rows
// (NB_pair = N/256 per token tile), each SM stages q/2 token rows, and the
// pairs are the workers.
MG_HD int pick_tile_pair(bool fp8, const int64_t (&token_tiles)[kNumTileCand], int64_t NB_pair,
                         int64_t KB, int num_pairs) {
  int best_q = tile_candidate(fp8, kNumTileCand - 1);
  int64_t best = -1;
  for (int i = 0; i < kNumTileCand; ++i) {
    const int q = tile_candidate(fp8, i);
    const int64_t T = token_tiles[i] * NB_pair;
    const int64_t waves = cdiv64(T, num_pairs);
    const int64_t cost = waves * tile_cost_cycles(q, KB, q / 2);
    if (best < 0 || cost <= best) {
      best = cost;
      best_q = q;
    }
  }
  return best_q;
}

}  // namespace mg
