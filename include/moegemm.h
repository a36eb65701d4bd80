/*
 * moegemm.h -- C ABI of libmoegemm.so: the MoE grouped GEMM on one GB300.
 *
 * In an MoE layer every expert has the same weight shape, so N and K are
 * fixed and only the token dimension varies per expert ("flops/deepgemm-
 * grouped-masked-moe-gemm", "Arithmetic intensity").  The library provides the
 * planning step ("MoE GroupGEMM padding under expert skew", "Calculate padded
 * token columns" and "Summarize skew without losing the histogram") and the
 * three grouped GEMM forms ("flops/deepgemm-grouped-masked-moe-gemm",
 * "Workarounds"): M-grouped contiguous, masked, and K-grouped weight
 * gradient.  Every GEMM is a CUDA kernel for sm_103a.
 *
 * Conventions used by every call:
 *   - Tokens are rows.  Expert weights are B[e] of shape [N, K] with K
 *     contiguous (the nn.Linear layout); each expert computes
 *     D_e = A_e * B[e]^T, D_e row-major [rows, N].
 *   - "d_" pointers are device pointers (cudaMalloc / torch CUDA memory);
 *     all other pointers are host pointers.  The caller allocates and owns
 *     every buffer; the library allocates no device memory and keeps no
 *     per-call state.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device calls only enqueue work on it: they never synchronise
 *     and never read device memory from the host, so they can be captured in
 *     a CUDA graph.
 *   - Errors the host can see (null pointers, bad sizes, bad alignment) are
 *     returned at once and nothing is launched.  Errors only the device can
 *     see (a negative count, a count beyond a buffer, a timed-out wait) are
 *     written to *d_status (int32, device) with the first error winning; the
 *     caller reads it when it chooses.  d_status may be NULL, in which case
 *     device-side errors are dropped.  Nothing aborts, traps or throws.
 *   - Every wait inside a kernel is bounded (see mg_set_wait_limit_ns): a
 *     kernel that cannot make progress writes MG_ERR_TIMEOUT to *d_status,
 *     drains its own in-flight copies, frees its tensor memory and returns.
 *   - Global base addresses must be 16-byte aligned; N and K must be
 *     multiples of 128.  The GEMM calls take at most 1024 experts and
 *     E * N < 2^31 (weight rows are 32-bit coordinates); FP8 forms take
 *     K <= 16384.  Beyond these limits a call returns MG_ERR_UNSUPPORTED.
 */
#ifndef MOEGEMM_H
#define MOEGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MG_OK = 0,
  MG_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad value      */
  MG_ERR_UNSUPPORTED = 2,  /* valid request this library does not handle      */
  MG_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed               */
  MG_ERR_CAPACITY = 4,     /* output or tile list too small for the counts     */
  MG_ERR_TIMEOUT = 5,      /* a device wait ran past the wait limit            */
  MG_ERR_DEVICE_ARG = 6    /* device-resident argument invalid (count < 0, ...) */
} mg_status;

typedef enum {
  MG_BF16 = 0,             /* bf16 operands, fp32 accumulate                   */
  MG_FP8_E4M3_UE8M0 = 1,   /* E4M3 operands with UE8M0 per-128 block scales    */
  MG_FP8_X_FP4_E2M1 = 2    /* E4M3 activations as above x E2M1 (FP4) weights
                              with one UE8M0 scale per (row, 32 K)             */
} mg_dtype;

/* Padding accounting of one histogram at one token tile q ("MoE GroupGEMM
 * padding under expert skew", "Calculate padded token columns", "Summarize
 * skew without losing the histogram").  48 bytes, naturally aligned. */
typedef struct {
  int64_t P;           /* padded token rows  sum_e q*ceil(t_e/q)             */
  int64_t U;           /* useful token rows  sum_e t_e                        */
  int64_t sumsq;       /* sum_e t_e^2; INT64_MAX when it is 2^63 or more      */
  int32_t active;      /* experts with t_e > 0                                */
  int32_t num_tiles;   /* sum_e ceil(t_e/q); 2^31-1 when it is that or more   */
  double pad_frac;     /* (double)(P-U) / (double)P; 0.0 when P == 0          */
  double eff_experts;  /* ((double)U*(double)U) / (double)(exact sum_e t_e^2),
                          every conversion and operation rounded to nearest;
                          0.0 if no expert has tokens                         */
} mg_plan_stats;

/* Human-readable name of a status code (static string, never NULL). */
const char* mg_status_str(mg_status s);

/* ------------------------------------------------------------------------
 * Planning.  Defined by "MoE GroupGEMM padding under expert skew",
 * "Calculate padded token columns": with t_e tokens for expert e and token
 * tile q, expert e executes q*ceil(t_e/q) rows; P sums them, U sums t_e, the
 * padding fraction is (P-U)/P; effective experts is U^2 / sum t_e^2
 * ("Summarize skew without losing the histogram").  The offsets are the
 * M-grouped contiguous layout: expert segments concatenated in expert order,
 * each starting on a multiple of q ("flops/deepgemm-grouped-masked-moe-gemm",
 * "Arithmetic intensity").
 *
 *   counts / d_counts  int32 [E], t_e >= 0; 1 <= E <= 2^20 and q >= 1
 *                      (else MG_ERR_INVALID_ARG).
 *   offsets            int64 [E+1]: offsets[e] = sum_{e'<e} q*ceil(t_e'/q),
 *                      offsets[E] = P.  Expert e's rows: [offsets[e],
 *                      offsets[e] + t_e).
 *   tiles              int32 [3*max_tiles] or NULL: triples (e, first_row,
 *                      rows) for e ascending and j ascending over
 *                      0..ceil(t_e/q)-1: (e, offsets[e] + j*q,
 *                      min(q, t_e - j*q)).  Experts with t_e = 0 get none.
 *   max_tiles          capacity of `tiles` in triples.
 *   stats              the accounting above.
 *
 * A caller that does not know how many tiles to expect calls once with
 * tiles = NULL and max_tiles = 0 (only offsets and stats are written) and
 * sizes the list from stats.num_tiles.
 *
 * If there are more than max_tiles tiles, the first max_tiles are written,
 * offsets and stats are complete, and the call reports MG_ERR_CAPACITY.
 * Tile rows are int32: when a tile list is requested and P exceeds 2^31-1,
 * only tiles whose first row fits are written and the call reports
 * MG_ERR_UNSUPPORTED (offsets and stats stay complete).
 * A negative count is MG_ERR_INVALID_ARG (host) / MG_ERR_DEVICE_ARG (device,
 * that expert counted as 0).  P and U are exact in int64 for E <= 2^20 and
 * t_e < 2^31; sum_e t_e^2 is formed exactly in two words, so sumsq is exact
 * whenever it fits int64 (three experts at 2^31-1 tokens do not: sumsq then
 * reads INT64_MAX) and eff_experts is correct either way.  The two doubles
 * are correctly rounded IEEE operations in the order written above,
 * identical on host and device.
 * ------------------------------------------------------------------------ */

/* Host, synchronous, touches no GPU. */
mg_status moe_plan_host(const int32_t* counts, int32_t E, int32_t q,
                        int64_t* offsets, int32_t* tiles, int32_t max_tiles,
                        mg_plan_stats* stats);

/* Device, stream-ordered; all pointers are device pointers (d_tiles may be
 * NULL).  One small kernel; the host never reads the counts. */
mg_status moe_plan(const int32_t* d_counts, int32_t E, int32_t q,
                   int64_t* d_offsets, int32_t* d_tiles, int32_t max_tiles,
                   mg_plan_stats* d_stats, int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * Token-tile selection.  The tile along the token dimension is chosen from
 * the count histogram, on the GPU, with no host round trip ("MoE GroupGEMM
 * padding under expert skew", "Adapt kernels without adding a CPU stall").
 * Candidates are priced by padded MMA work, weight/activation traffic and
 * per-tile scheduling cost ("Padding is not the whole cost model"); the
 * constants were measured on GB300.  This is the choice mgemm_contiguous
 * makes when called with tile_q = 0, and mgemm_masked always.
 *
 *   dt, N, K      as for mgemm_contiguous.
 *   d_counts      int32 [E] (device) / counts (host).
 *   d_tile_q      int32 (device): the chosen token tile, one of 32, 64, 128,
 *                 256 (bf16) or 32, 64, 128, 240 (fp8).
 *   num_sms       (host variant) SM count to price waves against; <= 0 uses
 *                 152.
 * ------------------------------------------------------------------------ */
mg_status moe_select_tile(mg_dtype dt, const int32_t* d_counts, int32_t E,
                          int32_t N, int32_t K, int32_t* d_tile_q,
                          int32_t* d_status, void* stream);
mg_status moe_select_tile_host(mg_dtype dt, const int32_t* counts, int32_t E,
                               int32_t N, int32_t K, int32_t num_sms,
                               int32_t* tile_q);

/* ------------------------------------------------------------------------
 * Exemplar selector ("MoE GroupGEMM padding under expert skew", "Adapt
 * kernels without adding a CPU stall": sort and normalise the per-expert
 * count vector, match it against exemplars tuned offline on the GPU, and add
 * guardrails so neighbouring histograms do not switch kernels every layer;
 * "Padding is not the whole cost model": the table comes from measurement,
 * not from the padding formula).  The pages give the steps; the integer
 * definitions below are this library's, so host and device agree exactly.
 *
 * Features of counts c[0..E) (negative counts read as 0), U = sum c:
 *   share[k-1] = floor(65536 * (sum of the m_k largest counts) / U),
 *                m_k = ceil(k*E/16), k = 1..16  (all 0 when U = 0);
 *   lu         = 16*e + floor(16*(U - 2^e) / 2^e), e = floor(log2 U)
 *                (0 when U = 0).
 * Distance to exemplar x: sum_k |share[k] - x.share[k]| + 2048*|lu - x.lu|.
 * Choice: the smallest distance, the lowest index on ties.  Hysteresis: with
 * a state word holding the previous choice p (>= 0), p is kept while
 * dist(p) - dist(best) <= margin; the state then holds the choice.
 *
 * The tactic written for the GEMM calls below: int32 [3] = {tile_q, blocks,
 * exemplar index}; tile_q a multiple of 16 in [16, 256], blocks 1 or 2
 * (weight blocks of 128 rows per tile).  A chosen exemplar with other
 * values writes {0, 0, index} and MG_ERR_DEVICE_ARG.
 * ------------------------------------------------------------------------ */
#define MG_EXEMPLAR_SHARES 16
typedef struct {
  int32_t lu;
  int32_t share[MG_EXEMPLAR_SHARES];
  int32_t tile_q;      /* token tile to use for histograms near this one      */
  int32_t blocks;      /* weight blocks per tile: 1 or 2                       */
  int32_t reserved;    /* 0                                                    */
} mg_exemplar;         /* 80 bytes */

/* Host: the features of one histogram (for building tables); 1 <= E <= 4096
 * (MG_ERR_UNSUPPORTED above, the device call's limit). */
mg_status moe_exemplar_features_host(const int32_t* counts, int32_t E, int32_t* lu,
                                     int32_t* share /* [16] */);
/* Host: the choice for one histogram (prev < 0: no history); E as above. */
mg_status moe_select_exemplar_host(const int32_t* counts, int32_t E, const mg_exemplar* table,
                                   int32_t n, int32_t margin, int32_t prev, int32_t* choice);
/* Device, one small kernel.  d_table: n entries in device memory (n <= 1024);
 * E <= 4096; d_state: int32 or NULL (no hysteresis; initialise to -1);
 * d_tactic: int32 [3] as above. */
mg_status moe_select_exemplar(const int32_t* d_counts, int32_t E, const mg_exemplar* d_table,
                              int32_t n, int32_t margin, int32_t* d_state, int32_t* d_tactic,
                              int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * M-grouped contiguous grouped GEMM ("flops/deepgemm-grouped-masked-moe-
 * gemm", "Workarounds": contiguous layout for prefill/training; "Arithmetic
 * intensity": segments aligned to the M block; "MoE GroupGEMM padding under
 * expert skew", "Grouped execution does not require padded experts": tiles
 * are built from each expert's actual count, zero-sized experts load no
 * weights, tail rows are excluded).
 *
 * For every expert e with t_e = d_counts[e] > 0 and every r < t_e:
 *     D[off_e + r, :] = A[off_e + r, :] * B[e]^T
 * where off_e = sum_{e'<e} align_q*ceil(t_e'/align_q) (moe_plan at q =
 * align_q).  No other row of D is written: padding rows keep whatever the
 * caller left there.
 *
 *   A     [rows_cap, K]   bf16, or E4M3 bytes (dt = MG_FP8_E4M3_UE8M0).
 *   SFA   uint8 [K/128, rows_cap]: UE8M0 scale of (row, 128-wide K block),
 *         K-block major so one block's scales for consecutive rows are
 *         contiguous.  fp8 only; NULL for bf16.
 *   B     [E, N, K]       bf16 or E4M3 bytes.
 *   SFB   uint8 [E, K/128, N/128]: UE8M0 scale of each 128x128 weight block.
 *         fp8 only; NULL for bf16.
 *   D     [rows_cap, N]   bf16 (fp32 accumulation, one final rounding).
 *   align_q  layout alignment of expert segments (>= 1; a multiple of 16
 *            for fp8).  rows_cap must be < 2^31.
 *   tile_q   token tile of the kernel: 0 = chosen on the device from the
 *            counts (moe_select_tile); otherwise a multiple of 16 in
 *            [16, 256] (fp8: [16, 240] or 256).  The result does not depend
 *            on it.
 *
 * Value of an E4M3 element: e4m3(x) * 2^(s-127) with s its block's scale
 * byte.
 *
 * FP8 x FP4 (dt = MG_FP8_X_FP4_E2M1; "flops/deepgemm-grouped-masked-moe-
 * gemm", "Workarounds": FP8xFP4 linear layers; the weight format follows the
 * OCP Microscaling convention, the pages give none).  A and SFA as for
 * E4M3.  B is uint8 [E, N, K/2]: two E2M1 codes per byte, element 2i of a
 * row in the low nibble of byte i, value (-1)^s * {0, 0.5, 1, 1.5, 2, 3, 4,
 * 6}.  SFB is uint8 [E, N, K/32]: the UE8M0 scale of (weight row, 32
 * consecutive K).  K must be a multiple of 512 (else MG_ERR_UNSUPPORTED) and
 * B 32-byte aligned.  Weight bytes read from HBM are half those of E4M3.
 * The SM-pair kernel families are not used (policies 3 and 4 run 2).
 *
 * Device errors: t_e < 0 -> MG_ERR_DEVICE_ARG (expert skipped);
 * aligned segments beyond rows_cap -> MG_ERR_CAPACITY (experts that do not
 * fit are skipped).
 * ------------------------------------------------------------------------ */
mg_status mgemm_contiguous(mg_dtype dt, const void* A, const uint8_t* SFA,
                           const void* B, const uint8_t* SFB, void* D,
                           const int32_t* d_counts, int32_t E,
                           int64_t rows_cap, int32_t N, int32_t K,
                           int32_t align_q, int32_t tile_q,
                           int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * Masked grouped GEMM ("flops/deepgemm-grouped-masked-moe-gemm",
 * "Workarounds": masked grouped GEMM for decode under CUDA graphs;
 * "Arithmetic intensity": each expert owns a fixed-size buffer and a
 * per-expert row count on the device tells the kernel how many of its rows
 * to compute, so the host never waits for the routing result).
 *
 * For every e and every r < v_e = d_valid_m[e]:
 *     D[e, r, :] = A[e, r, :] * B[e]^T
 * Rows r >= v_e are not written; experts with v_e = 0 load nothing.
 *
 *   A     [E, M_max, K]    bf16 or E4M3 bytes.
 *   SFA   uint8 [E, K/128, M_max] (fp8 and fp8 x fp4; M_max a multiple of 16).
 *   B, SFB  as for mgemm_contiguous (all three dtypes).
 *   D     [E, M_max, N]    bf16.
 *   E*M_max must be < 2^31.
 * Device errors: v_e < 0 or v_e > M_max -> MG_ERR_DEVICE_ARG (expert
 * skipped).
 * ------------------------------------------------------------------------ */
mg_status mgemm_masked(mg_dtype dt, const void* A, const uint8_t* SFA,
                       const void* B, const uint8_t* SFB, void* D,
                       const int32_t* d_valid_m, int32_t E, int32_t M_max,
                       int32_t N, int32_t K, int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * Grouped GEMM with the expert's SwiGLU fused into the epilogue
 * ("flops/deepgemm-grouped-masked-moe-gemm", "Workarounds": the fused MoE
 * kernel runs SwiGLU between the two grouped GEMMs, and the FP8 path hands
 * the second GEMM E4M3 activations with UE8M0 per-128 scales).  The pages
 * name SwiGLU without writing it out; this is the standard definition
 *     y = SiLU(g) * u,   SiLU(x) = x / (1 + exp(-x)).
 *
 * B holds GEMM1's gate and up weights interleaved in 128-row blocks: for
 * feature block j (features 128j..128j+127 of I = N/2), rows 256j..256j+127
 * are the gate rows and rows 256j+128..256j+255 the up rows.  With
 * H = A * B[e]^T (fp32 accumulation, as in mgemm_contiguous / mgemm_masked):
 *     Y[row, 128j + i] = SiLU(H[row, 256j + i]) * H[row, 256j + 128 + i]
 * computed in fp32, for the same rows the plain call would write; no other
 * row of Y (or column of SFY) is written.  SiLU uses the fast exponential
 * and division (relative error below (8 + 1.2|g|) 2^-23), and a SiLU whose
 * true value is below |g| 2^-126 comes out as 0.
 *
 *   out = MG_SWIGLU_BF16:  Y bf16 [rows, I] (round to nearest even); SFY
 *         unused (may be NULL).
 *   out = MG_SWIGLU_FP8_E4M3_UE8M0:  Y E4M3 bytes [rows, I] and SFY uint8:
 *         for each (row, 128-feature block j) the scale byte s is the
 *         smallest with max|y| <= 448 * 2^(s-127), clamped to [1, 254]
 *         (127 for an all-zero block), and each code is the nearest E4M3
 *         value of y * 2^(127-s), ties to even, magnitudes past 448
 *         saturating to 448.  SFY is laid out like the activation scales of
 *         the next GEMM: [I/128, rows_cap] (contiguous) or [E, I/128, M_max]
 *         (masked), so Y and SFY feed mgemm_contiguous / mgemm_masked with
 *         K = I directly (rows_cap, align_q and M_max multiples of 16).
 *
 * rows = rows_cap (contiguous) or E*M_max (masked).  All other arguments,
 * requirements and device errors are those of mgemm_contiguous /
 * mgemm_masked.  N must be a multiple of 256 (else MG_ERR_UNSUPPORTED).
 * mgemm_contiguous_swiglu runs CTA pairs (a tile: two feature blocks, each
 * SM one gate block and its up block) where mgemm_contiguous would run the
 * pair two-block family (N % 512 == 0, E4M3 or bf16 weights, default or
 * pair-dual policy); otherwise, and for mgemm_masked_swiglu always, the
 * single-SM two-block kernel (tile = one gate block and its up block).
 * ------------------------------------------------------------------------ */
typedef enum {
  MG_SWIGLU_BF16 = 1,
  MG_SWIGLU_FP8_E4M3_UE8M0 = 2
} mg_swiglu_out;

mg_status mgemm_contiguous_swiglu(mg_dtype dt, mg_swiglu_out out, const void* A,
                                  const uint8_t* SFA, const void* B, const uint8_t* SFB,
                                  void* Y, uint8_t* SFY, const int32_t* d_counts, int32_t E,
                                  int64_t rows_cap, int32_t N, int32_t K, int32_t align_q,
                                  int32_t tile_q, int32_t* d_status, void* stream);
mg_status mgemm_masked_swiglu(mg_dtype dt, mg_swiglu_out out, const void* A, const uint8_t* SFA,
                              const void* B, const uint8_t* SFB, void* Y, uint8_t* SFY,
                              const int32_t* d_valid_m, int32_t E, int32_t M_max, int32_t N,
                              int32_t K, int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * The contiguous and masked forms with the token tile and the blocks per
 * tile read from a device tactic (int32 [3], e.g. written by
 * moe_select_exemplar): no host round trip between the choice and the GEMM,
 * and both launches can be captured in one CUDA graph.  Arguments, results
 * and errors are those of mgemm_contiguous / mgemm_masked (with tile_q taken
 * from the tactic; tiles wider than the kernel allows are narrowed, which
 * does not change the result).  These calls run the kernel family that
 * mg_set_kernel_policy selects for mgemm_contiguous / mgemm_masked, with
 * tiles of one or two of that family's weight blocks (`blocks`: 128 rows on
 * one SM, 256 on an SM pair); a tactic that is not valid is reported as
 * MG_ERR_DEVICE_ARG and the kernel's own choice is used.
 * ------------------------------------------------------------------------ */
mg_status mgemm_contiguous_tactic(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                                  const uint8_t* SFB, void* D, const int32_t* d_counts, int32_t E,
                                  int64_t rows_cap, int32_t N, int32_t K, int32_t align_q,
                                  const int32_t* d_tactic, int32_t* d_status, void* stream);
mg_status mgemm_masked_tactic(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                              const uint8_t* SFB, void* D, const int32_t* d_valid_m, int32_t E,
                              int32_t M_max, int32_t N, int32_t K, const int32_t* d_tactic,
                              int32_t* d_status, void* stream);

/* The masked form with the exemplar matched inside the GEMM ("MoE GroupGEMM
 * padding under expert skew", "Adapt kernels without adding a CPU stall":
 * the choice stays on the GPU, here without a kernel of its own, which on
 * decode batches cost more than the tile choice saves).  Every CTA computes
 * the features of d_valid_m and picks the nearest exemplar exactly as
 * moe_select_exemplar does with margin 0 and no history (no state is
 * shared between CTAs), then runs with its tile_q and blocks.  E <= 32
 * (decode batches; MG_ERR_UNSUPPORTED above), 1 <= n <= 1024, d_table and
 * d_tactic_out 16-byte aligned.  d_tactic_out: int32 [3] or NULL; if given,
 * the first CTA writes {tile_q, blocks, index} of the choice.  A table entry
 * with an invalid tactic is reported as MG_ERR_DEVICE_ARG and the kernel's
 * own choice is used.  Other arguments, results and errors as mgemm_masked. */
mg_status mgemm_masked_exemplar(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                                const uint8_t* SFB, void* D, const int32_t* d_valid_m, int32_t E,
                                int32_t M_max, int32_t N, int32_t K, const mg_exemplar* d_table,
                                int32_t n, int32_t* d_tactic_out, int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * K-grouped weight-gradient GEMM ("flops/deepgemm-grouped-masked-moe-gemm",
 * "Workarounds": K-grouped GEMM for MoE weight backward, M and N fixed and
 * the contraction length varying per expert).
 *
 * With tok_e = sum_{e'<e} t_e' (tokens packed by expert, no alignment):
 *     dW[e] = sum_{t in [tok_e, tok_e + t_e)} dY[t, :]^T X[t, :]   ([N, K])
 * dW is overwritten; experts with t_e = 0 get dW[e] = 0 with no loads.
 *
 *   dY    bf16 [T_cap, N];  X  bf16 [T_cap, K];  dW  fp32 [E, N, K].
 *   T_cap < 2^31.
 * Device errors: t_e < 0 -> MG_ERR_DEVICE_ARG; sum t_e > T_cap ->
 * MG_ERR_CAPACITY; dW[e] of an expert that does not fit is not written.
 * ------------------------------------------------------------------------ */
mg_status kgemm_grouped(const void* dY, const void* X, float* dW,
                        const int32_t* d_counts, int32_t E, int64_t T_cap,
                        int32_t N, int32_t K, int32_t* d_status, void* stream);

/* ------------------------------------------------------------------------
 * Bounded waits.  Every kernel spin-wait gives up after this many
 * nanoseconds of wall time measured from the CTA's start (default 2e9),
 * writing MG_ERR_TIMEOUT.  Process-wide; not thread-safe against concurrent
 * launches.  ns <= 0 restores the default.
 * ------------------------------------------------------------------------ */
mg_status mg_set_wait_limit_ns(int64_t ns);
int64_t mg_get_wait_limit_ns(void);

/* ------------------------------------------------------------------------
 * Kernel family for the contiguous and masked forms.  A tile is one or two
 * weight blocks against one token tile; a block is 128 weight rows on one SM
 * or 256 rows on the two SMs of a cluster sharing each MMA (cta_group::2).
 * Families 1-4 put the tokens on the MMA's N axis (token tiles up to 240
 * rows for E4M3, 256 for bf16); family 5 puts them on its M axis (token
 * tiles of up to 128 rows against 256 weight rows per MMA).
 *   0 (default): contiguous form: SM pair, two blocks when N % 512 == 0,
 *      else as 2; masked form and E2M1 weights: as 2 (the fastest families
 *      measured on GB300 for prefill and decode shapes);
 *   1: single SM, one block (128 rows);
 *   2: single SM, two blocks (256 rows; needs N % 256 == 0);
 *   3: SM pair, one block (256 rows; needs N % 256 == 0);
 *   4: SM pair, two blocks (512 rows; needs N % 512 == 0);
 *   5: single SM, tokens on M, 256 weight rows (needs N % 256 == 0).
 * A family whose tile does not divide N falls back to the next narrower one
 * (4 -> 3 -> 1, 2 -> 1, 5 -> 1, 0 -> 1).  The two-block families run
 * one-block tiles where the device finds them cheaper from the counts
 * (contiguous form: when two-block tiles would not fill two waves of
 * workers; masked form: priced together with the token tile, E2M1 weights
 * always two blocks).  Results are identical up to fp32 summation order.
 * Process-wide.  Returns MG_ERR_INVALID_ARG for other values.
 * ------------------------------------------------------------------------ */
mg_status mg_set_kernel_policy(int32_t policy);
int32_t mg_get_kernel_policy(void);

/* Self-test of the bounded wait: one CTA waits on a shared-memory barrier
 * that nothing will ever complete, with a limit of limit_ns, and must write
 * MG_ERR_TIMEOUT to *d_status and return.  Faults nothing. */
mg_status mg_wait_selftest(int32_t* d_status, int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOEGEMM_H */
