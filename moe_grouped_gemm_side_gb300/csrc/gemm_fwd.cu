// Contiguous and masked MoE grouped GEMM for sm_103a (bf16, and E4M3 with
// UE8M0 per-128 block scales).
//
// "flops/deepgemm-grouped-masked-moe-gemm", "Arithmetic intensity" and
// "Workarounds": N and K are shared by all experts; the contiguous form
// concatenates each expert's token rows on M-block boundaries, the masked
// form keeps fixed per-expert buffers and computes only the first valid_m[e]
// rows.  "MoE GroupGEMM padding under expert skew", "Grouped execution does
// not require padded experts": a persistent kernel builds its tiles from the
// actual counts, experts with no tokens produce no tiles (so their weights are
// never loaded) and tail rows are not written.
//
// Tile shape.  Tokens sit on the MMA N axis and weight rows on the MMA M
// axis.  A tile is kBlocks weight blocks x q_n token rows, q_n any multiple
// of 16 up to 256 chosen per tile at run time: full tiles use the selected
// token tile q, an expert's last tile is trimmed to round_up(rows, 16).  The
// instruction descriptor and the TMA box count are runtime values, so one
// launch serves every tile size with no host round trip ("Adapt kernels
// without adding a CPU stall").  A weight block is 128 rows on one SM
// (cta_group::1) or 256 rows on the two SMs of a cluster (kPair,
// cta_group::2: each SM holds 128 weight rows and half of the token rows,
// and the MMA reads the other half from the peer).  With kTokM the roles
// swap: 128 token rows on M, the tile's 256 weight rows on N, one MMA per
// K-step for both blocks, one issuing warp.
//
// Why bigger tiles.  Every MMA reads both operands from shared memory while
// TMA writes the next stages into it; with one 128-row block a K-block stage
// moves ~94 KB through an SM's shared memory for 3.9 M fp8 multiply-adds and
// the tensor pipe waits.  Two blocks against the same token tile, and the
// pair's split of the token operand, cut the bytes per multiply-add.  Two
// 240/256-column fp32 accumulators fill TMEM, so the next tile's MMAs wait
// until the epilogue has read the accumulators; the epilogue then parks most
// of the tile in registers (as bf16) and stores it while they run.
//
// CTA = 16 warps: warp 0 issues TMA; warps 1 and 11 issue the tcgen05.mma
// and tcgen05.cp (below; on a CTA pair those of the first CTA); warps 2-5,
// 7-10 and 12-15 drain the fp32 accumulators from TMEM (three warps per
// 32-lane quadrant, every third 16-token chunk) and store bf16 rows; warp 6
// (fp8 only) turns the raw UE8M0 bytes into the TMEM scale-word layout, four
// K-blocks per word.
//
// MMA issue.  The tensor pipe queues only about two MMAs, so whatever the
// issuing thread does between MMAs (a barrier test ~90 cycles, a commit ~60,
// address arithmetic) shows up as idle pipe time: with one issuing thread a
// stage of eight 128 x 240 x 32 block-scaled MMAs took ~1530 cycles against
// ~1300 of MMA work (in-kernel clock stamps).  So on one SM two warps issue,
// each into a 256-column TMEM allocation of its own holding its accumulator
// and its copy of the scale words: for two-block tiles warp 1 issues block
// 0's MMAs and warp 11 block 1's; for one-block tiles each issues two of
// every stage's four K-steps into its own accumulator, and the epilogue adds
// the two partial sums (one fp32 addition, then the single bf16 rounding).
// One thread's barrier tests and commits then overlap the other's queued
// MMAs.  The issuing warps run their loops with all 32 lanes and lane 0
// alone executes each tcgen05 instruction: descriptors and addresses stay
// warp-uniform, which made issue cheaper again (FP8 GEMM1 of the skewed
// prefill: 0.844 ms with one single-lane issuer, 0.811 with two, 0.788 with
// two warp-wide; BF16 GEMM2: 0.841, 0.797, 0.743).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "mg_internal.h"
#include "sched.cuh"

namespace mg {
namespace fwd {

constexpr int kThreads = 512;
constexpr int kSfWarp = 6;
// Second MMA-issuing warp of single-SM two-block tiles (block 1's MMAs).
constexpr int kMma2Warp = 11;
// warps 2-5, 7-10 and 12-15: three per TMEM lane quadrant
constexpr int kEpiWarps = 12;
// plain epilogue: chunks of 16 tokens a warp parks in registers (as bf16)
// before it releases the accumulator
constexpr int kParked = 4;
constexpr int kMaxStages = 16;
constexpr int kCtaRows = 128;                    // weight rows of one block on one SM
constexpr int kRowBytes = 128;                   // K bytes per stage and row
constexpr int kWTileBytes = kCtaRows * kRowBytes;  // 16 KB
constexpr int kSfRaw = kSfRawBytes;              // [4][256] token scale bytes
// per-stage scale area: raw bytes, weight words of block 0, token words,
// weight words of block 1
constexpr int kSfStage = kSfStageBytes + 512;
constexpr int kSfW1 = kSfStageBytes;             // offset of block-1 weight words
// FP4 weights, per stage after the fp8 scale area: each block's scale box
// as loaded (128 rows x 16 bytes: K-blocks kb..kb+3 of the stage's group,
// four 32-K sub-blocks each), then each block's TMEM scale atom for the
// stage's K-block (32 lanes x 16 bytes: lane i, word j = the four sub-block
// scales of row i + 32 j), the layout tcgen05.cp.32x128b.warpx4 expects.
constexpr int kWsfBytes = kCtaRows * 16;
constexpr int kWsfAtom = 32 * 16;
// The boxes arrive once per group of four K-blocks, into a ring of
// kW4Groups group slots (both blocks' boxes per slot) ahead of the stage
// ring; every stage keeps only its two atoms.  (A box in every stage took
// 8 KB of scale data per stage: one stage fewer in the ring, and the decode
// waited on its loads.)  The scale warp releases a slot (sf_grp) when it
// starts the next group, and the producer reloads it only after that.  Two
// slots hold 8 KB where the boxes took 4 KB in every stage: two-block tiles
// of 128 tokens keep four stages in the ring instead of three.
constexpr int kW4Groups = 2;
constexpr int kW4GroupBytes = 2 * kWsfBytes;
constexpr int kW4Area = kW4Groups * kW4GroupBytes;
constexpr int kW4StageBytes = 2 * kWsfAtom;
static_assert(kSfStage % 1024 == 0 && kWsfBytes % 1024 == 0 && kWsfAtom % 16 == 0,
              "TMA and tcgen05.cp sources stay aligned");
constexpr int kGroupTiles = 8;                   // token tiles per raster group
// CTA pairs, fp8: slots of the ring of scale groups (raw token scales and
// scale words of four K-blocks each), loaded one group ahead of the stage
// that consumes them
constexpr int kGRing = 8;
// Launches with one-block tiles and at most this many token tiles deal their
// tiles by cost (see balanced_position)
constexpr int kBalMax = 512;
// Token-tile widths the producer publishes for the MMA thread, one slot per
// tile; more slots than stages, so a slot is rewritten only after the MMA
// thread has read it.
constexpr int kInfoRing = 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBytes = 227 * 1024;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

struct Params {
  const int32_t* counts;
  const uint8_t* sfb;
  void* D;           // bf16 [rows, N]; with a SwiGLU epilogue Y [rows, N/2] (bf16 or E4M3)
  uint8_t* sfy;      // SwiGLU to E4M3: UE8M0 scales of Y, [z][N/256][sfy_ld]
  int32_t* status;
  int64_t wait_ns;
  int32_t E, N, K;
  int32_t masked, fp8;
  int32_t rows_total, M_max, align_q, tile_q;
  int32_t epi;       // kEpiPlain, kEpiSwigluBf16 or kEpiSwigluFp8
  int32_t sfy_ld;
  const int32_t* tactic;  // device {tile_q, blocks} chosen elsewhere on the GPU, or null
  const mg_exemplar* table;  // exemplar table to match in the prologue (E <= 32), or null
  int32_t n_table;
  int32_t* tactic_out;    // with a table: the first CTA writes {tile_q, blocks, index}
};

struct Shared {
  uint64_t full[kMaxStages];      // operand bytes (of both CTAs of a pair) landed
  uint64_t empty[kMaxStages];     // the MMAs reading the stage are done
  uint64_t sf_full[kMaxStages];   // fp8: this CTA's raw scale bytes of the stage landed
  uint64_t acc_full[1];
  uint64_t acc_empty[1];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t tmem_base2;  // two issuers: block 1's own TMEM allocation
  int32_t abort_flag;
  int32_t q;         // token tile of full tiles
  int32_t qn_max;    // widest tile of this launch
  int32_t total;     // tiles of this launch
  int32_t nblk;      // weight blocks per tile of this launch
  int32_t bal;       // tiles dealt by cost (ttab) rather than in raster order
  int32_t tile_qn[kInfoRing];
  // SwiGLU to E4M3: per-token maxima of each lane quadrant over the tile's
  // tokens, exchanged between the four epilogue warps of one half
  uint64_t amax_bar[2];
  float amax[4][256];
  // pairs, fp8: group slot s of the scale ring: raw bytes landed (g_full),
  // words built in both CTAs (sf_grp, on the first CTA)
  uint64_t g_full[kGRing];
  uint64_t sf_grp[kGRing];
};

struct Tile {
  int32_t e, nb, row0, rows, qn, sf_x, sf_z;
};

template <int V>
struct IntC {
  static constexpr int value = V;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t deadline,
                                          volatile int32_t* abort_flag, int32_t* status) {
  const bool ok = wait_bounded(bar, parity, deadline, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Where the CTA that walks positions unit, unit + n_units, ... finds its
// tiles when they are dealt by cost: position t (round r = t / n_units)
// takes the (t mod n_units)-th tile of round r counted from the front in even
// rounds and from the back in odd ones (a snake), over the launch's tiles in
// order of decreasing cost (ttab: token tiles by decreasing width, each with
// its weight blocks).  Every CTA then holds a similar mix of wide and narrow
// tiles: with one-block decode tiles the token rows a tile streams differ by
// up to 8x between experts, and the round-robin deal left CTAs finishing from
// 54 to 85 us on the 16-expert decode (in-kernel global-timer stamps).
__device__ __forceinline__ int32_t balanced_position(int32_t t, int32_t total, int32_t n_units) {
  const int32_t r = t / n_units, u = t - r * n_units;
  const int32_t in_round = min(n_units, total - r * n_units);
  return r * n_units + ((r & 1) ? in_round - 1 - u : u);
}

// Tile t of the launch.  Raster order: experts in order; inside an expert,
// groups of kGroupTiles token tiles sweep all weight blocks before moving on,
// so CTAs working at the same time share weight and activation tiles in L2.
// With `even` (FP8) an expert's ceil(t_e / q) token tiles split its rows
// evenly, widths rounded up to 16 and the last tile trimmed (t_e = 445,
// q = 240: two tiles of 224 rather than 240 and 208); measured on the
// skewed FP8 prefill, GEMM1 0.726 -> 0.717 ms, GEMM2 unchanged, while the
// BF16 GEMMs came out within +-1 % either way, so they keep full tiles of q.
// Dealt by cost (bal): token tile ttab[k / NB], weight block k % NB, with k
// the balanced position of t, full tiles of width q.
__device__ __forceinline__ Tile decode_tile(int32_t t, const int32_t* tpre, const int32_t* cnt,
                                            const int32_t* rowbase, int32_t E, int32_t NB,
                                            int32_t q, int32_t masked, const int32_t* ttab, int32_t bal,
                                            int32_t total, int32_t n_units, int32_t even) {
  if (bal) {
    const int32_t k = balanced_position(t, total, n_units);
    const int32_t j = k / NB;
    const int32_t ent = ttab[j];
    Tile tl;
    tl.e = ent >> 16;
    tl.nb = k - j * NB;
    const int32_t in_e = (ent & 0xFFFF) * q;
    tl.rows = min(q, cnt[tl.e] - in_e);
    tl.qn = round_up16(tl.rows);
    tl.row0 = rowbase[tl.e] + in_e;
    tl.sf_x = masked ? in_e : tl.row0;
    tl.sf_z = masked ? tl.e : 0;
    return tl;
  }
  int32_t lo = 0, hi = E;  // tpre[lo] <= t < tpre[hi]
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (tpre[mid] <= t) lo = mid; else hi = mid;
  }
  Tile tl;
  tl.e = lo;
  const int32_t mt = (tpre[lo + 1] - tpre[lo]) / NB;
  const int32_t l = t - tpre[lo];
  const int32_t g = l / (kGroupTiles * NB);
  const int32_t gbase = g * kGroupTiles;
  const int32_t gsz = min(kGroupTiles, mt - gbase);
  const int32_t r = l - g * kGroupTiles * NB;
  tl.nb = r / gsz;
  const int32_t j = gbase + r % gsz;
  const int32_t c = cnt[lo];
  const int32_t w = even ? round_up16((int32_t)cdiv_u32((uint32_t)c, (uint32_t)mt)) : q;
  const int32_t in_e = j * w;
  tl.rows = min(w, c - in_e);
  tl.qn = round_up16(tl.rows);
  tl.row0 = rowbase[lo] + in_e;
  tl.sf_x = masked ? in_e : tl.row0;
  tl.sf_z = masked ? lo : 0;
  return tl;
}

// The packed weight scale word of K-block group g (bytes: K-blocks 4g..4g+3,
// 127 past the end) for g = this lane, from a tile's scales held as lane l
// owning K-blocks l, l+32, l+64, l+96.  Warp-collective; built once per tile
// (16 shuffles), after which a group's word is one shuffle away.  Building
// it per group on the scale warp took ~470 cycles per block and delayed the
// stage's scale words by ~1100 cycles (in-kernel clock stamps).
__device__ __forceinline__ uint32_t group_weight_word(const uint32_t (&wsf)[4], uint32_t lane, int32_t KB) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < kSfGroup; ++i) {
    const int32_t k = 4 * (int32_t)lane + i;
    const uint32_t src = (uint32_t)k & 31u;
    const uint32_t v0 = __shfl_sync(0xffffffffu, wsf[0], src);
    const uint32_t v1 = __shfl_sync(0xffffffffu, wsf[1], src);
    const uint32_t v2 = __shfl_sync(0xffffffffu, wsf[2], src);
    const uint32_t v3 = __shfl_sync(0xffffffffu, wsf[3], src);
    const int32_t sel = (k >> 5) & 3;
    const uint32_t v = sel == 1 ? v1 : sel == 2 ? v2 : sel == 3 ? v3 : v0;
    w |= (k < KB ? (v & 0xFFu) : 127u) << (8 * i);
  }
  return w;
}

// kind::mxf8f6f4 instruction-descriptor A / B format E2M1 (FP4), bits 7-9 / 10-12.
constexpr uint32_t kIdescAE2M1 = 5u << 7;
constexpr uint32_t kIdescBE2M1 = 5u << 10;

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// SwiGLU epilogue of a two-block tile ("flops/deepgemm-grouped-masked-moe-
// gemm", "Workarounds": the expert's SwiGLU runs between the two grouped
// GEMMs, and the FP8 path hands the second GEMM per-128 UE8M0-scaled E4M3
// activations).  GEMM1's weight rows are interleaved in 128-row blocks (gate
// rows of features 128j..128j+127, then their up rows), and each SM loads
// the gate block of its feature group fgrp as its block 0 and the up block
// as its block 1 (one SM: fgrp = tile nb; a CTA pair: fgrp = 2 nb + rank,
// the pair's M = 256 rows being two SMs' gate blocks, then their up blocks),
// so the thread owning TMEM lane l has both halves of one feature:
// y = SiLU(g) * u = g / (1 + e^-g) * u  in fp32.  The two warps of a lane
// quadrant take alternate 16-token chunks, as in the plain epilogue.
__device__ __forceinline__ float swiglu_f32(uint32_t g, uint32_t u) {
  const float gf = __uint_as_float(g);
  return __fdividef(gf, 1.0f + __expf(-gf)) * __uint_as_float(u);
}

// To bf16: lane pairs exchange so each store writes two features.
__device__ __forceinline__ void swiglu_bf16_tile(const Params& p, const Tile& tl, int32_t fgrp, uint32_t taddr,
                                                 uint32_t taddr_up, uint32_t quad, int32_t half,
                                                 uint32_t lane) {
  const int32_t I = p.N >> 1;
  const int32_t f = fgrp * kCtaRows + (int32_t)(quad * 32u + lane);  // this thread's feature
  const bool odd = (lane & 1u) != 0;
  __nv_bfloat16* ypair = static_cast<__nv_bfloat16*>(p.D) + (int64_t)tl.row0 * I + (f & ~1);
  for (int32_t c0 = 16 * half; c0 < tl.qn; c0 += 32) {
    uint32_t g[16], u[16];
    tmem_ld16(taddr + (uint32_t)c0, g);
    tmem_ld16(taddr_up + (uint32_t)c0, u);
    tmem_ld_wait();
    tmem_regs_ready(g);
    tmem_regs_ready(u);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const float y0 = swiglu_f32(g[i], u[i]), y1 = swiglu_f32(g[i + 1], u[i + 1]);
      const int32_t row = c0 + i + (odd ? 1 : 0);
      const float mine = odd ? y1 : y0;
      const float recv = __shfl_xor_sync(0xffffffffu, odd ? y0 : y1, 1);
      const __nv_bfloat162 v = odd ? __floats2bfloat162_rn(recv, mine) : __floats2bfloat162_rn(mine, recv);
      if (row < tl.rows) *reinterpret_cast<__nv_bfloat162*>(ypair + (int64_t)row * I) = v;
    }
  }
}

// To E4M3.  The scale of (token, 128 features) needs the maximum over all
// four lane quadrants, held by the four warps of this half, so the tile is
// drained in two passes with one exchange between them.  Pass 1: y of every
// chunk goes back into TMEM over the gate values, and each warp reduces its
// 32 features per token with a transposing butterfly (16 shuffles for 16
// tokens) into shared memory.  Then the half's 128 threads complete an
// mbarrier (bounded wait; one per tile, parity = tile count).  Pass 2: y is
// read back, and per token the scale byte is the smallest s with
// amax <= 448 * 2^(s-127), clamped to [1, 254] (127 for an all-zero block);
// codes round y * 2^(127-s) to the nearest E4M3 value, saturating; a byte
// transpose inside groups of four lanes turns each lane's 16 one-byte codes
// (one feature, 16 tokens) into four 4-byte stores (four features of one
// token), a quarter of the store instructions of byte stores.  The next
// tile's pass 1 cannot start before every epilogue warp has released this
// tile's accumulator, so one buffer of maxima suffices.  Returns false if
// the wait gave up.
__device__ __forceinline__ bool swiglu_fp8_tile(const Params& p, Shared& sh, const Tile& tl, int32_t fgrp,
                                                uint32_t taddr, uint32_t taddr_up, uint32_t quad,
                                                int32_t half, uint32_t lane, uint32_t tile_par,
                                                uint64_t deadline) {
  const int32_t I = p.N >> 1;
  const int32_t f = fgrp * kCtaRows + (int32_t)(quad * 32u + lane);
  const bool odd = (lane & 1u) != 0;
  const int32_t t = (int32_t)(lane >> 1);
  for (int32_t c0 = 16 * half; c0 < tl.qn; c0 += 32) {
    uint32_t g[16], u[16];
    tmem_ld16(taddr + (uint32_t)c0, g);
    tmem_ld16(taddr_up + (uint32_t)c0, u);
    tmem_ld_wait();
    tmem_regs_ready(g);
    tmem_regs_ready(u);
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float y = swiglu_f32(g[i], u[i]);
      g[i] = __float_as_uint(y);
      m[i] = fabsf(y);
    }
    tmem_st16(taddr + (uint32_t)c0, g);
    // each step halves the live values; afterwards lanes 2t and 2t+1 hold
    // token t's maximum over the warp's 32 features
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
      const bool hi = (lane & (uint32_t)(2 * w)) != 0;
#pragma unroll
      for (int j = 0; j < w; ++j) {
        const float keep = hi ? m[j + w] : m[j];
        const float send = hi ? m[j] : m[j + w];
        m[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 2 * w));
      }
    }
    m[0] = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));
    if (!odd) sh.amax[quad][c0 + t] = m[0];
  }
  tmem_st_wait();
  mbar_arrive(&sh.amax_bar[half]);
  if (!warp_wait(&sh.amax_bar[half], tile_par, deadline, &sh.abort_flag, p.status)) return false;
  uint8_t* yq4 = static_cast<uint8_t*>(p.D) + (int64_t)tl.row0 * I + (f & ~3);
  for (int32_t c0 = 16 * half; c0 < tl.qn; c0 += 32) {
    uint32_t y[16];
    tmem_ld16(taddr + (uint32_t)c0, y);
    tmem_ld_wait();
    tmem_regs_ready(y);
    const int32_t tok = c0 + t;
    const float amax = fmaxf(fmaxf(sh.amax[0][tok], sh.amax[1][tok]), fmaxf(sh.amax[2][tok], sh.amax[3][tok]));
    // amax = 1.m * 2^(E-127); 448 = 1.75 * 2^8: s = E - 8, plus one when 1.m > 1.75
    const uint32_t bits = __float_as_uint(amax);
    int32_t sc = (int32_t)(bits >> 23) - 8 + ((bits & 0x7fffffu) > 0x600000u ? 1 : 0);
    sc = min(max(sc, 1), 254);
    if (amax == 0.0f) sc = 127;
    // 2^(127-s): a normal float for s <= 253, the subnormal 2^-127 for s = 254
    const float inv = sc < 254 ? __uint_as_float((uint32_t)(254 - sc) << 23) : __uint_as_float(0x00400000u);
    if (quad == 0 && !odd && tok < tl.rows)
      p.sfy[((int64_t)tl.sf_z * (I / kCtaRows) + fgrp) * p.sfy_ld + tl.sf_x + tok] = (uint8_t)sc;
    // codes of tokens 4w..4w+3 of this lane's feature, one word per w
    uint32_t wd[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float2 a, b;
      a.x = __uint_as_float(y[4 * w]) * __shfl_sync(0xffffffffu, inv, 8 * w);
      a.y = __uint_as_float(y[4 * w + 1]) * __shfl_sync(0xffffffffu, inv, 8 * w + 2);
      b.x = __uint_as_float(y[4 * w + 2]) * __shfl_sync(0xffffffffu, inv, 8 * w + 4);
      b.y = __uint_as_float(y[4 * w + 3]) * __shfl_sync(0xffffffffu, inv, 8 * w + 6);
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
      wd[w] = (lo & 0xffffu) | (hi << 16);
    }
    // 4x4 byte transpose inside each group of four lanes (features 4a..4a+3):
    // afterwards lane 4a+r holds, per w, the codes of token 4w+r for the
    // group's four features, stored as one word
    const bool b1 = (lane & 2u) != 0, b0 = (lane & 1u) != 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t v = wd[w];
      uint32_t r = __shfl_xor_sync(0xffffffffu, v, 2);
      v = b1 ? __byte_perm(r, v, 0x7632) : __byte_perm(v, r, 0x5410);
      r = __shfl_xor_sync(0xffffffffu, v, 1);
      v = b0 ? __byte_perm(r, v, 0x7351) : __byte_perm(v, r, 0x6240);
      const int32_t row = c0 + 4 * w + (int32_t)(lane & 3u);
      if (row < tl.rows) *reinterpret_cast<uint32_t*>(yq4 + (int64_t)row * I) = v;
    }
  }
  return true;
}

template <int kBlocks, bool kPair, bool kW4, bool kTokM>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA64,
               const __grid_constant__ CUtensorMap tmA16, const __grid_constant__ CUtensorMap tmA8,
               const __grid_constant__ CUtensorMap tmSF, const __grid_constant__ CUtensorMap tmSFW,
               const Params p) {
  static_assert(kBlocks == 1 || kBlocks == 2, "one or two weight blocks per tile");
  static_assert(!(kW4 && kPair), "FP4 weights run on single-SM tiles");
  static_assert(!kTokM || (kBlocks == 2 && !kPair), "tokens-on-M tiles: two blocks on one SM");
  constexpr int kBlockRows = kPair ? 2 * kCtaRows : kCtaRows;  // rows of one weight block (MMA M)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Shared& sh = *reinterpret_cast<Shared*>(smem);
  const int32_t E = p.E;
  int32_t* cnt = reinterpret_cast<int32_t*>(smem + ((sizeof(Shared) + 15) & ~size_t(15)));
  int32_t* rowbase = cnt + E;
  int32_t* tpre = rowbase + E;
  int32_t* ttab = tpre + E + 1;  // token tiles by decreasing width: expert << 16 | tile in expert
  const uintptr_t sched_end = reinterpret_cast<uintptr_t>(ttab + kBalMax);
  uint8_t* sf_area = reinterpret_cast<uint8_t*>((sched_end + 1023) & ~uintptr_t(1023));

  const uint32_t warp = warp_id(), lane = lane_id();
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  // workers: CTAs, or CTA pairs
  const int32_t unit = kPair ? (int32_t)(blockIdx.x >> 1) : (int32_t)blockIdx.x;
  const int32_t n_units = kPair ? (int32_t)(gridDim.x >> 1) : (int32_t)gridDim.x;
  const uint64_t deadline = globaltimer_ns() + (uint64_t)p.wait_ns;
  const int32_t NB128 = p.N / kCtaRows;
  const int32_t KB = p.K / (p.fp8 ? 128 : 64);
  // widest token tile: 256, but 240 for fp8 wherever an accumulator shares
  // its 256 TMEM columns with the scale words
  // (tokens on M: the MMA's M, 128 rows)
  const int32_t q_cap = kTokM ? 128 : (p.fp8 ? 240 : 256);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      // single SM, fp8: the scale warp's arrival completes the stage's
      // operand barrier too, so the MMA thread tests one barrier per stage
      mbar_init(&sh.full[i], (!kPair && p.fp8) ? 2 : 1);
      mbar_init(&sh.sf_full[i], 1);
    }
    mbar_init(&sh.acc_empty[0], kEpiWarps * (kPair ? 2 : 1));  // one arrival per epilogue warp
    // (empty, acc_full and drain count one commit per MMA-issuing thread:
    // initialised once the block count of the launch is known)
    for (int i = 0; i < 2; ++i) mbar_init(&sh.amax_bar[i], 4 * 32);
    for (int i = 0; i < kGRing; ++i) {
      // pairs: both CTAs' scale warps publish a group; FP4 weights on one SM:
      // the scale warp releases a weight-scale group slot
      mbar_init(&sh.sf_grp[i], kPair ? 2 : 1);
      mbar_init(&sh.g_full[i], 1);
    }
    sh.abort_flag = 0;
    fence_barrier_init();
  }

  // ---- validated counts
  for (int32_t e = threadIdx.x; e < E; e += kThreads) {
    int32_t c = __ldg(p.counts + e);
    if (c < 0 || (p.masked && c > p.M_max)) {
      set_status(p.status, MG_ERR_DEVICE_ARG);
      c = 0;
    }
    cnt[e] = c;
  }
  __syncthreads();

  // One SM: the issuing warps allocate their TMEM while warp 0 builds the
  // schedule (allocation and schedule each took ~1500 and ~19000 cycles of
  // the prologue, one after the other).
  if constexpr (!kPair) {
    if (warp == 1) tmem_alloc_keep_permit(&sh.tmem_base, !kTokM ? 256u : kTmemCols);
    if (!kTokM && warp == kMma2Warp) tmem_alloc_keep_permit(&sh.tmem_base2, 256u);
  }

  // ---- schedule (warp 0): row bases, token tile, tile prefix
  if (warp == 0) {
    if (p.masked) {
      for (int32_t e = lane; e < E; e += 32) rowbase[e] = e * p.M_max;
    } else {
      int64_t carry = 0;
      for (int32_t b = 0; b < E; b += 32) {
        const int32_t e = b + lane;
        const int64_t own = e < E ? (int64_t)p.align_q * cdiv_u32((uint32_t)cnt[e], (uint32_t)p.align_q) : 0;
        int64_t v = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t n = __shfl_up_sync(0xffffffffu, v, o);
          if ((int)lane >= o) v += n;
        }
        if (e < E) {
          const int64_t start = carry + v - own;
          if (start + cnt[e] > p.rows_total) {
            cnt[e] = 0;  // segment does not fit: skip the expert
            rowbase[e] = 0;
          } else {
            rowbase[e] = (int32_t)start;
          }
        }
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0 && carry > p.rows_total) set_status(p.status, MG_ERR_CAPACITY);
    }
    __syncwarp();
    int32_t q = p.tile_q;
    int32_t want_blocks = 0;  // 0: decided below from the tile count
    if (p.table != nullptr) {
      // The exemplar choice of the separate select kernel (no history),
      // made by every CTA's warp 0 for E <= 32: lane e holds expert e's
      // count; the warp sorts them (descending, bitonic), forms the prefix
      // sums, the 16 shares and the log feature, and takes the nearest
      // exemplar (L1, ties to the lower index).  Integer arithmetic only,
      // so every CTA makes the same choice.
      int64_t c = (int32_t)lane < E ? (int64_t)cnt[lane] : 0;
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
          const int64_t o = __shfl_xor_sync(0xffffffffu, c, j);
          const bool desc = (lane & (uint32_t)k) == 0, lower = (lane & (uint32_t)j) == 0;
          c = (desc == lower) ? max(c, o) : min(c, o);
        }
      }
      int64_t v = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t nv = __shfl_up_sync(0xffffffffu, v, o);
        if ((int)lane >= o) v += nv;
      }
      const int64_t U = __shfl_sync(0xffffffffu, v, E - 1);
      int32_t share[kExemplarShares];
#pragma unroll
      for (int k = 0; k < kExemplarShares; ++k) {
        const int32_t m = ((k + 1) * E + kExemplarShares - 1) / kExemplarShares;
        const int64_t vm = __shfl_sync(0xffffffffu, v, m - 1);
        share[k] = U > 0 ? (int32_t)((int64_t)kShareOne * vm / U) : 0;
      }
      int32_t lu = 0;
      if (U > 0) {
        const int e = 63 - __clzll(U);
        lu = 16 * e + (int32_t)((16 * (U - (int64_t(1) << e))) >> e);
      }
      int64_t bd = INT64_MAX;
      int32_t bi = 0x7fffffff;
      for (int32_t i = (int32_t)lane; i < p.n_table; i += 32) {
        int64_t d = (int64_t)kLuWeight * llabs((int64_t)lu - p.table[i].lu);
#pragma unroll
        for (int k = 0; k < kExemplarShares; ++k) d += llabs((int64_t)share[k] - p.table[i].share[k]);
        if (d < bd) {
          bd = d;
          bi = i;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const int64_t od = __shfl_xor_sync(0xffffffffu, bd, o);
        const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (od < bd || (od == bd && oi < bi)) {
          bd = od;
          bi = oi;
        }
      }
      const int32_t tq = p.table[bi].tile_q, tb = p.table[bi].blocks;
      const bool ok = tq >= 16 && tq <= 256 && tq % 16 == 0 && (tb == 1 || tb == 2);
      if (ok) {
        q = tq;
        want_blocks = min(tb, kBlocks);
      } else if (lane == 0) {
        set_status(p.status, MG_ERR_DEVICE_ARG);
      }
      if (blockIdx.x == 0 && lane == 0 && p.tactic_out != nullptr) {
        p.tactic_out[0] = ok ? tq : 0;
        p.tactic_out[1] = ok ? tb : 0;
        p.tactic_out[2] = bi;
      }
    } else if (p.tactic != nullptr) {
      const int32_t tq = p.tactic[0], tb = p.tactic[1];
      if (tq >= 16 && tq <= 256 && tq % 16 == 0 && (tb == 1 || tb == 2)) {
        q = tq;
        want_blocks = min(tb, kBlocks);
      } else if (lane == 0) {
        set_status(p.status, MG_ERR_DEVICE_ARG);
      }
    }
    // Both forms price the candidate tiles on the histogram (the masked
    // decode case took the widest tile before; the priced choice, 128 on the
    // decode histogram, measured 8 % faster: the widest expert splits and
    // the narrower ring stages leave room for more of them).
    if (kTokM && q == 0) q = 128;  // the MMA computes 128 token rows whatever the tile
    if (q == 0) {
      // token tiles per candidate (32, 64, 128, then 240 or 256): shifts
      // for the powers of two, one division for 240
      int64_t tiles[kNumTileCand] = {0, 0, 0, 0};
      static_assert(kNumTileCand == 4, "four tile candidates");
      for (int32_t e = lane; e < E; e += 32) {
        const uint32_t c = (uint32_t)cnt[e];
        tiles[0] += (c + 31u) >> 5;
        tiles[1] += (c + 63u) >> 6;
        tiles[2] += (c + 127u) >> 7;
        tiles[3] += p.fp8 ? cdiv_u32(c, 240u) : (c + 255u) >> 8;
      }
#pragma unroll
      for (int i = 0; i < kNumTileCand; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tiles[i] += __shfl_xor_sync(0xffffffffu, tiles[i], o);
      }
      const int variant = kPair ? (kBlocks == 2 ? kFwdPairDual : kFwdPair) : (kBlocks == 2 ? kFwdDual : kFwdSingle);
      if (p.masked && kBlocks == 2 && !kPair && !kTokM && p.epi == kEpiPlain && want_blocks == 0) {
        // masked: tile and blocks per tile priced together
        int pb = 2;
        // the ring's bytes and per-stage scale bytes as laid out below
        const int64_t ring = kSmemBytes - 2048 - (kW4 ? kW4Area : 0) -
                             (int64_t)(reinterpret_cast<uintptr_t>(sf_area) - reinterpret_cast<uintptr_t>(smem));
        const int64_t sfb = p.fp8 ? kSfStage + (kW4 ? kW4StageBytes : 0) : 0;
        pick_tile_blocks_warp(p.fp8 != 0, kW4, tiles, p.N, sel_kblocks(p.fp8 != 0, p.K), (int)gridDim.x, ring, sfb,
                              kMaxStages, &q, &pb);
        want_blocks = pb;
      } else {
        q = pick_tile(p.fp8 != 0, tiles, variant, p.N, sel_kblocks(p.fp8 != 0, p.K), (int)gridDim.x);
      }
    }
    q = min(q, q_cap);
    // The two-block kernel runs one-block tiles when two-block tiles would
    // not fill two waves of workers: with few tiles (decode) the finer
    // split balances the SMs, which all stream weights from DRAM then.
    int32_t nblk = kBlocks;
    if (kTokM) {
      // tokens on M: a tile is always 256 weight rows (the MMA's N)
    } else if (kBlocks == 2 && p.epi == kEpiPlain && want_blocks != 0) {
      nblk = want_blocks;
    } else if (kBlocks == 2 && p.epi == kEpiPlain) {  // a SwiGLU epilogue needs gate and up in one tile
      int64_t tt = 0;
      for (int32_t e = lane; e < E; e += 32) tt += cdiv_u32((uint32_t)cnt[e], (uint32_t)q);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tt += __shfl_xor_sync(0xffffffffu, tt, o);
      if (tt * (p.N / (2 * kBlockRows)) < 2 * (int64_t)n_units) nblk = 1;
    }
    const int32_t NB = p.N / (nblk * kBlockRows);
    int32_t carry = 0, qmax = 0;
    for (int32_t b = 0; b < E; b += 32) {
      const int32_t e = b + lane;
      const int32_t c = e < E ? cnt[e] : 0;
      const int32_t own = (int32_t)cdiv_u32((uint32_t)c, (uint32_t)q) * NB;
      if (c > 0) qmax = max(qmax, min(q, round_up16(c)));
      int32_t v = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xffffffffu, v, o);
        if ((int)lane >= o) v += n;
      }
      if (e < E) tpre[e] = carry + v - own;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qmax = max(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
    // Cost order for one-block launches with few token tiles: the full
    // tiles (width q) in expert order, then each expert's trimmed last tile
    // by decreasing width (ties: lower expert first).  Built the same way
    // in every CTA (warp scans and ballots, no atomics).
    const int32_t T_tok = carry / NB;
    const int32_t bal = ((nblk == 1 || kTokM) && T_tok <= kBalMax) ? 1 : 0;
    if (bal) {
      int32_t fcarry = 0;
      for (int32_t b = 0; b < E; b += 32) {
        const int32_t e = b + lane;
        const int32_t c = e < E ? cnt[e] : 0;
        const int32_t nt = (int32_t)cdiv_u32((uint32_t)c, (uint32_t)q);
        const int32_t nfull = c % q == 0 ? nt : nt - 1;
        int32_t v = nfull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t n = __shfl_up_sync(0xffffffffu, v, o);
          if ((int)lane >= o) v += n;
        }
        const int32_t pos = fcarry + v - nfull;
        for (int32_t jj = 0; jj < nfull; ++jj) ttab[pos + jj] = (e << 16) | jj;
        fcarry += __shfl_sync(0xffffffffu, v, 31);
      }
      int32_t pcarry = fcarry;
      if (E <= 32) {
        // one expert per lane: its trimmed last tile's width, found once
        const int32_t c = (int32_t)lane < E ? cnt[lane] : 0;
        const int32_t nt = (int32_t)cdiv_u32((uint32_t)c, (uint32_t)q);
        const int32_t lw = (c % q != 0) ? round_up16(c - (nt - 1) * q) : 0;
        for (int32_t w = round_up16(q); w >= 16; w -= 16) {
          const bool hit = lw == w;
          const uint32_t m = __ballot_sync(0xffffffffu, hit);
          if (hit) ttab[pcarry + __popc(m & ((1u << lane) - 1u))] = ((int32_t)lane << 16) | (nt - 1);
          pcarry += __popc(m);
        }
      } else {
        for (int32_t w = round_up16(q); w >= 16; w -= 16) {
          for (int32_t b = 0; b < E; b += 32) {
            const int32_t e = b + lane;
            const int32_t c = e < E ? cnt[e] : 0;
            const int32_t nt = (int32_t)cdiv_u32((uint32_t)c, (uint32_t)q);
            const bool hit = c % q != 0 && round_up16(c - (nt - 1) * q) == w;
            const uint32_t m = __ballot_sync(0xffffffffu, hit);
            if (hit) ttab[pcarry + __popc(m & ((1u << lane) - 1u))] = (e << 16) | (nt - 1);
            pcarry += __popc(m);
          }
        }
      }
    }
    if (lane == 0) {
      sh.bal = bal;
      tpre[E] = carry;
      sh.total = carry;
      sh.q = q;
      sh.qn_max = max(qmax, 16);
      sh.nblk = nblk;
      // one commit per MMA-issuing thread frees a stage, fills an
      // accumulator and drains the CTA's tensor work
      const uint32_t issuers = kTokM ? 1u : 2u;
      for (int i = 0; i < kMaxStages; ++i) mbar_init(&sh.empty[i], issuers);
      mbar_init(&sh.acc_full[0], issuers);
      mbar_init(&sh.drain, issuers);
      fence_barrier_init();
    }
  }
  __syncthreads();
  // On one SM two warps issue the MMAs (of block 0 and block 1 for
  // two-block tiles, of the first and the last two K-steps of every stage
  // for one-block tiles), each into a 256-column TMEM allocation of its own:
  // its accumulator at columns 0-239 (bf16: 0-255) and the scale words its
  // MMAs read at 240-251.  A CTA pair makes the same two allocations in
  // each of its CTAs (cta_group::2), one at a time.
  // Tokens on M: one issuer; its accumulator fills 256 columns and the scale
  // words follow at 256-267.
  const bool two_issuers = !kTokM;
  if constexpr (!kPair) {
    // (allocated before the schedule; both allocations are made by now)
    if (warp == 1) tmem_relinquish();
  } else {
    // pair allocations are made by one warp in each CTA; one at a time, so
    // both CTAs pair up the same two requests
    cluster_sync();
    if (warp == 1) tmem_alloc_pair_keep_permit(&sh.tmem_base, 256u);
    cluster_sync();
    if (warp == kMma2Warp) tmem_alloc_pair_keep_permit(&sh.tmem_base2, 256u);
    cluster_sync();
    if (warp == 1) tmem_relinquish_pair();
  }
  tc_fence_after();
  // barriers of both CTAs are initialised before any cross-CTA traffic
  if constexpr (kPair) cluster_sync();

  // ---- ring layout, identical in every CTA
  const int32_t q = sh.q;
  const int32_t total = sh.total;
  const int32_t nblk = sh.nblk;
  const int32_t bal = sh.bal;
  const int32_t NB = p.N / (nblk * kBlockRows);  // tiles per token tile
  const int32_t tile_rows = nblk * kBlockRows;
  // Weight rows of this SM's blocks: tile_rows * nb + rank * wrank + b * wstep.
  // A pair with a SwiGLU epilogue takes each SM's gate block and its up
  // block (128 rows apart in GEMM1's interleaved layout) rather than each
  // SM's half of two 256-row blocks.
  const bool swiglu_pair = kPair && p.epi != kEpiPlain;
  const int32_t wrank = swiglu_pair ? 2 * kCtaRows : kCtaRows;
  const int32_t wstep = swiglu_pair ? kCtaRows : kBlockRows;
  // Runs body with the launch's block count as a compile-time constant.
  auto with_blocks = [&](auto&& body) {
    if constexpr (kBlocks == 2) {
      if (nblk == 2) body(IntC<2>{});
      else body(IntC<1>{});
    } else {
      body(IntC<1>{});
    }
  };
  // token rows this CTA stages per tile: all of them, or its half of a pair
  const int32_t stage_bytes =
      nblk * kWTileBytes + (kTokM ? 128 : (kPair ? sh.qn_max / 2 : sh.qn_max)) * kRowBytes;
  // scale data: per stage on one SM; a ring of groups for a pair
  const bool gring = kPair && p.fp8;
  const int32_t sf_bytes = (p.fp8 && !kPair) ? kSfStage + (kW4 ? kW4StageBytes : 0) : 0;
  // a pair's ring of scale groups, or (FP4 weights) the weight-scale group ring
  const int32_t grp_area = gring ? kGRing * kSfStage : (kW4 ? kW4Area : 0);
  uint8_t* gbuf = sf_area;
  uint8_t* sfst = sf_area + grp_area;  // one SM: the stages' scale areas
  const int32_t avail = kSmemBytes - 1024 - (int32_t)(reinterpret_cast<uintptr_t>(sf_area) -
                                                     reinterpret_cast<uintptr_t>(smem)) - 1024 - grp_area;
  int32_t S = avail / (stage_bytes + sf_bytes);
  S = min(S, kMaxStages);
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sf_area) + (uintptr_t)grp_area + (uintptr_t)S * sf_bytes + 1023) &
      ~uintptr_t(1023));
  const int32_t NG = (KB + kSfGroup - 1) / kSfGroup;   // scale groups per tile
  // one accumulator per issuer: the tile's next MMAs wait for the epilogue
  // to drain it
  const uint32_t tmem = sh.tmem_base;
  // the second issuer's allocation (block 1, or the last two K-steps)
  const uint32_t tacc1 = sh.tmem_base2;

  if (warp == 0) {
    // ================================================= TMA producer
    if (lane == 0 && S > 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmA64);
      tma_prefetch_desc(&tmA16);
      if (kPair) tma_prefetch_desc(&tmA8);
      if (p.fp8) tma_prefetch_desc(&tmSF);
      if (kW4) tma_prefetch_desc(&tmSFW);
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      int64_t gload = 0;  // pairs, fp8: scale groups loaded into the ring
      int64_t w4load = 0;  // FP4 weights: weight-scale groups loaded
      auto load_group = [&](const Tile& gt, int32_t g) {
        const uint32_t slot = (uint32_t)(gload % kGRing);
        mbar_arrive_expect_tx(&sh.g_full[slot], (uint32_t)kSfRaw);
        tma_load_3d(gbuf + (size_t)slot * kSfStage, &tmSF, &sh.g_full[slot], gt.sf_x, g * kSfGroup, gt.sf_z);
        ++gload;
      };
      bool ok = true;
      // The next tile is decoded right after the current tile's first stage
      // is issued, while the thread would wait for a free slot anyway.
      Tile nxt{};
      if (unit < total) nxt = decode_tile(unit, tpre, cnt, rowbase, E, NB, q, p.masked, ttab, bal, total, n_units, p.fp8);
      for (int32_t t = unit, ti = 0; ok && t < total; t += n_units, ++ti) {
        const Tile tl = nxt;
        const int32_t qc = kPair ? tl.qn >> 1 : tl.qn;   // token rows staged here
        const int32_t wy = tl.e * p.N + tl.nb * tile_rows + (int32_t)rank * wrank;
        const int32_t ty = tl.row0 + (int32_t)rank * qc;
        // A packed E2M1 box counts its 8 KB of global data toward the barrier,
        // although it fills 16 KB of shared memory
        const int32_t w_tx = kW4 ? kWTileBytes / 2 : kWTileBytes;
        const uint32_t bytes = (kPair ? 2u : 1u) * (uint32_t)(nblk * w_tx + qc * kRowBytes);
        for (int32_t kb = 0; kb < KB; ++kb) {
          const bool group = p.fp8 && (kb % kSfGroup) == 0;
          if (!wait_bounded(&sh.empty[stage], phase ^ 1u, deadline, &sh.abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (kW4 && group && w4load >= kW4Groups) {
            // the scale warp has moved past the group this slot held
            const uint32_t slot = (uint32_t)(w4load % kW4Groups);
            if (!wait_bounded(&sh.sf_grp[slot], (uint32_t)(((w4load / kW4Groups) - 1) & 1), deadline, &sh.abort_flag,
                              p.status)) {
              ok = false;
              break;
            }
            fence_proxy_async_smem();
          }
          uint8_t* sw = ring + (size_t)stage * stage_bytes;
          uint8_t* sa = sw + nblk * kWTileBytes;
          if (leader) {
            // the stage's barrier publishes the tile's width with its bytes
            if (kb == 0) sh.tile_qn[ti % kInfoRing] = tl.qn;
            mbar_arrive_expect_tx(&sh.full[stage], bytes);
          }
          // The raw scale bytes have a barrier of their own and are issued
          // first: the 1 KB lands well before the operands, so warp 6 builds
          // the scale words while the operands are still in flight.
          if (p.fp8 && !gring) {
            uint8_t* sfs = sfst + (size_t)stage * sf_bytes;
            mbar_arrive_expect_tx(&sh.sf_full[stage], group ? (uint32_t)kSfRaw : 0u);
            if (group) tma_load_3d(sfs, &tmSF, &sh.sf_full[stage], tl.sf_x, kb, tl.sf_z);
            if (kW4 && group) {
              // FP4 weights: each block's scale box of the group of four
              // K-blocks (16 bytes per row: the TMA minimum), once per group
              const uint32_t slot = (uint32_t)(w4load % kW4Groups);
              mbar_arrive_expect_tx(&sh.g_full[slot], (uint32_t)(nblk * kWsfBytes));
              for (int32_t b = 0; b < nblk; ++b)
                tma_load_2d(gbuf + (size_t)slot * kW4GroupBytes + b * kWsfBytes, &tmSFW, &sh.g_full[slot],
                            (kb & ~3) * 4, wy + b * kBlockRows);
              ++w4load;
            }
          }
          const int32_t kx = kb * (p.fp8 ? 128 : 64);
          if constexpr (kPair) {
            // operand bytes of both CTAs complete the first CTA's barrier
            const uint32_t bar = mapa_shared(smem_u32(&sh.full[stage]), 0);
#pragma unroll
            for (int b = 0; b < kBlocks; ++b)
              if (b < nblk) tma_load_2d_pair(sw + b * kWTileBytes, &tmW, bar, kx, wy + b * wstep);
            for (int32_t r = 0; r < qc;) {
              const int32_t left = qc - r;
              const CUtensorMap* m = left >= 64 ? &tmA64 : (left >= 16 ? &tmA16 : &tmA8);
              tma_load_2d_pair(sa + r * kRowBytes, m, bar, kx, ty + r);
              r += left >= 64 ? 64 : (left >= 16 ? 16 : 8);
            }
          } else {
#pragma unroll
            for (int b = 0; b < kBlocks; ++b)
              if (b < nblk) tma_load_2d(sw + b * kWTileBytes, &tmW, &sh.full[stage], kx, wy + b * kBlockRows);
            for (int32_t r = 0; r < qc;) {
              const bool wide = qc - r >= 64;
              tma_load_2d(sa + r * kRowBytes, wide ? &tmA64 : &tmA16, &sh.full[stage], kx, ty + r);
              r += wide ? 64 : 16;
            }
          }
          if (kb == 0 && t + n_units < total) nxt = decode_tile(t + n_units, tpre, cnt, rowbase, E, NB, q, p.masked, ttab, bal, total, n_units, p.fp8);
          if (gring && (kb % kSfGroup) == 0) {
            // a pair's scale groups run one group ahead of their first stage:
            // the words then reach both CTAs' shared memory well before the
            // copies that read them (loaded with the stage, the handshake
            // between the pair's scale warps delayed every fourth stage by
            // ~700 cycles)
            const int32_t g = kb / kSfGroup;
            if (gload == 0) load_group(tl, 0);
            if (g + 1 < NG) load_group(tl, g + 1);
            else if (t + n_units < total) load_group(nxt, 0);
          }
          ++issued;
          if (++stage == (uint32_t)S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every copy this CTA can observe lands before it can exit (a pair's
      // second CTA signals its operand copies on the first CTA's barriers,
      // which the first CTA drains)
      const uint64_t dl = globaltimer_ns() + kDrainNs;
      for (int64_t i = issued > S ? issued - S : 0; i < issued; ++i) {
        if (leader) wait_drain(&sh.full[i % S], (uint32_t)((i / S) & 1), dl);
        if (p.fp8 && !gring) wait_drain(&sh.sf_full[i % S], (uint32_t)((i / S) & 1), dl);
      }
      for (int64_t i = gload > kGRing ? gload - kGRing : 0; i < gload; ++i)
        wait_drain(&sh.g_full[i % kGRing], (uint32_t)((i / kGRing) & 1), dl);
      for (int64_t i = w4load > kW4Groups ? w4load - kW4Groups : 0; i < w4load; ++i)
        wait_drain(&sh.g_full[i % kW4Groups], (uint32_t)((i / kW4Groups) & 1), dl);
      if (kPair && !ok) {
        // give the second CTA's operand copies still in flight time to land
        const uint64_t until = globaltimer_ns() + 100000ull;
        while (globaltimer_ns() < until) {
        }
      }
    }
  } else if (warp == 1 || (two_issuers && warp == kMma2Warp)) {
    // ================================================= MMA issuers
    // Warps 1 and 11 on one SM (two-block tiles: block 0 and block 1;
    // one-block tiles: K-steps 0-1 and 2-3 of every stage), warp 1 of the
    // first CTA for a pair.  All lanes run the loop; lane 0 (e0) executes the
    // tcgen05 instructions.
    const int32_t me = warp == 1 ? 0 : 1;   // issuer index
    const uint32_t e0 = lane == 0 ? 1u : 0u;
    if (leader && S > 0) {
      // a stage is ready once its operands landed and (fp8, one SM) its scale
      // words are built: both complete the stage's barrier (each test of a
      // barrier costs the issuing thread ~80 cycles).  A pair's scale words
      // are built in both CTAs and published once per group of four K-blocks
      // on sf_grp, which the copies below wait for.  (Publishing every stage
      // with a cluster-scope release cost each scale warp 1300-2800 cycles
      // per stage: the pairs ran 25 % slower than one SM.)
      auto ready = [&](uint32_t st, uint32_t ph) {
        return wait_bounded(&sh.full[st], ph, deadline, &sh.abort_flag, p.status);
      };
      if constexpr (kTokM) {
        // Tokens on M (one issuer): D[token, weight row] += A[token, k] W[row, k]
        // with M = 128 token rows (rows past the tile's tokens hold stale
        // data; their output rows are never stored) and N = 256 weight rows,
        // so one MMA covers both weight blocks: half the MMAs per weight
        // byte of the swapped layout, which on decode-sized token tiles is
        // bound by MMA issue, not by the narrow token dimension.  Scale
        // words: tokens at column 256 (A), weights at 260-267 (B: block 0,
        // then block 1).
        const uint32_t sf_tok = tmem + 256u, sf_w = tmem + 260u;
        uint32_t stage = 0, phase = 0, acc_phase = 0;
        bool ok = true;
        const uint32_t idesc0 = p.fp8 ? (idesc_mxf8(128, 256) | (kW4 ? kIdescBE2M1 : 0u)) : idesc_bf16(128, 256, 0, 0);
        for (int32_t t = unit; ok && t < total; t += n_units) {
          if (!wait_bounded(&sh.acc_empty[0], acc_phase ^ 1u, deadline, &sh.abort_flag, p.status)) break;
          tc_fence_after();
          if (!ready(stage, phase)) break;
#pragma unroll 2
          for (int32_t kb = 0; kb < KB; ++kb) {
            uint8_t* sw = ring + (size_t)stage * stage_bytes;
            const uint32_t w0 = smem_u32(sw), a0 = smem_u32(sw + 2 * kWTileBytes);
            const uint32_t sid = (uint32_t)(kb & 3);
            // token scales: byte kb & 3 of their word (A scale id); E4M3
            // weights the same byte of theirs, E2M1 weights byte ks of the
            // stage's atom (B scale id)
            const uint32_t idesc = p.fp8 ? (idesc0 | (sid << 29) | (kW4 ? 0u : (sid << 4))) : idesc0;
            if (kW4) {
              const uint32_t atoms = smem_u32(sfst + (size_t)stage * sf_bytes + kSfStage);
              tmem_cp_32x128b_x4_e(e0, sf_w, desc_sf_32x16(atoms));
              tmem_cp_32x128b_x4_e(e0, sf_w + 4, desc_sf_32x16(atoms + kWsfAtom));
            }
            if (p.fp8 && sid == 0) {
              const uint32_t sfs = smem_u32(sfst + (size_t)stage * sf_bytes);
              tmem_cp_32x128b_x4_e(e0, sf_tok, desc_sf_32x16(sfs + kSfRaw + 512));
              if (!kW4) {
                tmem_cp_32x128b_x4_e(e0, sf_w, desc_sf_32x16(sfs + kSfRaw));
                tmem_cp_32x128b_x4_e(e0, sf_w + 4, desc_sf_32x16(sfs + kSfW1));
              }
            }
            auto kstep = [&](int ks, uint32_t accum) {
              const uint64_t ad = desc_kmajor_sw128(a0 + ks * 32), bd = desc_kmajor_sw128(w0 + ks * 32);
              if (p.fp8) mma_mxf8_e(e0, tmem, ad, bd, idesc | (kW4 ? (uint32_t)ks << 4 : 0u), sf_tok, sf_w, accum);
              else mma_f16_e(e0, tmem, ad, bd, idesc, accum);
            };
#pragma unroll
            for (int ks = 0; ks < 3; ++ks) kstep(ks, (kb | ks) != 0 ? 1u : 0u);
            const uint32_t nstage = stage + 1 == (uint32_t)S ? 0u : stage + 1;
            const uint32_t nphase = stage + 1 == (uint32_t)S ? phase ^ 1u : phase;
            if (kb + 1 < KB && !ready(nstage, nphase)) ok = false;
            kstep(3, 1u);
            mma_commit_e(e0, &sh.empty[stage]);
            stage = nstage;
            phase = nphase;
            if (!ok) break;
          }
          if (!ok) break;
          mma_commit_e(e0, &sh.acc_full[0]);
          acc_phase ^= 1u;
        }
        mma_commit_e(e0, &sh.drain);
      } else {
      // this thread's TMEM: its accumulator(s) and scale-word columns
      const uint32_t my_tmem = me == 0 ? tmem : tacc1;
      const uint32_t my_sfa = my_tmem + 240u;  // weight words
      const uint32_t my_sfb = my_tmem + 244u;  // token words
      uint32_t grp = 0;  // pairs: groups of scale words consumed
      with_blocks([&](auto bc) {
      constexpr int kB = decltype(bc)::value;
      // blocks this thread issues: all kB, or block `me` alone
      const int b_lo = kB == 2 ? me : 0, b_hi = kB == 2 ? me + 1 : kB;
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      for (int32_t t = unit, ti = 0; ok && t < total; t += n_units, ++ti) {
        if (!wait_bounded(&sh.acc_empty[0], acc_phase ^ 1u, deadline, &sh.abort_flag, p.status)) break;
        tc_fence_after();
        // The wait for stage kb+1 sits between the third and the fourth
        // K-step of stage kb, so the tensor pipe holds queued work while the
        // thread waits.  No tcgen05 fence follows the stage waits: the
        // stage's bytes are published by the mbarrier.
        if (!ready(stage, phase)) break;
        // The tile's width comes from the producer through the first stage's
        // barrier: decoding the tile here (a binary search and several
        // divisions) left the tensor pipe idle at every tile boundary.
        const int32_t qn = *reinterpret_cast<volatile int32_t*>(&sh.tile_qn[ti % kInfoRing]);
        // FP4 weights (the MMA's A operand): A format E2M1
        const uint32_t idesc0 = p.fp8 ? (idesc_mxf8(kBlockRows, qn) | (kW4 ? kIdescAE2M1 : 0u))
                                      : idesc_bf16(kBlockRows, qn, 0, 0);
        // Unrolled twice: the jump back to the loop top cost the issuing
        // thread ~200 cycles per iteration (measured with in-kernel clock
        // stamps), time in which the shallow tensor-pipe queue runs dry.
#pragma unroll 2
        for (int32_t kb = 0; kb < KB; ++kb) {
          uint8_t* sw = ring + (size_t)stage * stage_bytes;
          const uint32_t a0 = smem_u32(sw), b0 = smem_u32(sw + kB * kWTileBytes);
          const uint32_t sid = (uint32_t)(kb & 3);
          // scale bytes: tokens use byte kb & 3 of their word, fp8 weights the
          // same byte of theirs; FP4 weights byte ks of this stage's atom
          const uint32_t idesc = p.fp8 ? (idesc0 | (sid << 4) | (kW4 ? 0u : (sid << 29))) : idesc0;
          if constexpr (!kPair) {
            if (kW4) {
              const uint32_t atoms = smem_u32(sfst + (size_t)stage * sf_bytes + kSfStage);
              for (int b = b_lo; b < b_hi; ++b)
                tmem_cp_32x128b_x4_e(e0, my_sfa + 4 * (b - b_lo), desc_sf_32x16(atoms + b * kWsfAtom));
            }
          }
          if (p.fp8 && sid == 0) {
            if constexpr (kPair) {
              const uint32_t slot = grp % kGRing;
              const uint32_t sfs = smem_u32(gbuf + (size_t)slot * kSfStage);
              if (!wait_bounded(&sh.sf_grp[slot], (grp / kGRing) & 1, deadline, &sh.abort_flag, p.status)) {
                ok = false;
                break;
              }
              ++grp;
              for (int b = b_lo; b < b_hi; ++b)
                tmem_cp_32x128b_x4_pair_e(e0, my_sfa + 4 * (b - b_lo), desc_sf_32x16(sfs + (b == 0 ? kSfRaw : kSfW1)));
              tmem_cp_32x128b_x4_pair_e(e0, my_sfb, desc_sf_32x16(sfs + kSfRaw + 512));
              if (qn > 128) tmem_cp_32x128b_x4_pair_e(e0, my_sfb + 4, desc_sf_32x16(sfs + kSfRaw + 1024));
            } else {
              const uint32_t sfs = smem_u32(sfst + (size_t)stage * sf_bytes);
              if (!kW4) {
                // weight words of block b: at kSfRaw (block 0) or kSfW1 (block 1)
                for (int b = b_lo; b < b_hi; ++b)
                  tmem_cp_32x128b_x4_e(e0, my_sfa + 4 * (b - b_lo), desc_sf_32x16(sfs + (b == 0 ? kSfRaw : kSfW1)));
              }
              tmem_cp_32x128b_x4_e(e0, my_sfb, desc_sf_32x16(sfs + kSfRaw + 512));
              if (qn > 128) tmem_cp_32x128b_x4_e(e0, my_sfb + 4, desc_sf_32x16(sfs + kSfRaw + 1024));
            }
          }
          auto kstep = [&](int ks, uint32_t accum) {
            const uint64_t bd = desc_kmajor_sw128(b0 + ks * 32);
#pragma unroll
            for (int b = 0; b < kB; ++b) {
              if (b < b_lo || b >= b_hi) continue;
              const uint64_t ad = desc_kmajor_sw128(a0 + b * kWTileBytes + ks * 32);
              const uint32_t d = my_tmem;
              if constexpr (kPair) {
                if (p.fp8) mma_mxf8_pair_e(e0, d, ad, bd, idesc, my_sfa + 4 * (b - b_lo), my_sfb, accum);
                else mma_f16_pair_e(e0, d, ad, bd, idesc, accum);
              } else {
                if (p.fp8)
                  mma_mxf8_e(e0, d, ad, bd, idesc | (kW4 ? (uint32_t)ks << 29 : 0u), my_sfa + 4 * (b - b_lo),
                           my_sfb, accum);
                else mma_f16_e(e0, d, ad, bd, idesc, accum);
              }
            }
          };
          const uint32_t nstage = stage + 1 == (uint32_t)S ? 0u : stage + 1;
          const uint32_t nphase = stage + 1 == (uint32_t)S ? phase ^ 1u : phase;
          if constexpr (kB == 1) {
            // one-block tiles: this thread's two K-steps of the stage
            kstep(2 * me, kb != 0 ? 1u : 0u);
            if (kb + 1 < KB && !ready(nstage, nphase))
              ok = false;
            kstep(2 * me + 1, 1u);
          } else {
#pragma unroll
            for (int ks = 0; ks < 3; ++ks) kstep(ks, (kb | ks) != 0 ? 1u : 0u);
            if (kb + 1 < KB && !ready(nstage, nphase))
              ok = false;
            kstep(3, 1u);
          }
          if constexpr (kPair) mma_commit_pair_e(e0, &sh.empty[stage], 0x3);
          else mma_commit_e(e0, &sh.empty[stage]);
          stage = nstage;
          phase = nphase;
          if (!ok) break;
        }
        if (!ok) break;
        if constexpr (kPair) mma_commit_pair_e(e0, &sh.acc_full[0], 0x3);
        else mma_commit_e(e0, &sh.acc_full[0]);
        acc_phase ^= 1u;
      }
      });
      // all tcgen05 work of the CTA (pair) completes before TMEM is released
      if constexpr (kPair) mma_commit_pair_e(e0, &sh.drain, 0x3);
      else mma_commit_e(e0, &sh.drain);
      }
    }
    if (warp == 1 && lane == 0 && S > 0) wait_drain(&sh.drain, 0, globaltimer_ns() + kDrainNs);
    __syncwarp();
  } else if (warp == kSfWarp) {
    // ================================================= fp8 scale words
    // One SM: for every stage, in the order the MMA threads consume them,
    // wait until its raw scale bytes have landed; on the first K-block of
    // each group of four, write the TMEM scale words (weights of each block,
    // tokens) next to the raw bytes (FP4 weights: rearrange the stage's
    // weight-scale atom), then arrive on the stage's operand barrier.  A
    // stage's words are rewritten only after it has been refilled, i.e. after
    // the MMAs and copies that read them.  A pair: the same words once per
    // group, in the group ring, published on the first CTA's sf_grp.
    if (p.fp8 && S > 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      const uint32_t grp0 = mapa_shared(smem_u32(&sh.sf_grp[0]), 0);
      uint32_t wgrp = 0;  // groups of words published
      int64_t w4use = 0;    // FP4 weights: weight-scale groups read
      uint32_t w4slot = 0;
      // weight scales of a tile's blocks: lane l holds K-blocks l + 32 i;
      // the next tile's are fetched while the current tile streams
      with_blocks([&](auto bc) {
      constexpr int kB = decltype(bc)::value;
      uint32_t wsf[kB][4], wsf_nxt[kB][4];
      auto fetch_wsf = [&](int32_t t, uint32_t (&w)[kB][4]) {
        const Tile tl = decode_tile(t, tpre, cnt, rowbase, E, NB, q, p.masked, ttab, bal, total, n_units, p.fp8);
#pragma unroll
        for (int b = 0; b < kB; ++b) {
          const int32_t nb128 = (tl.nb * tile_rows + (int32_t)rank * wrank + b * wstep) / kCtaRows;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int32_t kb = (int32_t)lane + 32 * i;
            w[b][i] = kb < KB ? __ldg(p.sfb + ((int64_t)tl.e * KB + kb) * NB128 + nb128) : 127u;
          }
        }
      };
      if (unit < total && !kW4) fetch_wsf(unit, wsf_nxt);
      for (int32_t t = unit; ok && t < total; t += n_units) {
#pragma unroll
        for (int b = 0; b < kB; ++b)
#pragma unroll
          for (int i = 0; i < 4; ++i) wsf[b][i] = wsf_nxt[b][i];
        // lane g: the word of group g of each block (K <= 16384: 32 groups)
        uint32_t gword[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) gword[b] = kW4 ? 0u : group_weight_word(wsf[b], lane, KB);
        if constexpr (kPair) {
          // a pair: the tile's scale groups in order, as they land in the ring
          for (int32_t g = 0; g < NG; ++g) {
            const uint32_t slot = wgrp % kGRing;
            if (!warp_wait(&sh.g_full[slot], (wgrp / kGRing) & 1, deadline, &sh.abort_flag, p.status)) {
              ok = false;
              break;
            }
            uint8_t* gb = gbuf + (size_t)slot * kSfStage;
            sf_build_words(gb, __shfl_sync(0xffffffffu, gword[0], g), lane);
            if (kB == 2) {
              const uint32_t w1 = __shfl_sync(0xffffffffu, gword[kB - 1], g);
              *reinterpret_cast<uint4*>(gb + kSfW1 + lane * 16) = make_uint4(w1, w1, w1, w1);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(grp0 + slot * (uint32_t)sizeof(uint64_t));
            ++wgrp;
            if (g == 0 && t + n_units < total) fetch_wsf(t + n_units, wsf_nxt);
          }
        } else {
        for (int32_t kb = 0; kb < KB; ++kb) {
          if (!warp_wait(&sh.sf_full[stage], phase, deadline, &sh.abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sfs = sfst + (size_t)stage * sf_bytes;
          if ((kb % kSfGroup) == 0) {
            // lane l, column c of a word block holds the word of row c*32 + l
            // (FP4 weights: only the token words are built here)
            const int32_t g = kb / kSfGroup;
            sf_build_words(sfs, __shfl_sync(0xffffffffu, gword[0], g), lane);
            if (kB == 2 && !kW4) {
              const uint32_t w1 = __shfl_sync(0xffffffffu, gword[kB - 1], g);
              *reinterpret_cast<uint4*>(sfs + kSfW1 + lane * 16) = make_uint4(w1, w1, w1, w1);
            }
          }
          if (kW4) {
            if ((kb % kSfGroup) == 0) {
              // release the previous group's slot, then take the group's boxes
              __syncwarp();
              if (w4use > 0 && lane == 0) mbar_arrive(&sh.sf_grp[w4slot]);
              w4slot = (uint32_t)(w4use % kW4Groups);
              if (!warp_wait(&sh.g_full[w4slot], (uint32_t)((w4use / kW4Groups) & 1), deadline, &sh.abort_flag,
                             p.status)) {
                ok = false;
                break;
              }
              ++w4use;
            }
            // this K-block's word of rows lane + 32 j, from the group's box
#pragma unroll
            for (int b = 0; b < kB; ++b) {
              const uint8_t* box = gbuf + (size_t)w4slot * kW4GroupBytes + b * kWsfBytes + 4 * (kb & 3);
              uint32_t w[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const uint32_t*>(box + 16 * (lane + 32 * j));
              *reinterpret_cast<uint4*>(sfs + kSfStage + b * kWsfAtom + lane * 16) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
          if ((kb % kSfGroup) == 0 || kW4) fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.full[stage]);
          if (kb == 0 && t + n_units < total && !kW4) fetch_wsf(t + n_units, wsf_nxt);
          if (++stage == (uint32_t)S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        }
      }
      });
    }
  } else if (warp == kMma2Warp) {
    // second MMA issuer: idle with tokens on M (one issuer)
  } else {
    // ================================================= epilogue
    const uint32_t quad = warp & 3u;  // TMEM lanes this warp may access
    // which of the quadrant's three warps (the SwiGLU and tokens-on-M
    // epilogues use the first two, as halves)
    const int32_t third = warp < kSfWarp ? 0 : (warp < kMma2Warp ? 1 : 2);
    const int32_t half = third;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(&sh.acc_empty[0]), 0);
    const bool odd = (lane & 1u) != 0;
    with_blocks([&](auto bc) {
    constexpr int kB = decltype(bc)::value;
    uint32_t acc_phase = 0;
    [[maybe_unused]] uint32_t tile_par = 0;  // SwiGLU to E4M3: parity of tiles done, the exchange barrier's phase
    for (int32_t t = unit; S > 0 && t < total; t += n_units) {
      const Tile tl = decode_tile(t, tpre, cnt, rowbase, E, NB, q, p.masked, ttab, bal, total, n_units, p.fp8);
      if (!warp_wait(&sh.acc_full[0], acc_phase, deadline, &sh.abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + ((quad * 32u) << 16);
      // block 1's accumulator (the up half of a SwiGLU tile)
      [[maybe_unused]] const uint32_t taddr1 = tacc1 + ((quad * 32u) << 16);
      bool released = false;  // this warp's arrival on acc_empty is made
      bool swiglu = false;
      if constexpr (kB == 2 && !kTokM) swiglu = p.epi != kEpiPlain;
      if (kTokM && third == 2) {
        // (not needed by this epilogue)
      } else if constexpr (kTokM) {
        // Tokens on M: TMEM lane = the tile's token, column = weight row, so
        // each thread holds one output row; the two warps of a lane quadrant
        // take 128 of the 256 columns each and store 16 bytes at a time.
        const int32_t tok = (int32_t)(quad * 32u + lane);
        const int32_t c_lo = 128 * half;
        __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.D) + (int64_t)(tl.row0 + tok) * p.N +
                              tl.nb * (2 * kCtaRows) + c_lo;
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t r0[16], r1[16];
          tmem_ld16(taddr + (uint32_t)(c_lo + c), r0);
          tmem_ld16(taddr + (uint32_t)(c_lo + c + 16), r1);
          tmem_ld_wait();
          tmem_regs_ready(r0);
          tmem_regs_ready(r1);
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
            const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
            v[i] = *reinterpret_cast<const uint32_t*>(&a);
            v[8 + i] = *reinterpret_cast<const uint32_t*>(&b);
          }
          if (tok < tl.rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(drow + c + 8 * j) = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          }
        }
      } else if (swiglu) {
        if (third == 2) {
          // (not needed by this epilogue)
        } else if (p.epi == kEpiSwigluBf16) {
          swiglu_bf16_tile(p, tl, kPair ? 2 * tl.nb + (int32_t)rank : tl.nb, taddr, taddr1, quad, half, lane);
        } else if (!swiglu_fp8_tile(p, sh, tl, kPair ? 2 * tl.nb + (int32_t)rank : tl.nb, taddr, taddr1, quad,
                                    half, lane, tile_par, deadline)) {
          break;
        }
        tile_par ^= 1u;
      } else {
        // this thread's output column of block 0; block b is b * kBlockRows further
        const int32_t n = tl.nb * tile_rows + (int32_t)(rank * kCtaRows + quad * 32 + lane);
        __nv_bfloat16* dpair = static_cast<__nv_bfloat16*>(p.D) + (int64_t)tl.row0 * p.N + (n & ~1);
        // The quadrant's three warps take every third 16-token chunk.  A
        // warp reads its first kParked chunks into registers (rounded to
        // bf16, two tokens per register) and releases the accumulator before
        // storing them, so the next tile's MMAs run during the stores.
        // Chunks past those (only the widest tiles have them) are stored
        // before the release.
        auto load_chunk = [&](int32_t c0, uint32_t (&r)[kB][16]) {
#pragma unroll
          for (int b = 0; b < kB; ++b) tmem_ld16((b == 0 ? taddr : taddr1) + (uint32_t)c0, r[b]);
          if constexpr (kB == 1) {
            // the two issuers' partial sums (K-steps 0-1 and 2-3 of every stage)
            uint32_t r2[16];
            tmem_ld16(taddr1 + (uint32_t)c0, r2);
            tmem_ld_wait();
            tmem_regs_ready(r[0]);
            tmem_regs_ready(r2);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              r[0][i] = __float_as_uint(__uint_as_float(r[0][i]) + __uint_as_float(r2[i]));
          } else {
            tmem_ld_wait();
          }
#pragma unroll
          for (int b = 0; b < kB; ++b) tmem_regs_ready(r[b]);
        };
        // Lanes 2j and 2j+1 hold adjacent output columns, a register two
        // tokens of one column.  One exchange per register gives the even
        // lane both columns of the first token and the odd lane both
        // columns of the second, so each store writes 4 bytes.
        auto store_chunk = [&](int32_t c0, const uint32_t (&v)[kB][8]) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int32_t row = c0 + 2 * i + (odd ? 1 : 0);
#pragma unroll
            for (int b = 0; b < kB; ++b) {
              const uint32_t mine = v[b][i];
              const uint32_t recv = __shfl_xor_sync(0xffffffffu, mine, 1);
              const uint32_t out = odd ? __byte_perm(recv, mine, 0x7632) : __byte_perm(mine, recv, 0x5410);
              if (row < tl.rows)
                *reinterpret_cast<uint32_t*>(dpair + (int64_t)row * p.N + b * kBlockRows) = out;
            }
          }
        };
        auto pack_chunk = [&](const uint32_t (&r)[kB][16], uint32_t (&v)[kB][8]) {
#pragma unroll
          for (int b = 0; b < kB; ++b)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[b][2 * i]), __uint_as_float(r[b][2 * i + 1]));
              v[b][i] = *reinterpret_cast<const uint32_t*>(&h);
            }
        };
        for (int32_t c0 = 16 * third + 48 * kParked; c0 < tl.qn; c0 += 48) {
          uint32_t r[kB][16], v[kB][8];
          load_chunk(c0, r);
          pack_chunk(r, v);
          store_chunk(c0, v);
        }
        uint32_t park[kParked][kB][8];
#pragma unroll
        for (int j = 0; j < kParked; ++j) {
          const int32_t c0 = 16 * third + 48 * j;
          if (c0 < tl.qn) {
            uint32_t r[kB][16];
            load_chunk(c0, r);
            pack_chunk(r, park[j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) mbar_arrive_cluster_relaxed(acc_empty0);
          else mbar_arrive_relaxed(&sh.acc_empty[0]);
        }
#pragma unroll
        for (int j = 0; j < kParked; ++j) {
          const int32_t c0 = 16 * third + 48 * j;
          if (c0 < tl.qn) store_chunk(c0, park[j]);
        }
        released = true;
      }
      if (!released) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (kPair) mbar_arrive_cluster_relaxed(acc_empty0);
          else mbar_arrive_relaxed(&sh.acc_empty[0]);
        }
      }
      acc_phase ^= 1u;
    }
    });
  }

  __syncthreads();
  // neither CTA of a pair releases TMEM or exits while the pair shares work
  if constexpr (kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem, 256u);
    else tmem_dealloc(tmem, two_issuers ? 256u : kTmemCols);
  }
  // a pair's two deallocations, like its allocations, one at a time
  if constexpr (kPair) cluster_sync();
  if (two_issuers && warp == kMma2Warp) {
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tacc1, 256u);
    else tmem_dealloc(tacc1, 256u);
  }
}

template <int kBlocks, bool kPair, bool kW4, bool kTokM = false>
cudaError_t launch(const FwdArgs& a, cudaStream_t s) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  auto kernel = fwd_kernel<kBlocks, kPair, kW4, kTokM>;
  if (dev < 64 && !attr_done[dev]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_done[dev] = true;
  }
  // the SwiGLU epilogue pairs the gate and up blocks of a two-block tile
  if (a.epi != kEpiPlain && (kBlocks != 2 || kTokM)) return cudaErrorInvalidValue;
  if (a.w4 != kW4) return cudaErrorInvalidValue;
  Params p;
  p.counts = a.counts;
  p.sfb = a.sfb;
  p.D = a.D;
  p.sfy = a.sfy;
  p.epi = a.epi;
  p.sfy_ld = a.sfy_ld;
  p.tactic = a.tactic;
  p.table = a.table;
  p.n_table = a.n_table;
  p.tactic_out = a.tactic_out;
  p.status = a.status;
  p.wait_ns = a.wait_ns;
  p.E = a.E;
  p.N = a.N;
  p.K = a.K;
  p.masked = a.masked ? 1 : 0;
  p.fp8 = a.fp8 ? 1 : 0;
  p.rows_total = a.rows_total;
  p.M_max = a.M_max;
  p.align_q = a.align_q;
  p.tile_q = a.tile_q;
  const int sms = num_sms_current_device();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kPair ? (unsigned)(sms / 2) * 2u : (unsigned)sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  unsigned n_attr = 0;
  if (kPair) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = 2;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr].val.clusterDim.z = 1;
    ++n_attr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  return cudaLaunchKernelEx(&cfg, kernel, a.tmW, a.tmA64, a.tmA16, a.tmA8, a.tmSF, a.tmSFW, p);
}

}  // namespace fwd

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s, int variant) {
  if (a.w4) {  // FP4 weights: single-SM families only
    switch (variant) {
      case kFwdSingle: return fwd::launch<1, false, true>(a, s);
      case kFwdDual: return fwd::launch<2, false, true>(a, s);
      case kFwdTokM: return fwd::launch<2, false, true, true>(a, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (variant) {
    case kFwdSingle: return fwd::launch<1, false, false>(a, s);
    case kFwdDual: return fwd::launch<2, false, false>(a, s);
    case kFwdPair: return fwd::launch<1, true, false>(a, s);
    case kFwdPairDual: return fwd::launch<2, true, false>(a, s);
    case kFwdTokM: return fwd::launch<2, false, false, true>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mg
