// K-grouped MoE weight-gradient GEMM for sm_103a ("flops/deepgemm-grouped-
// masked-moe-gemm", "Workarounds": K-grouped GEMM for MoE weight backward, M
// and N fixed while the contraction length -- the expert's token count --
// varies).
//
//   dW[e] = sum over expert e's tokens t of dY[t, :]^T X[t, :]    ([N, K], fp32)
//
// Tokens are packed by expert with no alignment, so both operands arrive
// MN-major: a TMA box is 64 tokens x 64 contiguous columns of dY or X, and
// the MMA reads them through transposed (MN-major) descriptors.  A tile is a
// kBlocks*128 x 256 block of dW (two 128-row blocks when N allows: the token
// block of X is then shared by two MMAs, 1.5x the multiply-adds per staged
// byte); its main loop walks the expert's tokens 64 at a time.  The last,
// partial block of an expert may hold the next expert's tokens: warp 6
// zeroes those rows of the staged operands in shared memory, and the MMA
// thread issues only the 16-token steps that still hold valid tokens.
//
// Schedule.  An expert's tiles all stream the same token range of dY and X,
// so they read it from DRAM once only if they run at the same time.  When
// one expert's NT tiles fit the grid, the first floor(P / NT) * NT CTAs form
// groups of NT, and a group runs its experts one after another, all NT tiles
// of an expert side by side (tile l on the group's CTA l); the remaining
// P mod NT CTAs take the smallest experts, whose token ranges stay in L2
// while those CTAs go over them in several rounds.  Experts are split
// between the two by their cost (64-token stages plus a fixed epilogue
// share per tile), smallest first into the leftover CTAs while they stay
// within the grid's average load; the groups take the rest, largest first,
// each to the least loaded group.  Otherwise (an expert has more tiles than
// the grid, or the leftover CTAs would get nothing) the tiles of all experts,
// by descending token count, are dealt in a snake order.  Experts with no
// tokens produce zero tiles that the epilogue writes without any load or
// MMA.
//
// CTA = 11 warps: warp 0 issues TMA; warp 1 owns TMEM and one of its threads
// issues every tcgen05.mma (nothing else runs between MMAs, so the tensor
// pipe's short queue stays fed); warps 2-5 and 7-10 drain the accumulators
// (two warps per TMEM lane quadrant); warp 6 zeroes the tail rows.
#include "common.cuh"
#include "mg_internal.h"
#include "sched.cuh"

namespace mg {
namespace kg {

constexpr int kThreads = 352;
constexpr int kFixWarp = 6;
constexpr int kEpiWarps = 8;
constexpr int kMaxStages = 8;
constexpr int kBlockT = 64;               // tokens per stage
constexpr int kBoxBytes = kBlockT * 128;  // one 64 x 64 bf16 box
constexpr int kBlockM = 128;              // dW rows per block (MMA M)
constexpr int kTileN = 256;               // dW columns per tile (max, MMA N)
constexpr int kOutBox = 32 * 32 * 4;      // epilogue staging box: 32 rows x 32 fp32
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;
constexpr int kSmemBytes = 227 * 1024;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;
constexpr int kMaxGroups = 256;           // expert groups of the schedule
constexpr int kTileOverhead = 8;          // a tile's epilogue, in 64-token stages
static_assert((2 * kMaxExperts + kMaxGroups) * 4 <= kEpiWarps * kOutBox, "schedule scratch fits the staging area");

struct Params {
  const int32_t* counts;
  float* dW;
  int32_t* status;
  int64_t wait_ns;
  int32_t E, N, K, T_cap;
};

struct Shared {
  uint64_t full[kMaxStages];
  uint64_t fixed[kMaxStages];  // warp 6 has zeroed the stage's tail rows (if any)
  uint64_t empty[kMaxStages];  // the MMAs reading the stage are done and warp 6 is past it
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t n_valid;
  // schedule: mode 1 = expert groups, 0 = snake over all tiles
  int32_t mode, n_grp, n_left, nA;
  int32_t goff[kMaxGroups + 1];  // group g's experts: order[goff[g] .. goff[g+1])
};

struct Tile {
  int32_t e, mb, nb, w, cnt, tok0;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t deadline,
                                          volatile int32_t* abort_flag, int32_t* status) {
  const bool ok = wait_bounded(bar, parity, deadline, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Position `pos` of the CTA's snake walk -> tile.
__device__ __forceinline__ Tile decode_tile(int32_t pos, const int32_t* order, const int32_t* cnt,
                                            const int32_t* tokoff, int32_t NBk, int32_t NT,
                                            int32_t K) {
  Tile tl;
  const int32_t pe = pos / NT, l = pos - pe * NT;
  tl.e = order[pe];
  tl.mb = l / NBk;
  tl.nb = l - tl.mb * NBk;
  tl.w = min(kTileN, K - tl.nb * kTileN);
  tl.cnt = cnt[tl.e];
  tl.tok0 = tokoff[tl.e];
  return tl;
}

// Position of the CTA's r-th tile: rounds of gridDim.x tiles, alternating
// direction.  Returns -1 past the end of the list.
__device__ __forceinline__ int32_t snake_pos(int32_t r, int32_t total) {
  const int64_t base = (int64_t)r * gridDim.x;
  if (base >= total) return -1;
  const int64_t pos = base + ((r & 1) ? (int64_t)(gridDim.x - 1 - blockIdx.x) : (int64_t)blockIdx.x);
  return pos < total ? (int32_t)pos : -2;
}

template <int kBlocks>
__global__ void __launch_bounds__(kThreads, 1)
    kg_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmX,
              const __grid_constant__ CUtensorMap tmDW, const Params p) {
  static_assert(kBlocks == 1 || kBlocks == 2, "one or two 128-row blocks per tile");
  constexpr int kTileM = kBlocks * kBlockM;                              // dW rows per tile
  constexpr int kBoxesY = kTileM / 64;                                   // dY boxes per stage
  constexpr int kStageBytes = (kBoxesY + kTileN / 64) * kBoxBytes;       // 48 or 64 KB
  constexpr uint32_t kNAcc = kBlocks == 1 ? 2u : 1u;                     // accumulator sets
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Shared& sh = *reinterpret_cast<Shared*>(smem);
  const int32_t E = p.E;
  int32_t* cnt = reinterpret_cast<int32_t*>(smem + ((sizeof(Shared) + 15) & ~size_t(15)));
  int32_t* tokoff = cnt + E;
  int32_t* order = tokoff + E;
  // epilogue staging: one 32 x 32 fp32 box (4 KB, 128-byte swizzle) per warp
  uint8_t* stage_out = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(order + E) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = stage_out + kEpiWarps * kOutBox;

  const uint32_t warp = warp_id(), lane = lane_id();
  const uint64_t deadline = globaltimer_ns() + (uint64_t)p.wait_ns;
  const int32_t NBk = (p.K + kTileN - 1) / kTileN;
  const int32_t NT = (p.N / kTileM) * NBk;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.fixed[i], 1);
      // two arrivals free a stage: the MMA commit and warp 6, so the ring
      // never runs a whole cycle ahead of warp 6 (a warp that fell that far
      // behind would test a barrier phase that has already come round again)
      mbar_init(&sh.empty[i], 2);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.acc_full[i], 1);
      mbar_init(&sh.acc_empty[i], kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(&sh.drain, 1);
    sh.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sh.tmem_base, kTmemCols);

  // ---- counts (-1 marks an expert that is skipped)
  for (int32_t e = threadIdx.x; e < E; e += kThreads) {
    int32_t c = __ldg(p.counts + e);
    if (c < 0) {
      set_status(p.status, MG_ERR_DEVICE_ARG);
      c = -1;
    }
    cnt[e] = c;
  }
  __syncthreads();
  if (warp == 0) {
    int64_t carry = 0;
    for (int32_t b = 0; b < E; b += 32) {
      const int32_t e = b + lane;
      const int64_t own = (e < E && cnt[e] > 0) ? cnt[e] : 0;
      int64_t v = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, v, o);
        if ((int)lane >= o) v += n;
      }
      if (e < E) {
        const int64_t start = carry + v - own;
        if (start + own > p.T_cap) {
          set_status(p.status, MG_ERR_CAPACITY);
          cnt[e] = -1;
          tokoff[e] = 0;
        } else {
          tokoff[e] = (int32_t)start;
        }
      }
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  // ---- experts by descending count (ties: lower index first), skipped last
  for (int32_t e = threadIdx.x; e < E; e += kThreads) {
    const int32_t c = cnt[e];
    if (c < 0) continue;
    int32_t rank = 0;
    for (int32_t f = 0; f < E; ++f) {
      const int32_t d = cnt[f];
      rank += (d > c) || (d == c && f < e);
    }
    order[rank] = e;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t nv = 0;
    for (int32_t e = 0; e < E; ++e) nv += cnt[e] >= 0;
    sh.n_valid = nv;
    // ---- schedule (see the header comment)
    const int32_t P = (int32_t)gridDim.x;
    int32_t ng = NT <= P ? P / NT : 0;
    if (ng > kMaxGroups) ng = 0;
    const int32_t nl = P - ng * NT;
    auto cost = [&](int32_t e) { return (int64_t)((cnt[e] + kBlockT - 1) / kBlockT) + kTileOverhead; };
    int64_t tot = 0;
    for (int32_t r = 0; r < nv; ++r) tot += cost(order[r]);
    int32_t nA = nv;
    if (ng > 0 && nl > 0) {
      // leftover CTAs: NT * load / nl per CTA against the average NT * tot / P
      int64_t sl = 0;
      while (nA > 0 && (sl + cost(order[nA - 1])) * P <= tot * nl) sl += cost(order[--nA]);
    }
    const int32_t mode = (ng > 0 && nv > 0 && (nl == 0 || nA < nv)) ? 1 : 0;
    sh.mode = mode;
    sh.n_grp = ng;
    sh.n_left = nl;
    sh.nA = nA;
    if (mode == 1) {
      // group of each of order[0 .. nA): least loaded group (ties: lowest),
      // in a snake over the groups when there are many; then order[0 .. nA)
      // regrouped by group (counting sort, stable), in the epilogue staging
      // area, which is unused until the main loops (2 * E + ng ints: at
      // most 2 * 1024 + 256, a quarter of it)
      int32_t* grp = reinterpret_cast<int32_t*>(stage_out);
      int32_t* tmp = grp + E;
      int64_t load[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int32_t g = 0; g <= ng; ++g) sh.goff[g] = 0;
      for (int32_t r = 0; r < nA; ++r) {
        int32_t g;
        if (ng <= 8) {
          g = 0;
          for (int32_t h = 1; h < ng; ++h) if (load[h] < load[g]) g = h;
          load[g] += cost(order[r]);
        } else {
          const int32_t k = r % ng;
          g = ((r / ng) & 1) ? ng - 1 - k : k;
        }
        grp[r] = g;
        ++sh.goff[g + 1];
      }
      for (int32_t g = 0; g < ng; ++g) sh.goff[g + 1] += sh.goff[g];
      int32_t* put = tmp + E;
      for (int32_t g = 0; g < ng; ++g) put[g] = sh.goff[g];
      for (int32_t r = 0; r < nA; ++r) tmp[put[grp[r]]++] = order[r];
      for (int32_t r = 0; r < nA; ++r) order[r] = tmp[r];
    }
  }
  __syncthreads();
  tc_fence_after();

  const int32_t total = sh.n_valid * NT;
  // position (order index * NT + tile) of this CTA's r-th tile; -1: no more,
  // -2: none in this round
  const int32_t mode = sh.mode, ng = sh.n_grp, nl = sh.n_left, nA = sh.nA;
  auto tile_pos = [&](int32_t r) -> int32_t {
    if (mode == 0) return snake_pos(r, total);
    const int32_t c = (int32_t)blockIdx.x;
    if (c < ng * NT) {
      const int32_t g = c / NT, l = c - g * NT;
      const int32_t k = sh.goff[g] + r;
      return k < sh.goff[g + 1] ? k * NT + l : -1;
    }
    const int32_t b = c - ng * NT;
    const int32_t nlt = (sh.n_valid - nA) * NT;  // the leftover CTAs' tiles
    const int64_t base = (int64_t)r * nl;
    if (base >= nlt) return -1;
    const int64_t i = base + ((r & 1) ? nl - 1 - b : b);
    return i < nlt ? nA * NT + (int32_t)i : -2;
  };
  const int32_t avail = kSmemBytes - 1024 - (int32_t)(reinterpret_cast<uintptr_t>(ring) -
                                                     reinterpret_cast<uintptr_t>(smem));
  if (threadIdx.x == 0 && avail < kStageBytes) set_status(p.status, MG_ERR_UNSUPPORTED);
  const int32_t S = min(kMaxStages, avail / kStageBytes);
  const uint32_t tmem = sh.tmem_base;
  auto next_stage = [&](uint32_t& stage, uint32_t& phase) {
    if (++stage == (uint32_t)S) {
      stage = 0;
      phase ^= 1u;
    }
  };

  if (warp == 0) {
    // ================================================= TMA producer
    if (lane == 0 && S > 0) {
      tma_prefetch_desc(&tmY);
      tma_prefetch_desc(&tmX);
      tma_prefetch_desc(&tmDW);
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int32_t r = 0; ok; ++r) {
        const int32_t pos = tile_pos(r);
        if (pos == -1) break;
        if (pos < 0) continue;
        const Tile tl = decode_tile(pos, order, cnt, tokoff, NBk, NT, p.K);
        if (tl.cnt == 0) continue;
        const int32_t nkb = (tl.cnt + kBlockT - 1) / kBlockT;
        const uint32_t bytes = (uint32_t)(kBoxesY + tl.w / 64) * kBoxBytes;
        for (int32_t kb = 0; kb < nkb; ++kb) {
          if (!wait_bounded(&sh.empty[stage], phase ^ 1u, deadline, &sh.abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* sa = ring + (size_t)stage * kStageBytes;
          uint8_t* sb = sa + kBoxesY * kBoxBytes;
          mbar_arrive_expect_tx(&sh.full[stage], bytes);
          const int32_t y = tl.tok0 + kb * kBlockT;
#pragma unroll
          for (int i = 0; i < kBoxesY; ++i)
            tma_load_2d(sa + i * kBoxBytes, &tmY, &sh.full[stage], tl.mb * kTileM + i * 64, y);
          for (int i = 0; i < tl.w / 64; ++i)
            tma_load_2d(sb + i * kBoxBytes, &tmX, &sh.full[stage], tl.nb * kTileN + i * 64, y);
          ++issued;
          next_stage(stage, phase);
        }
      }
      const uint64_t dl = globaltimer_ns() + kDrainNs;
      for (int64_t i = issued > S ? issued - S : 0; i < issued; ++i)
        wait_drain(&sh.full[i % S], (uint32_t)((i / S) & 1), dl);
    }
  } else if (warp == 1) {
    // ================================================= MMA issuer (one thread)
    if (lane == 0 && S > 0) {
      // A stage is ready once its operands landed; a stage holding an
      // expert's last, partial token block must also have its rows past the
      // expert zeroed by warp 6.  Testing `fixed` only there saves the
      // issuing thread a barrier test (~80 cycles) on every other stage.
      // Warp 6 arrives on `fixed` and `empty` for every stage: it cannot be
      // a cycle ahead of this thread (the stage's refill waits for this
      // thread's commit) nor a cycle behind it (the refill waits for warp 6
      // too), so the parity of each wait is unambiguous.
      auto ready = [&](uint32_t st, uint32_t ph, int32_t rem) {
        const bool fix = rem < kBlockT && (rem & 15) != 0;
        return wait_bounded(&sh.full[st], ph, deadline, &sh.abort_flag, p.status) &&
               (!fix || wait_bounded(&sh.fixed[st], ph, deadline, &sh.abort_flag, p.status));
      };
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int32_t r = 0; ok; ++r) {
        const int32_t pos = tile_pos(r);
        if (pos == -1) break;
        if (pos < 0) continue;
        const Tile tl = decode_tile(pos, order, cnt, tokoff, NBk, NT, p.K);
        if (tl.cnt == 0) continue;
        const int32_t nkb = (tl.cnt + kBlockT - 1) / kBlockT;
        if (!wait_bounded(&sh.acc_empty[acc], acc_phase ^ 1u, deadline, &sh.abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + acc * kAccStride;  // block b accumulates at d0 + b * 256
        const uint32_t idesc = idesc_bf16(kBlockM, (uint32_t)tl.w, 1, 1);
        // The wait for stage kb+1 sits between the third and the fourth
        // 16-token step of stage kb, so the tensor pipe holds queued work
        // while the thread waits.
        if (!ready(stage, phase, tl.cnt)) break;
        // unrolled twice: the jump back to the loop top costs the issuing
        // thread ~200 cycles
#pragma unroll 2
        for (int32_t kb = 0; kb < nkb; ++kb) {
          const uint32_t a0 = smem_u32(ring + (size_t)stage * kStageBytes);
          const uint32_t b0 = a0 + kBoxesY * kBoxBytes;
          const int32_t rem = tl.cnt - kb * kBlockT;
          const int nks = rem >= kBlockT ? 4 : (rem + 15) >> 4;
          auto kstep = [&](int ks) {
            const uint64_t bd = desc_mnmajor_sw128(b0 + ks * 2048, kBoxBytes);
#pragma unroll
            for (int b = 0; b < kBlocks; ++b) {
              const uint64_t ad = desc_mnmajor_sw128(a0 + b * 2 * kBoxBytes + ks * 2048, kBoxBytes);
              mma_f16(d0 + b * kAccStride, ad, bd, idesc, (kb | ks) != 0 ? 1u : 0u);
            }
          };
          for (int ks = 0; ks < nks && ks < 3; ++ks) kstep(ks);
          uint32_t nstage = stage, nphase = phase;
          next_stage(nstage, nphase);
          if (kb + 1 < nkb && !ready(nstage, nphase, rem - kBlockT)) ok = false;
          if (nks == 4) kstep(3);
          mma_commit(&sh.empty[stage]);
          stage = nstage;
          phase = nphase;
          if (!ok) break;
        }
        if (!ok) break;
        mma_commit(&sh.acc_full[acc]);
        if (++acc == kNAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all tcgen05 work of this CTA completes before TMEM is released
      mma_commit(&sh.drain);
      wait_drain(&sh.drain, 0, globaltimer_ns() + kDrainNs);
    }
    __syncwarp();
  } else if (warp == kFixWarp) {
    // ================================================= tail rows
    // Every stage, in order: once it has landed, zero the rows of a partial
    // token block that belong to no token of the expert (up to the next
    // multiple of 16, the last rows an MMA step reads), then mark it fixed
    // and give the producer this warp's half of the stage's release.
    if (S > 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int32_t r = 0; ok; ++r) {
        const int32_t pos = tile_pos(r);
        if (pos == -1) break;
        if (pos < 0) continue;
        const Tile tl = decode_tile(pos, order, cnt, tokoff, NBk, NT, p.K);
        if (tl.cnt == 0) continue;
        const int32_t nkb = (tl.cnt + kBlockT - 1) / kBlockT;
        const int32_t nbox = kBoxesY + tl.w / 64;
        for (int32_t kb = 0; kb < nkb; ++kb) {
          if (!warp_wait(&sh.full[stage], phase, deadline, &sh.abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int32_t rem = tl.cnt - kb * kBlockT;
          if (rem < kBlockT) {
            const int32_t z0 = rem, z1 = ((rem + 15) >> 4) * 16;
            if (z1 > z0) {
              uint8_t* sa = ring + (size_t)stage * kStageBytes;
              const int32_t per_box = (z1 - z0) * 8;  // 16-byte chunks
              for (int32_t i = lane; i < per_box * nbox; i += 32) {
                const int32_t box = i / per_box, c = i - box * per_box;
                *reinterpret_cast<uint4*>(sa + box * kBoxBytes + z0 * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();
            }
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sh.fixed[stage]);
            mbar_arrive(&sh.empty[stage]);
          }
          next_stage(stage, phase);
        }
      }
    }
  } else {
    // ================================================= epilogue
    const uint32_t quad = warp & 3u;
    const int32_t half = warp >= kFixWarp ? 1 : 0;
    uint8_t* out_box = stage_out + ((warp - 2) - (half ? 1 : 0)) * kOutBox;  // warps 2-5, 7-10 -> 0-7
    bool out_pending = false;
    uint32_t acc = 0, acc_phase = 0;
    for (int32_t r = 0; S > 0; ++r) {
      const int32_t pos = tile_pos(r);
      if (pos == -1) break;
      if (pos < 0) continue;
      const Tile tl = decode_tile(pos, order, cnt, tokoff, NBk, NT, p.K);
      if (tl.cnt == 0) {
        // empty expert: dW = 0, split over the eight warps
#pragma unroll
        for (int b = 0; b < kBlocks; ++b) {
          const int32_t row = tl.mb * kTileM + b * kBlockM + (int32_t)(quad * 32 + lane);
          float* dst = p.dW + ((int64_t)tl.e * p.N + row) * p.K + tl.nb * kTileN;
          for (int32_t c = 4 * half; c < tl.w; c += 8)
            *reinterpret_cast<float4*>(dst + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        continue;
      }
      if (!warp_wait(&sh.acc_full[acc], acc_phase, deadline, &sh.abort_flag, p.status)) break;
      tc_fence_after();
#pragma unroll
      for (int b = 0; b < kBlocks; ++b) {
        const int32_t row0 = tl.mb * kTileM + b * kBlockM + (int32_t)(quad * 32);  // the warp's 32 rows
        const uint32_t taddr = tmem + ((quad * 32u) << 16) + acc * kAccStride + b * kAccStride;
        // The two warps of a lane quadrant take alternate 32-column chunks.
        // Each chunk goes through this warp's staging box and a TMA store:
        // full 128-byte rows reach L2, instead of one 16-byte piece of 32
        // different rows per store instruction.
        for (int32_t c0 = 32 * half; c0 < tl.w; c0 += 64) {
          uint32_t v[32];
          tmem_ld32(taddr + (uint32_t)c0, v);
          tmem_ld_wait();
          if (lane == 0 && out_pending) bulk_wait_read_all();  // the box is free again
          __syncwarp();
          // row `lane`, 16-byte chunk j at position j ^ (lane & 7) (128-byte swizzle)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(out_box + lane * 128 + ((j ^ (int)(lane & 7u)) * 16)) =
                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmDW, out_box, tl.nb * kTileN + c0, tl.e * p.N + row0);
            bulk_commit_group();
          }
          out_pending = true;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acc_empty[acc]);
      if (++acc == kNAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // every store has landed before the CTA exits
    if (lane == 0 && out_pending) bulk_wait_all();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int kBlocks>
cudaError_t launch(const KgArgs& a, cudaStream_t s) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !attr_done[dev]) {
    err = cudaFuncSetAttribute(kg_kernel<kBlocks>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_done[dev] = true;
  }
  Params p;
  p.counts = a.counts;
  p.dW = a.dW;
  p.status = a.status;
  p.wait_ns = a.wait_ns;
  p.E = a.E;
  p.N = a.N;
  p.K = a.K;
  p.T_cap = a.T_cap;
  kg_kernel<kBlocks><<<num_sms_current_device(), kThreads, kSmemBytes, s>>>(a.tmY, a.tmX, a.tmDW, p);
  return cudaGetLastError();
}

}  // namespace kg

// Two 128-row blocks of dW per tile when N allows it.
cudaError_t launch_kgrouped(const KgArgs& a, cudaStream_t s) {
  return a.N % 256 == 0 ? kg::launch<2>(a, s) : kg::launch<1>(a, s);
}

}  // namespace mg
