// Contiguous and masked MoE grouped GEMM on CTA pairs (cta_group::2), sm_103a.
//
// Same computation and tile order as the single-CTA kernel in gemm_fwd.cu
// ("flops/deepgemm-grouped-masked-moe-gemm", "Workarounds"; "MoE GroupGEMM
// padding under expert skew", "Grouped execution does not require padded
// experts"), with two CTAs of a cluster sharing each MMA:
//
//   * a tile is 256 weight rows (MMA M; 128 per CTA) x q_n tokens (MMA N;
//     each CTA stages q_n/2 of them), so each SM streams half as many token
//     bytes per FLOP from L2 and a pipeline stage is ~32 KB instead of ~48,
//     which buys 6-7 stages in shared memory;
//   * the leader CTA (rank 0) issues every tcgen05.mma for the pair; the
//     peer's TMA loads signal the leader's stage barrier, and the leader's
//     commits are multicast to both CTAs' stage and accumulator barriers;
//   * each CTA's epilogue drains its own TMEM (its own 128 weight rows) and
//     releases the accumulator on the leader's barrier.

//
// FP8 block scales are packed four K-blocks per 32-bit TMEM word: one
// tcgen05.cp per four K-blocks, the MMA selecting the byte with the scale
// ids of its instruction descriptor.  Each CTA builds the words for its own
// rows (tcgen05.cp of a pair copies each CTA's own shared memory into its own
// TMEM), and the peer signals the leader when its words are ready.
#include <cuda_bf16.h>

#include "common.cuh"
#include "mg_internal.h"
#include "sched.cuh"

namespace mg {
namespace fwd2 {

constexpr int kThreads = 192;
constexpr int kMaxStages = 12;
constexpr int kWRows = 128;                      // weight rows per CTA
constexpr int kPairRows = 256;                   // weight rows per pair tile (MMA M)
constexpr int kRowBytes = 128;
constexpr int kWTileBytes = kWRows * kRowBytes;  // 16 KB
constexpr int kMaxQ = 256;
constexpr int kSfRaw = kSfRawBytes;
constexpr int kSfStage = kSfStageBytes;
constexpr int kGroupTiles = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;
constexpr uint32_t kSfaCol = 496, kSfbCol = 500;
constexpr int kSmemBytes = 227 * 1024;
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;

struct Params {
  const int32_t* counts;
  const uint8_t* sfb;
  __nv_bfloat16* D;
  int32_t* status;
  int64_t wait_ns;
  int32_t E, N, K;
  int32_t masked, fp8;
  int32_t rows_total, M_max, align_q, tile_q;
};

struct Shared {
  uint64_t full[kMaxStages];      // leader: both CTAs' operand bytes landed
  uint64_t empty[kMaxStages];     // both: the pair's MMAs on the stage are done
  uint64_t sf_full[kMaxStages];   // peer: its own token-scale bytes landed
  uint64_t sf_ready[kMaxStages];  // leader: the peer's scale words are written
  uint64_t acc_full[2];
  uint64_t acc_empty[2];          // leader: both CTAs drained the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t q;
  int32_t qn_max;
  int32_t total;
};

struct Tile {
  int32_t e, nb, row0, rows, qn, sf_x, sf_z;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t deadline,
                                          volatile int32_t* abort_flag, int32_t* status) {
  const bool ok = wait_bounded(bar, parity, deadline, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ Tile decode_tile(int32_t t, const int32_t* tpre, const int32_t* cnt,
                                            const int32_t* rowbase, int32_t E, int32_t NB,
                                            int32_t q, int32_t masked) {
  int32_t lo = 0, hi = E;
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
  const int32_t in_e = j * q;
  tl.rows = min(q, cnt[lo] - in_e);
  tl.qn = round_up16(tl.rows);
  tl.row0 = rowbase[lo] + in_e;
  tl.sf_x = masked ? in_e : tl.row0;
  tl.sf_z = masked ? lo : 0;
  return tl;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fwd2_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA64,
                const __grid_constant__ CUtensorMap tmA16, const __grid_constant__ CUtensorMap tmA8,
                const __grid_constant__ CUtensorMap tmSF, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Shared& sh = *reinterpret_cast<Shared*>(smem);
  const int32_t E = p.E;
  int32_t* cnt = reinterpret_cast<int32_t*>(smem + ((sizeof(Shared) + 15) & ~size_t(15)));
  int32_t* rowbase = cnt + E;
  int32_t* tpre = rowbase + E;
  const uintptr_t sched_end = reinterpret_cast<uintptr_t>(tpre + E + 1);
  uint8_t* sf_area = reinterpret_cast<uint8_t*>((sched_end + 1023) & ~uintptr_t(1023));

  const uint32_t warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int32_t pair_id = (int32_t)(blockIdx.x >> 1), n_pairs = (int32_t)(gridDim.x >> 1);
  const uint64_t deadline = globaltimer_ns() + (uint64_t)p.wait_ns;
  const int32_t NB = p.N / kPairRows;       // pair tiles per token tile
  const int32_t NB128 = p.N / kWRows;
  const int32_t KB = p.K / (p.fp8 ? 128 : 64);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
      mbar_init(&sh.sf_full[i], 1);
      mbar_init(&sh.sf_ready[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.acc_full[i], 1);
      mbar_init(&sh.acc_empty[i], 2 * 4);  // one arrival per epilogue warp of each CTA
    }
    mbar_init(&sh.drain, 1);
    sh.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc_pair(&sh.tmem_base, kTmemCols);

  for (int32_t e = threadIdx.x; e < E; e += kThreads) {
    int32_t c = __ldg(p.counts + e);
    if (c < 0 || (p.masked && c > p.M_max)) {
      set_status(p.status, MG_ERR_DEVICE_ARG);
      c = 0;
    }
    cnt[e] = c;
  }
  __syncthreads();

  if (warp == 0) {
    if (p.masked) {
      for (int32_t e = lane; e < E; e += 32) rowbase[e] = e * p.M_max;
    } else {
      int64_t carry = 0;
      for (int32_t b = 0; b < E; b += 32) {
        const int32_t e = b + lane;
        const int64_t own = e < E ? (int64_t)p.align_q * cdiv64(cnt[e], p.align_q) : 0;
        int64_t v = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t n = __shfl_up_sync(0xffffffffu, v, o);
          if ((int)lane >= o) v += n;
        }
        if (e < E) {
          const int64_t start = carry + v - own;
          if (start + cnt[e] > p.rows_total) {
            cnt[e] = 0;
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
    if (p.masked) {
      q = kMaxQ;
    } else if (q == 0) {
      int64_t tiles[kNumTileCand];
#pragma unroll
      for (int i = 0; i < kNumTileCand; ++i) {
        int64_t s = 0;
        for (int32_t e = lane; e < E; e += 32) s += cdiv64(cnt[e], tile_candidate(p.fp8, i));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        tiles[i] = s;
      }
      q = pick_tile(p.fp8 != 0, tiles, kFwdPair, p.N, sel_kblocks(p.fp8 != 0, p.K), 2 * n_pairs);
    }
    int32_t carry = 0, qmax = 0;
    for (int32_t b = 0; b < E; b += 32) {
      const int32_t e = b + lane;
      const int32_t c = e < E ? cnt[e] : 0;
      const int32_t own = (int32_t)cdiv64(c, q) * NB;
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
    if (lane == 0) {
      tpre[E] = carry;
      sh.total = carry;
      sh.q = q;
      sh.qn_max = max(qmax, 16);
    }
  }
  __syncthreads();
  tc_fence_after();
  // barriers of both CTAs are initialised before any cross-CTA traffic
  cluster_sync();

  const int32_t q = sh.q;
  const int32_t total = sh.total;
  const int32_t stage_bytes = kWTileBytes + (sh.qn_max / 2) * kRowBytes;
  const int32_t sf_bytes = p.fp8 ? kSfStage : 0;
  const int32_t avail = kSmemBytes - 1024 - (int32_t)(reinterpret_cast<uintptr_t>(sf_area) -
                                                     reinterpret_cast<uintptr_t>(smem)) - 1024;
  int32_t S = avail / (stage_bytes + sf_bytes);
  S = min(S, kMaxStages);
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sf_area) + (uintptr_t)S * sf_bytes + 1023) & ~uintptr_t(1023));
  // fp8 scale words sit at columns 496-507, so a second accumulator at column
  // 256 needs N <= 240 there.
  const uint32_t n_acc = (!p.fp8 || sh.qn_max <= 240) ? 2u : 1u;
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ================================================= TMA producer (both CTAs)
    if (lane == 0 && S > 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmA64);
      tma_prefetch_desc(&tmA16);
      tma_prefetch_desc(&tmA8);
      if (p.fp8) tma_prefetch_desc(&tmSF);
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int32_t t = pair_id; ok && t < total; t += n_pairs) {
        const Tile tl = decode_tile(t, tpre, cnt, rowbase, E, NB, q, p.masked);
        const int32_t qh = tl.qn >> 1;
        const int32_t wy = tl.e * p.N + tl.nb * kPairRows + (int32_t)rank * kWRows;
        const int32_t ty = tl.row0 + (int32_t)rank * qh;
        for (int32_t kb = 0; kb < KB; ++kb) {
          if (!wait_bounded(&sh.empty[stage], phase ^ 1u, deadline, &sh.abort_flag, p.status)) {
            ok = false;
            break;
          }
          const bool group = p.fp8 && (kb % kSfGroup) == 0;
          uint8_t* sw = ring + (size_t)stage * stage_bytes;
          uint8_t* sa = sw + kWTileBytes;
          uint8_t* sfs = sf_area + (size_t)stage * kSfStage;
          const uint32_t bar_data = mapa_shared(smem_u32(&sh.full[stage]), 0);
          if (leader) {
            mbar_arrive_expect_tx(&sh.full[stage],
                                  2u * (uint32_t)(kWTileBytes + qh * kRowBytes) + (group ? kSfRaw : 0u));
          } else if (p.fp8) {
            mbar_arrive_expect_tx(&sh.sf_full[stage], group ? kSfRaw : 0u);
          }
          const int32_t kx = kb * (p.fp8 ? 128 : 64);
          tma_load_2d_pair(sw, &tmW, bar_data, kx, wy);
          for (int32_t r = 0; r < qh;) {
            const int32_t left = qh - r;
            const CUtensorMap* m = left >= 64 ? &tmA64 : (left >= 16 ? &tmA16 : &tmA8);
            tma_load_2d_pair(sa + r * kRowBytes, m, bar_data, kx, ty + r);
            r += left >= 64 ? 64 : (left >= 16 ? 16 : 8);
          }
          if (group)
            tma_load_3d(sfs, &tmSF, leader ? &sh.full[stage] : &sh.sf_full[stage], tl.sf_x, kb, tl.sf_z);
          ++issued;
          if (++stage == (uint32_t)S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      const uint64_t dl = globaltimer_ns() + kDrainNs;
      for (int64_t i = issued > S ? issued - S : 0; i < issued; ++i) {
        if (leader)
          wait_drain(&sh.full[i % S], (uint32_t)((i / S) & 1), dl);
        else if (p.fp8)
          wait_drain(&sh.sf_full[i % S], (uint32_t)((i / S) & 1), dl);
      }
      if (!ok) {
        // the peer's operand copies signal the leader; give any still in
        // flight time to land before the CTA can exit
        const uint64_t until = globaltimer_ns() + 100000ull;
        while (globaltimer_ns() < until) {
        }
      }
    }
  } else if (warp == 1) {
    // ================================================= MMA (leader) / scale words (peer)
    if (S > 0 && (leader || p.fp8)) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      const uint32_t sf_ready_leader = mapa_shared(smem_u32(&sh.sf_ready[0]), 0);
      for (int32_t t = pair_id; ok && t < total; t += n_pairs) {
        const Tile tl = decode_tile(t, tpre, cnt, rowbase, E, NB, q, p.masked);
        uint32_t wsf[4] = {127u, 127u, 127u, 127u};
        if (p.fp8) {
          const int32_t nb128 = tl.nb * 2 + (int32_t)rank;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int32_t kb = (int32_t)lane + 32 * i;
            if (kb < KB) wsf[i] = __ldg(p.sfb + ((int64_t)tl.e * KB + kb) * NB128 + nb128);
          }
        }
        uint32_t d_tmem = 0, idesc0 = 0;
        if (leader) {
          if (!warp_wait(&sh.acc_empty[acc], acc_phase ^ 1u, deadline, &sh.abort_flag, p.status)) break;
          tc_fence_after();
          d_tmem = tmem + acc * kAccStride;
          idesc0 = p.fp8 ? idesc_mxf8(kPairRows, tl.qn) : idesc_bf16(kPairRows, tl.qn, 0, 0);
        }
        if (!leader) {
          // peer: scale words of each group, then tell the leader
          for (int32_t kb = 0; kb < KB; ++kb) {
            uint8_t* sfs = sf_area + (size_t)stage * kSfStage;
            if (!warp_wait(&sh.sf_full[stage], phase, deadline, &sh.abort_flag, p.status)) {
              ok = false;
              break;
            }
            if (kb % kSfGroup == 0) {
              sf_build_words(sfs, sf_weight_word(wsf, kb, KB), lane);
              fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(sf_ready_leader + (uint32_t)(stage * sizeof(uint64_t)));
            __syncwarp();
            if (++stage == (uint32_t)S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        } else {
          // leader: the wait for stage kb+1 (operands of both CTAs and, for
          // fp8, the peer's scale words) sits between the third and fourth
          // K-step MMA of stage kb, so the tensor pipe holds queued work while
          // the warp waits.
          ok = warp_wait(&sh.full[stage], phase, deadline, &sh.abort_flag, p.status) &&
               (!p.fp8 || warp_wait(&sh.sf_ready[stage], phase, deadline, &sh.abort_flag, p.status));
          tc_fence_after();
          for (int32_t kb = 0; ok && kb < KB; ++kb) {
            uint8_t* sfs = sf_area + (size_t)stage * kSfStage;
            const bool group = p.fp8 && (kb % kSfGroup) == 0;
            if (group) {
              sf_build_words(sfs, sf_weight_word(wsf, kb, KB), lane);
              fence_proxy_async_smem();
              __syncwarp();
            }
            uint8_t* sw = ring + (size_t)stage * stage_bytes;
            const uint32_t a0 = smem_u32(sw), b0 = smem_u32(sw + kWTileBytes);
            const uint32_t sid = (uint32_t)(kb & 3);
            const uint32_t idesc = p.fp8 ? (idesc0 | (sid << 4) | (sid << 29)) : idesc0;
            if (lane == 0) {
              if (group) {
                tmem_cp_32x128b_x4_pair(tmem + kSfaCol, desc_sf_32x16(smem_u32(sfs + kSfRaw)));
                tmem_cp_32x128b_x4_pair(tmem + kSfbCol, desc_sf_32x16(smem_u32(sfs + kSfRaw + 512)));
                if (tl.qn > 128)
                  tmem_cp_32x128b_x4_pair(tmem + kSfbCol + 4, desc_sf_32x16(smem_u32(sfs + kSfRaw + 1024)));
              }
#pragma unroll
              for (int ks = 0; ks < 3; ++ks) {
                const uint64_t ad = desc_kmajor_sw128(a0 + ks * 32);
                const uint64_t bd = desc_kmajor_sw128(b0 + ks * 32);
                const uint32_t accum = (kb | ks) != 0 ? 1u : 0u;
                if (p.fp8)
                  mma_mxf8_pair(d_tmem, ad, bd, idesc, tmem + kSfaCol, tmem + kSfbCol, accum);
                else
                  mma_f16_pair(d_tmem, ad, bd, idesc, accum);
              }
            }
            const uint32_t nstage = stage + 1 == (uint32_t)S ? 0u : stage + 1;
            const uint32_t nphase = stage + 1 == (uint32_t)S ? phase ^ 1u : phase;
            if (kb + 1 < KB)
              ok = warp_wait(&sh.full[nstage], nphase, deadline, &sh.abort_flag, p.status) &&
                   (!p.fp8 || warp_wait(&sh.sf_ready[nstage], nphase, deadline, &sh.abort_flag, p.status));
            tc_fence_after();
            if (lane == 0) {
              const uint64_t ad = desc_kmajor_sw128(a0 + 96);
              const uint64_t bd = desc_kmajor_sw128(b0 + 96);
              if (p.fp8)
                mma_mxf8_pair(d_tmem, ad, bd, idesc, tmem + kSfaCol, tmem + kSfbCol, 1u);
              else
                mma_f16_pair(d_tmem, ad, bd, idesc, 1u);
              mma_commit_pair(&sh.empty[stage], 0x3);
            }
            __syncwarp();
            stage = nstage;
            phase = nphase;
          }
        }
        if (!ok) break;
        if (leader) {
          if (lane == 0) mma_commit_pair(&sh.acc_full[acc], 0x3);
          __syncwarp();
          if (++acc == n_acc) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
      }
    }
    if (leader && lane == 0) mma_commit_pair(&sh.drain, 0x3);
    if (lane == 0) wait_drain(&sh.drain, 0, globaltimer_ns() + kDrainNs);
    __syncwarp();
  } else {
    // ================================================= epilogue (both CTAs)
    const uint32_t quad = warp & 3u;
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(&sh.acc_empty[0]), 0);
    uint32_t acc = 0, acc_phase = 0;
    for (int32_t t = pair_id; S > 0 && t < total; t += n_pairs) {
      const Tile tl = decode_tile(t, tpre, cnt, rowbase, E, NB, q, p.masked);
      if (!warp_wait(&sh.acc_full[acc], acc_phase, deadline, &sh.abort_flag, p.status)) break;
      tc_fence_after();
      const int32_t n = tl.nb * kPairRows + (int32_t)(rank * kWRows + quad * 32 + lane);
      const uint32_t taddr = tmem + ((quad * 32u) << 16) + acc * kAccStride;
      __nv_bfloat16* dcol = p.D + (int64_t)tl.row0 * p.N + n;
      for (int32_t c0 = 0; c0 < tl.qn; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + (uint32_t)c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c0 + i < tl.rows) dcol[(int64_t)(c0 + i) * p.N] = __float2bfloat16_rn(__uint_as_float(r[i]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty_leader + acc * (uint32_t)sizeof(uint64_t));
      if (++acc == n_acc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  __syncthreads();
  // neither CTA releases TMEM or exits while the pair still shares work
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace fwd2

cudaError_t launch_fwd2(const FwdArgs& a, cudaStream_t s) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !attr_done[dev]) {
    err = cudaFuncSetAttribute(fwd2::fwd2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               fwd2::kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_done[dev] = true;
  }
  fwd2::Params p;
  p.counts = a.counts;
  p.sfb = a.sfb;
  p.D = static_cast<__nv_bfloat16*>(a.D);
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
  const int grid = (num_sms_current_device() / 2) * 2;
  fwd2::fwd2_kernel<<<grid, fwd2::kThreads, fwd2::kSmemBytes, s>>>(a.tmW, a.tmA64, a.tmA16, a.tmA8,
                                                                    a.tmSF, p);
  return cudaGetLastError();
}

}  // namespace mg
