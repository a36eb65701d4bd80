// Device-side planning ("MoE GroupGEMM padding under expert skew", "Calculate
// padded token columns" and "Summarize skew without losing the histogram"),
// the device token-tile selector ("Adapt kernels without adding a CPU
// stall"), and the bounded-wait self-test.
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <vector>

#include "common.cuh"
#include "mg_internal.h"
#include "plan_sums.cuh"
#include "sched.cuh"

namespace mg {

namespace {

constexpr int kPlanThreads = 1024;

// Exclusive block-wide prefix sum; `total` receives the block total.  All
// threads of the block must call it.
template <typename T>
__device__ T block_exclusive_scan(T v, T* scratch, T& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T s = lane < nwarps ? scratch[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    scratch[lane] = s;
  }
  __syncthreads();
  const T before = warp == 0 ? T(0) : scratch[warp - 1];
  total = scratch[nwarps - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t* __restrict__ counts, int32_t E, int32_t q,
                int64_t* __restrict__ offsets, int32_t* __restrict__ tiles, int32_t max_tiles,
                mg_plan_stats* __restrict__ stats, int32_t* status) {
  __shared__ int64_t scratch[32];
  int64_t carry_rows = 0, carry_tiles = 0, U = 0, sq_hi_sum = 0, sq_lo_sum = 0, active = 0;
  for (int32_t base = 0; base < E; base += kPlanThreads) {
    const int32_t e = base + threadIdx.x;
    int64_t c = 0;
    if (e < E) {
      c = counts[e];
      if (c < 0) {
        set_status(status, MG_ERR_DEVICE_ARG);
        c = 0;
      }
    }
    const int64_t nt = cdiv64(c, q);
    int64_t tot_rows, tot_tiles, tot;
    const int64_t off = carry_rows + block_exclusive_scan<int64_t>(nt * q, scratch, tot_rows);
    const int64_t t0 = carry_tiles + block_exclusive_scan<int64_t>(nt, scratch, tot_tiles);
    if (e < E) {
      offsets[e] = off;
      if (tiles != nullptr) {
        for (int64_t j = 0; j < nt && t0 + j < max_tiles; ++j) {
          if (off + j * q > 2147483647LL) break;
          int32_t* tp = tiles + 3 * (t0 + j);
          tp[0] = e;
          tp[1] = (int32_t)(off + j * q);
          tp[2] = (int32_t)min((int64_t)q, c - j * q);
        }
      }
    }
    carry_rows += tot_rows;
    carry_tiles += tot_tiles;
    block_exclusive_scan<int64_t>(c, scratch, tot);
    U += tot;
    block_exclusive_scan<int64_t>(sq_hi(c), scratch, tot);
    sq_hi_sum += tot;
    block_exclusive_scan<int64_t>(sq_lo(c), scratch, tot);
    sq_lo_sum += tot;
    block_exclusive_scan<int64_t>(c > 0 ? 1 : 0, scratch, tot);
    active += tot;
  }
  if (threadIdx.x == 0) {
    offsets[E] = carry_rows;
    const SumSq sq = sumsq_finish(sq_hi_sum, sq_lo_sum);
    mg_plan_stats s;
    s.P = carry_rows;
    s.U = U;
    s.sumsq = sq.value;
    s.active = (int32_t)active;
    s.num_tiles = carry_tiles > 2147483647LL ? 2147483647 : (int32_t)carry_tiles;  // saturates
    s.pad_frac = plan_pad_frac(carry_rows, U);
    s.eff_experts = plan_eff_experts_exact(U, sq.f64);
    *stats = s;
    if (tiles != nullptr && carry_tiles > max_tiles) set_status(status, MG_ERR_CAPACITY);
    if (tiles != nullptr && max_tiles > 0 && carry_rows > 2147483647LL) set_status(status, MG_ERR_UNSUPPORTED);
  }
}

__global__ void select_kernel(const int32_t* __restrict__ counts, int32_t E, int32_t fp8,
                              int32_t variant, int32_t N, int32_t KB, int32_t num_sms,
                              int32_t* tile_q, int32_t* status) {
  const int lane = threadIdx.x;
  int64_t tiles[kNumTileCand];
#pragma unroll
  for (int i = 0; i < kNumTileCand; ++i) {
    int64_t s = 0;
    for (int32_t e = lane; e < E; e += 32) {
      int32_t c = counts[e];
      if (c < 0) {
        if (i == 0) set_status(status, MG_ERR_DEVICE_ARG);
        c = 0;
      }
      s += cdiv64(c, tile_candidate(fp8 != 0, i));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    tiles[i] = s;
  }
  if (lane == 0)
    *tile_q = pick_tile(fp8 != 0, tiles, variant, N, KB, num_sms);
}

// Exemplar choice ("MoE GroupGEMM padding under expert skew", "Adapt kernels
// without adding a CPU stall": sort and normalise the count vector, match it
// against exemplars tuned offline, guard against switching on neighbouring
// histograms).  One CTA: bitonic sort of the counts (descending), in-place
// prefix sums, the 16-point cumulative top-share curve and the log2(U)
// feature (integers, the definitions in moegemm.h), the L1 distance to every
// exemplar, the smallest distance (lowest index on ties), then the
// hysteresis rule against the call site's state.
__global__ void __launch_bounds__(kPlanThreads)
    exemplar_kernel(const int32_t* __restrict__ counts, int32_t E, const mg_exemplar* __restrict__ table,
                    int32_t n, int32_t margin, int32_t* state, int32_t* tactic, int32_t* status) {
  __shared__ int64_t v[kSelMaxExperts];
  __shared__ int64_t dist[kSelMaxExemplars];
  __shared__ int64_t scratch[32];
  __shared__ int32_t feat[kExemplarShares + 1];      // shares, then lu
  __shared__ int64_t best_d[32];
  __shared__ int32_t best_i[32];
  const int tid = threadIdx.x;
  int32_t P = 2;
  while (P < E) P <<= 1;
  for (int32_t i = tid; i < P; i += kPlanThreads) v[i] = i < E ? (int64_t)max(counts[i], 0) : 0;
  __syncthreads();
  for (int32_t k = 2; k <= P; k <<= 1) {
    for (int32_t j = k >> 1; j > 0; j >>= 1) {
      for (int32_t i = tid; i < P; i += kPlanThreads) {
        const int32_t ixj = i ^ j;
        if (ixj > i) {
          const int64_t a = v[i], b = v[ixj];
          if ((i & k) == 0 ? (a < b) : (a > b)) {
            v[i] = b;
            v[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // inclusive prefix sums in place: each thread owns R consecutive values
  const int32_t R = (P + kPlanThreads - 1) / kPlanThreads;
  const int32_t lo = tid * R, hi = min(P, lo + R);
  int64_t own = 0;
  for (int32_t i = lo; i < hi; ++i) own += v[i];
  int64_t total;
  int64_t run = block_exclusive_scan<int64_t>(own, scratch, total);
  for (int32_t i = lo; i < hi; ++i) {
    run += v[i];
    v[i] = run;
  }
  __syncthreads();
  const int64_t U = v[E - 1];
  if (tid < kExemplarShares) {
    const int32_t m = ((tid + 1) * E + kExemplarShares - 1) / kExemplarShares;
    feat[tid] = U > 0 ? (int32_t)((int64_t)kShareOne * v[m - 1] / U) : 0;
  }
  if (tid == 0) {
    int32_t lu = 0;
    if (U > 0) {
      const int e = 63 - __clzll(U);
      lu = 16 * e + (int32_t)((16 * (U - (int64_t(1) << e))) >> e);
    }
    feat[kExemplarShares] = lu;
  }
  __syncthreads();
  int64_t bd = INT64_MAX;
  int32_t bi = 0x7fffffff;
  for (int32_t i = tid; i < n; i += kPlanThreads) {
    int64_t d = (int64_t)kLuWeight * llabs((int64_t)feat[kExemplarShares] - table[i].lu);
#pragma unroll
    for (int k = 0; k < kExemplarShares; ++k) d += llabs((int64_t)feat[k] - table[i].share[k]);
    dist[i] = d;
    if (d < bd) {  // i increases: the first minimum of this thread's subset
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
  if ((tid & 31) == 0) {
    best_d[tid >> 5] = bd;
    best_i[tid >> 5] = bi;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < kPlanThreads / 32; ++w)
      if (best_d[w] < bd || (best_d[w] == bd && best_i[w] < bi)) {
        bd = best_d[w];
        bi = best_i[w];
      }
    int32_t c = bi;
    const int32_t prev = state != nullptr ? *state : -1;
    if (prev >= 0 && prev < n && dist[prev] - bd <= (int64_t)margin) c = prev;
    const mg_exemplar& x = table[c];
    const bool ok = x.tile_q >= 16 && x.tile_q <= 256 && x.tile_q % 16 == 0 && (x.blocks == 1 || x.blocks == 2);
    if (!ok) set_status(status, MG_ERR_DEVICE_ARG);
    tactic[0] = ok ? x.tile_q : 0;
    tactic[1] = ok ? x.blocks : 0;
    tactic[2] = c;
    if (state != nullptr) *state = c;
  }
}

__global__ void wait_selftest_kernel(int32_t* status, int64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the wait must give up at the deadline.
  const uint64_t deadline = globaltimer_ns() + (uint64_t)limit_ns;
  wait_bounded(&bar, 0, deadline, &abort_flag, status);
  __syncthreads();
}

}  // namespace

int num_sms_current_device() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev < 64) cached[dev] = n;
  return n;
}

cudaError_t launch_plan(const int32_t* counts, int32_t E, int32_t q, int64_t* offsets,
                        int32_t* tiles, int32_t max_tiles, mg_plan_stats* stats, int32_t* status,
                        cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(counts, E, q, offsets, tiles, max_tiles, stats, status);
  return cudaGetLastError();
}

cudaError_t launch_select(bool fp8, int variant, const int32_t* counts, int32_t E, int32_t N,
                          int32_t K, int32_t* tile_q, int32_t* status, cudaStream_t s) {
  select_kernel<<<1, 32, 0, s>>>(counts, E, fp8 ? 1 : 0, variant, N,
                                 (int32_t)sel_kblocks(fp8, K), num_sms_current_device(), tile_q,
                                 status);
  return cudaGetLastError();
}

cudaError_t launch_exemplar(const int32_t* counts, int32_t E, const mg_exemplar* table, int32_t n,
                            int32_t margin, int32_t* state, int32_t* tactic, int32_t* status,
                            cudaStream_t s) {
  exemplar_kernel<<<1, kPlanThreads, 0, s>>>(counts, E, table, n, margin, state, tactic, status);
  return cudaGetLastError();
}

void exemplar_features_host(const int32_t* counts, int32_t E, int32_t* lu, int32_t* share) {
  std::vector<int64_t> c((size_t)E);
  for (int32_t e = 0; e < E; ++e) c[(size_t)e] = counts[e] > 0 ? counts[e] : 0;
  std::sort(c.begin(), c.end(), [](int64_t a, int64_t b) { return a > b; });
  std::vector<int64_t> prefix((size_t)E + 1, 0);
  for (int32_t e = 0; e < E; ++e) prefix[(size_t)e + 1] = prefix[(size_t)e] + c[(size_t)e];
  const int64_t U = prefix[(size_t)E];
  *lu = 0;
  for (int k = 0; k < kExemplarShares; ++k) {
    const int32_t m = ((k + 1) * E + kExemplarShares - 1) / kExemplarShares;
    share[k] = U > 0 ? (int32_t)((int64_t)kShareOne * prefix[(size_t)m] / U) : 0;
  }
  if (U > 0) {
    int e = 0;
    while ((U >> (e + 1)) != 0) ++e;
    *lu = 16 * e + (int32_t)((16 * (U - (int64_t(1) << e))) >> e);
  }
}

int32_t exemplar_choose_host(const int32_t* counts, int32_t E, const mg_exemplar* table, int32_t n,
                             int32_t margin, int32_t prev, int64_t* dist_out) {
  int32_t lu, share[kExemplarShares];
  exemplar_features_host(counts, E, &lu, share);
  int64_t bd = INT64_MAX;
  int32_t bi = 0;
  std::vector<int64_t> d((size_t)n);
  for (int32_t i = 0; i < n; ++i) {
    int64_t x = (int64_t)kLuWeight * std::llabs((int64_t)lu - table[i].lu);
    for (int k = 0; k < kExemplarShares; ++k) x += std::llabs((int64_t)share[k] - table[i].share[k]);
    d[(size_t)i] = x;
    if (x < bd) {
      bd = x;
      bi = i;
    }
  }
  if (prev >= 0 && prev < n && d[(size_t)prev] - bd <= (int64_t)margin) bi = prev;
  if (dist_out != nullptr) *dist_out = d[(size_t)bi];
  return bi;
}

cudaError_t launch_wait_selftest(int32_t* status, int64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace mg
