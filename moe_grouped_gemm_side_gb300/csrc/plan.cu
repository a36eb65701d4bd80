// Device-side planning ("MoE GroupGEMM padding under expert skew", "Calculate
// padded token columns" and "Summarize skew without losing the histogram"),
// the device token-tile selector ("Adapt kernels without adding a CPU
// stall"), and the bounded-wait self-test.
#include "common.cuh"
#include "mg_internal.h"
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
  int64_t carry_rows = 0, carry_tiles = 0, U = 0, sumsq = 0, active = 0;
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
    block_exclusive_scan<int64_t>(c * c, scratch, tot);
    sumsq += tot;
    block_exclusive_scan<int64_t>(c > 0 ? 1 : 0, scratch, tot);
    active += tot;
  }
  if (threadIdx.x == 0) {
    offsets[E] = carry_rows;
    mg_plan_stats s;
    s.P = carry_rows;
    s.U = U;
    s.sumsq = sumsq;
    s.active = (int32_t)active;
    s.num_tiles = (int32_t)carry_tiles;
    s.pad_frac = plan_pad_frac(carry_rows, U);
    s.eff_experts = plan_eff_experts(U, sumsq);
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

cudaError_t launch_wait_selftest(int32_t* status, int64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace mg
