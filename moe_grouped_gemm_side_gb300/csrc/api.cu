// C ABI of libmoegemm.so (declared in include/moegemm.h): argument checks,
// TMA tensor-map encoding, launches.  The host planner lives here too; it is
// plain C++ and touches no GPU.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <climits>
#include <cstring>

#include "mg_internal.h"
#include "moegemm.h"
#include "plan_sums.cuh"
#include "sched.cuh"

using namespace mg;

namespace {

constexpr int64_t kDefaultWaitNs = 2000000000LL;
std::atomic<int64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int32_t> g_policy{0};

// Kernel family for N.  Policy 0 (default): for the contiguous form two
// 256-row weight blocks per CTA pair (cta_group::2) when N % 512 == 0, else
// two 128-row blocks on one SM; for the masked form two 128-row blocks on
// one SM (their one-block split for decode-sized histograms).  Measured on
// GB300 these are the fastest families for prefill and decode shapes; FP4
// weights run on one SM.  (Tokens on the MMA's M axis halve the MMAs per
// weight byte, but on the 16-expert decode its 224 tiles leave half the SMs
// with two tiles and the others with one: no faster end to end.)  Policies
// 1-5 force single, dual, pair, pair-dual or tokens-on-M, falling back to
// the widest family N allows when N is not a multiple of the family's tile
// rows.
int fwd_variant(int32_t N, bool w4 = false, bool masked = false) {
  const int32_t pol = g_policy.load();
  const int dflt = (!masked && !w4 && N % 512 == 0) ? kFwdPairDual : kFwdDual;
  int v = pol == 0 ? dflt
        : pol == 1 ? kFwdSingle : pol == 2 ? kFwdDual : pol == 3 ? kFwdPair : pol == 4 ? kFwdPairDual : kFwdTokM;
  if (w4 && (v == kFwdPair || v == kFwdPairDual)) v = kFwdDual;  // FP4 weights: single-SM families
  if (v == kFwdPairDual && N % 512 != 0) v = kFwdPair;
  if ((v == kFwdPair || v == kFwdDual || v == kFwdTokM) && N % 256 != 0) v = kFwdSingle;
  return v;
}

cudaError_t launch_fwd_any(const FwdArgs& a, cudaStream_t s) {
  return launch_fwd(a, s, fwd_variant(a.N, a.w4, a.masked));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once.  A failed lookup is not
// cached: the first call of a process may come before this library's CUDA
// runtime has a context, so the context is made current first (cudaFree of
// nothing creates the device's primary context when there is none).
EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (f != nullptr) return f;
  (void)cudaFree(nullptr);
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return nullptr;
  }
  f = reinterpret_cast<EncodeTiledFn>(p);
  fn.store(f);
  return f;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor map over a row-major [outer, inner] matrix, rows `row_bytes` apart.
mg_status encode_2d_rows(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                         uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MG_ERR_CUDA;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MG_OK : MG_ERR_CUDA;
}

// Tensor map over a row-major [outer, inner] matrix of `elem`-byte elements.
mg_status encode_2d(CUtensorMap* m, CUtensorMapDataType dt, uint32_t elem, const void* base,
                    uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MG_ERR_CUDA;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * elem};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MG_OK : MG_ERR_CUDA;
}

// Tensor map over uint8 block scales [d2, d1, d0] (d0 contiguous), box
// {box0, box1, 1}.
mg_status encode_sf_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint32_t box0, uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return MG_ERR_CUDA;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0, d0 * d1};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MG_OK : MG_ERR_CUDA;
}

mg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MG_OK : MG_ERR_CUDA; }

bool valid_dtype(mg_dtype dt) {
  return dt == MG_BF16 || dt == MG_FP8_E4M3_UE8M0 || dt == MG_FP8_X_FP4_E2M1;
}
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Operand checks shared by the contiguous and masked forms.
mg_status check_fwd_common(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                           const uint8_t* SFB, const void* D, const int32_t* counts, int32_t E,
                           int32_t N, int32_t K) {
  if (!valid_dtype(dt)) return MG_ERR_INVALID_ARG;
  const bool fp8 = dt != MG_BF16;
  if (A == nullptr || B == nullptr || D == nullptr || counts == nullptr) return MG_ERR_INVALID_ARG;
  if (fp8 && (SFA == nullptr || SFB == nullptr)) return MG_ERR_INVALID_ARG;
  if (E <= 0 || N <= 0 || K <= 0) return MG_ERR_INVALID_ARG;
  if (E > kMaxExperts) return MG_ERR_UNSUPPORTED;
  if (N % 128 != 0 || K % 128 != 0) return MG_ERR_UNSUPPORTED;
  if (fp8 && K > 16384) return MG_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= (int64_t(1) << 31)) return MG_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !aligned16(counts))
    return MG_ERR_INVALID_ARG;
  if (fp8 && (!aligned16(SFA) || !aligned16(SFB))) return MG_ERR_INVALID_ARG;
  if (dt == MG_FP8_X_FP4_E2M1) {
    // weight-scale rows (K/32 bytes) must be whole 16-byte units for TMA;
    // packed 4-bit weights need a 32-byte aligned base
    if (K % 512 != 0) return MG_ERR_UNSUPPORTED;
    if (!aligned32(B)) return MG_ERR_INVALID_ARG;
  }
  return MG_OK;
}

// sf_kblocks: K-blocks of token scales per TMA box (both kernels pack four
// K-blocks per scale word and load their scales four K-blocks at a time).
mg_status encode_operands(FwdArgs& a, const void* A, const uint8_t* SFA, const void* B,
                          int64_t rows_total, int64_t sf_rows, int64_t sf_groups,
                          uint32_t sf_kblocks) {
  const CUtensorMapDataType dt = a.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t elem = a.fp8 ? 1 : 2;
  const uint32_t box_k = 128 / elem;  // one 128-byte swizzle row
  mg_status st;
  if (a.w4) {
    // packed E2M1: TMA spreads each 16 codes (8 bytes) over 16 bytes of
    // shared memory, the operand layout of kind::mxf8f6f4, so a 128-code box
    // fills one 128-byte swizzle row like E4M3
    st = encode_2d_rows(&a.tmW, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, B, (uint64_t)a.K,
                        (uint64_t)a.E * a.N, (uint64_t)a.K / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != MG_OK) return st;
    st = encode_2d_rows(&a.tmSFW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.sfb, (uint64_t)a.K / 32,
                        (uint64_t)a.E * a.N, (uint64_t)a.K / 32, 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    st = encode_2d(&a.tmW, dt, elem, B, (uint64_t)a.K, (uint64_t)a.E * a.N, box_k, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    std::memset(&a.tmSFW, 0, sizeof(a.tmSFW));
  }
  if (st != MG_OK) return st;
  st = encode_2d(&a.tmA64, dt, elem, A, (uint64_t)a.K, (uint64_t)rows_total, box_k, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MG_OK) return st;
  st = encode_2d(&a.tmA16, dt, elem, A, (uint64_t)a.K, (uint64_t)rows_total, box_k, 16,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MG_OK) return st;
  st = encode_2d(&a.tmA8, dt, elem, A, (uint64_t)a.K, (uint64_t)rows_total, box_k, 8,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MG_OK) return st;
  if (a.fp8) {
    st = encode_sf_3d(&a.tmSF, SFA, (uint64_t)sf_rows, (uint64_t)a.K / 128, (uint64_t)sf_groups, 256,
                      sf_kblocks);
    if (st != MG_OK) return st;
  } else {
    std::memset(&a.tmSF, 0, sizeof(a.tmSF));
  }
  return MG_OK;
}

mg_status prep_contiguous(FwdArgs& a, mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                          const uint8_t* SFB, void* D, const int32_t* d_counts, int32_t E,
                          int64_t rows_cap, int32_t N, int32_t K, int32_t align_q, int32_t tile_q,
                          int32_t* d_status) {
  mg_status st = check_fwd_common(dt, A, SFA, B, SFB, D, d_counts, E, N, K);
  if (st != MG_OK) return st;
  const bool fp8 = dt != MG_BF16;
  if (rows_cap <= 0 || rows_cap >= (int64_t(1) << 31) || align_q <= 0) return MG_ERR_INVALID_ARG;
  if (fp8 && (align_q % 16 != 0 || rows_cap % 16 != 0)) return MG_ERR_UNSUPPORTED;
  if (tile_q != 0) {
    if (tile_q < 16 || tile_q > 256 || tile_q % 16 != 0) return MG_ERR_INVALID_ARG;
    if (fp8 && tile_q > 240 && tile_q != 256) return MG_ERR_INVALID_ARG;
  }
  a.fp8 = fp8;
  a.w4 = dt == MG_FP8_X_FP4_E2M1;
  a.masked = false;
  a.counts = d_counts;
  a.E = E;
  a.N = N;
  a.K = K;
  a.rows_total = (int32_t)rows_cap;
  a.align_q = align_q;
  a.tile_q = tile_q;
  a.sfb = SFB;
  a.D = D;
  a.status = d_status;
  a.wait_ns = g_wait_ns.load();
  return encode_operands(a, A, SFA, B, rows_cap, rows_cap, 1, 4u);
}

mg_status prep_masked(FwdArgs& a, mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                      const uint8_t* SFB, void* D, const int32_t* d_valid_m, int32_t E, int32_t M_max,
                      int32_t N, int32_t K, int32_t* d_status) {
  mg_status st = check_fwd_common(dt, A, SFA, B, SFB, D, d_valid_m, E, N, K);
  if (st != MG_OK) return st;
  const bool fp8 = dt != MG_BF16;
  if (M_max <= 0 || (int64_t)E * M_max >= (int64_t(1) << 31)) return MG_ERR_INVALID_ARG;
  if (fp8 && M_max % 16 != 0) return MG_ERR_UNSUPPORTED;
  a.fp8 = fp8;
  a.w4 = dt == MG_FP8_X_FP4_E2M1;
  a.masked = true;
  a.counts = d_valid_m;
  a.E = E;
  a.N = N;
  a.K = K;
  a.rows_total = E * M_max;
  a.M_max = M_max;
  a.sfb = SFB;
  a.D = D;
  a.status = d_status;
  a.wait_ns = g_wait_ns.load();
  return encode_operands(a, A, SFA, B, (int64_t)E * M_max, M_max, E, 4u);
}

// The SwiGLU epilogue pairs a gate block with its up block in every SM's
// two-block tile, so N must hold whole 256-row gate/up pairs.
mg_status check_swiglu(mg_swiglu_out out, int32_t N, const uint8_t* SFY) {
  if (out != MG_SWIGLU_BF16 && out != MG_SWIGLU_FP8_E4M3_UE8M0) return MG_ERR_INVALID_ARG;
  if (N <= 0) return MG_ERR_INVALID_ARG;
  if (N % 256 != 0) return MG_ERR_UNSUPPORTED;
  if (out == MG_SWIGLU_FP8_E4M3_UE8M0 && SFY == nullptr) return MG_ERR_INVALID_ARG;
  return MG_OK;
}

void set_swiglu(FwdArgs& a, mg_swiglu_out out, uint8_t* SFY, int64_t sfy_ld) {
  a.epi = out == MG_SWIGLU_BF16 ? kEpiSwigluBf16 : kEpiSwigluFp8;
  a.sfy = out == MG_SWIGLU_BF16 ? nullptr : SFY;
  a.sfy_ld = (int32_t)sfy_ld;
}

}  // namespace

extern "C" {

const char* mg_status_str(mg_status s) {
  switch (s) {
    case MG_OK: return "MG_OK";
    case MG_ERR_INVALID_ARG: return "MG_ERR_INVALID_ARG";
    case MG_ERR_UNSUPPORTED: return "MG_ERR_UNSUPPORTED";
    case MG_ERR_CUDA: return "MG_ERR_CUDA";
    case MG_ERR_CAPACITY: return "MG_ERR_CAPACITY";
    case MG_ERR_TIMEOUT: return "MG_ERR_TIMEOUT";
    case MG_ERR_DEVICE_ARG: return "MG_ERR_DEVICE_ARG";
  }
  return "MG_ERR_UNKNOWN";
}

mg_status moe_plan_host(const int32_t* counts, int32_t E, int32_t q, int64_t* offsets,
                        int32_t* tiles, int32_t max_tiles, mg_plan_stats* stats) {
  if (counts == nullptr || offsets == nullptr || stats == nullptr) return MG_ERR_INVALID_ARG;
  if (E <= 0 || E > (1 << 20) || q <= 0 || max_tiles < 0) return MG_ERR_INVALID_ARG;
  if (tiles == nullptr && max_tiles > 0) return MG_ERR_INVALID_ARG;
  for (int32_t e = 0; e < E; ++e)
    if (counts[e] < 0) return MG_ERR_INVALID_ARG;
  int64_t P = 0, U = 0, sq_hi_sum = 0, sq_lo_sum = 0, ntiles = 0;
  int32_t active = 0;
  for (int32_t e = 0; e < E; ++e) {
    const int64_t c = counts[e];
    const int64_t nt = cdiv64(c, q);
    offsets[e] = P;
    for (int64_t j = 0; j < nt && tiles != nullptr && ntiles + j < max_tiles; ++j) {
      if (P + j * q > INT32_MAX) break;
      int32_t* tp = tiles + 3 * (ntiles + j);
      tp[0] = e;
      tp[1] = (int32_t)(P + j * q);
      tp[2] = (int32_t)(c - j * q < q ? c - j * q : q);
    }
    ntiles += nt;
    P += nt * q;
    U += c;
    sq_hi_sum += sq_hi(c);
    sq_lo_sum += sq_lo(c);
    active += c > 0;
  }
  offsets[E] = P;
  stats->P = P;
  stats->U = U;
  const SumSq sq = sumsq_finish(sq_hi_sum, sq_lo_sum);
  stats->sumsq = sq.value;
  stats->active = active;
  stats->num_tiles = ntiles > INT32_MAX ? INT32_MAX : (int32_t)ntiles;  // saturates
  stats->pad_frac = plan_pad_frac(P, U);
  stats->eff_experts = plan_eff_experts_exact(U, sq.f64);
  if (tiles != nullptr && ntiles > max_tiles) return MG_ERR_CAPACITY;
  if (tiles != nullptr && max_tiles > 0 && P > INT32_MAX) return MG_ERR_UNSUPPORTED;
  return MG_OK;
}

mg_status moe_plan(const int32_t* d_counts, int32_t E, int32_t q, int64_t* d_offsets,
                   int32_t* d_tiles, int32_t max_tiles, mg_plan_stats* d_stats, int32_t* d_status,
                   void* stream) {
  if (d_counts == nullptr || d_offsets == nullptr || d_stats == nullptr) return MG_ERR_INVALID_ARG;
  if (E <= 0 || E > (1 << 20) || q <= 0 || max_tiles < 0) return MG_ERR_INVALID_ARG;
  if (d_tiles == nullptr && max_tiles > 0) return MG_ERR_INVALID_ARG;
  return from_cuda(launch_plan(d_counts, E, q, d_offsets, d_tiles, max_tiles, d_stats, d_status,
                               static_cast<cudaStream_t>(stream)));
}

mg_status moe_select_tile(mg_dtype dt, const int32_t* d_counts, int32_t E, int32_t N, int32_t K,
                          int32_t* d_tile_q, int32_t* d_status, void* stream) {
  if (!valid_dtype(dt) || d_counts == nullptr || d_tile_q == nullptr) return MG_ERR_INVALID_ARG;
  if (E <= 0 || N <= 0 || K <= 0) return MG_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return MG_ERR_UNSUPPORTED;
  return from_cuda(launch_select(dt != MG_BF16, fwd_variant(N, dt == MG_FP8_X_FP4_E2M1), d_counts, E, N, K,
                                 d_tile_q, d_status, static_cast<cudaStream_t>(stream)));
}

mg_status moe_select_tile_host(mg_dtype dt, const int32_t* counts, int32_t E, int32_t N, int32_t K,
                               int32_t num_sms, int32_t* tile_q) {
  if (!valid_dtype(dt) || counts == nullptr || tile_q == nullptr) return MG_ERR_INVALID_ARG;
  if (E <= 0 || N <= 0 || K <= 0) return MG_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return MG_ERR_UNSUPPORTED;
  const bool fp8 = dt != MG_BF16;
  int64_t tiles[kNumTileCand] = {};
  for (int i = 0; i < kNumTileCand; ++i)
    for (int32_t e = 0; e < E; ++e) tiles[i] += cdiv64(counts[e] > 0 ? counts[e] : 0, tile_candidate(fp8, i));
  const int sms = num_sms > 0 ? num_sms : 152;
  *tile_q = pick_tile(fp8, tiles, fwd_variant(N, dt == MG_FP8_X_FP4_E2M1), N, sel_kblocks(fp8, K), sms);
  return MG_OK;
}

mg_status mgemm_contiguous(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                           const uint8_t* SFB, void* D, const int32_t* d_counts, int32_t E,
                           int64_t rows_cap, int32_t N, int32_t K, int32_t align_q, int32_t tile_q,
                           int32_t* d_status, void* stream) {
  FwdArgs a;
  const mg_status st = prep_contiguous(a, dt, A, SFA, B, SFB, D, d_counts, E, rows_cap, N, K, align_q,
                                       tile_q, d_status);
  if (st != MG_OK) return st;
  return from_cuda(launch_fwd_any(a, static_cast<cudaStream_t>(stream)));
}

mg_status mgemm_masked(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                       const uint8_t* SFB, void* D, const int32_t* d_valid_m, int32_t E,
                       int32_t M_max, int32_t N, int32_t K, int32_t* d_status, void* stream) {
  FwdArgs a;
  const mg_status st = prep_masked(a, dt, A, SFA, B, SFB, D, d_valid_m, E, M_max, N, K, d_status);
  if (st != MG_OK) return st;
  return from_cuda(launch_fwd_any(a, static_cast<cudaStream_t>(stream)));
}

mg_status mgemm_contiguous_swiglu(mg_dtype dt, mg_swiglu_out out, const void* A, const uint8_t* SFA,
                                  const void* B, const uint8_t* SFB, void* Y, uint8_t* SFY,
                                  const int32_t* d_counts, int32_t E, int64_t rows_cap, int32_t N,
                                  int32_t K, int32_t align_q, int32_t tile_q, int32_t* d_status,
                                  void* stream) {
  mg_status st = check_swiglu(out, N, SFY);
  if (st != MG_OK) return st;
  FwdArgs a;
  st = prep_contiguous(a, dt, A, SFA, B, SFB, Y, d_counts, E, rows_cap, N, K, align_q, tile_q, d_status);
  if (st != MG_OK) return st;
  set_swiglu(a, out, SFY, rows_cap);
  // two-block tiles only: CTA pairs (two gate/up pairs per tile) where the
  // plain call would run them, else one SM
  const int v = fwd_variant(N, a.w4, false);
  return from_cuda(launch_fwd(a, static_cast<cudaStream_t>(stream), v == kFwdPairDual ? kFwdPairDual : kFwdDual));
}

mg_status mgemm_masked_swiglu(mg_dtype dt, mg_swiglu_out out, const void* A, const uint8_t* SFA,
                              const void* B, const uint8_t* SFB, void* Y, uint8_t* SFY,
                              const int32_t* d_valid_m, int32_t E, int32_t M_max, int32_t N, int32_t K,
                              int32_t* d_status, void* stream) {
  mg_status st = check_swiglu(out, N, SFY);
  if (st != MG_OK) return st;
  FwdArgs a;
  st = prep_masked(a, dt, A, SFA, B, SFB, Y, d_valid_m, E, M_max, N, K, d_status);
  if (st != MG_OK) return st;
  set_swiglu(a, out, SFY, M_max);
  return from_cuda(launch_fwd(a, static_cast<cudaStream_t>(stream), kFwdDual));
}

mg_status moe_exemplar_features_host(const int32_t* counts, int32_t E, int32_t* lu, int32_t* share) {
  if (counts == nullptr || lu == nullptr || share == nullptr || E <= 0) return MG_ERR_INVALID_ARG;
  if (E > kSelMaxExperts) return MG_ERR_UNSUPPORTED;  // keeps 65536 * (top-m sum) within int64
  exemplar_features_host(counts, E, lu, share);
  return MG_OK;
}

mg_status moe_select_exemplar_host(const int32_t* counts, int32_t E, const mg_exemplar* table, int32_t n,
                                   int32_t margin, int32_t prev, int32_t* choice) {
  if (counts == nullptr || table == nullptr || choice == nullptr || E <= 0 || n <= 0 || margin < 0)
    return MG_ERR_INVALID_ARG;
  if (E > kSelMaxExperts) return MG_ERR_UNSUPPORTED;
  *choice = exemplar_choose_host(counts, E, table, n, margin, prev, nullptr);
  return MG_OK;
}

mg_status moe_select_exemplar(const int32_t* d_counts, int32_t E, const mg_exemplar* d_table, int32_t n,
                              int32_t margin, int32_t* d_state, int32_t* d_tactic, int32_t* d_status,
                              void* stream) {
  if (d_counts == nullptr || d_table == nullptr || d_tactic == nullptr) return MG_ERR_INVALID_ARG;
  if (E <= 0 || n <= 0 || margin < 0) return MG_ERR_INVALID_ARG;
  if (E > kSelMaxExperts || n > kSelMaxExemplars) return MG_ERR_UNSUPPORTED;
  return from_cuda(launch_exemplar(d_counts, E, d_table, n, margin, d_state, d_tactic, d_status,
                                   static_cast<cudaStream_t>(stream)));
}

mg_status mgemm_contiguous_tactic(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                                  const uint8_t* SFB, void* D, const int32_t* d_counts, int32_t E,
                                  int64_t rows_cap, int32_t N, int32_t K, int32_t align_q,
                                  const int32_t* d_tactic, int32_t* d_status, void* stream) {
  if (d_tactic == nullptr) return MG_ERR_INVALID_ARG;
  FwdArgs a;
  const mg_status st = prep_contiguous(a, dt, A, SFA, B, SFB, D, d_counts, E, rows_cap, N, K, align_q, 0,
                                       d_status);
  if (st != MG_OK) return st;
  a.tactic = d_tactic;
  return from_cuda(launch_fwd_any(a, static_cast<cudaStream_t>(stream)));
}

mg_status mgemm_masked_tactic(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                              const uint8_t* SFB, void* D, const int32_t* d_valid_m, int32_t E,
                              int32_t M_max, int32_t N, int32_t K, const int32_t* d_tactic,
                              int32_t* d_status, void* stream) {
  if (d_tactic == nullptr) return MG_ERR_INVALID_ARG;
  FwdArgs a;
  const mg_status st = prep_masked(a, dt, A, SFA, B, SFB, D, d_valid_m, E, M_max, N, K, d_status);
  if (st != MG_OK) return st;
  a.tactic = d_tactic;
  return from_cuda(launch_fwd_any(a, static_cast<cudaStream_t>(stream)));
}

mg_status mgemm_masked_exemplar(mg_dtype dt, const void* A, const uint8_t* SFA, const void* B,
                                const uint8_t* SFB, void* D, const int32_t* d_valid_m, int32_t E,
                                int32_t M_max, int32_t N, int32_t K, const mg_exemplar* d_table,
                                int32_t n, int32_t* d_tactic_out, int32_t* d_status, void* stream) {
  if (d_table == nullptr || n <= 0) return MG_ERR_INVALID_ARG;
  if (!aligned16(d_table) || (d_tactic_out != nullptr && !aligned16(d_tactic_out))) return MG_ERR_INVALID_ARG;
  if (E > kFusedExemplarMaxExperts || n > kSelMaxExemplars) return MG_ERR_UNSUPPORTED;
  FwdArgs a;
  const mg_status st = prep_masked(a, dt, A, SFA, B, SFB, D, d_valid_m, E, M_max, N, K, d_status);
  if (st != MG_OK) return st;
  a.table = d_table;
  a.n_table = n;
  a.tactic_out = d_tactic_out;
  return from_cuda(launch_fwd_any(a, static_cast<cudaStream_t>(stream)));
}

mg_status kgemm_grouped(const void* dY, const void* X, float* dW, const int32_t* d_counts,
                        int32_t E, int64_t T_cap, int32_t N, int32_t K, int32_t* d_status,
                        void* stream) {
  if (dY == nullptr || X == nullptr || dW == nullptr || d_counts == nullptr) return MG_ERR_INVALID_ARG;
  if (E <= 0 || N <= 0 || K <= 0 || T_cap <= 0 || T_cap >= (int64_t(1) << 31)) return MG_ERR_INVALID_ARG;
  if (E > kMaxExperts) return MG_ERR_UNSUPPORTED;
  if (N % 128 != 0 || K % 128 != 0) return MG_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= (int64_t(1) << 31)) return MG_ERR_UNSUPPORTED;  // dW rows are int32 coordinates
  if (!aligned16(dY) || !aligned16(X) || !aligned16(dW) || !aligned16(d_counts)) return MG_ERR_INVALID_ARG;
  KgArgs a;
  a.counts = d_counts;
  a.E = E;
  a.N = N;
  a.K = K;
  a.T_cap = (int32_t)T_cap;
  a.dW = dW;
  a.status = d_status;
  a.wait_ns = g_wait_ns.load();
  mg_status st = encode_2d(&a.tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dY, (uint64_t)N,
                           (uint64_t)T_cap, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MG_OK) return st;
  st = encode_2d(&a.tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, (uint64_t)K, (uint64_t)T_cap, 64,
                 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MG_OK) return st;
  // dW as [E*N, K] fp32, stored by the epilogue in 32 x 32 boxes
  st = encode_2d(&a.tmDW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW, (uint64_t)K, (uint64_t)E * N, 32, 32,
                 CU_TENSOR_MAP_SWIZZLE_128B);
  if (st != MG_OK) return st;
  return from_cuda(launch_kgrouped(a, static_cast<cudaStream_t>(stream)));
}

mg_status mg_set_wait_limit_ns(int64_t ns) {
  g_wait_ns.store(ns > 0 ? ns : kDefaultWaitNs);
  return MG_OK;
}

int64_t mg_get_wait_limit_ns(void) { return g_wait_ns.load(); }

mg_status mg_set_kernel_policy(int32_t policy) {
  if (policy < 0 || policy > 5) return MG_ERR_INVALID_ARG;
  g_policy.store(policy);
  return MG_OK;
}

int32_t mg_get_kernel_policy(void) { return g_policy.load(); }

mg_status mg_wait_selftest(int32_t* d_status, int64_t limit_ns, void* stream) {
  if (d_status == nullptr || limit_ns <= 0 || limit_ns > 10000000000LL) return MG_ERR_INVALID_ARG;
  return from_cuda(launch_wait_selftest(d_status, limit_ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
