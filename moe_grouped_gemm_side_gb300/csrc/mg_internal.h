// Internal host-side interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "moegemm.h"

namespace mg {

// Epilogue of the contiguous/masked kernel: plain bf16 D, or SwiGLU of
// interleaved gate/up blocks stored as bf16 or as E4M3 with UE8M0 scales.
enum FwdEpilogue { kEpiPlain = 0, kEpiSwigluBf16 = 1, kEpiSwigluFp8 = 2 };

// Contiguous and masked forms share one kernel: both place an expert's
// token rows at a known row base of a 2-D [rows_total, K] activation view and
// compute only its first t_e rows.
struct FwdArgs {
  bool fp8 = false;                 // E4M3 activations (and weights unless w4)
  bool w4 = false;                  // E2M1 weights, UE8M0 per (row, 32 K)
  bool masked = false;
  const int32_t* counts = nullptr;  // t_e (contiguous) or valid_m (masked)
  int32_t E = 0, N = 0, K = 0;
  int32_t rows_total = 0;           // contiguous: rows_cap; masked: E*M_max
  int32_t M_max = 0;                // masked only
  int32_t align_q = 1;              // contiguous only
  int32_t tile_q = 0;               // 0: choose on the device
  const uint8_t* sfb = nullptr;     // fp8 weight scales [E, K/128, N/128]
  void* D = nullptr;
  int32_t epi = kEpiPlain;
  uint8_t* sfy = nullptr;           // kEpiSwigluFp8: scales [z][N/256][sfy_ld]
  int32_t sfy_ld = 0;
  int32_t* status = nullptr;
  const int32_t* tactic = nullptr;  // device {tile_q, blocks} or null
  const mg_exemplar* table = nullptr;  // exemplar table matched in the prologue, or null
  int32_t n_table = 0;
  int32_t* tactic_out = nullptr;    // with a table: {tile_q, blocks, index} of the choice, or null
  int64_t wait_ns = 0;
  CUtensorMap tmW{}, tmA64{}, tmA16{}, tmA8{}, tmSF{};
  CUtensorMap tmSFW{};              // w4: weight scales [E*N, K/32]
};
// Contiguous/masked kernel of one family (FwdVariant in sched.cuh).
cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t s, int variant);

struct KgArgs {
  const int32_t* counts = nullptr;
  int32_t E = 0, N = 0, K = 0;
  int32_t T_cap = 0;
  float* dW = nullptr;
  int32_t* status = nullptr;
  int64_t wait_ns = 0;
  CUtensorMap tmY{}, tmX{}, tmDW{};
};
cudaError_t launch_kgrouped(const KgArgs& a, cudaStream_t s);

cudaError_t launch_plan(const int32_t* counts, int32_t E, int32_t q, int64_t* offsets,
                        int32_t* tiles, int32_t max_tiles, mg_plan_stats* stats,
                        int32_t* status, cudaStream_t s);
cudaError_t launch_select(bool fp8, int variant, const int32_t* counts, int32_t E, int32_t N,
                          int32_t K, int32_t* tile_q, int32_t* status, cudaStream_t s);
cudaError_t launch_wait_selftest(int32_t* status, int64_t limit_ns, cudaStream_t s);

// Exemplar selector: integer features and choice, host and device.
constexpr int kExemplarShares = MG_EXEMPLAR_SHARES;
constexpr int32_t kShareOne = 65536;
constexpr int32_t kLuWeight = 2048;
constexpr int kSelMaxExperts = 4096;
constexpr int kSelMaxExemplars = 1024;
constexpr int kFusedExemplarMaxExperts = 32;  // mgemm_masked_exemplar: one warp per CTA
cudaError_t launch_exemplar(const int32_t* counts, int32_t E, const mg_exemplar* table, int32_t n,
                            int32_t margin, int32_t* state, int32_t* tactic, int32_t* status,
                            cudaStream_t s);
void exemplar_features_host(const int32_t* counts, int32_t E, int32_t* lu, int32_t* share);
int32_t exemplar_choose_host(const int32_t* counts, int32_t E, const mg_exemplar* table, int32_t n,
                             int32_t margin, int32_t prev, int64_t* dist_out);

int num_sms_current_device();

constexpr int kMaxExperts = 1024;

}  // namespace mg
