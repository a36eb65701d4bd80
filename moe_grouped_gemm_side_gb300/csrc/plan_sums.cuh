// Sum of squared expert counts for the effective expert count U^2 / sum t^2
// ("MoE GroupGEMM padding under expert skew", "Summarize skew without losing
// the histogram"), kept exact where int64 is not wide enough: three experts
// at 2^31 - 1 tokens already pass 2^63.  Each t^2 (t < 2^31, so t^2 < 2^62)
// is split into its high and low 32-bit halves and the halves are summed
// separately; for up to 2^20 experts the two sums stay below 2^50 and 2^52,
// exact in int64 and in double.  Shared by the host planner and the device
// plan kernel so that both round the same way.
#pragma once

#include <climits>
#include <cstdint>

#include "sched.cuh"

namespace mg {

MG_HD int64_t sq_hi(int64_t c) { return (int64_t)((uint64_t)(c * c) >> 32); }
MG_HD int64_t sq_lo(int64_t c) { return (int64_t)((uint64_t)(c * c) & 0xffffffffull); }

MG_HD double f64_add(double a, double b) {
#ifdef __CUDA_ARCH__
  return __dadd_rn(a, b);
#else
  return a + b;
#endif
}

struct SumSq {
  int64_t value;  // the exact sum, or INT64_MAX when it does not fit
  double f64;     // the exact sum rounded to nearest
};

// hi = sum of sq_hi, lo = sum of sq_lo.  hi * 2^32 and lo are exact doubles,
// so their one rounded addition is the exact sum rounded to nearest.
MG_HD SumSq sumsq_finish(int64_t hi, int64_t lo) {
  SumSq r;
  if (hi >= (int64_t(1) << 31)) {
    r.value = INT64_MAX;
  } else {
    const uint64_t v = ((uint64_t)hi << 32) + (uint64_t)lo;
    r.value = v > (uint64_t)INT64_MAX ? INT64_MAX : (int64_t)v;
  }
  r.f64 = f64_add(f64_mul(i64_to_f64(hi), 4294967296.0), i64_to_f64(lo));
  return r;
}

// U^2 / sum t^2 in the order of the definition; 0 if no expert has tokens.
MG_HD double plan_eff_experts_exact(int64_t U, double sumsq_f64) {
  if (sumsq_f64 == 0.0) return 0.0;
  const double u = i64_to_f64(U);
  return f64_div(f64_mul(u, u), sumsq_f64);
}

}  // namespace mg
