// cbq_draft.cpp -- the draft length of the next verify round (host only).
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section
// "Adaptive speculation / Adaptive draft length": with acceptance probability
// q per drafted token and c the added cost of one more draft token, a round
// of d drafted tokens yields E[N_d] = sum_{j=0..d} q^j tokens on average (the
// drafted tokens accepted before the first rejection, plus one token the
// target model produces itself) in time
// T(d) = 1 + c (d - 1) relative to d = 1; the round drafts
// d* = argmax_{1 <= d <= dmax} E[N_d] / T(d) tokens, so the verify round that
// follows multiplies d* + 1 token rows per request by the weights.
//
// Ties go to the shorter draft (the page is silent); the sum is accumulated
// in increasing j in double precision, which also covers q = 1.
#include <cmath>
#include <cstdint>

#include "cbq_internal.h"

namespace {
constexpr int32_t kMaxDraft = 63;
}

extern "C" int cbq_draft_length(double q, double c, int32_t dmax, int32_t* d_star, double* expected_tokens,
                                double* tokens_per_time) {
  // dmax <= 63: a verify round multiplies d* + 1 token rows per request and
  // cbq_gemm takes at most 64 rows, so a longer draft could not be verified.
  if (!d_star || dmax < 1 || dmax > kMaxDraft || !(q >= 0.0 && q <= 1.0) || !(c >= 0.0) || !std::isfinite(c))
    return CBQ_EINVAL;
  double sum = 1.0, power = 1.0;                  // E[N_0] = q^0
  int32_t best_d = 0;
  double best_e = 0.0, best_r = 0.0;
  for (int32_t d = 1; d <= dmax; ++d) {
    power *= q;
    sum += power;                                 // E[N_d]
    const double r = sum / (1.0 + c * static_cast<double>(d - 1));
    if (best_d == 0 || r > best_r) {
      best_d = d;
      best_e = sum;
      best_r = r;
    }
  }
  *d_star = best_d;
  if (expected_tokens) *expected_tokens = best_e;
  if (tokens_per_time) *tokens_per_time = best_r;
  return CBQ_OK;
}
