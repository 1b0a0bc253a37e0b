// Hardware-aware prefix scheduler of the verify lengths (host code).
//
// DSpark summary, "Confidence-Scheduled Verification": each request r carries
// per-position confidences c_{r,i} (the probability that draft i survives
// given that drafts 1 .. i-1 did), so its survival probabilities
// a_{r,j} = prod_{i <= j} c_{r,i} never increase with j. The expected tokens
// of a step that verifies L_r drafts of every request are
//   tau(L) = sum_r (1 + sum_{j <= L_r} a_{r,j})        (accepted + one more)
// and the step verifies M = sum_r (L_r + 1) rows, costing T(M) from a table
// measured once on the device (the "SPS" table: steps per second 1 / T(M)).
// The scheduler maximizes the throughput Theta = tau / T(M). For a fixed M
// the best tau takes the M - B largest survival probabilities, and since
// a_{r,j} never increases with j, any such set is a prefix of every
// request's drafts; so one global sort of the a_{r,j}, admitted greedily,
// visits the best L for every M, each step an O(1) table lookup.
// With early stopping the scan ends at the first admission that lowers Theta
// (the global maximum when Theta is unimodal in M); without it the scan
// covers every M and keeps the best, which the summary's deployment section
// prefers because measured step costs fall in steps, not smoothly.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <vector>

#include "internal.h"

extern "C" sv_status sv_schedule_prefix(int32_t batch, int32_t gamma, const float* conf, const float* step_us,
                                        int32_t n_cost, int32_t early_stop, int32_t* verify_lens,
                                        double* expected_tokens, double* throughput) {
  if (batch < 1 || gamma < 0 || !conf || !step_us || !verify_lens || n_cost < 1) {
    sv::record_error("sv_schedule_prefix: NULL pointer or bad size");
    return SV_ERR_INVALID_ARG;
  }
  if (n_cost < batch) {
    sv::record_error("sv_schedule_prefix: the cost table must cover M = batch (every request's anchor row)");
    return SV_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_cost; ++i)
    if (!(step_us[i] > 0.f) || std::isinf(step_us[i])) {
      sv::record_error("sv_schedule_prefix: step costs must be finite and positive");
      return SV_ERR_INVALID_ARG;
    }
  struct Cand {
    double a;  // survival probability a_{r,j}
    int r, j;
  };
  std::vector<Cand> cand;
  cand.reserve(static_cast<size_t>(batch) * gamma);
  for (int r = 0; r < batch; ++r) {
    double a = 1.0;
    for (int j = 1; j <= gamma; ++j) {
      const float c = conf[static_cast<size_t>(r) * gamma + (j - 1)];
      if (!(c >= 0.f && c <= 1.f)) {
        sv::record_error("sv_schedule_prefix: confidences must lie in [0, 1]");
        return SV_ERR_INVALID_ARG;
      }
      a *= c;
      cand.push_back({a, r, j});
    }
  }
  // descending survival; ties by position then request, so a request's drafts
  // enter in order even where its survival stays flat
  std::stable_sort(cand.begin(), cand.end(), [](const Cand& x, const Cand& y) {
    if (x.a != y.a) return x.a > y.a;
    if (x.j != y.j) return x.j < y.j;
    return x.r < y.r;
  });
  double tau = batch;
  int M = batch;
  double best = tau / step_us[M - 1];
  size_t best_k = 0;
  for (size_t k = 0; k < cand.size(); ++k) {
    if (M + 1 > n_cost) break;  // no measured cost beyond the table
    tau += cand[k].a;
    ++M;
    const double th = tau / step_us[M - 1];
    if (th > best) {
      best = th;
      best_k = k + 1;
    } else if (early_stop && th < best) {
      break;
    }
  }
  for (int r = 0; r < batch; ++r) verify_lens[r] = 0;
  double t_best = batch;
  for (size_t k = 0; k < best_k; ++k) {
    verify_lens[cand[k].r] = std::max(verify_lens[cand[k].r], cand[k].j);
    t_best += cand[k].a;
  }
  if (expected_tokens) *expected_tokens = t_best;
  if (throughput) *throughput = best * 1e6;  // tokens per second
  return SV_OK;
}
