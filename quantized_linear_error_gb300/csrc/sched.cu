// SLO-constrained, compensator-aware chunk scheduler ("SPEAR: A System for
// Post-Quantization Error-Adaptive Recovery", section 2.2C): a latency lookup
// table of measured step times, indexed by the share of layers that carry a
// compensator (the EC density) and by the tokens in the step, predicts the
// time of a step; the scheduler picks the largest prefill chunk whose step,
// batched with the pending decode tokens, meets an inter-token-latency target.
// Host code only.
#include <algorithm>
#include <new>
#include <vector>

#include "../../include/spear.h"

struct spear_sched_s {
  std::vector<double> dens;  // ascending, in [0, 1]
  std::vector<int> toks;     // ascending, >= 1
  std::vector<double> ms;    // [dens][toks]
};

namespace {

// Piecewise-linear in the token count (linear extrapolation past either end
// of the table, from its first or last two points), at one density row.
double row_predict(const spear_sched_s* s, size_t i, double m) {
  const std::vector<int>& t = s->toks;
  const double* row = s->ms.data() + i * t.size();
  if (t.size() == 1) return row[0];
  size_t j = 1;
  while (j + 1 < t.size() && m > t[j]) ++j;
  const double t0 = t[j - 1], t1 = t[j];
  return row[j - 1] + (row[j] - row[j - 1]) * (m - t0) / (t1 - t0);
}

double predict(const spear_sched_s* s, int M, double d) {
  const std::vector<double>& ds = s->dens;
  if (d <= ds.front() || ds.size() == 1) return row_predict(s, 0, M);
  if (d >= ds.back()) return row_predict(s, ds.size() - 1, M);
  size_t i = 1;
  while (i + 1 < ds.size() && d > ds[i]) ++i;
  const double a = row_predict(s, i - 1, M), b = row_predict(s, i, M);
  return a + (b - a) * (d - ds[i - 1]) / (ds[i] - ds[i - 1]);
}

}  // namespace

extern "C" {

spear_status_t spear_sched_create(const double* densities, int32_t n_d, const int32_t* tokens, int32_t n_m,
                                  const double* ms, spear_sched_t* out) {
  if (!out) return SPEAR_ERR_INVALID_ARG;
  *out = nullptr;
  if (!densities || !tokens || !ms || n_d < 1 || n_m < 1) return SPEAR_ERR_INVALID_ARG;
  for (int i = 0; i < n_d; ++i)
    if (!(densities[i] >= 0.0 && densities[i] <= 1.0) || (i > 0 && !(densities[i] > densities[i - 1])))
      return SPEAR_ERR_INVALID_ARG;
  for (int j = 0; j < n_m; ++j)
    if (tokens[j] < 1 || (j > 0 && tokens[j] <= tokens[j - 1])) return SPEAR_ERR_INVALID_ARG;
  for (long k = 0; k < (long)n_d * n_m; ++k)
    if (!(ms[k] >= 0.0)) return SPEAR_ERR_INVALID_ARG;
  spear_sched_s* s = new (std::nothrow) spear_sched_s();
  if (!s) return SPEAR_ERR_OOM;
  s->dens.assign(densities, densities + n_d);
  s->toks.assign(tokens, tokens + n_m);
  s->ms.assign(ms, ms + (long)n_d * n_m);
  *out = s;
  return SPEAR_OK;
}

double spear_sched_predict(spear_sched_t s, int32_t M, double density) {
  if (!s || M < 0) return -1.0;
  return predict(s, M, density);
}

spear_status_t spear_sched_pick_chunk(spear_sched_t s, int32_t n_decode, double density, double itl_ms,
                                      const int32_t* candidates, int32_t n_c, int32_t* chunk_out) {
  if (!s || !candidates || !chunk_out || n_c < 0 || n_decode < 0) return SPEAR_ERR_INVALID_ARG;
  int32_t best = 0;
  for (int k = 0; k < n_c; ++k) {
    const int32_t c = candidates[k];
    if (c < 0) return SPEAR_ERR_INVALID_ARG;
    if (c > best && predict(s, n_decode + c, density) <= itl_ms) best = c;
  }
  *chunk_out = best;
  return SPEAR_OK;
}

spear_status_t spear_sched_destroy(spear_sched_t s) {
  delete s;
  return SPEAR_OK;
}

}  // extern "C"
