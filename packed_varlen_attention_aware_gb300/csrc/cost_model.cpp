// Cost models of "ByteScale: Communication-Efficient Scaling of LLM Training
// with a 2048K Context Length on 16384 GPUs" (research digest):
//   section 3.2  ring timing model: per-step compute t_c and ring time T_attn;
//   section 3.3  profiled models T(s), Act(s) and Eq. 3 (offload ratio and
//                rank count of a long sequence).
// Host arithmetic only.  Every entry point validates its arguments and
// reports through the status code; nothing allocates.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <utility>

#include "internal.h"

namespace {

// A quotient within this relative distance above an integer counts as that
// integer when Eq. 3 takes its ceiling, so exact multiples of C are not pushed
// up by the rounding of the double-precision products.
constexpr double kCeilRelTol = 1e-9;

int64_t ceil_tol(double x) {
  const double k = std::floor(x);
  if (x == k) return static_cast<int64_t>(k);
  if (k > 0 && (x - k) <= kCeilRelTol * x) return static_cast<int64_t>(k);
  return static_cast<int64_t>(k) + 1;
}

// Solves the n x n system a x = b in place (Gaussian elimination with partial
// pivoting); false when a pivot vanishes.
bool solve_small(double* a, double* b, int n) {
  for (int c = 0; c < n; ++c) {
    int piv = c;
    for (int r = c + 1; r < n; ++r)
      if (std::fabs(a[r * n + c]) > std::fabs(a[piv * n + c])) piv = r;
    if (a[piv * n + c] == 0.0) return false;
    if (piv != c) {
      for (int k = 0; k < n; ++k) std::swap(a[c * n + k], a[piv * n + k]);
      std::swap(b[c], b[piv]);
    }
    for (int r = c + 1; r < n; ++r) {
      const double f = a[r * n + c] / a[c * n + c];
      for (int k = c; k < n; ++k) a[r * n + k] -= f * a[c * n + k];
      b[r] -= f * b[c];
    }
  }
  for (int c = n - 1; c >= 0; --c) {
    double v = b[c];
    for (int k = c + 1; k < n; ++k) v -= a[c * n + k] * b[k];
    b[c] = v / a[c * n + c];
  }
  return true;
}

}  // namespace

extern "C" {

hdp_status_t hdp_ring_step_compute(const int32_t* lengths, int32_t n, int32_t num_ranks, int32_t capacity,
                                   double t_blk, double* t_c) {
  if (!lengths || !t_c) return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_ring_step_compute: null pointer");
  if (n < 1 || num_ranks < 1 || capacity < 1 || !(t_blk >= 0.0))
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_ring_step_compute: n, num_ranks, capacity >= 1 and t_blk >= 0");
  const int64_t ring_tokens = static_cast<int64_t>(num_ranks) * capacity;
  int64_t sum = 0;
  // sum of s_i^2 exactly in 128-bit integers, then one division
  unsigned __int128 sq = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (lengths[i] < 1) return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_ring_step_compute: every length >= 1");
    sum += lengths[i];
    sq += static_cast<unsigned __int128>(static_cast<uint64_t>(lengths[i]) * static_cast<uint64_t>(lengths[i]));
  }
  if (sum > ring_tokens)
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_ring_step_compute: the pack exceeds num_ranks * capacity tokens");
  const long double frac = static_cast<long double>(sq) /
                           (static_cast<long double>(ring_tokens) * static_cast<long double>(ring_tokens));
  *t_c = static_cast<double>(static_cast<long double>(t_blk) * frac);
  return HDP_OK;
}

hdp_status_t hdp_ring_attention_time(int32_t num_ranks, double t_c, double t_x, double* t_attn) {
  if (!t_attn) return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_ring_attention_time: null pointer");
  if (num_ranks < 1 || !(t_c >= 0.0) || !(t_x >= 0.0))
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_ring_attention_time: num_ranks >= 1, t_c >= 0, t_x >= 0");
  const long double step = t_c > t_x ? t_c : t_x;
  *t_attn = static_cast<double>(static_cast<long double>(num_ranks - 1) * step + t_c);
  return HDP_OK;
}

hdp_status_t hdp_offload_ranks(const hdp_offload_model_t* m, int64_t s, int64_t capacity, double* r_out,
                               int64_t* ranks) {
  if (!m || !r_out || !ranks) return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_offload_ranks: null pointer");
  if (s < 1 || capacity < 1 || m->layers < 3 || !(m->bw_d2h >= 0.0) || !(m->bw_h2d >= 0.0))
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT,
                     "hdp_offload_ranks: s >= 1, capacity >= 1, layers >= 3, bandwidths >= 0");
  const long double l = m->layers;
  const long double ss = static_cast<long double>(s), cc = static_cast<long double>(capacity);
  const long double act_s = static_cast<long double>(m->alpha2) * ss + m->beta2;
  const long double act_c = static_cast<long double>(m->alpha2) * cc + m->beta2;
  const long double t_s = static_cast<long double>(m->alpha1) * ss * ss + static_cast<long double>(m->beta1) * ss +
                          m->gamma;
  if (!(act_s > 0) || !(act_c > 0))
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_offload_ranks: Act(s) and Act(C) must be positive");
  // Eq. 3, third line: admissible ratios
  long double r_lo = l * act_c / ((l - 2) * act_s);
  if (r_lo > 1) r_lo = 1;
  // second line: the copy hides behind compute
  const long double bmin = m->bw_d2h < m->bw_h2d ? m->bw_d2h : m->bw_h2d;
  long double r = t_s * bmin / act_s;
  if (r > 1) r = 1;
  if (r < r_lo) r = 0;  // nothing admissible: no offloading
  // first line: D does not grow with r, so the largest admissible r is the best
  const long double q = (2 * act_s + (1 - r) * (l - 2) * act_s) / (l * act_c);
  *r_out = static_cast<double>(r);
  *ranks = ceil_tol(static_cast<double>(q));
  return HDP_OK;
}

hdp_status_t hdp_fit_cost_model(const double* x, const double* y, const double* w, int32_t n, int32_t degree,
                                double* coef) {
  if (!x || !y || !coef) return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_fit_cost_model: null pointer");
  if (degree < 1 || degree > 2 || n <= degree)
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_fit_cost_model: degree 1 or 2 and n > degree");
  double scale = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (!std::isfinite(x[i]) || !std::isfinite(y[i]) || (w && !(w[i] >= 0.0 && std::isfinite(w[i]))))
      return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_fit_cost_model: non-finite point or negative weight");
    if (!w || w[i] > 0) scale = std::fmax(scale, std::fabs(x[i]));
  }
  if (scale == 0) return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_fit_cost_model: all weighted x are zero");
  // at least degree + 1 distinct x values with positive weight
  {
    double seen[2] = {0, 0};
    int distinct = 0;
    for (int32_t i = 0; i < n && distinct <= degree; ++i) {
      if (w && !(w[i] > 0)) continue;
      bool fresh = true;
      for (int k = 0; k < distinct; ++k) fresh = fresh && x[i] != seen[k];
      if (fresh) {
        if (distinct < 2) seen[distinct] = x[i];
        ++distinct;
      }
    }
    if (distinct <= degree)
      return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_fit_cost_model: fewer than degree + 1 distinct x values");
  }
  // weighted normal equations in u = x / scale, accumulated in long double
  const int m = degree + 1;
  long double ata[9] = {0}, aty[3] = {0};
  for (int32_t i = 0; i < n; ++i) {
    const long double wi = w ? w[i] : 1.0;
    if (!(wi > 0)) continue;
    const long double u = static_cast<long double>(x[i]) / scale;
    long double p[3] = {1, u, u * u};
    for (int r = 0; r < m; ++r) {
      aty[r] += wi * p[r] * y[i];
      for (int c = 0; c < m; ++c) ata[r * m + c] += wi * p[r] * p[c];
    }
  }
  double a[9], b[3];
  for (int k = 0; k < m * m; ++k) a[k] = static_cast<double>(ata[k]);
  for (int k = 0; k < m; ++k) b[k] = static_cast<double>(aty[k]);
  if (!solve_small(a, b, m))
    return hdp::fail(HDP_ERR_INVALID_ARGUMENT, "hdp_fit_cost_model: fewer than degree + 1 distinct x values");
  double sk = 1;
  for (int k = 0; k < m; ++k) {
    coef[k] = b[k] / sk;
    sk *= scale;
  }
  return HDP_OK;
}

}  // extern "C"
