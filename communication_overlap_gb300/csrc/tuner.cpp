// Wave-group partition tuning: the latency predictor of Algorithm 1 and an
// exact search over all partitions.
//
// Page: "FlashOverlap: 信号驱动计算通信重叠论文详解", 四、实时调优 (Algorithm 1):
// per group t_p = duration / T * |G_i|, t_m = the communication latency
// interpolated at the group's data size, t_acc_m = max(t_acc_p, t_acc_m) +
// t_m.  Read with a group's communication starting once its own compute is
// done:  E_i = max(C_i, E_{i-1}) + t_m(G_i),  C_i = compute end of G_1..G_i.
//
// The pages enumerate all 2^(T-1) candidates (128 at T = 8).  E_i depends on
// the earlier groups only through E_{i-1}, and the rest of the recurrence is
// non-decreasing in E_{i-1}; so the smallest final E is found exactly by a
// dynamic program over group boundaries: best[w] = the smallest E of any
// partition of waves [0, w), best[w] = min_v max(w d, best[v]) + t_m(v..w).
// O(T^2) instead of O(2^T), which makes T = 98 (the grouped workload)
// tractable.
//
// Interference (the _ex entry points; not in the pages, whose compute and
// communication use separate hardware): on one GPU the GEMM and the consumer
// share memory and SMs, so each slows the other while both run.  While a
// communication runs the GEMM advances at 1 / sigma (gemm_slowdown) of its
// rate; while the GEMM runs a communication advances at 1 / rho
// (comm_slowdown) of the curve's rate.  The GEMM's progress then depends on
// the whole schedule of earlier communications, so the dynamic program no
// longer applies: with factors other than 1 the search is exhaustive up to
// T = 20 waves and a local search beyond (single cuts toggled from the best
// of the plain optimum, the finest partition and one wave then groups of
// two).  sigma = rho = 1 is the pages' predictor and the exact search.
#include <algorithm>
#include <cmath>
#include <limits>
#include <utility>
#include <vector>

#include "fo_internal.h"

namespace fo {

namespace {

struct Curve {
  std::vector<std::pair<double, double>> pts;  // (bytes, latency), sorted

  // Piecewise linear; the first latency below the first sample; the last
  // segment's slope above the last sample.
  double at(double bytes) const {
    if (bytes <= pts.front().first) return pts.front().second;
    for (size_t i = 1; i < pts.size(); ++i)
      if (bytes <= pts[i].first) {
        const auto& a = pts[i - 1];
        const auto& b = pts[i];
        return a.second + (b.second - a.second) * (bytes - a.first) / (b.first - a.first);
      }
    const auto& a = pts[pts.size() - 2];
    const auto& b = pts.back();
    return b.second + (b.second - a.second) * (bytes - b.first) / (b.first - a.first);
  }
};

fo_status make_curve(const double* bytes, const double* us, int32_t n, Curve* c) {
  if (!bytes || !us || n < 2) return FO_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    if (!(bytes[i] >= 0) || !(us[i] >= 0) || !std::isfinite(bytes[i]) || !std::isfinite(us[i]))
      return FO_ERR_ARG;
    c->pts.emplace_back(bytes[i], us[i]);
  }
  std::sort(c->pts.begin(), c->pts.end());
  for (int i = 1; i < n; ++i)
    if (c->pts[i].first == c->pts[i - 1].first) return FO_ERR_ARG;  // duplicate size
  return FO_OK;
}

struct Shape {
  int32_t W = 0, tiles = 0, waves = 0;
  double tile_bytes = 0;
  // bytes of the tiles in waves [v, w)
  double bytes(int32_t v, int32_t w) const {
    const int64_t first = int64_t(v) * W;
    const int64_t last = std::min<int64_t>(tiles, int64_t(w) * W);
    return double(last - first) * tile_bytes;
  }
};

fo_status make_shape(const fo_plan_desc* d, Shape* s) {
  const fo_status st = check_shape(d, &s->W, &s->tiles, &s->waves);
  if (st != FO_OK) return st;
  s->tile_bytes = double(d->tile_m) * d->tile_n * 2.0;
  return FO_OK;
}

// Predicted latency of one partition (waves per group).  sigma = rho = 1:
// the pages' recurrence.  Otherwise the schedule is simulated event by event:
// while a communication runs the GEMM advances at 1 / sigma of its rate,
// while the GEMM runs a communication advances at 1 / rho of the curve's
// rate; a group's communication starts once its waves are computed and the
// previous one has ended; between events both rates are constant.
double predict_parts(const Shape& sh, const Curve& cv, double gemm_us, double sigma, double rho,
                     const std::vector<int32_t>& parts) {
  const int32_t T = sh.waves;
  const double d = gemm_us / T;
  if (sigma == 1.0 && rho == 1.0) {
    double e = 0.0;
    int32_t w = 0;
    for (int32_t g : parts) {
      const int32_t v = w;
      w += g;
      e = std::max(d * w, e) + cv.at(sh.bytes(v, w));
    }
    return e;
  }
  const size_t P = parts.size();
  std::vector<double> ready(P), lat(P);
  {
    int32_t w = 0;
    for (size_t j = 0; j < P; ++j) {
      const int32_t v = w;
      w += parts[j];
      ready[j] = d * w;
      lat[j] = cv.at(sh.bytes(v, w));
    }
  }
  const double eps = 1e-9 * std::max(1.0, gemm_us);
  double t = 0.0, done = 0.0;   // time; GEMM work done (us alone)
  size_t j = 0;                 // next group to communicate
  size_t next_ready = 0;        // first group not yet computed
  double left = -1.0;           // running communication's curve work left; < 0: none
  while (true) {
    while (next_ready < P && done >= ready[next_ready] - eps) ++next_ready;
    const bool gemm_on = done < gemm_us - eps;
    if (left < 0.0 && j < P && j < next_ready) left = lat[j];
    const bool comm_on = left >= 0.0;
    if (!gemm_on && !comm_on) return t;
    const double gr = gemm_on ? (comm_on ? 1.0 / sigma : 1.0) : 0.0;
    const double cr = comm_on ? (gemm_on ? 1.0 / rho : 1.0) : 0.0;
    double dt = std::numeric_limits<double>::infinity();
    double target = gemm_us;
    if (gemm_on) {
      if (next_ready < P) target = std::min(target, ready[next_ready]);
      dt = (target - done) / gr;
    }
    if (comm_on) dt = std::min(dt, left / cr);
    t += dt;
    if (gemm_on) {
      done += gr * dt;
      if (std::fabs(done - target) <= eps) done = target;
    }
    if (comm_on) {
      left -= cr * dt;
      if (left <= eps) {
        left = -1.0;
        ++j;
      }
    }
  }
}

bool factors_ok(double sigma, double rho) {
  return std::isfinite(sigma) && std::isfinite(rho) && sigma > 0.0 && rho > 0.0;
}

fo_status predict_impl(const fo_plan_desc* desc, double gemm_us, const double* curve_bytes,
                       const double* curve_us, int32_t n_points, double sigma, double rho,
                       double* predicted_us) {
  if (!desc || !predicted_us || !(gemm_us >= 0) || !factors_ok(sigma, rho)) return FO_ERR_ARG;
  Shape sh;
  Curve cv;
  fo_status st = make_shape(desc, &sh);
  if (st == FO_OK) st = make_curve(curve_bytes, curve_us, n_points, &cv);
  if (st != FO_OK) return st;
  if (desc->n_groups < 1 || !desc->group_waves) return FO_ERR_ARG;
  int64_t sum = 0;
  for (int j = 0; j < desc->n_groups; ++j) {
    if (desc->group_waves[j] < 1) return FO_ERR_ARG;
    sum += desc->group_waves[j];
  }
  if (sum != sh.waves) return FO_ERR_ARG;
  *predicted_us = predict_parts(sh, cv, gemm_us, sigma, rho,
                                std::vector<int32_t>(desc->group_waves,
                                                     desc->group_waves + desc->n_groups));
  return FO_OK;
}

// The pages' recurrence: exact dynamic program over group boundaries.
std::vector<int32_t> tune_plain(const Shape& sh, const Curve& cv, double gemm_us) {
  const int32_t T = sh.waves;
  const double d = gemm_us / T;
  std::vector<double> best(T + 1, std::numeric_limits<double>::infinity());
  std::vector<int32_t> prev(T + 1, -1);
  best[0] = 0.0;
  for (int32_t w = 1; w <= T; ++w)
    for (int32_t v = 0; v < w; ++v) {
      const double e = std::max(d * w, best[v]) + cv.at(sh.bytes(v, w));
      if (e < best[w]) {
        best[w] = e;
        prev[w] = v;
      }
    }
  std::vector<int32_t> parts;
  for (int32_t w = T; w > 0; w = prev[w]) parts.push_back(w - prev[w]);
  std::reverse(parts.begin(), parts.end());
  return parts;
}

// Partition of T waves from the cut mask (bit i: a cut after wave i + 1),
// in the enumeration order of the design space: the mask's highest bit is
// the cut after the first wave.
std::vector<int32_t> parts_of_mask(int32_t T, uint64_t mask) {
  std::vector<int32_t> parts;
  int32_t run = 0;
  for (int32_t k = 0; k < T; ++k) {
    ++run;
    if (k == T - 1 || ((mask >> (T - 2 - k)) & 1u)) {
      parts.push_back(run);
      run = 0;
    }
  }
  return parts;
}

// The largest T searched exhaustively with the interference factors
// (2^(T-1) candidates); beyond it a local search.
constexpr int32_t kExhaustiveWaves = 20;

fo_status tune_impl(const fo_plan_desc* desc, double gemm_us, const double* curve_bytes,
                    const double* curve_us, int32_t n_points, double sigma, double rho,
                    int32_t* group_waves, int32_t capacity, int32_t* n_groups,
                    double* predicted_us) {
  if (!desc || !group_waves || !n_groups || !(gemm_us >= 0) || !factors_ok(sigma, rho))
    return FO_ERR_ARG;
  Shape sh;
  Curve cv;
  fo_status st = make_shape(desc, &sh);
  if (st == FO_OK) st = make_curve(curve_bytes, curve_us, n_points, &cv);
  if (st != FO_OK) return st;
  const int32_t T = sh.waves;
  std::vector<int32_t> best = tune_plain(sh, cv, gemm_us);
  double best_e = predict_parts(sh, cv, gemm_us, sigma, rho, best);
  if (!(sigma == 1.0 && rho == 1.0)) {
    if (T <= kExhaustiveWaves) {
      // every candidate, in the design space's order (the first on ties)
      best_e = std::numeric_limits<double>::infinity();
      for (uint64_t m = 0; m < (uint64_t(1) << (T - 1)); ++m) {
        std::vector<int32_t> c = parts_of_mask(T, m);
        const double e = predict_parts(sh, cv, gemm_us, sigma, rho, c);
        if (e < best_e) {
          best_e = e;
          best.swap(c);
        }
      }
    } else {
      // local search: from the best of the plain optimum, the finest
      // partition and one wave then groups of two, toggle single cuts
      // while that lowers the prediction
      std::vector<int32_t> finest(T, 1), otwo{1};
      for (int32_t left = T - 1; left > 0; left -= otwo.back()) otwo.push_back(std::min(2, left));
      for (const auto& c : {finest, otwo}) {
        const double e = predict_parts(sh, cv, gemm_us, sigma, rho, c);
        if (e < best_e) {
          best_e = e;
          best = c;
        }
      }
      std::vector<char> cut(T, 0);   // cut[k]: a group ends after wave k + 1
      {
        int32_t w = 0;
        for (int32_t g : best) cut[(w += g) - 1] = 1;
      }
      auto parts_of_cuts = [&]() {
        std::vector<int32_t> p;
        int32_t run = 0;
        for (int32_t k = 0; k < T; ++k) {
          ++run;
          if (cut[k] || k == T - 1) {
            p.push_back(run);
            run = 0;
          }
        }
        return p;
      };
      for (bool improved = true; improved;) {
        improved = false;
        for (int32_t k = 0; k + 1 < T; ++k) {
          cut[k] ^= 1;
          const std::vector<int32_t> c = parts_of_cuts();
          const double e = predict_parts(sh, cv, gemm_us, sigma, rho, c);
          if (e < best_e - 1e-9) {
            best_e = e;
            best = c;
            improved = true;
          } else {
            cut[k] ^= 1;
          }
        }
      }
    }
  } else {
    best_e = predict_parts(sh, cv, gemm_us, 1.0, 1.0, best);
  }
  *n_groups = int32_t(best.size());
  if (predicted_us) *predicted_us = best_e;
  if (capacity < int32_t(best.size())) return FO_ERR_ARG;
  std::copy(best.begin(), best.end(), group_waves);
  return FO_OK;
}

}  // namespace

}  // namespace fo

extern "C" {

fo_status fo_predict_partition(const fo_plan_desc* desc, double gemm_us,
                               const double* curve_bytes, const double* curve_us,
                               int32_t n_points, double* predicted_us) {
  return fo::predict_impl(desc, gemm_us, curve_bytes, curve_us, n_points, 1.0, 1.0,
                          predicted_us);
}

fo_status fo_predict_partition_ex(const fo_plan_desc* desc, double gemm_us,
                                  const double* curve_bytes, const double* curve_us,
                                  int32_t n_points, double gemm_slowdown, double comm_slowdown,
                                  double* predicted_us) {
  return fo::predict_impl(desc, gemm_us, curve_bytes, curve_us, n_points, gemm_slowdown,
                          comm_slowdown, predicted_us);
}

fo_status fo_tune_partition(const fo_plan_desc* desc, double gemm_us,
                            const double* curve_bytes, const double* curve_us,
                            int32_t n_points, int32_t* group_waves, int32_t capacity,
                            int32_t* n_groups, double* predicted_us) {
  return fo::tune_impl(desc, gemm_us, curve_bytes, curve_us, n_points, 1.0, 1.0, group_waves,
                       capacity, n_groups, predicted_us);
}

fo_status fo_tune_partition_ex(const fo_plan_desc* desc, double gemm_us,
                               const double* curve_bytes, const double* curve_us,
                               int32_t n_points, double gemm_slowdown, double comm_slowdown,
                               int32_t* group_waves, int32_t capacity, int32_t* n_groups,
                               double* predicted_us) {
  return fo::tune_impl(desc, gemm_us, curve_bytes, curve_us, n_points, gemm_slowdown,
                       comm_slowdown, group_waves, capacity, n_groups, predicted_us);
}

}  // extern "C"
