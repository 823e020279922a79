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

}  // namespace

}  // namespace fo

extern "C" {

fo_status fo_predict_partition(const fo_plan_desc* desc, double gemm_us,
                               const double* curve_bytes, const double* curve_us,
                               int32_t n_points, double* predicted_us) {
  using namespace fo;
  if (!desc || !predicted_us || !(gemm_us >= 0)) return FO_ERR_ARG;
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
  const double d = gemm_us / sh.waves;
  double e = 0.0;
  int32_t w = 0;
  for (int j = 0; j < desc->n_groups; ++j) {
    const int32_t v = w;
    w += desc->group_waves[j];
    e = std::max(d * w, e) + cv.at(sh.bytes(v, w));
  }
  *predicted_us = e;
  return FO_OK;
}

fo_status fo_tune_partition(const fo_plan_desc* desc, double gemm_us,
                            const double* curve_bytes, const double* curve_us,
                            int32_t n_points, int32_t* group_waves, int32_t capacity,
                            int32_t* n_groups, double* predicted_us) {
  using namespace fo;
  if (!desc || !group_waves || !n_groups || !(gemm_us >= 0)) return FO_ERR_ARG;
  Shape sh;
  Curve cv;
  fo_status st = make_shape(desc, &sh);
  if (st == FO_OK) st = make_curve(curve_bytes, curve_us, n_points, &cv);
  if (st != FO_OK) return st;
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
  *n_groups = int32_t(parts.size());
  if (predicted_us) *predicted_us = best[T];
  if (capacity < int32_t(parts.size())) return FO_ERR_ARG;
  std::copy(parts.begin(), parts.end(), group_waves);
  return FO_OK;
}

}  // extern "C"
