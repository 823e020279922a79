// Host planner: launch order, waves, wave groups, counting-table sizes,
// mapping tables and the reordered layout of one GEMM shape.
//
// Pages: "FlashOverlap: 信号驱动计算通信重叠论文详解" -- 一、信号机制 (waves are
// tiles / SMs; block swizzling interleaves the tiles of a wave; a wave group
// holds consecutive waves; the counting table has one entry per group and
// the tile's index identifies its group), 二、重排机制 (the mapping table
// makes a group's data contiguous; Figure 6's tile, subtile and sub-token
// units), 四、实时调优 Algorithm 1 (T = tile_num / (sm_num - comm_sm_num)).
//
// Readings where the pages are silent: the launch order is banded (bands of
// `swizzle` tile rows, each band walked column by column); wave = slot / W
// with W persistent GEMM CTAs; |G_j| counts tiles; a unit is one tile row.
#include <algorithm>
#include <cstring>
#include <numeric>

#include <cuda_runtime.h>

#include "fo_internal.h"

namespace fo {

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

// Tile rows of an expert's grid: ceil(rows / 128), the GEMM's output tiles.
// With pad_expert_tile_rows (an explicit plan input, All-to-All layout
// only), an odd count gets one empty tile row, so that every band of the
// launch order has an even height and launch slots 2i, 2i+1 can be
// vertically adjacent tiles (CTA pairs); the empty tiles take slots and are
// counted like the others.
int32_t expert_tile_rows(int32_t pad, int32_t rows) {
  const int32_t tm = int32_t(ceil_div(rows, kTileM));
  return pad ? tm + (tm & 1) : tm;
}

fo_status check_shape(const fo_plan_desc* d, int32_t* W_out, int32_t* tiles_out,
                      int32_t* waves_out) {
  if (!d) return FO_ERR_ARG;
  if (d->M <= 0 || d->N <= 0 || d->K <= 0) return FO_ERR_ARG;
  if (d->tile_m != kTileM) return FO_ERR_UNSUPPORTED;
  if (d->tile_n != 128 && d->tile_n != 256) return FO_ERR_UNSUPPORTED;
  if (d->N % d->tile_n != 0 || d->K % kBlockK != 0) return FO_ERR_ARG;
  if (d->swizzle < 1) return FO_ERR_ARG;
  if (d->band_order != FO_BAND_FORWARD && d->band_order != FO_BAND_SERPENTINE)
    return FO_ERR_ARG;
  if (d->n_experts < 0 || d->n_experts > kMaxExperts) return FO_ERR_ARG;
  if (d->pad_expert_tile_rows != 0 &&
      (d->pad_expert_tile_rows != 1 || d->layout != FO_LAYOUT_A2A_SUBTOKEN))
    return FO_ERR_ARG;
  const int32_t pad = d->pad_expert_tile_rows;
  int32_t W = d->wave_width;
  if (W <= 0) {
    if (d->host_only) return FO_ERR_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FO_ERR_CUDA;
    if (cudaDeviceGetAttribute(&W, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FO_ERR_CUDA;
  }
  int64_t tiles_m = 0;
  if (d->n_experts > 0) {
    if (!d->expert_rows) return FO_ERR_ARG;
    int64_t sum = 0;
    for (int e = 0; e < d->n_experts; ++e) {
      if (d->expert_rows[e] < 0) return FO_ERR_ARG;
      sum += d->expert_rows[e];
      tiles_m += expert_tile_rows(pad, d->expert_rows[e]);
    }
    if (sum != d->M) return FO_ERR_ARG;
  } else {
    tiles_m = expert_tile_rows(pad, d->M);
  }
  int64_t tiles = tiles_m * (d->N / d->tile_n);
  if (tiles <= 0 || tiles > (int64_t(1) << 24)) return FO_ERR_ARG;
  // units (tile rows) index the reordered buffer in int32
  if (int64_t(d->M) * (d->N / d->tile_n) >= (int64_t(1) << 31)) return FO_ERR_ARG;
  if (W_out) *W_out = W;
  if (tiles_out) *tiles_out = int32_t(tiles);
  if (waves_out) *waves_out = int32_t(ceil_div(tiles, W));
  return FO_OK;
}

// Build every host table.  The layout is computed arithmetically from the
// group and slot structure (prefix sums), not by walking units.
fo_status build_plan(const fo_plan_desc* d, fo_plan* p) {
  int32_t W = 0, tiles = 0, waves = 0;
  fo_status st = check_shape(d, &W, &tiles, &waves);
  if (st != FO_OK) return st;
  if (d->n_groups < 1 || !d->group_waves) return FO_ERR_ARG;
  int64_t wsum = 0;
  for (int j = 0; j < d->n_groups; ++j) {
    if (d->group_waves[j] < 1) return FO_ERR_ARG;
    wsum += d->group_waves[j];
  }
  if (wsum != waves) return FO_ERR_ARG;

  const int layout = d->layout;
  if (layout < FO_LAYOUT_TILE || layout > FO_LAYOUT_A2A_SUBTOKEN) return FO_ERR_ARG;
  int R = 1;
  if (layout != FO_LAYOUT_TILE) {
    R = d->n_dest;
    if (R < 1 || R > kMaxDest) return FO_ERR_ARG;
  }
  if (layout == FO_LAYOUT_RS_SUBTILE || layout == FO_LAYOUT_RS_ROWBLOCK) {
    if (d->n_experts > 1) return FO_ERR_ARG;
    if (d->M % kTileM != 0) return FO_ERR_ARG;
    if (layout == FO_LAYOUT_RS_SUBTILE && kTileM % R != 0) return FO_ERR_ARG;
    if (layout == FO_LAYOUT_RS_ROWBLOCK && (d->M % R != 0 || (d->M / R) % kTileM != 0))
      return FO_ERR_ARG;
  }
  if (layout == FO_LAYOUT_A2A_SUBTOKEN && (!d->row_token != !d->row_slot))
    return FO_ERR_ARG;   // both routing arrays or neither (every row empty)

  p->M = d->M; p->N = d->N; p->K = d->K;
  p->tile_m = d->tile_m; p->tile_n = d->tile_n; p->swizzle = d->swizzle;
  p->band_order = d->band_order;
  p->W = W; p->P = d->n_groups; p->R = R; p->layout = layout;
  p->n_dest = d->n_dest; p->n_experts = d->n_experts;
  p->tiles = tiles; p->waves = waves; p->tiles_n = d->N / d->tile_n;
  const int TN = p->tiles_n, P = p->P;

  if (d->n_experts > 0)
    p->expert_rows.assign(d->expert_rows, d->expert_rows + d->n_experts);
  else
    p->expert_rows.assign(1, d->M);
  const int E = int(p->expert_rows.size());
  p->expert_row0.assign(E, 0);
  p->expert_tile0.assign(E, 0);
  p->expert_tm.assign(E, 0);
  for (int e = 0; e < E; ++e)
    p->expert_tm[e] = expert_tile_rows(d->pad_expert_tile_rows, p->expert_rows[e]);
  for (int e = 1; e < E; ++e) {
    p->expert_row0[e] = p->expert_row0[e - 1] + p->expert_rows[e - 1];
    p->expert_tile0[e] = p->expert_tile0[e - 1] + p->expert_tm[e - 1] * TN;
  }

  // Launch order: experts in turn; inside an expert, band b covers tile rows
  // [b*S, b*S + h) with h = min(S, rows left); position o inside the band is
  // column o / h (serpentine: TN - 1 - o / h in the expert's odd bands), row
  // b*S + o % h.
  p->slot_tile.assign(tiles, 0);
  p->tile_slot.assign(tiles, 0);
  p->tile.assign(tiles, TileInfo{});
  {
    int32_t s = 0;
    for (int e = 0; e < E; ++e) {
      const int32_t tm_count = p->expert_tm[e];
      for (int32_t top = 0; top < tm_count; top += d->swizzle) {
        const int32_t h = std::min<int32_t>(d->swizzle, tm_count - top);
        for (int32_t o = 0; o < h * TN; ++o, ++s) {
          const bool back = d->band_order == FO_BAND_SERPENTINE && (top / d->swizzle) % 2;
          const int32_t tm = top + o % h, tn = back ? TN - 1 - o / h : o / h;
          const int32_t t = p->expert_tile0[e] + tm * TN + tn;
          p->slot_tile[s] = t;
          p->tile_slot[t] = s;
          TileInfo& ti = p->tile[s];
          ti.row0 = p->expert_row0[e] + tm * kTileM;
          ti.col0 = tn * d->tile_n;
          // (a padding tile row holds no rows)
          ti.rows = std::max<int32_t>(0, std::min<int32_t>(kTileM, p->expert_rows[e] - tm * kTileM));
          ti.expert = e;
        }
      }
    }
  }

  // Last-wave split: a last wave of n <= W / 2 tiles leaves at least n CTAs
  // idle; each of its tiles is then computed by two CTAs over halves of K.
  {
    const int32_t n_last = tiles - (waves - 1) * W;
    p->split_n = (waves >= 2 && 2 * n_last <= W && d->K / kBlockK >= 2) ? n_last : 0;
  }

  // CTA pairs: with W even, CTAs 2p and 2p+1 take slots 2i and 2i+1 of every
  // wave; they can share one M = 256 MMA when those are vertically adjacent
  // tiles of the same expert and column.
  p->pairable = (W % 2 == 0) && (tiles % 2 == 0);
  for (int32_t s = 0; p->pairable && s < tiles; s += 2) {
    const TileInfo& t0 = p->tile[s];
    const TileInfo& t1 = p->tile[s + 1];
    p->pairable = t0.expert == t1.expert && t0.col0 == t1.col0 && t1.row0 == t0.row0 + kTileM;
  }

  // Groups: consecutive wave ranges; slot ranges follow from W.
  p->group_waves.assign(d->group_waves, d->group_waves + P);
  p->group_slot_begin.assign(P + 1, 0);
  p->group_tiles.assign(P, 0);
  {
    int64_t wave_end = 0;
    for (int j = 0; j < P; ++j) {
      wave_end += p->group_waves[j];
      p->group_slot_begin[j + 1] = int32_t(std::min<int64_t>(tiles, wave_end * W));
      p->group_tiles[j] = p->group_slot_begin[j + 1] - p->group_slot_begin[j];
    }
  }
  p->slot_group.assign(tiles, 0);
  for (int j = 0; j < P; ++j)
    for (int32_t s = p->group_slot_begin[j]; s < p->group_slot_begin[j + 1]; ++s) {
      p->slot_group[s] = j;
      p->tile[s].group = j;
    }

  // Reordered layout.  A group's units start after all earlier groups'.
  p->part_start.assign(size_t(P) * R, 0);
  p->part_len.assign(size_t(P) * R, 0);
  p->part_dst.assign(size_t(P) * R, 0);
  p->group_unit_begin.assign(P + 1, 0);

  int64_t routed_rows = d->M;
  if (layout == FO_LAYOUT_A2A_SUBTOKEN) {
    // per routed row: destination rank, rank among the rows of its tile row
    // going to the same destination, and its row in that rank's output.  A
    // row with a negative token holds none (an expert's capacity left
    // unfilled by the routing): it goes nowhere and all three are -1.
    p->row_dest.assign(d->M, -1);
    p->row_rank.assign(d->M, -1);
    p->final_row.assign(d->M, -1);
    int32_t top_k = 1, n_tokens = 0;
    routed_rows = 0;
    for (int32_t r = 0; d->row_token && r < d->M; ++r) {
      if (d->row_token[r] < 0) continue;
      if (d->row_slot[r] < 0) return FO_ERR_ARG;
      top_k = std::max(top_k, d->row_slot[r] + 1);
      n_tokens = std::max(n_tokens, d->row_token[r] + 1);
      ++routed_rows;
    }
    p->top_k = top_k;
    p->n_tokens = n_tokens;
    for (int32_t r = 0; d->row_token && r < d->M; ++r) {
      if (d->row_token[r] < 0) continue;
      p->row_dest[r] = d->row_token[r] % R;
      p->final_row[r] = (d->row_token[r] / R) * top_k + d->row_slot[r];
    }
    // rows per (tile row, destination): tile rows are identified by row0
    std::vector<int32_t> cnt(R);
    for (int e = 0; e < E; ++e) {
      for (int32_t b = p->expert_row0[e]; b < p->expert_row0[e] + p->expert_rows[e];
           b += kTileM) {
        std::fill(cnt.begin(), cnt.end(), 0);
        const int32_t end = std::min(b + kTileM, p->expert_row0[e] + p->expert_rows[e]);
        for (int32_t r = b; r < end; ++r)
          if (p->row_dest[r] >= 0) p->row_rank[r] = cnt[p->row_dest[r]]++;
      }
    }
    // per slot and destination: rows of the tile bound there
    auto rows_to = [&](int32_t s, int k) {
      const TileInfo& ti = p->tile[s];
      int32_t c = 0;
      for (int32_t r = ti.row0; r < ti.row0 + ti.rows; ++r) c += (p->row_dest[r] == k);
      return c;
    };
    std::vector<int32_t> tile_cnt(size_t(tiles) * R);
    for (int32_t s = 0; s < tiles; ++s) {
      // tiles of one tile row share their rows: count once per row0 would
      // be enough, but the count is cheap
      for (int k = 0; k < R; ++k) tile_cnt[size_t(s) * R + k] = rows_to(s, k);
    }
    p->dest_base.assign(size_t(tiles) * R, 0);
    int32_t u = 0;
    for (int j = 0; j < P; ++j) {
      p->group_unit_begin[j] = u;
      for (int k = 0; k < R; ++k) {
        p->part_start[size_t(j) * R + k] = u;
        for (int32_t s = p->group_slot_begin[j]; s < p->group_slot_begin[j + 1]; ++s) {
          p->dest_base[size_t(s) * R + k] = u;
          u += tile_cnt[size_t(s) * R + k];
        }
        p->part_len[size_t(j) * R + k] = u - p->part_start[size_t(j) * R + k];
      }
    }
    p->group_unit_begin[P] = u;
    p->n_units = u;
    p->slot_live.assign(tiles, 0);
    for (int32_t s = 0; s < tiles; ++s)
      for (int k = 0; k < R; ++k) p->slot_live[s] |= tile_cnt[size_t(s) * R + k] > 0;
  } else if (layout == FO_LAYOUT_RS_SUBTILE) {
    const int32_t h = kTileM / R;
    for (int j = 0; j < P; ++j) {
      const int32_t n_j = p->group_tiles[j];
      const int32_t gb = p->group_slot_begin[j] * kTileM;  // all tiles are full
      p->group_unit_begin[j] = gb;
      for (int k = 0; k < R; ++k) {
        p->part_start[size_t(j) * R + k] = gb + k * n_j * h;
        p->part_len[size_t(j) * R + k] = n_j * h;
      }
      for (int32_t i = 0; i < n_j; ++i) {
        TileInfo& ti = p->tile[p->group_slot_begin[j] + i];
        ti.unit_base = gb + i * h;
        ti.sub_stride = n_j * h;
      }
    }
    p->group_unit_begin[P] = tiles * kTileM;
    p->n_units = tiles * kTileM;
  } else if (layout == FO_LAYOUT_RS_ROWBLOCK) {
    const int32_t rows_per = d->M / R;
    for (int32_t s = 0; s < tiles; ++s) p->tile[s].dest = p->tile[s].row0 / rows_per;
    int32_t u = 0;
    for (int j = 0; j < P; ++j) {
      p->group_unit_begin[j] = u;
      for (int k = 0; k < R; ++k) {
        p->part_start[size_t(j) * R + k] = u;
        for (int32_t s = p->group_slot_begin[j]; s < p->group_slot_begin[j + 1]; ++s)
          if (p->tile[s].dest == k) {
            p->tile[s].unit_base = u;
            u += kTileM;
          }
        p->part_len[size_t(j) * R + k] = u - p->part_start[size_t(j) * R + k];
      }
    }
    p->group_unit_begin[P] = u;
    p->n_units = u;
  } else {  // FO_LAYOUT_TILE: prefix sum of valid rows in slot order
    int32_t u = 0;
    for (int j = 0; j < P; ++j) {
      p->group_unit_begin[j] = u;
      p->part_start[j] = u;
      for (int32_t s = p->group_slot_begin[j]; s < p->group_slot_begin[j + 1]; ++s) {
        p->tile[s].unit_base = u;
        u += p->tile[s].rows;
      }
      p->part_len[j] = u - p->part_start[j];
    }
    p->group_unit_begin[P] = u;
    p->n_units = u;
  }

  // parts are appended, group after group, to their destination buffer
  p->dest_units.assign(R, 0);
  for (int k = 0; k < R; ++k) {
    int32_t off = 0;
    for (int j = 0; j < P; ++j) {
      p->part_dst[size_t(j) * R + k] = off;
      off += p->part_len[size_t(j) * R + k];
    }
    p->dest_units[k] = off;
  }
  if (int64_t(p->n_units) != routed_rows * TN) return FO_ERR_ARG;  // every row once

  // rows of each output of the post-communication reorder
  if (layout == FO_LAYOUT_TILE) {
    p->final_rows.assign(1, d->M);
  } else if (layout == FO_LAYOUT_A2A_SUBTOKEN) {
    set_a2a_outputs(p, p->n_tokens, p->top_k);
    // a routing with a (token, slot) pair twice could outgrow the buffers
    for (int k = 0; k < R; ++k)
      if (p->dest_units[k] > p->dest_capacity[k]) return FO_ERR_ARG;
  } else {
    p->final_rows.assign(R, d->M / R);
  }
  if (layout != FO_LAYOUT_A2A_SUBTOKEN) p->dest_capacity = p->dest_units;
  // The inverse of the unit layout at row granularity: which tile row each
  // unit holds (read by the fused consumer+reorder).  All-to-All: room for
  // every row, since fo_plan_route may route them all.
  p->unit_src.assign(layout == FO_LAYOUT_A2A_SUBTOKEN ? size_t(d->M) * TN : size_t(p->n_units), 0);
  // and each unit's final place, for the direct consumer+reorder
  p->place_ok = true;
  for (int32_t rows : p->final_rows)
    if (int64_t(rows) * (d->N / 8) >= (int64_t(1) << kPlaceShift)) p->place_ok = false;
  p->unit_place.assign(p->unit_src.size(), 0);
  for (int32_t s = 0; s < tiles; ++s)
    for (int32_t r = 0; r < p->tile[s].rows; ++r) {
      const int32_t u = unit_of(p, s, r);
      if (u < 0) continue;
      p->unit_src[u] = (s << 7) | r;
      if (p->place_ok) p->unit_place[u] = place_of(p, s, r);
    }
  return FO_OK;
}

// Final place of row r of the tile at slot s (a row that holds a token):
// output k << kPlaceShift | the 16-byte vector index, in output k, of the
// row's element at the tile's first column.  The rows are those of the
// post-communication reorder: TILE row row0 + r; RS_SUBTILE subtile k = r / h
// of tile row tm goes to slice row h tm + r - h k; RS_ROWBLOCK the tile's
// rank, row row0 + r - k M / R; A2A the row's rank and its final row.
int32_t place_of(const fo_plan* p, int32_t slot, int32_t r) {
  const TileInfo& ti = p->tile[slot];
  int32_t k = 0, row = ti.row0 + r;
  if (p->layout == FO_LAYOUT_RS_SUBTILE) {
    const int32_t h = kTileM / p->R;
    k = r / h;
    row = (ti.row0 / kTileM) * h + r - k * h;
  } else if (p->layout == FO_LAYOUT_RS_ROWBLOCK) {
    k = ti.dest;
    row = ti.row0 + r - k * (p->M / p->R);
  } else if (p->layout == FO_LAYOUT_A2A_SUBTOKEN) {
    k = p->row_dest[ti.row0 + r];
    row = p->final_row[ti.row0 + r];
  }
  return (k << kPlaceShift) | (row * (p->N / 8) + ti.col0 / 8);
}

// All-to-All outputs for routings of n_tokens tokens with top_k slots each:
// rank d receives the tokens t = d, d + R, ... and all their slots, so its
// output has ceil((n_tokens - d) / R) * top_k rows and its receive buffer
// at most that many rows of every column block.
void set_a2a_outputs(fo_plan* p, int32_t n_tokens, int32_t top_k) {
  p->n_tokens = n_tokens;
  p->top_k = top_k;
  p->final_rows.assign(p->R, 0);
  p->dest_capacity.assign(p->R, 0);
  for (int k = 0; k < p->R; ++k) {
    const int64_t toks = n_tokens > k ? (int64_t(n_tokens) - k + p->R - 1) / p->R : 0;
    p->final_rows[k] = int32_t(toks * top_k);
    p->dest_capacity[k] = int32_t(toks * top_k * p->tiles_n);
  }
}

// Unit of row r of the tile at `slot`, from the same per-slot / per-row
// fields the kernels read (-1 when the tile has no row r).
int32_t unit_of(const fo_plan* p, int32_t slot, int32_t r) {
  const TileInfo& ti = p->tile[slot];
  if (r >= ti.rows) return -1;
  switch (p->layout) {
    case FO_LAYOUT_RS_SUBTILE: {
      const int32_t h = kTileM / p->R;
      return ti.unit_base + (r / h) * ti.sub_stride + r % h;
    }
    case FO_LAYOUT_A2A_SUBTOKEN: {
      const int32_t rho = ti.row0 + r;
      if (p->row_dest[rho] < 0) return -1;   // the row holds no token
      return p->dest_base[size_t(slot) * p->R + p->row_dest[rho]] + p->row_rank[rho];
    }
    default:
      return ti.unit_base + r;
  }
}

namespace {

template <typename T>
size_t put(std::vector<char>& buf, const std::vector<T>& v) {
  size_t off = (buf.size() + 255) & ~size_t(255);
  buf.resize(off + std::max<size_t>(v.size() * sizeof(T), 16), 0);
  if (!v.empty()) std::memcpy(buf.data() + off, v.data(), v.size() * sizeof(T));
  return off;
}

}  // namespace

// One device allocation holds every table plus the consumer's scratch
// counters (zeroed by the consume call before each launch).
fo_status upload_plan(fo_plan* p) {
  if (cudaGetDevice(&p->device) != cudaSuccess) return FO_ERR_CUDA;
  if (cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) !=
      cudaSuccess)
    return FO_ERR_CUDA;
  std::vector<char> buf;
  const size_t o_tile = put(buf, p->tile);
  const size_t o_gt = put(buf, p->group_tiles);
  const size_t o_gub = put(buf, p->group_unit_begin);
  const size_t o_gsb = put(buf, p->group_slot_begin);
  const size_t o_ps = put(buf, p->part_start);
  const size_t o_pl = put(buf, p->part_len);
  const size_t o_pd = put(buf, p->part_dst);
  const size_t o_db = put(buf, p->dest_base);
  const size_t o_rd = put(buf, p->row_dest);
  const size_t o_rr = put(buf, p->row_rank);
  const size_t o_fr = put(buf, p->final_row);
  const size_t o_sl = put(buf, p->slot_live);
  const size_t o_us = put(buf, p->unit_src);
  const size_t o_up = put(buf, p->unit_place);
  const size_t o_work = put(buf, std::vector<int32_t>(p->P + 1, 0));
  const size_t o_fin = put(buf, std::vector<int32_t>(p->P, 0));
  const size_t o_cons = put(buf, std::vector<int32_t>(p->P, 0));
  const size_t o_rtile = put(buf, std::vector<int32_t>(2, 0));
  const size_t o_gst = put(buf, std::vector<int32_t>(1, 0));
  const size_t o_crd = put(buf, std::vector<int32_t>(2, 0));   // count_ready, gemm_exit
  const bool a2a = p->layout == FO_LAYOUT_A2A_SUBTOKEN;
  if (a2a) {
    p->route_blocks = 0;
    for (int32_t tm : p->expert_tm) p->route_blocks += tm;
  }
  const size_t o_sws = put(buf, std::vector<float>(size_t(p->split_n) * kTileM * p->tile_n, 0.f));
  const size_t o_sfl = put(buf, std::vector<int32_t>(size_t(p->split_n) * 4, 0));
  const size_t o_rc =
      put(buf, std::vector<int32_t>(a2a ? size_t(p->route_blocks) * (p->R + 1) : 1, 0));
  void* blob = nullptr;
  if (cudaMalloc(&blob, buf.size()) != cudaSuccess) return FO_ERR_CUDA;
  if (cudaMemcpy(blob, buf.data(), buf.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(blob);
    return FO_ERR_CUDA;
  }
  char* b = static_cast<char*>(blob);
  p->blob = blob;
  p->dev.tile = reinterpret_cast<TileInfo*>(b + o_tile);
  p->dev.group_tiles = reinterpret_cast<int32_t*>(b + o_gt);
  p->dev.group_unit_begin = reinterpret_cast<int32_t*>(b + o_gub);
  p->dev.group_slot_begin = reinterpret_cast<int32_t*>(b + o_gsb);
  p->dev.part_start = reinterpret_cast<int32_t*>(b + o_ps);
  p->dev.part_len = reinterpret_cast<int32_t*>(b + o_pl);
  p->dev.part_dst = reinterpret_cast<int32_t*>(b + o_pd);
  p->dev.dest_base = reinterpret_cast<int32_t*>(b + o_db);
  p->dev.row_dest = reinterpret_cast<int32_t*>(b + o_rd);
  p->dev.row_rank = reinterpret_cast<int32_t*>(b + o_rr);
  p->dev.final_row = reinterpret_cast<int32_t*>(b + o_fr);
  p->dev.slot_live = reinterpret_cast<int32_t*>(b + o_sl);
  p->dev.unit_src = reinterpret_cast<int32_t*>(b + o_us);
  p->dev.unit_place = reinterpret_cast<int32_t*>(b + o_up);
  p->dev.work = reinterpret_cast<int32_t*>(b + o_work);
  p->dev.finished = reinterpret_cast<int32_t*>(b + o_fin);
  p->dev.consumed = reinterpret_cast<uint32_t*>(b + o_cons);
  p->dev.rtile = reinterpret_cast<int32_t*>(b + o_rtile);
  p->dev.gemm_status = reinterpret_cast<int32_t*>(b + o_gst);
  p->dev.count_ready = reinterpret_cast<uint32_t*>(b + o_crd);
  p->dev.gemm_exit = reinterpret_cast<int32_t*>(b + o_crd) + 1;
  p->dev.route_cnt = reinterpret_cast<int32_t*>(b + o_rc);
  p->dev.split_ws = b + o_sws;
  p->dev.split_flag = reinterpret_cast<uint32_t*>(b + o_sfl);
  return FO_OK;
}

// Download the routing tables fo_plan_route built on the device (waits for
// the device first), so that the host copies and every table derived from
// them describe the routing the kernels now use.
fo_status refresh_routing(fo_plan* p) {
  if (!p->routing_on_device) return FO_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return FO_ERR_CUDA;
  auto get = [](std::vector<int32_t>& v, const int32_t* src) {
    return cudaMemcpy(v.data(), src, v.size() * sizeof(int32_t), cudaMemcpyDeviceToHost) ==
           cudaSuccess;
  };
  if (!get(p->part_start, p->dev.part_start) || !get(p->part_len, p->dev.part_len) ||
      !get(p->part_dst, p->dev.part_dst) || !get(p->group_unit_begin, p->dev.group_unit_begin) ||
      !get(p->dest_base, p->dev.dest_base) || !get(p->row_dest, p->dev.row_dest) ||
      !get(p->row_rank, p->dev.row_rank) || !get(p->final_row, p->dev.final_row) ||
      !get(p->slot_live, p->dev.slot_live) || !get(p->unit_place, p->dev.unit_place))
    return FO_ERR_CUDA;
  for (int k = 0; k < p->R; ++k) {
    int32_t off = 0;
    for (int j = 0; j < p->P; ++j) off += p->part_len[size_t(j) * p->R + k];
    p->dest_units[k] = off;
  }
  p->n_units = p->group_unit_begin[p->P];
  p->routing_on_device = false;
  return FO_OK;
}

}  // namespace fo
