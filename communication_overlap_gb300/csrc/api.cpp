// The extern "C" entry points of libfo.so (declared in include/fo.h):
// argument checks, plan ownership and dispatch to the kernel launchers.
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "fo_internal.h"

extern "C" {

fo_status fo_wave_count(const fo_plan_desc* desc, int32_t* tiles, int32_t* waves) {
  return fo::check_shape(desc, nullptr, tiles, waves);
}

fo_status fo_plan_groups(const fo_plan_desc* desc, fo_plan** out) {
  if (!out) return FO_ERR_ARG;
  *out = nullptr;
  fo_plan* p = new (std::nothrow) fo_plan();
  if (!p) return FO_ERR_ARG;
  fo_status st = fo::build_plan(desc, p);
  if (st == FO_OK && !desc->host_only) st = fo::upload_plan(p);
  if (st != FO_OK) {
    fo_plan_destroy(p);
    return st;
  }
  *out = p;
  return FO_OK;
}

fo_status fo_plan_info(const fo_plan* p, int32_t* tiles, int32_t* waves,
                       int32_t* n_groups, int32_t* group_tiles,
                       int32_t* tile_to_slot) {
  if (!p) return FO_ERR_ARG;
  if (tiles) *tiles = p->tiles;
  if (waves) *waves = p->waves;
  if (n_groups) *n_groups = p->P;
  if (group_tiles) std::memcpy(group_tiles, p->group_tiles.data(), sizeof(int32_t) * p->P);
  if (tile_to_slot)
    std::memcpy(tile_to_slot, p->tile_slot.data(), sizeof(int32_t) * p->tiles);
  return FO_OK;
}

fo_status fo_plan_table(const fo_plan* p, int32_t which, int32_t* out,
                        int64_t capacity, int64_t* length) {
  if (!p) return FO_ERR_ARG;
  if (p->routing_on_device) {
    // the routing tables were last built on the device: bring the host
    // copies up to date (the plan's contents do not change, only its cache)
    const fo_status st = fo::refresh_routing(const_cast<fo_plan*>(p));
    if (st != FO_OK) return st;
  }
  std::vector<int32_t> unit;
  const std::vector<int32_t>* v = nullptr;
  switch (which) {
    case FO_TAB_SLOT_TILE: v = &p->slot_tile; break;
    case FO_TAB_TILE_SLOT: v = &p->tile_slot; break;
    case FO_TAB_SLOT_GROUP: v = &p->slot_group; break;
    case FO_TAB_GROUP_TILES: v = &p->group_tiles; break;
    case FO_TAB_PART_START: v = &p->part_start; break;
    case FO_TAB_PART_LEN: v = &p->part_len; break;
    case FO_TAB_PART_DST: v = &p->part_dst; break;
    case FO_TAB_DEST_UNITS: v = &p->dest_units; break;
    case FO_TAB_FINAL_ROWS: v = &p->final_rows; break;
    case FO_TAB_DEST_CAPACITY: v = &p->dest_capacity; break;
    case FO_TAB_SLOT_LIVE:
      if (p->layout != FO_LAYOUT_A2A_SUBTOKEN) {
        unit.assign(p->tiles, 1);
        v = &unit;
      } else {
        v = &p->slot_live;
      }
      break;
    case FO_TAB_UNIT_PLACE:
      if (!p->place_ok) return FO_ERR_UNSUPPORTED;
      unit.assign(p->unit_place.begin(), p->unit_place.begin() + p->n_units);
      v = &unit;
      break;
    case FO_TAB_UNIT:
      unit.resize(size_t(p->tiles) * p->tile_m);
      for (int32_t s = 0; s < p->tiles; ++s)
        for (int32_t r = 0; r < p->tile_m; ++r)
          unit[size_t(s) * p->tile_m + r] = fo::unit_of(p, s, r);
      v = &unit;
      break;
    default: return FO_ERR_ARG;
  }
  if (length) *length = int64_t(v->size());
  if (!out) return FO_OK;
  if (capacity < int64_t(v->size())) return FO_ERR_ARG;
  if (!v->empty()) std::memcpy(out, v->data(), v->size() * sizeof(int32_t));
  return FO_OK;
}

fo_status fo_plan_set_launch(fo_plan* p, int32_t consumer_ctas, int32_t reorder_ctas,
                             int32_t overlap) {
  if (!p) return FO_ERR_ARG;
  p->consumer_ctas = consumer_ctas;
  p->reorder_ctas = reorder_ctas;
  p->overlap = overlap ? 1 : 0;
  return FO_OK;
}

fo_status fo_plan_set_pacing(fo_plan* p, int32_t ctas_during_gemm) {
  if (!p || ctas_during_gemm < 0) return FO_ERR_ARG;
  p->consumer_pace = ctas_during_gemm;
  return FO_OK;
}

fo_status fo_plan_set_consumer_placement(fo_plan* p, fo_consumer_placement placement) {
  if (!p) return FO_ERR_ARG;
  if (placement == FO_CONSUMER_SHARED) {
    p->consumer_smem = 0;
    return FO_OK;
  }
  if (placement != FO_CONSUMER_RESERVED) return FO_ERR_ARG;
  if (fo::reserved_sms(p) <= 0) return FO_ERR_UNSUPPORTED;
  int cap = 0, per_block = 0;
  if (cudaDeviceGetAttribute(&cap, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p->device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&per_block, cudaDevAttrReservedSharedMemoryPerBlock, p->device) !=
          cudaSuccess)
    return FO_ERR_CUDA;
  // more than an SM holding a GEMM CTA has left, counting the system's
  // reservation of each of the two CTAs; rounded up to 4 KB
  int need = cap - fo::gemm_smem_bytes() - 2 * per_block + 1;
  if (need < 1) need = 1;
  need = (need + 4095) / 4096 * 4096;
  if (need > 48 * 1024) return FO_ERR_UNSUPPORTED;   // above the default dynamic limit
  p->consumer_smem = need;
  return FO_OK;
}

fo_status fo_plan_set_gemm(fo_plan* p, fo_gemm_variant variant, int32_t* pairable,
                           int32_t* pair_capacity) {
  if (!p) return FO_ERR_ARG;
  const int cap = p->blob ? fo::gemm_pair_capacity(p) : 0;
  const int grid = p->W < p->tiles ? p->W : p->tiles;
  const bool ok = p->pairable && cap >= grid;
  if (pairable) *pairable = ok ? 1 : 0;
  if (pair_capacity) *pair_capacity = cap;
  if (variant < FO_GEMM_AUTO || variant > FO_GEMM_PAIRS) return FO_ERR_ARG;
  if (variant == FO_GEMM_PAIRS && !ok) return FO_ERR_UNSUPPORTED;
  p->gemm_variant = variant;
  return FO_OK;
}

fo_status fo_plan_set_split(fo_plan* p, int32_t enable, int32_t* split_tiles) {
  if (!p) return FO_ERR_ARG;
  p->split_enabled = enable != 0;
  // (split only when every CTA of the grid can be resident at once)
  const bool fits = p->blob == nullptr || p->W <= p->sm_count;
  if (split_tiles) *split_tiles = (p->split_enabled && fits) ? p->split_n : 0;
  return FO_OK;
}

fo_status fo_plan_set_trace(fo_plan* p, uint64_t* stamps, uint64_t* consumer_stamps) {
  if (!p || !fo::aligned8(stamps) || !fo::aligned8(consumer_stamps)) return FO_ERR_ARG;
  p->trace = stamps;
  p->consumer_trace = consumer_stamps;
  return FO_OK;
}

fo_status fo_plan_device_status(const fo_plan* p, int32_t* gemm_status, int32_t clear) {
  if (!p || !p->blob || !gemm_status) return FO_ERR_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return FO_ERR_CUDA;
  if (cudaMemcpy(gemm_status, p->dev.gemm_status, sizeof(int32_t), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return FO_ERR_CUDA;
  if (clear && cudaMemset(p->dev.gemm_status, 0, sizeof(int32_t)) != cudaSuccess)
    return FO_ERR_CUDA;
  return FO_OK;
}

void fo_plan_destroy(fo_plan* p) {
  if (!p) return;
  if (p->blob) cudaFree(p->blob);
  delete p;
}

fo_status fo_counting_table_init(const fo_plan* p, int32_t* count, void* stream) {
  if (!p || !count) return FO_ERR_ARG;
  return cudaMemsetAsync(count, 0, sizeof(int32_t) * p->P, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FO_OK
             : FO_ERR_CUDA;
}

fo_status fo_signaled_gemm(const fo_plan* p, const void* A, const void* const* B,
                           void* C_r, int32_t* count, uint32_t* flags,
                           uint32_t epoch, void* stream) {
  if (!p || !p->blob || !A || !B || !C_r) return FO_ERR_ARG;
  if ((count == nullptr) != (flags == nullptr)) return FO_ERR_ARG;
  if (!fo::aligned4(count) || !fo::aligned4(flags)) return FO_ERR_ARG;
  const fo_status st = fo::launch_signaled_gemm(p, A, B, C_r, count, flags, epoch, stream);
  if (st == FO_OK) fo::noalloc_note_ordinary_launch(p->device, stream);
  return st;
}

fo_status fo_consume_group(const fo_plan* p, int32_t group, fo_consumer kind,
                           const void* src, const void* const* partials,
                           int32_t n_partials, void* const* dst,
                           const uint32_t* flags, uint32_t epoch,
                           uint64_t spin_limit_ns, int32_t* dev_status,
                           void* stream) {
  if (!p || !p->blob || !src || !dst || !flags || !dev_status) return FO_ERR_ARG;
  if (!fo::aligned4(flags) || !fo::aligned4(dev_status)) return FO_ERR_ARG;
  if (group < -1 || group >= p->P) return FO_ERR_ARG;
  const int32_t g0 = group < 0 ? 0 : group, g1 = group < 0 ? p->P : group + 1;
  switch (kind) {
    case FO_CONS_COPY:
      if (n_partials != 0) return FO_ERR_ARG;
      break;
    case FO_CONS_SUM:
      if (n_partials < 0 || n_partials > fo::kMaxPartials) return FO_ERR_ARG;
      break;
    case FO_CONS_RS:
      if (n_partials < 0 || n_partials > fo::kMaxPartials) return FO_ERR_ARG;
      if (p->layout != FO_LAYOUT_RS_SUBTILE && p->layout != FO_LAYOUT_RS_ROWBLOCK)
        return FO_ERR_ARG;
      break;
    case FO_CONS_A2A:
      if (n_partials != 0 || p->layout != FO_LAYOUT_A2A_SUBTOKEN) return FO_ERR_ARG;
      break;
    default: return FO_ERR_ARG;
  }
  if (n_partials > 0 && !partials) return FO_ERR_ARG;
  // the kernels move 16-byte vectors: every buffer starts on a 16-byte boundary
  if (!fo::aligned16(src)) return FO_ERR_ARG;
  for (int i = 0; i < n_partials; ++i)
    if (!partials[i] || !fo::aligned16(partials[i])) return FO_ERR_ARG;
  const int n_dst = (kind == FO_CONS_RS || kind == FO_CONS_A2A) ? p->R : 1;
  for (int k = 0; k < n_dst; ++k)
    if (!dst[k] || !fo::aligned16(dst[k])) return FO_ERR_ARG;
  return fo::launch_consume(p, g0, g1, int(kind), src, partials, n_partials, dst,
                            flags, epoch, spin_limit_ns, dev_status, stream);
}

fo_status fo_consume_reorder(const fo_plan* p, int32_t group, fo_consumer kind,
                             const void* src, const void* const* partials, int32_t n_partials,
                             void* const* comm_dst, void* const* final_dst, const void* bias,
                             fo_activation act, const uint32_t* flags, uint32_t epoch,
                             uint64_t spin_limit_ns, int32_t* dev_status, void* stream) {
  if (!p || !p->blob || !src || !final_dst || !flags || !dev_status) return FO_ERR_ARG;
  if (!fo::aligned4(flags) || !fo::aligned4(dev_status)) return FO_ERR_ARG;
  if (group < -1 || group >= p->P) return FO_ERR_ARG;
  if (act < FO_ACT_NONE || act > FO_ACT_SILU) return FO_ERR_ARG;
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 15)) return FO_ERR_ARG;
  switch (kind) {
    case FO_CONS_COPY:
      if (n_partials != 0 || p->layout != FO_LAYOUT_TILE) return FO_ERR_ARG;
      break;
    case FO_CONS_SUM:
      if (n_partials < 0 || n_partials > fo::kMaxPartials || p->layout != FO_LAYOUT_TILE)
        return FO_ERR_ARG;
      break;
    case FO_CONS_RS:
      if (n_partials < 0 || n_partials > fo::kMaxPartials) return FO_ERR_ARG;
      if (p->layout != FO_LAYOUT_RS_SUBTILE && p->layout != FO_LAYOUT_RS_ROWBLOCK)
        return FO_ERR_ARG;
      break;
    case FO_CONS_A2A:
      if (n_partials != 0 || p->layout != FO_LAYOUT_A2A_SUBTOKEN) return FO_ERR_ARG;
      break;
    default: return FO_ERR_ARG;
  }
  if (n_partials > 0 && !partials) return FO_ERR_ARG;
  if (!fo::aligned16(src)) return FO_ERR_ARG;
  for (int i = 0; i < n_partials; ++i)
    if (!partials[i] || !fo::aligned16(partials[i])) return FO_ERR_ARG;
  const int n = (kind == FO_CONS_RS || kind == FO_CONS_A2A) ? p->R : 1;
  for (int k = 0; k < n; ++k) {
    if ((comm_dst && (!comm_dst[k] || !fo::aligned16(comm_dst[k]))) || !final_dst[k] ||
        !fo::aligned16(final_dst[k]))
      return FO_ERR_ARG;
  }
  const int32_t g0 = group < 0 ? 0 : group, g1 = group < 0 ? p->P : group + 1;
  return fo::launch_consume_reorder(p, g0, g1, int(kind), src, partials, n_partials, comm_dst,
                                    final_dst, bias, int(act), flags, epoch, spin_limit_ns,
                                    dev_status, stream);
}

fo_status fo_reorder_back_fused(const fo_plan* p, int32_t group_begin, int32_t group_end,
                                const void* const* src, void* const* dst, const void* bias,
                                fo_activation act, void* stream) {
  if (!p || !p->blob || !src || !dst) return FO_ERR_ARG;
  if (group_begin < 0 || group_end > p->P || group_begin > group_end) return FO_ERR_ARG;
  if (act < FO_ACT_NONE || act > FO_ACT_SILU) return FO_ERR_ARG;
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 15)) return FO_ERR_ARG;
  const int n = p->layout == FO_LAYOUT_TILE ? 1 : p->R;
  for (int k = 0; k < n; ++k)
    if (!src[k] || !dst[k]) return FO_ERR_ARG;
  if (group_begin == group_end) return FO_OK;
  return fo::launch_reorder_back(p, group_begin, group_end, src, dst, bias, int(act), stream);
}

fo_status fo_plan_route(fo_plan* p, const int32_t* row_token, const int32_t* row_slot,
                        int32_t n_tokens, int32_t top_k, int32_t* dev_status, void* stream) {
  if (!p || !p->blob || p->layout != FO_LAYOUT_A2A_SUBTOKEN) return FO_ERR_ARG;
  if (!row_token || !row_slot || !dev_status) return FO_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(row_token) | reinterpret_cast<uintptr_t>(row_slot) |
       reinterpret_cast<uintptr_t>(dev_status)) & 3)
    return FO_ERR_ARG;
  if (n_tokens < 0 || top_k < 1) return FO_ERR_ARG;
  // every output row and receive-buffer unit must stay addressable in int32
  const int64_t toks = (int64_t(n_tokens) + p->R - 1) / p->R;
  if (toks * top_k * p->tiles_n >= (int64_t(1) << 31)) return FO_ERR_ARG;
  // the kernels read the new output sizes from the plan; a failed launch
  // leaves the plan as it was
  const int32_t old_tokens = p->n_tokens, old_top_k = p->top_k;
  fo::set_a2a_outputs(p, n_tokens, top_k);
  const fo_status st = fo::launch_plan_route(p, row_token, row_slot, dev_status, stream);
  if (st != FO_OK) {
    fo::set_a2a_outputs(p, old_tokens, old_top_k);
    return st;
  }
  p->routing_on_device = true;
  return FO_OK;
}

fo_status fo_reorder_back(const fo_plan* p, int32_t group_begin, int32_t group_end,
                          const void* const* src, void* const* dst, void* stream) {
  return fo_reorder_back_fused(p, group_begin, group_end, src, dst, nullptr, FO_ACT_NONE,
                               stream);
}

fo_status fo_allgather_rows(const fo_plan* p, const void* const* slices, void* out,
                            const void* bias, fo_activation act, void* stream) {
  if (!p || !p->blob || !slices || !out) return FO_ERR_ARG;
  if (p->layout != FO_LAYOUT_RS_SUBTILE && p->layout != FO_LAYOUT_RS_ROWBLOCK) return FO_ERR_ARG;
  if (act < FO_ACT_NONE || act > FO_ACT_SILU) return FO_ERR_ARG;
  uintptr_t bits = reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(bias);
  for (int k = 0; k < p->R; ++k) {
    if (!slices[k]) return FO_ERR_ARG;
    bits |= reinterpret_cast<uintptr_t>(slices[k]);
  }
  if (bits & 15) return FO_ERR_ARG;
  return fo::launch_allgather_rows(p, slices, out, bias, int(act), stream);
}

const char* fo_status_string(fo_status s) {
  switch (s) {
    case FO_OK: return "ok";
    case FO_ERR_ARG: return "invalid argument";
    case FO_ERR_CUDA: return "CUDA error";
    case FO_ERR_TIMEOUT: return "device wait timed out";
    case FO_ERR_UNSUPPORTED: return "unsupported shape or device";
  }
  return "unknown status";
}

}  // extern "C"
