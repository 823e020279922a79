// Internal declarations shared by the host planner, the C ABI and the
// kernels of libfo.so.  Not installed; the public interface is include/fo.h.
#pragma once

#include <cstdint>
#include <vector>

#include "fo.h"

namespace fo {

constexpr int kTileM = 128;      // rows per tile (tcgen05 M = 128, one CTA)
constexpr int kBlockK = 64;      // K per pipeline stage (one 128-byte swizzle atom)
constexpr int kMaxDest = 16;     // ranks a layout may route to
constexpr int kMaxPartials = 8;  // partial buffers a SUM / RS consumer adds
constexpr int kMaxExperts = 16;  // B matrices of a grouped GEMM

// One entry per launch slot (32 bytes, read by the GEMM producer and
// epilogue and by the reorder kernel).
struct TileInfo {
  int32_t row0;        // first row of the tile in A and in the stacked C
  int32_t col0;        // first column
  int32_t rows;        // valid rows (an expert's last tile row may be ragged)
  int32_t expert;      // which B
  int32_t group;       // wave group j
  int32_t unit_base;   // unit of row 0 (RS_SUBTILE: of row 0 of subtile 0)
  int32_t sub_stride;  // RS_SUBTILE: units from subtile k to subtile k+1
  int32_t dest;        // RS_ROWBLOCK: the rank all rows of the tile go to
};
static_assert(sizeof(TileInfo) == 32, "TileInfo is 32 bytes");

// Device copies of the plan's tables: pointers into one allocation.
struct DeviceTables {
  TileInfo* tile = nullptr;            // [tiles]
  int32_t* group_tiles = nullptr;      // [P]       |G_j|
  int32_t* group_unit_begin = nullptr; // [P + 1]   unit range of each group
  int32_t* group_slot_begin = nullptr; // [P + 1]   slot range of each group
  int32_t* part_start = nullptr;       // [P * R]
  int32_t* part_len = nullptr;         // [P * R]
  int32_t* part_dst = nullptr;         // [P * R]
  int32_t* dest_base = nullptr;        // [tiles * R]  A2A: unit of the tile's
                                       //   first row bound for rank d
  int32_t* row_dest = nullptr;         // [M] A2A: rank of each routed row
  int32_t* row_rank = nullptr;         // [M] A2A: index among the rows of its
                                       //   tile row that go to the same rank
  int32_t* final_row = nullptr;        // [M] A2A: row in the rank's output
  int32_t* unit_src = nullptr;         // [units] slot << 7 | row of the tile row each
                                       //   unit holds (A2A: room for M * N / tile_n)
  int32_t* unit_place = nullptr;       // [units, as unit_src] final place of each unit:
                                       //   output k << 28 | 16-byte vector index of
                                       //   its first element there
  int32_t* slot_live = nullptr;        // [tiles] A2A: 1 if a row of the tile holds
                                       //   a token (else the GEMM skips it)
  int32_t* work = nullptr;             // [P + 1] scratch: consumer chunk counters
  int32_t* finished = nullptr;         // [P] scratch: chunks the consumer finished
  uint32_t* consumed = nullptr;        // [P] sequence number of the last consume
                                       //   that finished each group (read by the
                                       //   overlapped reorder)
  int32_t* rtile = nullptr;            // [2] scratch of the reorder: tile counter,
                                       //   CTAs done
  int32_t* gemm_status = nullptr;      // [1] sticky status of the GEMM's waits
  uint32_t* count_ready = nullptr;     // [1] launch seq once the GEMM zeroed the count table
  int32_t* gemm_exit = nullptr;        // [1] CTAs of the GEMM that finished (reset by the last)
  void* split_ws = nullptr;            // [split_n * 128 * tile_n] fp32 partial sums of
                                       //   the last wave's split tiles
  uint32_t* split_flag = nullptr;      // [split_n * 4] per tile quarter: launch seq
  int32_t* route_cnt = nullptr;        // [blocks * (R + 1)] A2A scratch of
                                       //   fo_plan_route: rows per (tile-row
                                       //   block, rank), then a flag per block
                                       //   that saw an invalid row
};

}  // namespace fo

struct fo_plan {
  // description
  int32_t M = 0, N = 0, K = 0, tile_m = 0, tile_n = 0, swizzle = 0, W = 0;
  int32_t band_order = 0;   // fo_band_order
  int32_t P = 0, R = 1, layout = 0, n_dest = 1, n_experts = 0, top_k = 1, n_tokens = 0;
  int32_t tiles = 0, tiles_n = 0, waves = 0, n_units = 0;
  std::vector<int32_t> expert_rows, expert_row0, expert_tile0;
  std::vector<int32_t> expert_tm;   // tile rows of each expert's grid (incl. padding)
  std::vector<int32_t> group_waves, group_tiles, group_slot_begin, group_unit_begin;
  std::vector<int32_t> slot_tile, tile_slot, slot_group;
  std::vector<fo::TileInfo> tile;
  std::vector<int32_t> part_start, part_len, part_dst, dest_units, final_rows, dest_capacity;
  std::vector<int32_t> dest_base, row_dest, row_rank, final_row, slot_live, unit_src;
  std::vector<int32_t> unit_place;
  // every output holds fewer than 2^28 16-byte vectors, so unit_place can
  // name any place in it (the direct consumer+reorder needs this)
  bool place_ok = false;
  int32_t route_blocks = 0;       // A2A: tile-row blocks (ceil(rows / 128) per expert)
  // fo_plan_route rebuilt the routing tables on the device: the host copies
  // above are stale until refresh_routing() downloads them
  bool routing_on_device = false;
  // device side
  int device = -1;
  int sm_count = 0;
  int consumer_ctas = 0, reorder_ctas = 0, overlap = 1;
  // fo_consume_reorder with overlap on: consumer CTAs with an index of at
  // least this many wait for the last group's flag before taking work
  // (0: every CTA works from the first flag on)
  int consumer_pace = 0;
  // FO_CONSUMER_RESERVED: the consumers launch with this much (unused)
  // dynamic shared memory, more than an SM holding a GEMM CTA has left, so
  // their CTAs run on the SMs the GEMM leaves free (0: shared placement)
  int consumer_smem = 0;
  int gemm_variant = 0;   // fo_gemm_variant
  // last-wave split: when the last wave holds split_n <= W / 2 tiles, each
  // is computed by two CTAs over halves of K (0: no split possible)
  int32_t split_n = 0;
  bool split_enabled = true;
  mutable uint32_t gemm_seq = 0;   // GEMM launches on this plan (never 0 once launched)
  // sequence number of the last consume launched on this plan: a reorder
  // launched as its programmatic dependent waits until consumed[j] holds it
  mutable uint32_t consume_seq = 0;
  mutable bool consume_published = false;   // that consume published its groups
  bool pairable = false;  // launch slots (2i, 2i+1) are vertically adjacent tiles
  uint64_t* trace = nullptr;           // caller's device buffers, see fo_plan_set_trace
  uint64_t* consumer_trace = nullptr;
  void* blob = nullptr;
  fo::DeviceTables dev;
};

namespace fo {

// planner.cpp
fo_status check_shape(const fo_plan_desc* d, int32_t* W, int32_t* tiles,
                      int32_t* waves);
fo_status build_plan(const fo_plan_desc* d, fo_plan* p);
int32_t expert_tile_rows(int32_t pad, int32_t rows);
fo_status upload_plan(fo_plan* p);
int32_t unit_of(const fo_plan* p, int32_t slot, int32_t r);
int32_t place_of(const fo_plan* p, int32_t slot, int32_t r);
// bits of unit_place that hold the vector index; the output is above them
constexpr int kPlaceShift = 28;
// The data kernels move 16-byte vectors: buffers must start on 16 bytes.
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// Counters, flags and status words are 32-bit atomics, stamps 64-bit.
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }
inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7) == 0; }

// SMs without a CTA of the plan's signaled GEMM while it runs (its grid is
// min(W, tiles) CTAs, one per SM).
inline int reserved_sms(const fo_plan* p) {
  return p->sm_count - (p->W < p->tiles ? p->W : p->tiles);
}

void set_a2a_outputs(fo_plan* p, int32_t n_tokens, int32_t top_k);
fo_status refresh_routing(fo_plan* p);

// route.cu
fo_status launch_plan_route(const fo_plan* p, const int32_t* row_token, const int32_t* row_slot,
                            int32_t* dev_status, void* stream);

// gemm.cu
int gemm_pair_capacity(const fo_plan* p);
int gemm_smem_bytes();
fo_status launch_signaled_gemm(const fo_plan* p, const void* A,
                               const void* const* B, void* C_r,
                               int32_t* count, uint32_t* flags, uint32_t epoch,
                               void* stream);

// comm.cu
fo_status launch_consume(const fo_plan* p, int32_t g0, int32_t g1, int kind,
                         const void* src, const void* const* partials,
                         int32_t n_partials, void* const* dst,
                         const uint32_t* flags, uint32_t epoch,
                         uint64_t spin_limit_ns, int32_t* dev_status,
                         void* stream);
fo_status launch_consume_reorder(const fo_plan* p, int32_t g0, int32_t g1, int kind,
                                 const void* src, const void* const* partials,
                                 int32_t n_partials, void* const* comm_dst,
                                 void* const* final_dst, const void* bias, int act,
                                 const uint32_t* flags, uint32_t epoch, uint64_t spin_limit_ns,
                                 int32_t* dev_status, void* stream);
fo_status launch_reorder_back(const fo_plan* p, int32_t g0, int32_t g1,
                              const void* const* src, void* const* dst,
                              const void* bias, int act, void* stream);
// An ordinary (not programmatic) launch of the library on `stream` (the
// signaled GEMM): every earlier kernel on the stream has finished before it
// starts, so a no-alloc consume issued after it cannot run beside an
// earlier one (comm.cu, fo_consume_group_noalloc).
void noalloc_note_ordinary_launch(int device, void* stream);
fo_status launch_allgather_rows(const fo_plan* p, const void* const* slices, void* out,
                                const void* bias, int act, void* stream);

}  // namespace fo
