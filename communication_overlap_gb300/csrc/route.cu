// Routing tables of the All-to-All layout, built on the device.
//
// Page: "FlashOverlap: 信号驱动计算通信重叠论文详解" -- 二、重排机制 (3) All-to-All:
// in an MoE layer tokens are routed to experts at run time; the sub-token
// (one tile row) is the reorder unit, the pre-communication reorder makes
// the sub-tokens bound for one GPU contiguous, the post-communication
// reorder puts them back through the mapping table, and that table has to
// follow the dynamic routing.
//
// The plan fixes each expert's capacity (its rows), hence the tiles, their
// launch order, the waves and the groups.  A routing says which token each
// row holds (or none).  From a routing in device memory, two kernels
// rebuild every table that depends on it -- the same tables the host
// planner builds from a host routing, bit for bit:
//
//  route_rows   one CTA per tile-row block (128 rows of one expert): per row
//               its destination rank d = token mod R, its rank among the
//               block's rows bound for d (a warp match plus per-warp counts)
//               and its output row (token / R) * top_k + slot; per block the
//               rows bound for each rank, and whether the routing is invalid.
//  route_parts  units are laid out group after group, part d of a group
//               holding, over its tiles in launch order, the rows bound for
//               d.  With BP[b][d] = rows for d in blocks before b (a scan over
//               blocks, redone in every CTA's shared memory), the units for d
//               before launch slot s follow in closed form from the banded
//               launch order (bands of `swizzle` tile rows walked column by
//               column; in a serpentine order the expert's odd bands walk
//               them right to left, and tn below is the column's position
//               in its band, TN - 1 - column there):
//                 E(s, d) = TN * BP[b0][d] + tn * (BP[b0 + h][d] - BP[b0][d])
//                           + BP[b][d] - BP[b0][d]
//               for the tile of block b, column tn, in the band of blocks
//               [b0, b0 + h).  Everything else is E at group boundaries:
//                 group_unit_begin[j] = sum_d E(gsb[j], d)
//                 part_dst[j][d]      = E(gsb[j], d)
//                 part_len[j][d]      = E(gsb[j + 1], d) - E(gsb[j], d)
//                 part_start[j][d]    = group_unit_begin[j] + sum_{d' < d} part_len[j][d']
//                 dest_base[s][d]     = part_start[j][d] + E(s, d) - E(gsb[j], d)
//               CTA 0 writes the per-group tables, all CTAs the per-slot ones
//               (dest_base, and whether any row of the tile holds a token:
//               the GEMM skips tiles that hold none) and the per-unit one
//               (which tile row each unit holds).
//
// An invalid routing (token >= n_tokens, slot outside [0, top_k), or more
// units for a rank than its receive buffer holds) routes nothing: every row
// is marked empty, every part is empty, and the caller's status word is set
// to FO_ERR_ARG.
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"

namespace fo {

namespace {

constexpr int kPartsThreads = 256;

struct RouteArgs {
  const int32_t* token;       // [M]
  const int32_t* slot;        // [M]
  const TileInfo* tile;       // [tiles]
  const int32_t* group_slot_begin;  // [P + 1]
  int32_t* row_dest;          // [M]
  int32_t* row_rank;          // [M]
  int32_t* final_row;         // [M]
  int32_t* cnt;               // [B * R] rows per (block, rank), then bad[B]
  int32_t* part_start;        // [P * R]
  int32_t* part_len;          // [P * R]
  int32_t* part_dst;          // [P * R]
  int32_t* group_unit_begin;  // [P + 1]
  int32_t* dest_base;         // [tiles * R]
  int32_t* slot_live;         // [tiles] 1 if a row of the tile holds a token
  int32_t* unit_src;          // [units] slot << 7 | row of the tile row each unit holds
  int32_t* unit_place;        // [units] final place: rank << kPlaceShift | vector index
                              //   (NULL: the plan's outputs are too large for it)
  int32_t* status;            // caller's status word
  int32_t expert_row0[kMaxExperts];
  int32_t expert_rows[kMaxExperts];
  int32_t expert_block0[kMaxExperts + 1];
  int32_t cap[kMaxDest];      // units each receive buffer holds
  int32_t n_experts, R, n_tokens, top_k, B, P, tiles, TN, swizzle, tile_n, M, N;
  int32_t serpentine;   // odd bands of each expert walk their columns right to left
};

__global__ void __launch_bounds__(kTileM) route_rows_kernel(const __grid_constant__ RouteArgs a) {
  constexpr int kWarps = kTileM / 32;
  __shared__ int32_t warp_cnt[kWarps][kMaxDest];
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int e = 0;
  while (e + 1 < a.n_experts && a.expert_block0[e + 1] <= b) ++e;
  const int32_t row0 = a.expert_row0[e] + (b - a.expert_block0[e]) * kTileM;
  // (a padding tile row of an expert's grid holds no rows)
  const int32_t rows = max(0, min(kTileM, a.expert_row0[e] + a.expert_rows[e] - row0));
  for (int i = tid; i < kWarps * kMaxDest; i += kTileM) (&warp_cnt[0][0])[i] = 0;
  int32_t d = -1, t = -1, q = 0;
  int bad = 0;
  if (tid < rows) {
    t = a.token[row0 + tid];
    q = a.slot[row0 + tid];
    if (t >= 0) {
      if (t >= a.n_tokens || q < 0 || q >= a.top_k)
        bad = 1;
      else
        d = t % a.R;
    }
  }
  __syncthreads();
  // rank among this warp's earlier rows bound for the same d, then the
  // earlier warps' counts
  const uint32_t peers = __match_any_sync(0xffffffffu, d);
  const int32_t rank_w = __popc(peers & ((1u << lane) - 1u));
  if (d >= 0 && rank_w == 0) warp_cnt[warp][d] = __popc(peers);
  __syncthreads();
  if (tid < rows) {
    int32_t rank = -1, fr = -1;
    if (d >= 0) {
      rank = rank_w;
      for (int w = 0; w < warp; ++w) rank += warp_cnt[w][d];
      fr = (t / a.R) * a.top_k + q;
    }
    a.row_dest[row0 + tid] = d;
    a.row_rank[row0 + tid] = rank;
    a.final_row[row0 + tid] = fr;
  }
  if (tid < a.R) {
    int32_t c = 0;
    for (int w = 0; w < kWarps; ++w) c += warp_cnt[w][tid];
    a.cnt[b * a.R + tid] = c;
  }
  bad = __syncthreads_or(bad);
  if (tid == 0) a.cnt[a.B * a.R + b] = bad ? 1 : 0;
}

// Units bound for rank d in the launch slots before the tile (row0, col0) of
// expert e, from the block prefix BP (shared memory).
__device__ __forceinline__ int32_t units_before(const RouteArgs& a, const int32_t* BP,
                                                int32_t row0, int32_t col0, int32_t e, int d) {
  const int32_t tm = (row0 - a.expert_row0[e]) / kTileM;
  const int32_t tm_count = a.expert_block0[e + 1] - a.expert_block0[e];
  const int32_t top = tm - tm % a.swizzle;
  const int32_t h = min(a.swizzle, tm_count - top);
  const int32_t b0 = a.expert_block0[e] + top, b = a.expert_block0[e] + tm;
  const int32_t col = col0 / a.tile_n;
  // the column's position in its band's order
  const int32_t tn = (a.serpentine && (top / a.swizzle) % 2) ? a.TN - 1 - col : col;
  const int32_t p0 = BP[b0 * a.R + d];
  return a.TN * p0 + tn * (BP[(b0 + h) * a.R + d] - p0) + (BP[b * a.R + d] - p0);
}

__device__ __forceinline__ int32_t units_before_slot(const RouteArgs& a, const int32_t* BP,
                                                     int32_t s, int d) {
  if (s >= a.tiles) return a.TN * BP[a.B * a.R + d];
  const TileInfo& ti = a.tile[s];
  return units_before(a, BP, ti.row0, ti.col0, ti.expert, d);
}

__global__ void __launch_bounds__(kPartsThreads) route_parts_kernel(const __grid_constant__ RouteArgs a) {
  extern __shared__ int32_t sm[];
  const int R = a.R, B = a.B, P = a.P, tid = threadIdx.x;
  const int nseg = kPartsThreads / R;
  int32_t* BP = sm;                    // [(B + 1) * R]
  int32_t* Eg = BP + (B + 1) * R;      // [(P + 1) * R]  E at group boundaries
  int32_t* off = Eg + (P + 1) * R;     // [P * R]        part_start - E(gsb[j])
  int32_t* seg = off + P * R;          // [nseg * R]     segment sums of the scan
  const int32_t* bad_of = a.cnt + B * R;

  // 1. BP: exclusive prefix over blocks, per rank, as a segmented scan
  const int d0 = tid % R, sg = tid / R;
  const int len = (B + nseg - 1) / nseg;
  const int b_lo = min(B, sg * len), b_hi = min(B, b_lo + len);
  int any_bad = 0;
  if (sg < nseg) {
    int32_t sum = 0;
    for (int b = b_lo; b < b_hi; ++b) sum += a.cnt[b * R + d0];
    seg[sg * R + d0] = sum;
    if (d0 == 0)
      for (int b = b_lo; b < b_hi; ++b) any_bad |= bad_of[b];
  }
  __syncthreads();
  if (tid < R) {
    int32_t run = 0;
    for (int g = 0; g < nseg; ++g) {
      const int32_t v = seg[g * R + tid];
      seg[g * R + tid] = run;
      run += v;
    }
    BP[tid] = 0;
  }
  __syncthreads();
  if (sg < nseg) {
    int32_t run = seg[sg * R + d0];
    for (int b = b_lo; b < b_hi; ++b) {
      run += a.cnt[b * R + d0];
      BP[(b + 1) * R + d0] = run;
    }
  }
  __syncthreads();

  // 2. E at the group boundaries; the routing is rejected if a rank would
  //    receive more units than its buffer holds
  for (int i = tid; i < (P + 1) * R; i += kPartsThreads) {
    const int j = i / R, d = i - j * R;
    Eg[i] = units_before_slot(a, BP, a.group_slot_begin[j], d);
  }
  __syncthreads();
  if (tid < R && Eg[P * R + tid] > a.cap[tid]) any_bad = 1;
  const bool bad = __syncthreads_or(any_bad) != 0;

  // 3. per-group tables
  for (int i = tid; i < P * R; i += kPartsThreads) {
    const int j = i / R, d = i - j * R;
    int32_t start = 0;
    for (int dd = 0; dd < R; ++dd) start += Eg[j * R + dd];
    for (int dd = 0; dd < d; ++dd) start += Eg[(j + 1) * R + dd] - Eg[j * R + dd];
    off[i] = start - Eg[i];
    if (blockIdx.x == 0) {
      a.part_start[i] = bad ? 0 : start;
      a.part_len[i] = bad ? 0 : Eg[(j + 1) * R + d] - Eg[i];
      a.part_dst[i] = bad ? 0 : Eg[i];
    }
  }
  if (blockIdx.x == 0) {
    for (int j = tid; j <= P; j += kPartsThreads) {
      int32_t g = 0;
      for (int d = 0; d < R; ++d) g += Eg[j * R + d];
      a.group_unit_begin[j] = bad ? 0 : g;
    }
    if (bad && tid == 0) atomicCAS(a.status, 0, int32_t(FO_ERR_ARG));
  }
  __syncthreads();

  // 4. per-slot bases; a rejected routing also empties every row
  const int32_t stride = int32_t(gridDim.x) * kPartsThreads;
  const int32_t first = int32_t(blockIdx.x) * kPartsThreads + tid;
  for (int32_t i = first; i < a.tiles * R; i += stride) {
    const int32_t s = i / R;
    const int d = i - s * R;
    int32_t v = 0;
    const TileInfo& ti = a.tile[s];
    if (!bad) v = off[ti.group * R + d] + units_before(a, BP, ti.row0, ti.col0, ti.expert, d);
    a.dest_base[i] = v;
    if (d == 0) {   // the tile's rows that hold a token: its block's count
      const int32_t b = a.expert_block0[ti.expert] + (ti.row0 - a.expert_row0[ti.expert]) / kTileM;
      int32_t n = 0;
      for (int dd = 0; dd < R; ++dd) n += BP[(b + 1) * R + dd] - BP[b * R + dd];
      a.slot_live[s] = (!bad && n > 0) ? 1 : 0;
    }
  }
  if (bad) {
    for (int32_t r = first; r < a.M; r += stride) {
      a.row_dest[r] = -1;
      a.row_rank[r] = -1;
      a.final_row[r] = -1;
    }
    return;
  }
  // 5. the inverse at row granularity: unit -> the tile row it holds (read by
  //    the fused consumer+reorder) and its final place (read by its direct
  //    variant); row r of the tile at slot s is unit dest_base[s][d] + rank,
  //    computed here from the same closed form
  //    Four entries per thread and pass, their table loads issued together:
  //    each entry is a chain of two dependent global loads (the tile, then
  //    the row's rank, destination and output row).
  constexpr int kE = 4;
  const int64_t n_entries = int64_t(a.tiles) * kTileM;
  for (int64_t i0 = first; i0 < n_entries; i0 += int64_t(stride) * kE) {
    TileInfo ti[kE];
    int32_t rho[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const int64_t i = i0 + int64_t(stride) * e;
      rho[e] = -1;
      if (i < n_entries) {
        ti[e] = a.tile[i / kTileM];
        const int32_t r = int32_t(i % kTileM);
        if (r < ti[e].rows) rho[e] = ti[e].row0 + r;
      }
    }
    int d[kE];
    int32_t rank[kE], frow[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      d[e] = -1;
      if (rho[e] >= 0) {
        d[e] = a.row_dest[rho[e]];
        rank[e] = a.row_rank[rho[e]];
        frow[e] = a.unit_place != nullptr ? a.final_row[rho[e]] : 0;
      }
    }
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      if (d[e] < 0) continue;
      const int64_t i = i0 + int64_t(stride) * e;
      const int32_t s = int32_t(i / kTileM), r = int32_t(i % kTileM);
      const int32_t u = off[ti[e].group * R + d[e]] +
                        units_before(a, BP, ti[e].row0, ti[e].col0, ti[e].expert, d[e]) + rank[e];
      a.unit_src[u] = (s << 7) | r;
      if (a.unit_place != nullptr)
        a.unit_place[u] = (d[e] << kPlaceShift) | (frow[e] * (a.N / 8) + ti[e].col0 / 8);
    }
  }
}

size_t parts_smem_bytes(const fo_plan* p) {
  const int nseg = kPartsThreads / p->R;
  return sizeof(int32_t) * (size_t(p->route_blocks + 1) * p->R + size_t(p->P + 1) * p->R +
                            size_t(p->P) * p->R + size_t(nseg) * p->R);
}

}  // namespace

fo_status launch_plan_route(const fo_plan* p, const int32_t* row_token, const int32_t* row_slot,
                            int32_t* dev_status, void* stream) {
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  static int smem_optin[64];
  const int dv = p->device < 64 ? p->device : 63;
  std::call_once(once[dv], [&] {
    attr_err[dv] = cudaDeviceGetAttribute(&smem_optin[dv],
                                          cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
    if (attr_err[dv] == cudaSuccess)
      attr_err[dv] = cudaFuncSetAttribute(route_parts_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          smem_optin[dv]);
  });
  if (attr_err[dv] != cudaSuccess) return FO_ERR_CUDA;
  const size_t smem = parts_smem_bytes(p);
  if (smem > size_t(smem_optin[dv])) return FO_ERR_UNSUPPORTED;
  if (p->route_blocks < 1) return FO_ERR_ARG;

  RouteArgs a{};
  a.token = row_token;
  a.slot = row_slot;
  a.tile = p->dev.tile;
  a.group_slot_begin = p->dev.group_slot_begin;
  a.row_dest = p->dev.row_dest;
  a.row_rank = p->dev.row_rank;
  a.final_row = p->dev.final_row;
  a.cnt = p->dev.route_cnt;
  a.part_start = p->dev.part_start;
  a.part_len = p->dev.part_len;
  a.part_dst = p->dev.part_dst;
  a.group_unit_begin = p->dev.group_unit_begin;
  a.dest_base = p->dev.dest_base;
  a.slot_live = p->dev.slot_live;
  a.unit_src = p->dev.unit_src;
  a.unit_place = p->place_ok ? p->dev.unit_place : nullptr;
  a.status = dev_status;
  const int E = int(p->expert_rows.size());
  int32_t blocks = 0;
  for (int e = 0; e < E; ++e) {
    a.expert_row0[e] = p->expert_row0[e];
    a.expert_rows[e] = p->expert_rows[e];
    a.expert_block0[e] = blocks;
    blocks += p->expert_tm[e];   // (incl. a padding tile row)
  }
  a.expert_block0[E] = blocks;
  for (int k = 0; k < p->R; ++k) a.cap[k] = p->dest_capacity[k];
  a.n_experts = E;
  a.R = p->R;
  a.n_tokens = p->n_tokens;
  a.top_k = p->top_k;
  a.B = p->route_blocks;
  a.P = p->P;
  a.tiles = p->tiles;
  a.TN = p->tiles_n;
  a.swizzle = p->swizzle;
  a.serpentine = p->band_order == FO_BAND_SERPENTINE ? 1 : 0;
  a.tile_n = p->tile_n;
  a.M = p->M;
  a.N = p->N;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  route_rows_kernel<<<a.B, kTileM, 0, st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return FO_ERR_CUDA;
  // enough CTAs that each thread takes a handful of the tiles x 128 rows of
  // the unit table (each needs a dependent global load), up to 4 per SM
  const int64_t entries = int64_t(p->tiles) * kTileM;
  int ctas = int((entries + 4 * kPartsThreads - 1) / (4 * kPartsThreads));
  ctas = ctas < 1 ? 1 : (ctas > 4 * p->sm_count ? 4 * p->sm_count : ctas);
  route_parts_kernel<<<ctas, kPartsThreads, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? FO_OK : FO_ERR_CUDA;
}

}  // namespace fo
