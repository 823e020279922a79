// Consumer kernels: the communication stand-in, alone (consume_kernel) and
// with the post-communication reorder fused in (consume_reorder_kernel,
// which either writes the communication buffers and moves each chunk on to
// its final place, or -- the direct variant -- stores every unit straight
// to its final place).
//
// Pages: "FlashOverlap: 信号驱动计算通信重叠论文详解" -- 核心设计 "通信侧" (the
// communication runs as its own kernel on another stream), 五、CUTLASS 扩展实现
// "专用监控内核" (a monitor kernel tracks progress through atomic counters) and
// "Epilogue 集成" (the reorder fused with element-wise operations), 二、重排机制
// (a group's data is contiguous so one collective call covers it).
//
// Both are HBM-bound streams of 16-byte vectors over each group's contiguous
// unit range (every warp instruction moves 512 contiguous bytes), launched as
// programmatic dependents of the GEMM so that they run beside it: per group,
// one thread polls the group's flag, then the CTAs take chunks of the range
// from a per-group counter.  The plain consumer also publishes when each
// group is fully written, for a reorder launched as its own dependent.
#include <cuda_runtime.h>

#include <mutex>
#include <utility>
#include <vector>

#include "device_common.cuh"
#include "row_map.cuh"

namespace fo {

namespace {

constexpr int kThreads = 256;

// Reserved placement with the default grid: default_ctas returns minus the
// number of SMs the GEMM leaves free, and the launch turns that into as many
// CTAs as those SMs hold at once (the kernel's own occupancy: threads,
// registers and the requested shared memory), so that no CTA waits for an
// SM and then lands on one a finished GEMM CTA left.
template <typename Kernel>
int resolve_grid(Kernel kernel, int ctas, int smem) {
  if (ctas > 0) return ctas;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, size_t(smem)) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm * (-ctas > 0 ? -ctas : 1);
}

// 16-byte vectors each lane keeps in flight per source (per iteration): the
// sums keep one per source, all sources at once (sum_partials).
template <int KIND>
constexpr int kUnroll = (KIND == FO_CONS_SUM || KIND == FO_CONS_RS) ? 1 : 8;
// Bytes of the source a CTA takes per chunk: one pass of U vectors per
// thread for the copies (32 KB), four passes for the sums (16 KB).
template <int KIND>
constexpr int kChunkBytes = (KIND == FO_CONS_SUM || KIND == FO_CONS_RS) ? 16 * 1024 : 32 * 1024;
// The fused consumer+reorder keeps fewer copy loads in flight per thread: it
// runs at 72 registers (two CTAs beside a GEMM CTA) and also holds the
// reorder's loads.
template <int KIND>
constexpr int kFusedUnroll = (KIND == FO_CONS_SUM || KIND == FO_CONS_RS) ? 1 : 4;
// Units of the largest chunk (32 KB of 256-byte units at tile_n = 128).
constexpr int kMaxChunkUnits = 32 * 1024 / 256;

struct ConsumeArgs {
  const uint4* src;
  const uint4* partials[kMaxPartials];
  uint4* dst[kMaxDest];
  const uint32_t* flags;
  int32_t* status;
  const int32_t* group_unit_begin;
  const int32_t* part_start;
  const int32_t* part_len;
  const int32_t* part_dst;
  int32_t* work;   // [P] chunk counters, then one "CTAs done" counter
  int32_t* finished;   // [P] chunks finished per group (NULL: no consumed flags)
  uint32_t* consumed;  // [P] = seq once every chunk of the group is written
  uint32_t seq;        // this launch's number on the plan (never 0)
  int32_t g0, g1, n_partials, R, P, vpu_shift, chunk_units;
  uint32_t epoch;
  uint64_t limit_ns;
  uint64_t* trace;  // optional: [P] group fully consumed, [P] group reordered
                    // (fused kernel), then [grid][4] CTA records
};

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], bf16lo(w[i]));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], bf16hi(w[i]));
  }
}

__device__ __forceinline__ void set_bf16x8(float (&acc)[8], const uint4& x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = bf16lo(w[i]);
    acc[2 * i + 1] = bf16hi(w[i]);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                    pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

// Partials a sum with U vectors per source and thread holds in registers:
// with two vectors (the direct kernel's sum of at most 4 partials) 4.
template <int U>
constexpr int kPartialsInFlight = U >= 2 ? 4 : kMaxPartials;

// x[i] (U vectors of the own buffer at base + kThreads * i, those below v1)
// becomes the fp32 sum of itself and the same vectors of every partial, in
// order, rounded once to bf16.  Every partial's loads are issued before the
// first addition (predicated per partial, no early exit), so a thread keeps
// all its sources' loads in flight at once instead of one source at a time.
template <int U>
__device__ __forceinline__ void sum_partials(const ConsumeArgs& a, int32_t base, int32_t v1,
                                             uint64_t pol, uint4 (&x)[U]) {
  constexpr int kP = kPartialsInFlight<U>;
  uint4 y[kP][U];
#pragma unroll
  for (int q = 0; q < kP; ++q)
#pragma unroll
    for (int i = 0; i < U; ++i)
      if (q < a.n_partials && base + kThreads * i < v1)
        y[q][i] = ld_once(a.partials[q] + base + kThreads * i, pol);
  float acc[U][8];
#pragma unroll
  for (int i = 0; i < U; ++i) set_bf16x8(acc[i], x[i]);
#pragma unroll
  for (int q = 0; q < kP; ++q)
    if (q < a.n_partials)
#pragma unroll
      for (int i = 0; i < U; ++i) add_bf16x8(acc[i], y[q][i]);
#pragma unroll
  for (int i = 0; i < U; ++i) x[i] = pack8(acc[i]);
}

// Where vector v (unit v >> vpu_shift) of the group goes: destination k's
// part (j, k) starts at unit part_dst there.
__device__ __forceinline__ uint4* route(const int32_t* ps, const int32_t* pl,
                                        const int32_t* pd, uint4* const* dst, int R,
                                        int vpu_shift, int32_t v) {
  const int32_t u = v >> vpu_shift;
  int k = 0;
  for (; k < R - 1; ++k)
    if (uint32_t(u - ps[k]) < uint32_t(pl[k])) break;
  const int32_t vu = (pd[k] + (u - ps[k])) << vpu_shift;
  return dst[k] + vu + (v & ((1 << vpu_shift) - 1));
}

// The CTA processes vectors [v0, v1) of the reordered buffer: thread t
// takes v0 + t + kThreads * i, so each warp instruction covers 512
// contiguous bytes and every thread keeps U loads (per source) in flight.
template <int KIND, int U>
__device__ __forceinline__ void consume_range(const ConsumeArgs& a, const int32_t* ps,
                                              const int32_t* pl, const int32_t* pd,
                                              uint4* const* dst, int32_t v0, int32_t v1,
                                              int tid) {
  constexpr bool kSum = (KIND == FO_CONS_SUM || KIND == FO_CONS_RS);
  constexpr int S = kThreads;
  // every source vector is read exactly once: evict-first in L2
  const uint64_t pol = l2_evict_first();
  for (int32_t base = v0 + tid; base < v1; base += S * U) {
    uint4 x[U];
#pragma unroll
    for (int i = 0; i < U; ++i)
      if (base + S * i < v1) x[i] = ld_once(a.src + base + S * i, pol);
    if constexpr (kSum) sum_partials<U>(a, base, v1, pol, x);
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int32_t v = base + S * i;
      if (v >= v1) break;
      // ordinary write-back stores: the post-communication reorder reads
      // these buffers next, so they may stay in L2
      if constexpr (KIND == FO_CONS_COPY || KIND == FO_CONS_SUM)
        dst[0][v] = x[i];
      else
        *route(ps, pl, pd, dst, a.R, a.vpu_shift, v) = x[i];
    }
  }
}

// Persistent consumer: for each group in order, thread 0 waits on the
// group's flag, then the CTA takes chunks of the group's unit range from a
// per-group counter until none are left (thread 0 fetches the next chunk
// index while the CTA works on the current one).  Chunks are small enough
// that every CTA gets work in every group, and dynamic so the work stays
// balanced whichever CTAs are resident while the GEMM still runs.
//
// The chunk counters clean up after themselves: the last CTA to finish
// (counted on work[P]) zeroes them, so the next launch needs no memset and
// can follow the GEMM directly as a programmatic dependent launch.
//
// Each finished chunk is counted per group; the CTA that finishes a group's
// last chunk publishes consumed[j] = epoch (release, after every chunk's
// stores), which a post-communication reorder launched as this kernel's
// programmatic dependent waits for before it moves the group.
template <int KIND, int U>
__global__ void __launch_bounds__(kThreads) consume_kernel(const __grid_constant__ ConsumeArgs a) {
  __shared__ int s_ok;
  __shared__ int32_t s_chunk[2];
  __shared__ int32_t s_ps[kMaxDest], s_pl[kMaxDest], s_pd[kMaxDest];
  __shared__ uint4* s_dst[kMaxDest];
  const int tid = threadIdx.x;
  // every CTA of this grid is resident from here on: a dependent reorder may
  // start (its CTAs can then never hold resources this grid still needs)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid < kMaxDest) s_dst[tid] = a.dst[tid];
  uint64_t t_start = 0;
  int32_t chunks_done = 0;
  if (a.trace != nullptr && tid == 0) t_start = globaltimer_ns();
  for (int j = a.g0; j < a.g1; ++j) {
    // the group's first chunk is taken before the wait on its flag
    if (tid == 0) {
      s_chunk[0] = atomicAdd(a.work + j, 1);
      s_ok = wait_flag(a.flags + j, a.epoch, a.limit_ns) ? 1 : 0;
    }
    if (tid < a.R) {
      s_ps[tid] = a.part_start[j * a.R + tid];
      s_pl[tid] = a.part_len[j * a.R + tid];
      s_pd[tid] = a.part_dst[j * a.R + tid];
    }
    __syncthreads();
    if (!s_ok) {
      if (tid == 0) atomicCAS(a.status, 0, int32_t(FO_ERR_TIMEOUT));
      break;
    }
    const int32_t ub = a.group_unit_begin[j], ue = a.group_unit_begin[j + 1];
    const int32_t n_chunks = (ue - ub + a.chunk_units - 1) / a.chunk_units;
    if (n_chunks == 0 && a.finished != nullptr && tid == 0)
      st_release_gpu(a.consumed + j, a.seq);   // an empty group is consumed at once
    int32_t group_chunks = 0;
    for (int buf = 0;; buf ^= 1) {
      const int32_t c = s_chunk[buf];
      if (c >= n_chunks) break;
      if (tid == 0) s_chunk[buf ^ 1] = atomicAdd(a.work + j, 1);
      const int32_t u0 = ub + c * a.chunk_units;
      const int32_t u1 = min(u0 + a.chunk_units, ue);
      consume_range<KIND, U>(a, s_ps, s_pl, s_pd, s_dst, u0 << a.vpu_shift,
                             u1 << a.vpu_shift, tid);
      __syncthreads();
      ++group_chunks;
      if (a.trace != nullptr && tid == 0) {
        // the latest chunk end of the group is when it is fully consumed
        atomicMax(reinterpret_cast<unsigned long long*>(a.trace + j),
                  static_cast<unsigned long long>(globaltimer_ns()));
        ++chunks_done;
      }
    }
    __syncthreads();
    if (a.finished != nullptr && tid == 0 && group_chunks > 0) {
      // this CTA's stores for the group (all threads, ordered by the
      // barrier) are visible before its chunks are counted, once per group;
      // the CTA that completes the count releases the group
      __threadfence();
      if (atomicAdd(a.finished + j, group_chunks) + group_chunks == n_chunks)
        st_release_gpu(a.consumed + j, a.seq);
    }
  }
  if (a.trace != nullptr) {
    if (tid == 0) {
      uint64_t* rec = a.trace + 2 * a.P + 4 * blockIdx.x;
      rec[3] = uint64_t(chunks_done);
      uint32_t smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      rec[0] = smid;
      rec[1] = t_start;
      rec[2] = globaltimer_ns();
    }
  }
  // A consume launched as the programmatic dependent of the kernel before
  // it on the stream (the GEMM, or with per-group calls an earlier consume
  // or reorder of this plan) can run beside that kernel: the scratch
  // counters below are shared between launches on one plan, so wait until
  // that kernel has completed before touching them.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // every CTA, finished or timed out, reports; the last one resets the
  // counters of this launch's groups and the report counter
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.work + a.P, 1) == int32_t(gridDim.x) - 1) {
      for (int j = a.g0; j < a.g1; ++j) {
        atomicExch(a.work + j, 0);
        if (a.finished != nullptr) atomicExch(a.finished + j, 0);
      }
      atomicExch(a.work + a.P, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// Consumer with the post-communication reorder (and the element-wise
// epilogue) fused in: one persistent kernel, on the GEMM's stream, that
// moves every group to its final layout while the GEMM still computes later
// groups.  A CTA that has written a chunk of units to the communication
// buffers reads them back from there -- still in L2 -- and moves each unit
// to its final place at once: unit_src names the tile row a unit holds, the
// inverse mapping gives its place.  No CTA waits for another, so a group is
// final one chunk after its flag rises.

struct FusedArgs {
  ConsumeArgs c;                  // the communication part (c.dst: its outputs)
  uint4* fin[kMaxDest];           // final outputs of the reorder
  RowMap map;
  const uint16_t* bias;
  const int32_t* unit_src;  // [units] slot << 7 | row of the tile row each unit holds
  const int32_t* unit_place;   // [units] output << kPlaceShift | vector index
  int32_t act, row_vec;
  int32_t direct;  // no communication buffers: each unit goes straight to its final place
  int32_t pace;    // > 0: CTAs from this index on first wait for the last group's flag
};

// Where the units of a chunk go, computed by threads t < units before the
// chunk is consumed (their loads overlap the other warps' consume loads):
// the communication buffer k and unit su it was written to, and its place
// in final output k (16-byte vector index of the row start) and column.
struct ChunkMap {
  int32_t k[kMaxChunkUnits];
  int32_t su[kMaxChunkUnits];
  int32_t col[kMaxChunkUnits];
  int64_t to[kMaxChunkUnits];
};

__device__ __forceinline__ void map_chunk_units(const FusedArgs& a, ChunkMap& m, int32_t u0,
                                                int32_t u1, int tid) {
  if (tid < u1 - u0) {
    const int32_t us = a.unit_src[u0 + tid];
    const int32_t s = us >> 7, r = us & (kTileM - 1);
    const TileInfo ti = a.map.tile[s];
    int k;
    int32_t su, dr;
    map_row(a.map, ti, s, r, &k, &su, &dr);
    m.k[tid] = k;
    m.su[tid] = su;
    m.col[tid] = ti.col0;
    m.to[tid] = int64_t(dr) * a.row_vec + (ti.col0 >> 3);
  }
}

// The chunk's units, just written to the communication buffers by this CTA,
// read back from there and stored to their final places: thread t moves
// vectors t, t + 256, ... (one unit per warp instruction), all loads in
// flight before the stores.
template <int VPU, int NV>
__device__ __forceinline__ void reorder_chunk_regs(const FusedArgs& a, const ChunkMap& m,
                                                   uint4* const* src, uint4* const* fin,
                                                   int32_t n_units, int tid) {
  const uint64_t pol = l2_evict_first();   // the received data is read once
  const int32_t n_vec = n_units * VPU;
  uint4 x[NV];
#pragma unroll
  for (int b = 0; b < NV; ++b) {
    const int32_t v = tid + kThreads * b;
    if (v < n_vec) {
      const int32_t i = v / VPU, vl = v % VPU;
      x[b] = ld_once(src[m.k[i]] + int64_t(m.su[i]) * VPU + vl, pol);
    }
  }
#pragma unroll
  for (int b = 0; b < NV; ++b) {
    const int32_t v = tid + kThreads * b;
    if (v < n_vec) {
      const int32_t i = v / VPU, vl = v % VPU;
      uint4 y = x[b];
      if (a.act != FO_ACT_NONE || a.bias != nullptr)
        y = epilogue8(y, a.bias, m.col[i] + vl * 8, a.act);
      st_cs(fin[m.k[i]] + m.to[i] + vl, y);
    }
  }
}

// The direct variant: the chunk's vectors [v0, v1) of the reordered buffer,
// consumed as in consume_range (same loads, same fp32 sums in the same
// order), then stored straight to their final places, so the communication
// buffers are neither written nor read back.  Each lane reads its unit's
// place from the plan's unit_place table (one load, which a warp's lanes
// share: a unit is 512 or 256 contiguous bytes), issued before the data
// loads so that both are in flight together.
template <int KIND, int U>
__device__ __forceinline__ void consume_direct(const FusedArgs& a, uint4* const* fin,
                                               int32_t v0, int32_t v1, int tid) {
  const ConsumeArgs& c = a.c;
  constexpr bool kSum = (KIND == FO_CONS_SUM || KIND == FO_CONS_RS);
  constexpr int S = kThreads;
  const uint64_t pol = l2_evict_first();
  const int32_t vmask = (1 << c.vpu_shift) - 1;
  for (int32_t base = v0 + tid; base < v1; base += S * U) {
    int32_t place[U];   // output << kPlaceShift | vector index; -1 past the chunk
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int32_t v = base + S * i;
      place[i] = v < v1 ? a.unit_place[v >> c.vpu_shift] + (v & vmask) : -1;
    }
    uint4 x[U];
#pragma unroll
    for (int i = 0; i < U; ++i)
      if (base + S * i < v1) x[i] = ld_once(c.src + base + S * i, pol);
    if constexpr (kSum) sum_partials<U>(c, base, v1, pol, x);
#pragma unroll
    for (int i = 0; i < U; ++i) {
      if (place[i] < 0) continue;   // past the chunk
      const int32_t to = place[i] & ((1 << kPlaceShift) - 1);
      uint4 y = x[i];
      if (a.act != FO_ACT_NONE || a.bias != nullptr)
        y = epilogue8(y, a.bias, (to % a.row_vec) * 8, a.act);
      st_cs(fin[place[i] >> kPlaceShift] + to, y);
    }
  }
}

// Launched with 256 threads.  Registers capped at 72: measured, two CTAs at
// 70 registers run beside each GEMM CTA while the GEMM runs, at 80 only one.
template <int KIND, int U, int VPU, bool DIRECT>
__global__ void __maxnreg__(72) consume_reorder_kernel(const __grid_constant__ FusedArgs a) {
  constexpr int kNV = kChunkBytes<KIND> / (16 * kThreads);   // vectors of a chunk per thread
  const ConsumeArgs& c = a.c;
  __shared__ ChunkMap s_map;
  __shared__ int s_ok;
  __shared__ int32_t s_chunk[2];
  __shared__ int32_t s_ps[kMaxDest], s_pl[kMaxDest], s_pd[kMaxDest];
  __shared__ uint4* s_dst[kMaxDest];
  __shared__ uint4* s_fin[kMaxDest];
  const int tid = threadIdx.x;
  if (tid < kMaxDest) {
    s_dst[tid] = c.dst[tid];
    s_fin[tid] = a.fin[tid];
  }
  uint64_t t_start = 0;
  int32_t chunks_done = 0;
  if (c.trace != nullptr && tid == 0) t_start = globaltimer_ns();

  // Pacing: while the GEMM still runs, only the first `pace` CTAs consume;
  // the others wait until the last group's flag rises (the GEMM's end) and
  // then take whatever chunks are left, from the first group on.
  bool paced_ok = true;
  if (a.pace > 0 && int32_t(blockIdx.x) >= a.pace && c.g1 > c.g0) {
    if (tid == 0) s_ok = wait_flag(c.flags + (c.g1 - 1), c.epoch, c.limit_ns) ? 1 : 0;
    __syncthreads();
    if (!s_ok) {
      if (tid == 0) atomicCAS(c.status, 0, int32_t(FO_ERR_TIMEOUT));
      paced_ok = false;
    }
  }

  for (int j = c.g0; paced_ok && j < c.g1; ++j) {
    // The group's first chunk is taken, and its unit map computed, before
    // the wait on the group's flag: when the group completes, only the data
    // moves are left.
    const int32_t ub = c.group_unit_begin[j], ue = c.group_unit_begin[j + 1];
    const int32_t n_chunks = (ue - ub + c.chunk_units - 1) / c.chunk_units;
    if (tid == 0) s_chunk[0] = atomicAdd(c.work + j, 1);
    if (tid < c.R) {
      s_ps[tid] = c.part_start[j * c.R + tid];
      s_pl[tid] = c.part_len[j * c.R + tid];
      s_pd[tid] = c.part_dst[j * c.R + tid];
    }
    __syncthreads();
    const int32_t first = s_chunk[0];
    if (!DIRECT && first < n_chunks) {
      const int32_t u0 = ub + first * c.chunk_units;
      map_chunk_units(a, s_map, u0, min(u0 + c.chunk_units, ue), tid);
    }
    if (tid == 0) s_ok = wait_flag(c.flags + j, c.epoch, c.limit_ns) ? 1 : 0;
    __syncthreads();
    if (!s_ok) {
      if (tid == 0) atomicCAS(c.status, 0, int32_t(FO_ERR_TIMEOUT));
      break;
    }
    for (int buf = 0, n = 0;; buf ^= 1, ++n) {
      const int32_t ch = s_chunk[buf];
      if (ch >= n_chunks) break;
      if (tid == 0) s_chunk[buf ^ 1] = atomicAdd(c.work + j, 1);
      const int32_t u0 = ub + ch * c.chunk_units;
      const int32_t u1 = min(u0 + c.chunk_units, ue);
      if constexpr (DIRECT) {
        consume_direct<KIND, U>(a, s_fin, u0 << c.vpu_shift, u1 << c.vpu_shift, tid);
        __syncthreads();   // the next chunk index is visible to the whole CTA
      } else {
        if (n > 0) map_chunk_units(a, s_map, u0, u1, tid);   // the first is mapped
        consume_range<KIND, U>(c, s_ps, s_pl, s_pd, s_dst, u0 << c.vpu_shift,
                               u1 << c.vpu_shift, tid);
        __syncthreads();   // the chunk's stores and its map are visible to the whole CTA
        reorder_chunk_regs<VPU, kNV>(a, s_map, s_dst, s_fin, u1 - u0, tid);
        __syncthreads();   // s_map is free for the next chunk
      }
      if (c.trace != nullptr && tid == 0) {
        const unsigned long long now = globaltimer_ns();
        atomicMax(reinterpret_cast<unsigned long long*>(c.trace + j), now);
        atomicMax(reinterpret_cast<unsigned long long*>(c.trace + c.P + j), now);
        ++chunks_done;
      }
    }
    __syncthreads();
  }
  if (c.trace != nullptr && tid == 0) {
    uint64_t* rec = c.trace + 2 * c.P + 4 * blockIdx.x;
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    rec[0] = smid;
    rec[1] = t_start;
    rec[2] = globaltimer_ns();
    rec[3] = uint64_t(chunks_done);
  }

  // the kernel this one depends on has completed before the shared
  // counters are touched (see consume_kernel)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // every CTA reports; the last one resets this launch's counters
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(c.work + c.P, 1) == int32_t(gridDim.x) - 1) {
      for (int j = c.g0; j < c.g1; ++j) atomicExch(c.work + j, 0);
      atomicExch(c.work + c.P, 0);
    }
  }
}

template <int KIND, int U, int VPU, bool DIRECT>
fo_status launch_fused_kind(const FusedArgs& a, int ctas, bool overlap, int device,
                            cudaStream_t st, int smem) {
  static std::once_flag once[64];
  static cudaError_t err[64];
  const int d = device < 64 ? device : 63;
  std::call_once(once[d], [&] {
    err[d] = cudaFuncSetAttribute(consume_reorder_kernel<KIND, U, VPU, DIRECT>,
                                  cudaFuncAttributePreferredSharedMemoryCarveout,
                                  int(cudaSharedmemCarveoutMaxShared));
  });
  if (err[d] != cudaSuccess) return FO_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(resolve_grid(consume_reorder_kernel<KIND, U, VPU, DIRECT>, ctas, smem));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, consume_reorder_kernel<KIND, U, VPU, DIRECT>, a) != cudaSuccess)
    return FO_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FO_OK : FO_ERR_CUDA;
}

// deep: at most one CTA per SM, so each thread may keep twice the copy
// vectors in flight (the same bytes in flight per SM as two CTAs of 4)
template <int VPU, bool DIRECT>
fo_status launch_fused_vpu(int kind, const FusedArgs& a, int ctas, bool ov, int dv,
                           cudaStream_t st, bool deep, int smem) {
  switch (kind) {
    case FO_CONS_COPY: return launch_fused_kind<FO_CONS_COPY, kFusedUnroll<FO_CONS_COPY>, VPU, DIRECT>(a, ctas, ov, dv, st, smem);
    // the direct sum of at most 4 partials keeps two vectors per source in
    // flight (measured: reducescatter's sum alone 3% faster; the step even)
    case FO_CONS_SUM:
      if constexpr (DIRECT)
        if (a.c.n_partials <= kPartialsInFlight<2>)
          return launch_fused_kind<FO_CONS_SUM, 2, VPU, true>(a, ctas, ov, dv, st, smem);
      return launch_fused_kind<FO_CONS_SUM, kFusedUnroll<FO_CONS_SUM>, VPU, DIRECT>(a, ctas, ov, dv, st, smem);
    case FO_CONS_RS:
      if constexpr (DIRECT)
        if (a.c.n_partials <= kPartialsInFlight<2>)
          return launch_fused_kind<FO_CONS_RS, 2, VPU, true>(a, ctas, ov, dv, st, smem);
      return launch_fused_kind<FO_CONS_RS, kFusedUnroll<FO_CONS_RS>, VPU, DIRECT>(a, ctas, ov, dv, st, smem);
    // the direct bucket runs at one CTA per SM beside the GEMM; there it
    // keeps 8 vectors per thread in flight (72 registers, no spills;
    // measured: alone at that grid 731 -> 568 us on the All-to-All layer, the
    // step no slower).  At 4 CTAs per SM that was slower (0.75 -> 0.64 of the
    // copy bandwidth), so larger grids keep 4.
    case FO_CONS_A2A:
      if constexpr (DIRECT)
        if (deep) return launch_fused_kind<FO_CONS_A2A, 8, VPU, true>(a, ctas, ov, dv, st, smem);
      return launch_fused_kind<FO_CONS_A2A, kFusedUnroll<FO_CONS_A2A>, VPU, DIRECT>(a, ctas, ov, dv, st, smem);
  }
  return FO_ERR_ARG;
}

// With overlap on, the consumer publishes each group's completion (per-group
// finished-chunk counters, then consumed[j] = the launch's sequence number,
// which no earlier launch on the plan used, so a flag left by one never
// passes for the next) for a reorder launched as its programmatic
// dependent.  Serially the reorder follows in stream order and nothing is
// published (the counting costs a fence per CTA and group).
void publish_consumed(const fo_plan* p, ConsumeArgs& a, int32_t* finished) {
  const bool on = p->overlap != 0;
  a.finished = on ? finished : nullptr;
  a.consumed = on ? p->dev.consumed : nullptr;
  if (on) {
    if (++p->consume_seq == 0) p->consume_seq = 1;
    a.seq = p->consume_seq;
  }
  p->consume_published = on;
}

int chunk_units_of(int kind, int tile_n) {
  const int bytes = (kind == FO_CONS_SUM || kind == FO_CONS_RS) ? kChunkBytes<FO_CONS_SUM>
                                                                 : kChunkBytes<FO_CONS_COPY>;
  return bytes / (tile_n * 2);
}

// The direct consumer+reorder's copy takes 16 KB chunks (one pass of its 4
// vectors per thread): the last group, which runs after the GEMM, is then
// shared by twice as many CTAs (measured: wave_pattern's step 1.5 us
// shorter); the bucket keeps 32 KB (no difference), the sums 16 KB.
int direct_chunk_units_of(int kind, int tile_n) {
  return kind == FO_CONS_COPY ? 16 * 1024 / (tile_n * 2) : chunk_units_of(kind, tile_n);
}

int log2_exact(int v) {
  int s = 0;
  while ((1 << s) < v) ++s;
  return s;
}

// Default grids, measured on GB300 beside the signaled GEMM (step time over
// 1, 2, 3 and 4 CTAs per SM): the sums are bandwidth-bound with a load per
// source in flight and want 4 CTAs per SM; the copy and bucket
// consumers keep 8 loads in flight per thread and interfere least with the
// GEMM at 1 per SM; the fused consumer+reorder does best at 3 per SM, and
// so does its direct variant except for the All-to-All bucket, where the
// GEMM dominates the step and 1 CTA per SM slows it least.
int default_ctas(const fo_plan* p, int requested, int kind, bool fused, bool direct) {
  if (requested > 0) return requested;
  // reserved placement: resolved at launch (resolve_grid)
  if (p->consumer_smem > 0) return -reserved_sms(p);
  if (fused) return (direct && kind == FO_CONS_A2A ? 1 : 3) * p->sm_count;
  return (kind == FO_CONS_SUM || kind == FO_CONS_RS) ? 4 * p->sm_count : p->sm_count;
}

// The consumer is launched as a programmatic dependent (when `overlap`):
// after fo_signaled_gemm on the same stream it starts once every GEMM CTA
// is resident and runs alongside it.  Its shared-memory carveout matches the
// GEMM's so its CTAs can share SMs with GEMM CTAs.
template <int KIND, int U>
fo_status launch_consume_kind(const ConsumeArgs& a, int ctas, bool overlap, int device,
                              cudaStream_t st, int smem) {
  static std::once_flag once[64];
  static cudaError_t err[64];
  const int d = device < 64 ? device : 63;
  std::call_once(once[d], [&] {
    err[d] = cudaFuncSetAttribute(consume_kernel<KIND, U>,
                                  cudaFuncAttributePreferredSharedMemoryCarveout,
                                  int(cudaSharedmemCarveoutMaxShared));
  });
  if (err[d] != cudaSuccess) return FO_ERR_CUDA;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(resolve_grid(consume_kernel<KIND, U>, ctas, smem));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, consume_kernel<KIND, U>, a) != cudaSuccess) return FO_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FO_OK : FO_ERR_CUDA;
}

}  // namespace

fo_status launch_consume(const fo_plan* p, int32_t g0, int32_t g1, int kind,
                         const void* src, const void* const* partials,
                         int32_t n_partials, void* const* dst, const uint32_t* flags,
                         uint32_t epoch, uint64_t spin_limit_ns, int32_t* dev_status,
                         void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ConsumeArgs a{};
  a.src = static_cast<const uint4*>(src);
  for (int i = 0; i < n_partials; ++i) a.partials[i] = static_cast<const uint4*>(partials[i]);
  const int n_dst = (kind == FO_CONS_RS || kind == FO_CONS_A2A) ? p->R : 1;
  for (int k = 0; k < n_dst; ++k) a.dst[k] = static_cast<uint4*>(dst[k]);
  a.flags = flags;
  a.status = dev_status;
  a.group_unit_begin = p->dev.group_unit_begin;
  a.part_start = p->dev.part_start;
  a.part_len = p->dev.part_len;
  a.part_dst = p->dev.part_dst;
  a.work = p->dev.work;
  publish_consumed(p, a, p->dev.finished);
  a.g0 = g0;
  a.g1 = g1;
  a.P = p->P;
  a.n_partials = n_partials;
  a.R = (kind == FO_CONS_RS || kind == FO_CONS_A2A) ? p->R : 1;
  a.vpu_shift = log2_exact(p->tile_n / 8);
  a.chunk_units = chunk_units_of(kind, p->tile_n);
  a.epoch = epoch;
  a.limit_ns = spin_limit_ns ? spin_limit_ns : 2000000000ull;
  a.trace = p->consumer_trace;
  const int ctas = default_ctas(p, p->consumer_ctas, kind, false, false);
  const bool ov = p->overlap != 0;
  const int dv = p->device;
  const int smem = p->consumer_smem;
  switch (kind) {
    case FO_CONS_COPY: return launch_consume_kind<FO_CONS_COPY, kUnroll<FO_CONS_COPY>>(a, ctas, ov, dv, st, smem);
    case FO_CONS_SUM: return launch_consume_kind<FO_CONS_SUM, kUnroll<FO_CONS_SUM>>(a, ctas, ov, dv, st, smem);
    case FO_CONS_RS: return launch_consume_kind<FO_CONS_RS, kUnroll<FO_CONS_RS>>(a, ctas, ov, dv, st, smem);
    case FO_CONS_A2A: return launch_consume_kind<FO_CONS_A2A, kUnroll<FO_CONS_A2A>>(a, ctas, ov, dv, st, smem);
  }
  return FO_ERR_ARG;
}

fo_status launch_consume_reorder(const fo_plan* p, int32_t g0, int32_t g1, int kind,
                                 const void* src, const void* const* partials,
                                 int32_t n_partials, void* const* comm_dst,
                                 void* const* final_dst, const void* bias, int act,
                                 const uint32_t* flags, uint32_t epoch, uint64_t spin_limit_ns,
                                 int32_t* dev_status, void* stream) {
  FusedArgs a{};
  ConsumeArgs& c = a.c;
  c.src = static_cast<const uint4*>(src);
  for (int i = 0; i < n_partials; ++i) c.partials[i] = static_cast<const uint4*>(partials[i]);
  const int n_comm = (kind == FO_CONS_RS || kind == FO_CONS_A2A) ? p->R : 1;
  a.direct = comm_dst == nullptr ? 1 : 0;
  // the direct variant names each place in 28 bits of 16-byte vectors
  if (a.direct && !p->place_ok) return FO_ERR_UNSUPPORTED;
  if (comm_dst != nullptr)
    for (int k = 0; k < n_comm; ++k) c.dst[k] = static_cast<uint4*>(comm_dst[k]);
  const int n_fin = p->layout == FO_LAYOUT_TILE ? 1 : p->R;
  for (int k = 0; k < n_fin; ++k) a.fin[k] = static_cast<uint4*>(final_dst[k]);
  c.flags = flags;
  c.status = dev_status;
  c.group_unit_begin = p->dev.group_unit_begin;
  c.part_start = p->dev.part_start;
  c.part_len = p->dev.part_len;
  c.part_dst = p->dev.part_dst;
  c.work = p->dev.work;
  c.g0 = g0;
  c.g1 = g1;
  c.P = p->P;
  c.n_partials = n_partials;
  c.R = n_comm;
  c.vpu_shift = log2_exact(p->tile_n / 8);
  c.chunk_units = comm_dst == nullptr ? direct_chunk_units_of(kind, p->tile_n)
                                      : chunk_units_of(kind, p->tile_n);
  c.epoch = epoch;
  c.limit_ns = spin_limit_ns ? spin_limit_ns : 2000000000ull;
  c.trace = p->consumer_trace;
  a.map = make_row_map(p);
  a.bias = static_cast<const uint16_t*>(bias);
  a.unit_src = p->dev.unit_src;
  a.unit_place = p->dev.unit_place;
  a.act = act;
  a.row_vec = p->N / 8;
  const int ctas = default_ctas(p, p->consumer_ctas, kind, true, a.direct != 0);
  a.pace = (p->overlap != 0 && p->consumer_pace > 0 && p->consumer_pace < ctas)
               ? p->consumer_pace : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool ov = p->overlap != 0;
  const bool deep = ctas > 0 && ctas <= p->sm_count;   // (reserved default: several per SM)
  if (a.direct)
    return p->tile_n == 256 ? launch_fused_vpu<32, true>(kind, a, ctas, ov, p->device, st, deep, p->consumer_smem)
                            : launch_fused_vpu<16, true>(kind, a, ctas, ov, p->device, st, deep, p->consumer_smem);
  return p->tile_n == 256 ? launch_fused_vpu<32, false>(kind, a, ctas, ov, p->device, st, deep, p->consumer_smem)
                          : launch_fused_vpu<16, false>(kind, a, ctas, ov, p->device, st, deep, p->consumer_smem);
}

}  // namespace fo

// ---------------------------------------------------------------------------
// Allocation-free consumer entry point.
//
// Some callers may not allocate device memory at the moment they run the
// overlap: code being captured into a CUDA graph (cudaMalloc is not allowed
// inside a capture), serving runtimes that hand all device memory to their
// own pool and forbid allocations on the request path, and latency-critical
// loops that cannot afford the synchronisation an allocation may cause.
// fo_consume_group keeps its chunk counters in scratch memory that
// fo_plan_groups allocated; this variant keeps them instead in a fixed
// array that lives in the library's own device image, so the call itself
// allocates nothing.  The plan's tables and every buffer are still the
// caller's, created beforehand.

// The shared scratch.  Layout for a plan of P groups (P <= MAX =
// FO_NOALLOC_MAX_GROUPS):
//   [MAX - P, MAX)        chunk counters of groups 0 .. P-1
//   [MAX]                 "CTAs done" counter (the same slot for every plan)
//   [MAX + 1, MAX + 1 + P) finished-chunk counters of groups 0 .. P-1
// Zero when the library is loaded; every launch leaves what it used at zero
// (its last CTA resets it, also after a timeout).  Every GPU that loads the
// library holds the array (32 KB) until the process exits.
static __device__ __align__(256) int32_t fo_noalloc_scratch[2 * FO_NOALLOC_MAX_GROUPS + 1] = {0};

namespace fo {
namespace {

std::mutex g_noalloc_mutex;
int32_t* g_noalloc_addr[64] = {};

// Streams (device, stream) on which a no-alloc consume was launched with no
// ordinary (non-programmatic) library launch after it.  A consume is a
// programmatic dependent launch that lets its own dependents start at once,
// so a second no-alloc consume issued on the same stream -- directly after
// the first, or after a reorder that is in turn the first's dependent --
// could start while the first still runs, and both would take chunks from
// the one array.  Such a consume is launched as an ordinary kernel instead:
// it starts once everything before it on the stream has finished.  An
// ordinary launch (fo_signaled_gemm) ends that: it waits for all earlier
// work, so a consume that depends on it cannot meet an earlier consume.
std::vector<std::pair<int, cudaStream_t>> g_noalloc_pending;

bool noalloc_take_pending(int device, cudaStream_t st) {
  for (auto& e : g_noalloc_pending)
    if (e.first == device && e.second == st) return true;
  g_noalloc_pending.emplace_back(device, st);
  return false;
}

// Device address of fo_noalloc_scratch on the current device.  In host code
// the array's name only stands for it; its address on a device comes from
// cudaGetSymbolAddress, taken once per device with that device current.
fo_status noalloc_scratch(int device, int32_t** out) {
  if (device < 0 || device >= 64) return FO_ERR_UNSUPPORTED;
  if (g_noalloc_addr[device] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, fo_noalloc_scratch) != cudaSuccess) return FO_ERR_CUDA;
    g_noalloc_addr[device] = static_cast<int32_t*>(ptr);
  }
  *out = g_noalloc_addr[device];
  return FO_OK;
}

}  // namespace

void noalloc_note_ordinary_launch(int device, void* stream) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (size_t i = 0; i < g_noalloc_pending.size(); ++i)
    if (g_noalloc_pending[i].first == device && g_noalloc_pending[i].second == st) {
      g_noalloc_pending[i] = g_noalloc_pending.back();
      g_noalloc_pending.pop_back();
      return;
    }
}

}  // namespace fo

extern "C" fo_status fo_consume_group_noalloc(const fo_plan* p, int32_t group,
                                              fo_consumer kind, const void* src,
                                              const void* const* partials,
                                              int32_t n_partials, void* const* dst,
                                              const uint32_t* flags, uint32_t epoch,
                                              uint64_t spin_limit_ns, int32_t* dev_status,
                                              void* stream) {
  using namespace fo;
  if (!p || !p->blob || !src || !dst || !flags || !dev_status) return FO_ERR_ARG;
  if (!aligned4(flags) || !aligned4(dev_status)) return FO_ERR_ARG;
  if (p->P > FO_NOALLOC_MAX_GROUPS) return FO_ERR_ARG;  // scratch too small for this plan
  if (group < -1 || group >= p->P) return FO_ERR_ARG;
  switch (kind) {
    case FO_CONS_COPY:
      if (n_partials != 0) return FO_ERR_ARG;
      break;
    case FO_CONS_SUM:
      if (n_partials < 0 || n_partials > kMaxPartials) return FO_ERR_ARG;
      break;
    case FO_CONS_RS:
      if (n_partials < 0 || n_partials > kMaxPartials) return FO_ERR_ARG;
      if (p->layout != FO_LAYOUT_RS_SUBTILE && p->layout != FO_LAYOUT_RS_ROWBLOCK)
        return FO_ERR_ARG;
      break;
    case FO_CONS_A2A:
      if (n_partials != 0 || p->layout != FO_LAYOUT_A2A_SUBTOKEN) return FO_ERR_ARG;
      break;
    default: return FO_ERR_ARG;
  }
  if (n_partials > 0 && !partials) return FO_ERR_ARG;
  if (!aligned16(src)) return FO_ERR_ARG;
  for (int i = 0; i < n_partials; ++i)
    if (!partials[i] || !aligned16(partials[i])) return FO_ERR_ARG;
  const int n_dst = (kind == FO_CONS_RS || kind == FO_CONS_A2A) ? p->R : 1;
  for (int k = 0; k < n_dst; ++k)
    if (!dst[k] || !aligned16(dst[k])) return FO_ERR_ARG;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return FO_ERR_CUDA;
  if (device != p->device) return FO_ERR_ARG;  // the plan's device must be current
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  int32_t* scratch = nullptr;
  const fo_status st = noalloc_scratch(device, &scratch);
  if (st != FO_OK) return st;

  ConsumeArgs a{};
  a.src = static_cast<const uint4*>(src);
  for (int i = 0; i < n_partials; ++i) a.partials[i] = static_cast<const uint4*>(partials[i]);
  for (int k = 0; k < n_dst; ++k) a.dst[k] = static_cast<uint4*>(dst[k]);
  a.flags = flags;
  a.status = dev_status;
  a.group_unit_begin = p->dev.group_unit_begin;
  a.part_start = p->dev.part_start;
  a.part_len = p->dev.part_len;
  a.part_dst = p->dev.part_dst;
  // work[j] for j < P just below the fixed "CTAs done" slot work[P] =
  // scratch[MAX]; consumed flags in the plan (allocated when it was built)
  a.work = scratch + (FO_NOALLOC_MAX_GROUPS - p->P);
  publish_consumed(p, a, scratch + FO_NOALLOC_MAX_GROUPS + 1);
  a.g0 = group < 0 ? 0 : group;
  a.g1 = group < 0 ? p->P : group + 1;
  a.P = p->P;
  a.n_partials = n_partials;
  a.R = n_dst;
  a.vpu_shift = log2_exact(p->tile_n / 8);
  a.chunk_units = chunk_units_of(kind, p->tile_n);
  a.epoch = epoch;
  a.limit_ns = spin_limit_ns ? spin_limit_ns : 2000000000ull;
  a.trace = p->consumer_trace;
  const int ctas = default_ctas(p, p->consumer_ctas, kind, false, false);
  // overlap as fo_consume_group does, unless a no-alloc consume launched
  // earlier on this stream may still be running (see g_noalloc_pending)
  const bool ov = p->overlap != 0 && !noalloc_take_pending(device, cs);
  switch (kind) {
    case FO_CONS_COPY: return launch_consume_kind<FO_CONS_COPY, kUnroll<FO_CONS_COPY>>(a, ctas, ov, device, cs, p->consumer_smem);
    case FO_CONS_SUM: return launch_consume_kind<FO_CONS_SUM, kUnroll<FO_CONS_SUM>>(a, ctas, ov, device, cs, p->consumer_smem);
    case FO_CONS_RS: return launch_consume_kind<FO_CONS_RS, kUnroll<FO_CONS_RS>>(a, ctas, ov, device, cs, p->consumer_smem);
    case FO_CONS_A2A: return launch_consume_kind<FO_CONS_A2A, kUnroll<FO_CONS_A2A>>(a, ctas, ov, device, cs, p->consumer_smem);
  }
  return FO_ERR_ARG;
}
