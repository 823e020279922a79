// Post-communication reorder kernel (TMA bulk copies).
//
// Pages: "FlashOverlap: 信号驱动计算通信重叠论文详解" -- 二、重排机制 "解决方案:
// 映射表重排" (after communication the inverse mapping table restores the
// original layout) and Figure 6's per-primitive patterns; "Efficient and
// Adaptable Overlapping ...", Figure 5 ("the tiles are reordered back when
// communication finishes").
//
// A CTA moves one tile at a time through 64 KB of shared memory using the
// Tensor Memory Accelerator, so almost no thread time goes into moving
// bytes:
//  * the tile's rows are contiguous in the communication buffer (one run
//    per destination part), so they arrive with one 1-D bulk copy per run
//    (a per-row copy for the All-to-All layout, whose rows are spread over
//    the receive buffers by rank);
//  * a full tile leaves with one 2-D tensor store of a 128 x tile_n box (a
//    32-row box per subtile for the ReduceScatter layout) into the
//    row-major output; ragged tiles and All-to-All rows leave as per-row
//    512-byte bulk stores.
// Three CTAs per SM keep ~192 KB per SM in flight.  Tiles are handed out in
// launch order by a counter; launched as the consumer's programmatic
// dependent, a CTA waits for its tile's group to be consumed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"
#include "row_map.cuh"
#include "tensor_map.h"

namespace fo {

namespace {

constexpr int kRThreads = kTileM;                  // one thread per tile row
constexpr int kRTileBytes = kTileM * 256 * 2;      // a full 128 x 256 bf16 tile
constexpr int kRSmem = 1024 + kRTileBytes + 64;    // alignment slack, tile, barrier
constexpr uint64_t kRWaitLimitNs = 1000000000ull;  // 1 s per wait

struct ReorderArgs {
  CUtensorMap dst_map[kMaxDest];  // outputs, boxes of box_rows x tile_n
  const uint8_t* src[kMaxDest];
  uint8_t* dst[kMaxDest];
  RowMap map;
  int32_t* status;
  const uint16_t* bias;   // optional bf16[N] added before the activation
  int32_t act;            // fo_activation
  int32_t unit_bytes, row_bytes, slot0, n_slots;
  int32_t* counters;         // [0] next tile, [1] CTAs done (reset by the last CTA)
  uint32_t* consumed;        // non-NULL: wait until consumed[group] == seq
  uint32_t seq;              // the preceding consume launch's number
  int32_t g0, g1;            // the groups this launch covers
};

// Wait (thread 0) until the consumer has finished the tile's group: acquire
// loads with __nanosleep back-off, bounded; gives up at once when another
// CTA already gave up (the status word is set).
__device__ __forceinline__ bool wait_consumed(const ReorderArgs& a, int32_t group) {
  const uint32_t* f = a.consumed + group;
  if (ld_acquire_gpu(f) == a.seq) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t backoff = 64;
  while (true) {
    __nanosleep(backoff);
    if (ld_acquire_gpu(f) == a.seq) return true;
    if (*reinterpret_cast<volatile int32_t*>(a.status) != 0) return false;
    if (globaltimer_ns() - t0 > kRWaitLimitNs) {
      atomicCAS(a.status, 0, int32_t(FO_ERR_TIMEOUT));
      return false;
    }
    if (backoff < 2048) backoff <<= 1;
  }
}

__device__ __forceinline__ void reorder_row(const ReorderArgs& a, const TileInfo& ti, int32_t s,
                                            int32_t r, int* k, int32_t* src_unit,
                                            int32_t* dst_row) {
  map_row(a.map, ti, s, r, k, src_unit, dst_row);
}

__global__ void __launch_bounds__(kRThreads) reorder_kernel(const __grid_constant__ ReorderArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* buf = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(buf + kRTileBytes);
  __shared__ int s_ok, s_ready;   // separate words: no barrier lies between
                                  // the last read of one and the next write
  __shared__ int32_t s_next[2];
  const int tid = threadIdx.x;
  const uint32_t sbuf = smem_u32(buf), sfull = smem_u32(full);
  // overlapped (waiting on the consumer): tiles come from a shared counter
  // in launch order; otherwise CTA b takes tiles b, b + grid, ...
  const bool dyn = a.consumed != nullptr;
  if (tid == 0) {
    mbar_init(sfull, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_next[0] = dyn ? atomicAdd(a.counters, 1) : int32_t(blockIdx.x);
  }
  __syncthreads();
  const int32_t ub = a.unit_bytes;
  const uint64_t pol = l2_evict_first();   // the received data is read once
  uint32_t phase = 0;
  // thread 0 fetches the next index while the CTA works; with the shared
  // counter, CTAs that start early -- beside a running GEMM and consumer --
  // take the groups that finish first
  for (int nb = 0;; nb ^= 1, phase ^= 1) {
    const int32_t t = s_next[nb];
    if (t >= a.n_slots) break;
    const int32_t s = a.slot0 + t;
    const TileInfo ti = a.map.tile[s];
    if (tid == 0) {
      s_next[nb ^ 1] = dyn ? atomicAdd(a.counters, 1) : t + int32_t(gridDim.x);
      int ok = 1;
      if (a.consumed != nullptr) {
        ok = wait_consumed(a, ti.group) ? 1 : 0;
        // the consumer's generic stores are read next by the TMA engine
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      s_ready = ok;
    }
    __syncthreads();
    if (!s_ready) break;
    const bool whole = (a.map.layout == FO_LAYOUT_TILE || a.map.layout == FO_LAYOUT_RS_ROWBLOCK);
    const bool a2a = a.map.layout == FO_LAYOUT_A2A_SUBTOKEN;
    // All-to-All: this thread's row (k = -1: it holds no token, moves nowhere)
    int rk = -1;
    int32_t rsu = 0, rdr = 0;
    if (a2a && tid < ti.rows) reorder_row(a, ti, s, tid, &rk, &rsu, &rdr);
    const int32_t in_rows = a2a ? __syncthreads_count(rk >= 0) : ti.rows;
    // the previous tile's stores have finished reading the buffer
    bulk_wait_read_all();
    __syncthreads();
    if (tid == 0) mbar_expect_tx(sfull, uint32_t(in_rows * ub));
    __syncthreads();
    if (whole) {
      if (tid == 0 && ti.rows > 0) {   // (a padding tile holds no rows)
        int k;
        int32_t su, dr;
        reorder_row(a, ti, s, 0, &k, &su, &dr);   // rows are contiguous from row 0
        bulk_load_hint(sbuf, a.src[k] + int64_t(su) * ub, uint32_t(ti.rows * ub), sfull, pol);
      }
    } else if (a.map.layout == FO_LAYOUT_RS_SUBTILE) {
      if (tid < a.map.R) {   // subtile tid: rows tid*h .. +h, contiguous in slice tid
        int k;
        int32_t su, dr;
        reorder_row(a, ti, s, tid * a.map.h, &k, &su, &dr);
        bulk_load_hint(sbuf + tid * a.map.h * ub, a.src[k] + int64_t(su) * ub,
                       uint32_t(a.map.h * ub), sfull, pol);
      }
    } else if (rk >= 0) {  // All-to-All: row by row
      bulk_load_hint(sbuf + tid * ub, a.src[rk] + int64_t(rsu) * ub, uint32_t(ub), sfull, pol);
    }
    // wait for the tile to land (bounded)
    if (tid == 0) {
      int ok = 1;
      if (!mbar_try_wait(sfull, phase)) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(sfull, phase))
          if (globaltimer_ns() - t0 > kRWaitLimitNs) {
            ok = 0;
            atomicCAS(a.status, 0, int32_t(FO_ERR_TIMEOUT));
            break;
          }
      }
      s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) break;
    if (a.act != FO_ACT_NONE || a.bias != nullptr) {
      // element-wise epilogue in place ([P1] 五: fused with the reorder):
      // row r of the tile is at r * ub in every layout
      const int vpr = ub / 16;
      for (int v = tid; v < ti.rows * vpr; v += kRThreads) {
        const int r = v / vpr, cv = v - r * vpr;
        uint4* pv = reinterpret_cast<uint4*>(buf + r * ub + cv * 16);
        *pv = epilogue8(*pv, a.bias, ti.col0 + cv * 8, a.act);
      }
      // generic writes to shared memory, read next by the TMA engine
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
    }
    if (whole && ti.rows == kTileM) {
      if (tid == 0) {
        int k;
        int32_t su, dr;
        reorder_row(a, ti, s, 0, &k, &su, &dr);
        tensor_store_2d(&a.dst_map[k], sbuf, ti.col0, dr);
        bulk_commit();
      }
    } else if (a.map.layout == FO_LAYOUT_RS_SUBTILE) {
      if (tid < a.map.R) {
        int k;
        int32_t su, dr;
        reorder_row(a, ti, s, tid * a.map.h, &k, &su, &dr);
        tensor_store_2d(&a.dst_map[k], sbuf + tid * a.map.h * ub, ti.col0, dr);
        bulk_commit();
      }
    } else if (a2a) {  // All-to-All rows: per row
      if (rk >= 0) {
        bulk_store(a.dst[rk] + int64_t(rdr) * a.row_bytes + int64_t(ti.col0) * 2,
                   sbuf + tid * ub, uint32_t(ub));
        bulk_commit();
      }
    } else if (tid < ti.rows) {  // ragged tiles: per row
      int k;
      int32_t su, dr;
      reorder_row(a, ti, s, tid, &k, &su, &dr);
      bulk_store(a.dst[k] + int64_t(dr) * a.row_bytes + int64_t(ti.col0) * 2, sbuf + tid * ub,
                 uint32_t(ub));
      bulk_commit();
    }
  }
  // every store has completed before the CTA (and its shared memory) ends
  bulk_wait_all();
  // Launched as the consumer's programmatic dependent, this grid completes
  // only after the consumer has: a later launch on the stream (a consume of
  // the next group) then never meets the consumer still running.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the last CTA resets the tile counter for the next launch
  if (!dyn) return;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.counters + 1, 1) == int32_t(gridDim.x) - 1) {
      // every tile is done: clear the groups' consumed flags too, so a
      // launch that carries the same sequence number (a replayed graph)
      // waits for its own consumer
      for (int32_t j = a.g0; j < a.g1; ++j) atomicExch(a.consumed + j, 0u);
      atomicExch(a.counters, 0);
      atomicExch(a.counters + 1, 0);
    }
  }
}

}  // namespace

fo_status launch_reorder_back(const fo_plan* p, int32_t g0, int32_t g1,
                              const void* const* src, void* const* dst, const void* bias,
                              int act, void* stream) {
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  const int dv = p->device < 64 ? p->device : 63;
  std::call_once(once[dv], [&] {
    attr_err[dv] = cudaFuncSetAttribute(reorder_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
  });
  if (attr_err[dv] != cudaSuccess) return FO_ERR_CUDA;

  ReorderArgs a{};
  const int n = p->layout == FO_LAYOUT_TILE ? 1 : p->R;
  for (int k = 0; k < n; ++k) {
    if ((reinterpret_cast<uintptr_t>(src[k]) | reinterpret_cast<uintptr_t>(dst[k])) & 15)
      return FO_ERR_ARG;
    a.src[k] = static_cast<const uint8_t*>(src[k]);
    a.dst[k] = static_cast<uint8_t*>(dst[k]);
    if (p->layout != FO_LAYOUT_A2A_SUBTOKEN) {
      const int box_rows = p->layout == FO_LAYOUT_RS_SUBTILE ? kTileM / p->R : kTileM;
      if (!encode_tensor_map_2d(&a.dst_map[k], dst[k], uint64_t(p->N),
                                uint64_t(p->final_rows[k]), uint32_t(p->tile_n),
                                uint32_t(box_rows), false))
        return FO_ERR_CUDA;
    }
  }
  a.map = make_row_map(p);
  a.status = p->dev.gemm_status;
  a.bias = static_cast<const uint16_t*>(bias);
  a.act = act;
  a.unit_bytes = p->tile_n * 2;
  a.row_bytes = p->N * 2;
  a.slot0 = p->group_slot_begin[g0];
  a.n_slots = p->group_slot_begin[g1] - a.slot0;
  a.counters = p->dev.rtile;
  a.g0 = g0;
  a.g1 = g1;
  int ctas = p->reorder_ctas > 0 ? p->reorder_ctas : 3 * p->sm_count;
  if (ctas > a.n_slots) ctas = a.n_slots;
  // With overlap on, the reorder is a programmatic dependent of the
  // consumer launched just before it on the stream: its CTAs start once all
  // the consumer's CTAs are resident (on SMs the GEMM leaves room on) and
  // move each group as soon as the consumer has finished it.
  const bool ov = p->overlap != 0 && p->consume_published;
  if (ov) {
    a.consumed = p->dev.consumed;
    a.seq = p->consume_seq;
    // this launch clears the consumed flags once it has used them: a later
    // reorder without a consume in between runs as an ordinary launch
    p->consume_published = false;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = kRSmem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = ov ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, reorder_kernel, a) != cudaSuccess) return FO_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FO_OK : FO_ERR_CUDA;
}

namespace {

struct GatherArgs {
  const uint4* src[kMaxDest];
  uint4* out;
  const uint16_t* bias;
  int32_t act, layout, h, rows_per, row_vec;
  int64_t total;  // 16-byte vectors of the M x N output
};

// The AllGather stand-in and the local row exchange in one pass ([P1] 二 (2):
// after ReduceScatter + AllGather the rows are fixed by a block-cyclic
// permutation that needs no mapping table and fuses with element-wise
// operations).  Output row g takes row rho of slice k:
//   subtile layout: g = tile_m * tm + h * k + i  <-  rho = h * tm + i
//   row-block layout: g = k * M/R + rho
// Both sides are read and written as contiguous rows (16-byte vectors,
// four in flight per thread).
__global__ void __launch_bounds__(256) allgather_kernel(const __grid_constant__ GatherArgs a) {
  constexpr int U = 4;
  __shared__ const uint4* s_src[kMaxDest];
  if (threadIdx.x < kMaxDest) s_src[threadIdx.x] = a.src[threadIdx.x];
  __syncthreads();
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t base = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; base < a.total;
       base += stride * U) {
    uint4 x[U];
    int32_t col[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + stride * u;
      if (v >= a.total) break;
      const int32_t g = int32_t(v / a.row_vec), cv = int32_t(v - int64_t(g) * a.row_vec);
      int32_t k, rho;
      if (a.layout == FO_LAYOUT_RS_SUBTILE) {
        const int32_t tm = g / kTileM, w = g - tm * kTileM;
        k = w / a.h;
        rho = tm * a.h + (w - k * a.h);
      } else {
        k = g / a.rows_per;
        rho = g - k * a.rows_per;
      }
      x[u] = ld_cg(s_src[k] + int64_t(rho) * a.row_vec + cv);
      col[u] = cv * 8;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = base + stride * u;
      if (v >= a.total) break;
      uint4 y = x[u];
      if (a.act != FO_ACT_NONE || a.bias != nullptr) y = epilogue8(y, a.bias, col[u], a.act);
      st_cs(a.out + v, y);
    }
  }
}

}  // namespace

fo_status launch_allgather_rows(const fo_plan* p, const void* const* slices, void* out,
                                const void* bias, int act, void* stream) {
  GatherArgs a{};
  for (int k = 0; k < p->R; ++k) a.src[k] = static_cast<const uint4*>(slices[k]);
  a.out = static_cast<uint4*>(out);
  a.bias = static_cast<const uint16_t*>(bias);
  a.act = act;
  a.layout = p->layout;
  a.h = kTileM / p->R;
  a.rows_per = p->M / p->R;
  a.row_vec = p->N / 8;
  a.total = int64_t(p->M) * a.row_vec;
  const int ctas = 4 * p->sm_count;
  allgather_kernel<<<ctas, 256, 0, static_cast<cudaStream_t>(stream)>>>(a);
  return cudaGetLastError() == cudaSuccess ? FO_OK : FO_ERR_CUDA;
}

}  // namespace fo
