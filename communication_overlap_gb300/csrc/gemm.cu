// The signaled GEMM: one persistent, warp-specialised tcgen05 kernel for
// sm_103a whose epilogue performs the pre-communication reorder and raises
// the wave-group signal.
//
// Pages: "FlashOverlap: 信号驱动计算通信重叠论文详解" -- 核心设计 "计算侧" (the GEMM
// stays a single kernel, not split), 一、信号机制 "实现方法: 组级 Tile 计数" (each
// finished tile adds 1 to its group's entry of the counting table; reaching
// |G_j| starts G_j's communication), 二、重排机制 (finished tiles are written to
// the contiguous range of their group), 五、CUTLASS 扩展实现 "Epilogue 集成"
// (the signal and the reorder live in the epilogue).  "Efficient and
// Adaptable Overlapping ...", Figure 5: reorder, then signal.
//
// Design for GB300 (the pages' CUTLASS kernel targets sm_80/sm_89):
//  * W persistent CTAs, one per SM; CTA c computes launch slots c, c+W, ...
//    so wave k is the k-th tile of every CTA (wave = slot / W exactly).
//  * warp 0: TMA producer; A tile 128x64 (K-major) and B tile 64xBN
//    (N-major) per stage, 128-byte swizzle, no multicast.
//  * warp 1: allocates tensor memory and issues tcgen05.mma (M=128, N=BN,
//    K=16, bf16 in, fp32 accumulate) from one thread; two accumulators of
//    BN columns so tile i+1's main loop runs while tile i drains.
//  * warps 2-5: epilogue; tcgen05.ld 32 lanes x 64 columns, round to bf16,
//    transpose through a swizzled 4 KB staging buffer per warp, and store
//    whole 128-byte row segments to the rows' units in C_r; then one
//    acq_rel atomic on the group's counter and, for the group's last tile,
//    a release store of the epoch into the group's flag.
//  * Every mbarrier wait is bounded (globaltimer); a wait that runs out
//    records FO_ERR_TIMEOUT in the plan's status word and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "device_common.cuh"
#include "tensor_map.h"

namespace fo {

namespace {

constexpr int kGemmThreads = 192;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait

// PAIR: two CTAs of a cluster compute vertically adjacent 128 x BN tiles with
// one tcgen05.mma.cta_group::2 (M = 256): each CTA stages its own A rows
// and half of B's columns, so a CTA loads 32 KB per 64-deep k-block instead
// of 48 KB (BN = 256).
template <int BN, bool PAIR>
struct Cfg {
  static constexpr int kBCols = PAIR ? BN / 2 : BN;       // B columns this CTA stages
  static constexpr int kABytes = kTileM * kBlockK * 2;
  static constexpr int kBBytes = kBlockK * kBCols * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  // as many stages as fit in 192 KB (4 of 48 KB, 6 of 32 KB, 8 of 24 KB)
  static constexpr int kStages = (196608 / kStageBytes) < 8 ? (196608 / kStageBytes) : 8;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kStagingBytes = 4 * 32 * 128;
  static constexpr int kBarOffset = kStages * kStageBytes + kStagingBytes;
  static constexpr int kSmemBytes = 1024 + kBarOffset + 256;
  static constexpr int kMmaM = PAIR ? 2 * kTileM : kTileM;
  // instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (bits
  // 7-9 = 1), B bf16 (bits 10-12 = 1), A K-major (bit 15 = 0), B MN-major
  // (bit 16 = 1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                     (uint32_t(BN >> 3) << 17) |
                                     (uint32_t(kMmaM >> 4) << 24);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(2 * kStages + 8 + 4 <= 32, "barrier area");
  // a split tile's partial sums, a quarter (32 rows) per epilogue warp, are
  // received into the pipeline stages (idle by then)
  static constexpr int kQuarterBytes = 32 * BN * 4;
  static_assert(4 * kQuarterBytes <= kStages * kStageBytes, "partial sums fit the stages");
  // when a quarter fills exactly one stage (pairs, BN = 256), the producer
  // receives quarter q into stage q as soon as that stage's last k-block has
  // been consumed, overlapping the copies with the owner's last MMAs
  static constexpr bool kEarlyPartial = kStageBytes == kQuarterBytes && kStages >= 4;
};

struct GemmArgs {
  CUtensorMap tmap_a;
  CUtensorMap tmap_b[kMaxExperts];
  const TileInfo* tile;
  const int32_t* group_tiles;
  const int32_t* dest_base;
  const int32_t* row_dest;
  const int32_t* row_rank;
  const int32_t* slot_live;  // A2A: [tiles] 0 = no row of the tile holds a token
  uint16_t* c_r;
  int32_t* count;
  uint32_t* count_ready;  // = seq once CTA 0 has zeroed count[0 .. P)
  int32_t* exit_count;    // CTAs finished; the last withdraws count_ready
  int32_t n_groups;
  uint32_t* flags;
  int32_t* status;
  uint64_t* trace;  // optional: [tiles] tile done times, then [grid] CTA starts
  // last-wave split (split_n > 0): the last wave's split_n tiles, from slot
  // split_slot0 on, are each computed by two CTAs over halves of K
  float4* split_ws;       // [split_n][4 quarters][BN / 64][16][32] fp32 partials
  uint32_t* split_flag;   // [split_n * 4] = seq once a quarter's partial is written
  int32_t split_n, split_slot0, split_wave;
  uint32_t seq;           // this launch's number on the plan (never 0)
  int32_t tiles, k_blocks, layout, R, h;
  uint32_t epoch;
};

// ---------------------------------------------------------------- PTX wrappers

// Bounded wait for the phase with the given parity.  Gives up when another
// role aborted (shared flag) or after kWaitLimitNs; then records the error.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicCAS(status, 0, int32_t(FO_ERR_TIMEOUT));
      return false;
    }
  }
}

// The same, with the first attempt inline: the pipeline loops call it once
// per k-block and almost always find the phase complete.
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag, int32_t* status) {
  return mbar_try_wait(bar, parity) || mbar_wait(bar, parity, abort_flag, status);
}

// Bounded wait that ignores the abort flag (used while winding down).
__device__ __noinline__ bool mbar_wait_plain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// TMA tile loads carry an L2 cache policy (`policy`, from createpolicy).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address >> 4 at bits
// 0-13, leading byte offset >> 4 at 16-29, stride byte offset >> 4 at
// 32-45, version 1 at bits 46-47, layout 2 (128-byte swizzle) at 61-63.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((addr >> 4) & 0x3FFF) | (uint64_t((lbo >> 4) & 0x3FFF) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFF) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- CTA pairs

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
               : "memory");
}

// Arrive on the leader's full barrier announcing this CTA's TMA bytes.  No
// release ordering is needed (the data is tracked by the transaction count),
// and a release at cluster scope would fence the producer on every stage.
__device__ __forceinline__ void mbar_expect_tx_cluster_relaxed(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(
                   addr),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on the
// pair leader's mbarrier (`bar` is a cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int32_t c0, int32_t c1,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Commit the pair's MMAs to the mbarrier at `bar` in both CTAs.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(uint16_t(3))
      : "memory");
}

// ---------------------------------------------------------------- the kernel

// Unit (row of the reordered buffer) of row r of a tile, or -1 past its rows
// (and, in the All-to-All layout, for a row that holds no token).
__device__ __forceinline__ int32_t row_unit(const GemmArgs& a, const TileInfo& ti, int32_t slot,
                                            int32_t r) {
  if (r >= ti.rows) return -1;
  if (a.layout == FO_LAYOUT_RS_SUBTILE) {
    const int32_t k = r / a.h;
    return ti.unit_base + k * ti.sub_stride + (r - k * a.h);
  }
  if (a.layout == FO_LAYOUT_A2A_SUBTOKEN) {
    const int32_t rho = ti.row0 + r;
    const int32_t d = a.row_dest[rho];
    if (d < 0) return -1;   // the row holds no token: it is sent nowhere
    return a.dest_base[slot * a.R + d] + a.row_rank[rho];
  }
  return ti.unit_base + r;
}

// One item of a CTA's work: the tile at `slot`, k-blocks [kb0, kb1), and
// its role: 0 a whole tile; 1 the owner of a split tile (first half of K;
// adds the helper's partial before its epilogue stores, then counts the
// tile); 2 the helper (second half of K; hands over its fp32 partial).
struct Work {
  int32_t slot, kb0, kb1, role;
};

// Item k of this CTA.  CTA c takes slots c, c + W, ... (wave = slot / W).
// When the last wave holds n <= W / 2 tiles, its tile c < n is split: CTA c
// computes the first half of K and CTA c + n (idle in that wave otherwise)
// the second.  With pairs n is even, so both CTAs of a pair help the two
// vertically adjacent tiles of one owner pair.
__device__ __forceinline__ bool next_work(const GemmArgs& a, int32_t k, Work& w) {
  const int32_t c = blockIdx.x, W = gridDim.x;
  if (a.split_n > 0 && k == a.split_wave) {
    // the owner takes 9/16 of K: the helper also has to hand its partial
    // sums over, so with equal halves the owner would wait for it
    const int32_t half = (a.k_blocks * 9 + 8) / 16;
    if (c < a.split_n) {
      w = Work{a.split_slot0 + c, 0, half, 1};
      return true;
    }
    if (c < 2 * a.split_n) {
      w = Work{a.split_slot0 + c - a.split_n, half, a.k_blocks, 2};
      return true;
    }
    return false;
  }
  const int32_t slot = c + k * W;
  if (slot >= a.tiles) return false;
  w = Work{slot, 0, a.k_blocks, 0};
  return true;
}

// The counting table is reset by the kernel itself: CTA 0 zeroes it at its
// start and publishes count_ready = seq; a CTA's first count waits (bounded)
// for that, which by then -- after its first tile -- has long happened.
__device__ __forceinline__ bool count_table_ready(const GemmArgs& a, bool& seen,
                                                  volatile int* abort_flag) {
  if (seen) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(a.count_ready) != a.seq) {
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicCAS(a.status, 0, int32_t(FO_ERR_TIMEOUT));
      return false;
    }
    __nanosleep(64);
  }
  seen = true;
  return true;
}

// Bounded wait (lane 0) for a helper's partial: flag == seq.
__device__ __noinline__ bool wait_partial(const uint32_t* flag, uint32_t seq,
                                          volatile int* abort_flag, int32_t* status) {
  if (ld_acquire_gpu(flag) == seq) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_gpu(flag) == seq) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicCAS(status, 0, int32_t(FO_ERR_TIMEOUT));
      return false;
    }
  }
}

// A tile none of whose rows holds a token (All-to-All capacity the routing
// left empty) has no output: its loads and MMAs are skipped and the tile is
// only counted.  A pair computes its two tiles with one MMA, so it skips only
// when both are empty (slots 2i and 2i+1; the partner is slot ^ 1).
template <bool PAIR>
__device__ __forceinline__ bool tile_skipped(const GemmArgs& a, int32_t slot) {
  if (a.slot_live == nullptr) return false;
  if (PAIR) return (a.slot_live[slot] | a.slot_live[slot ^ 1]) == 0;
  return a.slot_live[slot] == 0;
}

// 192 threads; registers capped at 112 so that two 256-thread consumer CTAs
// at 72 registers fit beside a GEMM CTA on an SM.
template <int BN, bool PAIR>
__global__ void __maxnreg__(112) signaled_gemm_kernel(const __grid_constant__ GemmArgs a) {
  using C = Cfg<BN, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle atoms (the same offsets in
  // both CTAs of a pair: the pair's MMA reads both at the leader's offsets)
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + C::kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* full = bars;                         // PAIR: used in the leader only
  uint64_t* empty = bars + C::kStages;
  uint64_t* acc_full = bars + 2 * C::kStages;
  uint64_t* acc_empty = bars + 2 * C::kStages + 2;   // PAIR: leader's counts both CTAs
  uint64_t* epi_done = bars + 2 * C::kStages + 4;
  uint64_t* drain = bars + 2 * C::kStages + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::kStages + 7);
  uint64_t* part_bar = bars + 2 * C::kStages + 8;   // [4] a quarter of partial sums landed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = PAIR ? cluster_rank() : 0;   // 0 = the pair's leader

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), PAIR ? 2 : 1);   // one producer per CTA
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&acc_full[b]), 1);
      mbar_init(smem_u32(&acc_empty[b]), PAIR ? 8 : 4);   // epilogue warps
      mbar_init(smem_u32(&epi_done[b]), 4);
    }
    mbar_init(smem_u32(drain), 1);
    for (int b = 0; b < 4; ++b) mbar_init(smem_u32(&part_bar[b]), 1);
    if (blockIdx.x == 0 && a.count != nullptr) {
      // [P1] 一 "组级 Tile 计数": the counting table starts at [0, ..., 0].
      // The flags are cleared too, before any consumer of this launch can
      // start (it starts once every CTA has passed launch_dependents below),
      // so a step replayed with the same epoch -- a captured CUDA graph --
      // never sees the previous replay's flags.
      for (int j = 0; j < a.n_groups; ++j) {
        a.count[j] = 0;
        a.flags[j] = 0;
      }
      __threadfence();
      st_release_gpu(a.count_ready, a.seq);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    prefetch_tmap(&a.tmap_a);
  }
  if (warp == 1) {
    // PAIR: one warp in each CTA of the pair allocates collectively; both
    // get the same columns in their own tensor memory
    if constexpr (PAIR) {
      asm volatile(
          "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
              smem_u32(tmem_slot)),
          "r"(uint32_t(C::kTmemCols))
          : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile(
          "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
              smem_u32(tmem_slot)),
          "r"(uint32_t(C::kTmemCols))
          : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();   // the peer's barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // This CTA is resident: a consumer launched as a programmatic dependent of
  // this grid may start once every CTA got here, so it can never hold an SM
  // that a GEMM CTA still needs while it waits for that CTA's tiles.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.trace != nullptr && threadIdx.x == 0) a.trace[a.tiles + blockIdx.x] = globaltimer_ns();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int64_t issued = 0;
      // A and B tiles are reused by the other tiles of their band and column
      // and the consumer's streams pass through L2 beside them (read once,
      // evict-first): keep the operands, evict them last.  Measured: the
      // overlapped step 1-2% shorter on every workload.
      uint64_t keep;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
      Work wk;
      int32_t owner_slot = -1;   // the split tile this CTA owns (its last item)
      for (int32_t item = 0; ok && next_work(a, item, wk); ++item) {
        const int32_t slot = wk.slot;
        const TileInfo ti = a.tile[slot];
        const CUtensorMap* mb = &a.tmap_b[ti.expert];
        if (item == 0)
          for (int e = 0; e <= ti.expert; ++e) prefetch_tmap(&a.tmap_b[e]);
        if (tile_skipped<PAIR>(a, slot)) continue;
        if (wk.role == 1) owner_slot = slot;
        for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
          if (!mbar_wait_fast(smem_u32(&empty[stage]), phase ^ 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
          if constexpr (PAIR) {
            // this CTA's A rows and its half of B land in its own shared
            // memory; the leader's full barrier counts both CTAs' bytes
            const uint32_t fb = map_to_rank(smem_u32(&full[stage]), 0);
            if (rank == 0)
              mbar_expect_tx(smem_u32(&full[stage]), C::kStageBytes);
            else
              mbar_expect_tx_cluster_relaxed(fb, C::kStageBytes);
            tma_load_2d_pair(sa, &a.tmap_a, fb, kb * kBlockK, ti.row0, keep);
#pragma unroll
            for (int c = 0; c < C::kBCols / 64; ++c)
              tma_load_2d_pair(sb + c * (kBlockK * 128), mb, fb,
                               ti.col0 + int32_t(rank) * C::kBCols + c * 64, kb * kBlockK, keep);
          } else {
            const uint32_t fb = smem_u32(&full[stage]);
            mbar_expect_tx(fb, C::kStageBytes);
            tma_load_2d(sa, &a.tmap_a, fb, kb * kBlockK, ti.row0, keep);
#pragma unroll
            for (int c = 0; c < C::kBCols / 64; ++c)
              tma_load_2d(sb + c * (kBlockK * 128), mb, fb, ti.col0 + c * 64, kb * kBlockK, keep);
          }
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if constexpr (C::kEarlyPartial) {
        if (ok && owner_slot >= 0) {
          // Continue around the ring: each stage is free once the MMA has
          // consumed its last k-block.  Stage q < 4 then receives quarter q
          // of the helper's partial sums (after the helper has published
          // it), while the owner's last MMAs still run; the epilogue waits
          // on part_bar[q].
          const int32_t i = owner_slot - a.split_slot0;
          uint32_t sent = 0;   // quarters whose copy was issued (bit q)
          for (int v = 0; v < C::kStages; ++v) {
            if (!mbar_wait_fast(smem_u32(&empty[stage]), phase ^ 1, abort_flag, a.status)) break;
            if (stage < 4) {
              const int q = stage;
              if (!wait_partial(a.split_flag + i * 4 + q, a.seq, abort_flag, a.status)) break;
              // taken: clear it for the next launch (a replay reuses a.seq)
              *reinterpret_cast<volatile uint32_t*>(a.split_flag + i * 4 + q) = 0u;
              // the helper's generic stores are read next by the TMA engine
              asm volatile("fence.proxy.async.global;" ::: "memory");
              const uint32_t pb = smem_u32(&part_bar[q]);
              mbar_expect_tx(pb, uint32_t(C::kQuarterBytes));
              bulk_load(smem_u32(smem + q * C::kQuarterBytes),
                        a.split_ws + size_t(i * 4 + q) * (BN / 64) * 16 * 32,
                        uint32_t(C::kQuarterBytes), pb);
              sent |= 1u << q;
            }
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          // the copies land before the CTA can exit, whatever happened
          for (int q = 0; q < 4; ++q)
            if ((sent >> q) & 1u) mbar_wait_plain(smem_u32(&part_bar[q]), 0, 10000000ull);
        }
      }
      if (!ok && !PAIR) {
        // wind-down: let copies already issued land before the CTA exits
        for (int st = 0; st < C::kStages; ++st) {
          const int64_t fills = issued / C::kStages + (st < issued % C::kStages ? 1 : 0);
          if (fills > 0)
            mbar_wait_plain(smem_u32(&full[st]), uint32_t((fills - 1) & 1), 10000000ull);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (PAIR: the leader's thread issues the pair's MMAs)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      Work wk;
      for (int32_t item = 0; ok && next_work(a, item, wk); ++item) {
        if (tile_skipped<PAIR>(a, wk.slot)) continue;
        if (!mbar_wait(smem_u32(&acc_empty[acc]), acc_phase ^ 1, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        for (int kb = wk.kb0; kb < wk.kb1; ++kb) {
          if (!mbar_wait_fast(smem_u32(&full[stage]), phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk) {
            // A: K-major, advance 16 elements (32 bytes) inside the swizzle
            // atom; SBO = 8 rows x 128 B.  B: N-major, advance 16 K rows
            // (two 1 KB atoms); LBO = 64 K rows x 128 B between 64-column
            // blocks, SBO = 8 K rows x 128 B.
            const uint64_t ad = smem_desc(sa + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc(sb + kk * 2048, kBlockK * 128, 1024);
            const uint32_t accumulate = (kb != wk.kb0 || kk != 0) ? 1u : 0u;
            if constexpr (PAIR)
              mma_bf16_pair(d_tmem, ad, bd, C::kIdesc, accumulate);
            else
              mma_bf16(d_tmem, ad, bd, C::kIdesc, accumulate);
          }
          if constexpr (PAIR)
            mma_commit_pair(smem_u32(&empty[stage]));
          else
            mma_commit(smem_u32(&empty[stage]));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          mma_commit_pair(smem_u32(&acc_full[acc]));
        else
          mma_commit(smem_u32(&acc_full[acc]));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stage_buf = staging + (warp - 2) * (32 * 128);
    const uint32_t stage_base = smem_u32(stage_buf);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool count_seen = false;   // (warp 2, lane 0) the table was reset
    Work wk;
    for (int32_t item = 0; next_work(a, item, wk); ++item) {
      const int32_t slot = wk.slot;
      const TileInfo ti = a.tile[slot];
      if (tile_skipped<PAIR>(a, slot)) {
        // nothing computed, nothing stored: only counted (and signalled),
        // by its owner
        if (warp == 2 && lane == 0 && wk.role != 2) {
          if (a.count != nullptr && count_table_ready(a, count_seen, abort_flag)) {
            const int32_t old = atom_add_acq_rel_gpu(a.count + ti.group, 1);
            if (old + 1 == a.group_tiles[ti.group]) st_release_gpu(a.flags + ti.group, a.epoch);
          }
          if (a.trace != nullptr) a.trace[slot] = globaltimer_ns();
        }
        __syncwarp();
        continue;
      }
      const int32_t my_unit = row_unit(a, ti, slot, q * 32 + lane);
      // one lane waits, the decision is warp-uniform (tcgen05.ld is .aligned)
      int ok = 0;
      if (lane == 0) ok = mbar_wait(smem_u32(&acc_full[acc]), acc_phase, abort_flag, a.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // a split tile's quarter q of the partial sums: [chunk][16 x 4 cols][lane]
      float4* part = nullptr;
      uint32_t* part_flag = nullptr;
      if (wk.role != 0) {
        const int32_t i = slot - a.split_slot0;
        part = a.split_ws + size_t(i * 4 + q) * (BN / 64) * 16 * 32;
        part_flag = a.split_flag + i * 4 + q;
      }
      // The owner waits for the helper's quarter and copies it (TMA, one
      // bulk copy per warp) into the pipeline stages: this is the CTA's last
      // item, so once its accumulator is full no stage is read or filled any
      // more.
      const float* part_smem = reinterpret_cast<const float*>(smem + q * C::kQuarterBytes);
      if (wk.role == 1) {
        if (a.trace != nullptr && lane == 0 && q == 0)   // the owner's half is computed
          a.trace[a.tiles + gridDim.x + 2 * (slot - a.split_slot0) + 1] = globaltimer_ns();
        const uint32_t pb = smem_u32(&part_bar[q]);
        if constexpr (!C::kEarlyPartial) {   // (else the producer sends it)
          if (lane == 0) {
            ok = wait_partial(part_flag, a.seq, abort_flag, a.status);
            if (ok) {
              // taken: clear it for the next launch (a replay reuses a.seq)
              *reinterpret_cast<volatile uint32_t*>(part_flag) = 0u;
              // the helper's generic stores are read next by the TMA engine
              asm volatile("fence.proxy.async.global;" ::: "memory");
              mbar_expect_tx(pb, uint32_t(C::kQuarterBytes));
              bulk_load(smem_u32(part_smem), part, uint32_t(C::kQuarterBytes), pb);
              ok = mbar_wait(pb, 0, abort_flag, a.status);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        // every lane observes the completed copy before reading it
        if (!mbar_wait(pb, 0, abort_flag, a.status)) break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
      if (wk.role == 2) {
        // the helper: hand this lane's row of fp32 partial sums over (each
        // warp instruction writes 512 contiguous bytes), then release the
        // accumulator and publish the quarter
#pragma unroll 1
        for (int cc = 0; cc < BN / 64; ++cc) {
          uint32_t v0[32], v1[32];
          tmem_ld32(t_row + cc * 64, v0);
          tmem_ld32(t_row + cc * 64 + 32, v1);
          tmem_wait_ld();
          float4* dst = part + cc * 16 * 32 + lane;
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const uint32_t* src = (c4 < 8) ? &v0[c4 * 4] : &v1[(c4 - 8) * 4];
            __stcg(dst + c4 * 32, make_float4(__uint_as_float(src[0]), __uint_as_float(src[1]),
                                              __uint_as_float(src[2]), __uint_as_float(src[3])));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          st_release_gpu(part_flag, a.seq);
          if (a.trace != nullptr && q == 0)   // when the helper handed its partial over
            a.trace[a.tiles + gridDim.x + 2 * (slot - a.split_slot0)] = globaltimer_ns();
          mbar_arrive(smem_u32(&epi_done[acc]));
          if (PAIR && rank != 0)
            mbar_arrive_cluster(map_to_rank(smem_u32(&acc_empty[acc]), 0));
          else
            mbar_arrive(smem_u32(&acc_empty[acc]));
        }
        __syncwarp();
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
        continue;
      }
#pragma unroll 1
      for (int cc = 0; cc < BN / 64; ++cc) {
        uint32_t v0[32], v1[32];
        tmem_ld32(t_row + cc * 64, v0);
        tmem_ld32(t_row + cc * 64 + 32, v1);
        tmem_wait_ld();
        if (wk.role == 1) {   // add the helper's half of K (fp32, from shared memory)
          const float4* src = reinterpret_cast<const float4*>(part_smem) + cc * 16 * 32 + lane;
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4) {
            const float4 h = src[c4 * 32];
            uint32_t* d = (c4 < 8) ? &v0[c4 * 4] : &v1[(c4 - 8) * 4];
            d[0] = __float_as_uint(__uint_as_float(d[0]) + h.x);
            d[1] = __float_as_uint(__uint_as_float(d[1]) + h.y);
            d[2] = __float_as_uint(__uint_as_float(d[2]) + h.z);
            d[3] = __float_as_uint(__uint_as_float(d[3]) + h.w);
          }
        }
        // round to bf16 and write this lane's row (128 B) into the staging
        // buffer, 16-byte pieces rotated by row to spread the banks
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* src = (c < 4) ? &v0[c * 8] : &v1[(c - 4) * 8];
          uint32_t w0 = pack_bf16x2(__uint_as_float(src[0]), __uint_as_float(src[1]));
          uint32_t w1 = pack_bf16x2(__uint_as_float(src[2]), __uint_as_float(src[3]));
          uint32_t w2 = pack_bf16x2(__uint_as_float(src[4]), __uint_as_float(src[5]));
          uint32_t w3 = pack_bf16x2(__uint_as_float(src[6]), __uint_as_float(src[7]));
          const uint32_t off = lane * 128 + ((c ^ (lane & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage_base + off),
                       "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                       : "memory");
        }
        __syncwarp();
        // read back four rows per instruction (8 lanes x 16 B = 128 B each)
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int row = it * 4 + (lane >> 3);
          const int piece = lane & 7;
          const int32_t u = __shfl_sync(0xffffffffu, my_unit, row);
          uint32_t w0, w1, w2, w3;
          const uint32_t off = row * 128 + ((piece ^ (row & 7)) << 4);
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                       : "r"(stage_base + off)
                       : "memory");
          if (u >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(a.c_r + int64_t(u) * BN + cc * 64 + piece * 8);
            *dst = make_uint4(w0, w1, w2, w3);
          }
        }
        __syncwarp();
      }
      // This warp's rows are stored: report it, then hand the accumulator
      // back to the MMA warp.  (The accumulator is released only after the
      // report, so no warp can report a later tile on this barrier before
      // every warp reported this one.)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&epi_done[acc]));
        if (PAIR && rank != 0)
          mbar_arrive_cluster(map_to_rank(smem_u32(&acc_empty[acc]), 0));
        else
          mbar_arrive(smem_u32(&acc_empty[acc]));
      }
      // Once all four warps have stored the tile, count it; the group's last
      // tile raises the group's flag.
      if (warp == 2 && lane == 0 && (a.count != nullptr || a.trace != nullptr)) {
        if (mbar_wait(smem_u32(&epi_done[acc]), acc_phase, abort_flag, a.status)) {
          if (a.count != nullptr && count_table_ready(a, count_seen, abort_flag)) {
            __threadfence();
            const int32_t old = atom_add_acq_rel_gpu(a.count + ti.group, 1);
            if (old + 1 == a.group_tiles[ti.group]) st_release_gpu(a.flags + ti.group, a.epoch);
          }
          if (a.trace != nullptr) a.trace[slot] = globaltimer_ns();
        }
      }
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  // Every tile of this CTA is counted.  The last CTA to get here withdraws
  // the table-ready word, so the next launch's CTAs wait for its own reset
  // even when it carries the same sequence number (a replayed graph).
  if (threadIdx.x == 0 && a.count != nullptr) {
    __threadfence();
    if (atomicAdd(a.exit_count, 1) == int32_t(gridDim.x) - 1) {
      atomicExch(a.count_ready, 0u);
      atomicExch(a.exit_count, 0);
    }
  }
  if (warp == 1) {
    // every MMA has completed before the tensor memory is released
    // (immediate on the normal path: the epilogue saw them all)
    if (lane == 0) {
      if constexpr (PAIR) {
        if (rank == 0) mma_commit_pair(smem_u32(drain));
      } else {
        mma_commit(smem_u32(drain));
      }
      mbar_wait_plain(smem_u32(drain), 0, 10000000ull);
    }
    __syncwarp();
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();   // neither CTA leaves while the pair still works
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(uint32_t(C::kTmemCols))
                   : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(uint32_t(C::kTmemCols))
                   : "memory");
  }
}

// ---------------------------------------------------------------- host side

template <int BN, bool PAIR>
fo_status launch_bn(const fo_plan* p, GemmArgs& a, cudaStream_t st) {
  static std::once_flag attr_once[64];
  static cudaError_t attr_err[64];
  const int dev = p->device < 64 ? p->device : 63;
  std::call_once(attr_once[dev], [&] {
    attr_err[dev] = cudaFuncSetAttribute(signaled_gemm_kernel<BN, PAIR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<BN, PAIR>::kSmemBytes);
  });
  if (attr_err[dev] != cudaSuccess) return FO_ERR_CUDA;
  const int grid = p->W < p->tiles ? p->W : p->tiles;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = Cfg<BN, PAIR>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, signaled_gemm_kernel<BN, PAIR>, a) != cudaSuccess)
    return FO_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FO_OK : FO_ERR_CUDA;
}

template <int BN>
int pair_capacity_bn(int device) {
  static std::once_flag once[64];
  static int cap[64];
  const int dev = device < 64 ? device : 63;
  std::call_once(once[dev], [&] {
    cap[dev] = 0;
    if (cudaFuncSetAttribute(signaled_gemm_kernel<BN, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<BN, true>::kSmemBytes) != cudaSuccess)
      return;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = Cfg<BN, true>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, signaled_gemm_kernel<BN, true>, &cfg) ==
        cudaSuccess)
      cap[dev] = 2 * clusters;
  });
  return cap[dev];
}

}  // namespace

// CTAs the device can hold at once as CTA pairs of the pair kernel (pairs
// need both SMs of a TPC; a device with partly disabled TPCs holds fewer
// pairs than half its SMs).
int gemm_pair_capacity(const fo_plan* p) {
  return p->tile_n == 256 ? pair_capacity_bn<256>(p->device) : pair_capacity_bn<128>(p->device);
}

// Dynamic shared memory of a GEMM CTA: the smallest over the kernel's
// variants (the ring is 192 KB in every variant, so they are all equal).
int gemm_smem_bytes() {
  int m = Cfg<256, true>::kSmemBytes;
  m = Cfg<256, false>::kSmemBytes < m ? Cfg<256, false>::kSmemBytes : m;
  m = Cfg<128, true>::kSmemBytes < m ? Cfg<128, true>::kSmemBytes : m;
  m = Cfg<128, false>::kSmemBytes < m ? Cfg<128, false>::kSmemBytes : m;
  return m;
}

fo_status launch_signaled_gemm(const fo_plan* p, const void* A, const void* const* B,
                               void* C_r, int32_t* count, uint32_t* flags, uint32_t epoch,
                               void* stream) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, p->device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, p->device) !=
          cudaSuccess)
    return FO_ERR_CUDA;
  if (major != 10 || minor != 3) return FO_ERR_UNSUPPORTED;
  const uintptr_t align_bits = reinterpret_cast<uintptr_t>(A) |
                               reinterpret_cast<uintptr_t>(C_r);
  if (align_bits & 15) return FO_ERR_ARG;
  GemmArgs a{};
  if (!encode_tensor_map_2d(&a.tmap_a, A, uint64_t(p->K), uint64_t(p->M), kBlockK, kTileM, true))
    return FO_ERR_CUDA;
  const int E = p->n_experts > 0 ? p->n_experts : 1;
  for (int e = 0; e < E; ++e) {
    if (!B[e] || (reinterpret_cast<uintptr_t>(B[e]) & 15)) return FO_ERR_ARG;
    if (!encode_tensor_map_2d(&a.tmap_b[e], B[e], uint64_t(p->N), uint64_t(p->K), 64, kBlockK, true))
      return FO_ERR_CUDA;
  }
  a.tile = p->dev.tile;
  a.group_tiles = p->dev.group_tiles;
  a.dest_base = p->dev.dest_base;
  a.row_dest = p->dev.row_dest;
  a.row_rank = p->dev.row_rank;
  a.slot_live = p->layout == FO_LAYOUT_A2A_SUBTOKEN ? p->dev.slot_live : nullptr;
  a.c_r = static_cast<uint16_t*>(C_r);
  a.count = count;
  a.count_ready = p->dev.count_ready;
  a.exit_count = p->dev.gemm_exit;
  a.n_groups = p->P;
  a.flags = flags;
  a.status = p->dev.gemm_status;
  a.trace = p->trace;
  a.tiles = p->tiles;
  a.k_blocks = p->K / kBlockK;
  if (++p->gemm_seq == 0) p->gemm_seq = 1;
  a.seq = p->gemm_seq;
  // an owner waits for its helper's partial sums, so the split needs every
  // CTA of the grid resident at once (W no larger than the SM count)
  if (p->split_n > 0 && p->split_enabled && p->W <= p->sm_count) {
    a.split_ws = static_cast<float4*>(p->dev.split_ws);
    a.split_flag = p->dev.split_flag;
    a.split_n = p->split_n;
    a.split_wave = p->waves - 1;
    a.split_slot0 = (p->waves - 1) * p->W;
  }
  a.layout = p->layout;
  a.R = p->R;
  a.h = kTileM / p->R;
  a.epoch = epoch;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // pairs only when every pair of the W CTAs can be resident at once:
  // otherwise the waves would not run side by side
  const bool fits = p->pairable && gemm_pair_capacity(p) >= (p->W < p->tiles ? p->W : p->tiles);
  bool pair = false;
  if (p->gemm_variant == FO_GEMM_PAIRS) {
    if (!fits) return FO_ERR_UNSUPPORTED;
    pair = true;
  } else if (p->gemm_variant == FO_GEMM_AUTO) {
    pair = fits;
  }
  if (p->tile_n == 256)
    return pair ? launch_bn<256, true>(p, a, st) : launch_bn<256, false>(p, a, st);
  return pair ? launch_bn<128, true>(p, a, st) : launch_bn<128, false>(p, a, st);
}

}  // namespace fo
