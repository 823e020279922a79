/*
 * fo.h -- C ABI of libfo.so: FlashOverlap's signaled GEMM + reorder path on
 * one GB300 (sm_103a).
 *
 * Pages followed (cited by title and section):
 *  [P1] "FlashOverlap: 信号驱动计算通信重叠论文详解" -- 核心设计 (system overview),
 *       一、信号机制 (waves, wave groups, counting table), 二、重排机制 (mapping
 *       table, pre-/post-communication reordering, Figure 6 patterns),
 *       五、CUTLASS 扩展实现 (epilogue + monitor kernel on its own stream).
 *  [P2] "Efficient and Adaptable Overlapping for Computation and
 *       Communication via Signaling and Reordering" -- abstract, Figure 5.
 *
 * The pages describe no library interface.  These calls follow their
 * statement of the problem: plan the wave groups, run one uninterrupted GEMM
 * that reorders each finished tile into its group's contiguous range and
 * signals when the group is complete, consume each group as soon as it is
 * signalled, and reorder the results back.
 *
 * Conventions for every call:
 *  - Matrices are bf16 (2-byte IEEE bfloat16), row-major.  A is M x K (for
 *    the grouped workload: the routed rows stacked expert after expert), B
 *    is K x N.  Accumulation is fp32; outputs are bf16 rounded to nearest
 *    even.
 *  - A "unit" is one tile row: tile_n consecutive bf16 values (512 bytes at
 *    tile_n = 256).  The reordered buffer and every consumer buffer are
 *    arrays of units.
 *  - Ownership: the caller owns every device buffer it passes (A, B, C_r,
 *    partials, destinations, counting table, flags, status word).  A plan
 *    owns its host tables, its device copies of them and a small device
 *    scratch area; fo_plan_destroy frees them.
 *  - Streams are cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every launch is asynchronous on that stream.
 *  - Argument errors return FO_ERR_ARG synchronously and launch nothing.
 *    A failed CUDA call returns FO_ERR_CUDA.  Device-side waits are bounded:
 *    a wait that runs out writes FO_ERR_TIMEOUT into the caller's status word
 *    (read it after synchronising); no kernel traps or asserts.
 *  - Device data buffers (A, B, C_reordered, partials, communication and
 *    final buffers, bias) must be 16-byte aligned; counting tables, flags,
 *    status words and routing arrays 4-byte aligned; trace stamps 8-byte
 *    aligned.  A misaligned pointer is an argument error (FO_ERR_ARG),
 *    checked before anything is launched.
 */
#ifndef FO_H
#define FO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FO_OK = 0,
  FO_ERR_ARG = 1,          /* invalid argument; nothing launched */
  FO_ERR_CUDA = 2,         /* a CUDA runtime call or launch failed */
  FO_ERR_TIMEOUT = 3,      /* a bounded device wait ran out (status word) */
  FO_ERR_UNSUPPORTED = 4   /* shape or device the kernels do not cover */
} fo_status;

/* How each wave group is laid out in the reordered buffer ([P1] 二,
 * Figure 6).  In every layout a group is one contiguous unit range, and the
 * group's part for destination k is one contiguous sub-range. */
typedef enum {
  FO_LAYOUT_TILE = 0,        /* AllReduce / copy: the group's tiles whole, in
                                launch order, rows in order */
  FO_LAYOUT_RS_SUBTILE = 1,  /* ReduceScatter: each tile cut along rows into
                                n_dest subtiles; part k = the k-th subtile of
                                each of the group's tiles, in launch order */
  FO_LAYOUT_RS_ROWBLOCK = 2, /* ReduceScatter, literal reading: part k = the
                                group's whole tiles whose rows lie in rank k's
                                block of M / n_dest rows */
  FO_LAYOUT_A2A_SUBTOKEN = 3 /* All-to-All: part d = the tile rows (sub-tokens)
                                whose token t has t mod n_dest == d, over the
                                group's tiles in launch order */
} fo_layout;

/* What stands in for the collective on one GPU ([P1] 二: the reordered
 * group is what a ncclAllReduce / ReduceScatter / AlltoAll call would send). */
typedef enum {
  FO_CONS_COPY = 0,  /* dst[0][u] = src[u] over the group's range */
  FO_CONS_SUM = 1,   /* dst[0][u] = bf16(((src[u] + P1[u]) + P2[u]) + ...),
                        every addition in fp32, one rounding */
  FO_CONS_RS = 2,    /* the same sum; part k of the group is appended to
                        dst[k] (group after group) */
  FO_CONS_A2A = 3    /* part d of the group is copied, appended to dst[d] */
} fo_consumer;

/* Plan description.  Host pointers are read during fo_plan_groups only. */
typedef struct {
  int32_t M, N, K;        /* C = A . B sizes; M = sum(expert_rows) if grouped */
  int32_t tile_m;         /* 128 */
  int32_t tile_n;         /* 128 or 256; N % tile_n == 0 */
  int32_t swizzle;        /* band height, in tile rows, of the launch order */
  int32_t wave_width;     /* W: persistent GEMM CTAs = tiles per wave;
                             <= 0 means the device's SM count */
  int32_t n_groups;       /* P */
  const int32_t* group_waves; /* [P] waves per group, each >= 1, sum = T */
  fo_layout layout;
  int32_t n_dest;         /* ranks the layout routes to (RS: R, A2A: D) */
  int32_t n_experts;      /* 0 = plain GEMM; >= 1 = grouped GEMM */
  const int32_t* expert_rows; /* [n_experts] routed rows of each expert */
  const int32_t* row_token;   /* [M] A2A: token id of each routed row; a
                                 negative id marks a row that holds no token
                                 (expert capacity the routing left unfilled:
                                 it is sent nowhere).  row_token and row_slot
                                 may both be NULL: every row starts empty,
                                 for a routing given by fo_plan_route */
  const int32_t* row_slot;    /* [M] A2A: top-k slot of each routed row */
  int32_t host_only;      /* 1: build host tables only (no device needed) */
  int32_t pad_expert_tile_rows; /* 0 (default): each expert's grid has
                                 ceil(rows / tile_m) tile rows, the GEMM's
                                 output tiles.  1 (A2A layout only): an odd
                                 count gets one empty tile row, so that every
                                 band of the launch order has an even height
                                 and CTA pairs (fo_plan_set_gemm) can take
                                 launch slots 2i, 2i+1; empty tiles take
                                 slots, count in waves and |G_j|, and are
                                 skipped by the GEMM.  Not in the pages: a
                                 choice of this library's pair kernel */
  int32_t band_order;     /* FO_BAND_FORWARD (0, default) or
                             FO_BAND_SERPENTINE, see fo_band_order */
} fo_plan_desc;

/* Column order inside the bands of the launch order.  Tiles are launched
 * band by band (`swizzle` tile rows per band, per expert); inside a band,
 * column by column, each column top to bottom.
 *  FO_BAND_FORWARD:    every band walks its columns left to right.
 *  FO_BAND_SERPENTINE: the odd bands of each expert walk them right to
 *      left, so a band starts on the columns of B the band before it ended
 *      on, while they may still be in L2.
 * Either way a band's tiles are consecutive launch slots, waves are slot / W
 * and the CTA pairs of fo_plan_set_gemm stay vertically adjacent. */
typedef enum { FO_BAND_FORWARD = 0, FO_BAND_SERPENTINE = 1 } fo_band_order;

typedef struct fo_plan fo_plan;   /* opaque, library-owned */

/* Tiles and waves of a description, T = ceil(tiles / W) ([P1] 一 "关键洞察",
 * 四 Algorithm 1).  Checks the shape fields only (group_waves may be NULL),
 * so a caller can choose a partition of T waves before planning. */
fo_status fo_wave_count(const fo_plan_desc* desc, int32_t* tiles, int32_t* waves);

/* Validate desc, build the launch order (banded swizzle), wave -> group map,
 * |G_j| in tiles, mapping and inverse mapping tables and the reordered
 * layout ([P1] 一 "组级 Tile 计数", 二 "映射表重排"), and upload the tables
 * (unless host_only).  On success *out owns them. */
fo_status fo_plan_groups(const fo_plan_desc* desc, fo_plan** out);

/* Sizes of a plan ([P1] 一: tiles, waves and |G_j|, the tiles of each
 * group).  Any output pointer may be NULL.  group_tiles: [P];
 * tile_to_slot: [tiles], row-major tile id -> launch slot. */
fo_status fo_plan_info(const fo_plan* plan, int32_t* tiles, int32_t* waves,
                       int32_t* n_groups, int32_t* group_tiles,
                       int32_t* tile_to_slot);

/* Host copies of a plan's tables, for inspection and tests. */
typedef enum {
  FO_TAB_SLOT_TILE = 0,   /* [tiles] inverse mapping: slot -> tile id */
  FO_TAB_TILE_SLOT = 1,   /* [tiles] mapping: tile id -> slot */
  FO_TAB_SLOT_GROUP = 2,  /* [tiles] group of each slot */
  FO_TAB_GROUP_TILES = 3, /* [P] |G_j| */
  FO_TAB_UNIT = 4,        /* [tiles * tile_m] unit of row r of the tile at
                             slot s (index s * tile_m + r); -1 = no row */
  FO_TAB_PART_START = 5,  /* [P * R] first unit of part (j, k) in C_r */
  FO_TAB_PART_LEN = 6,    /* [P * R] units of part (j, k) */
  FO_TAB_PART_DST = 7,    /* [P * R] offset (units) of part (j, k) in dst[k] */
  FO_TAB_DEST_UNITS = 8,  /* [R] units each destination buffer receives */
  FO_TAB_FINAL_ROWS = 9,  /* [R] rows of each output of fo_reorder_back
                             (each row has N values) */
  FO_TAB_DEST_CAPACITY = 10, /* [R] units a destination buffer must hold: A2A
                             final_rows[k] * (N / tile_n), enough for any
                             routing of the plan's tokens (see
                             fo_plan_route); other layouts DEST_UNITS */
  FO_TAB_SLOT_LIVE = 11,  /* [tiles] 1 if a row of the tile at slot s holds a
                             token.  A2A only can have 0s: the GEMM skips
                             such a tile's loads and MMAs (both tiles of a
                             CTA pair must be empty) and only counts it */
  FO_TAB_UNIT_PLACE = 12  /* [units] final place of each unit of C_r, as
                             the post-communication reorder puts it:
                             k << 28 | the 16-byte vector index, in output k,
                             of the unit's first element (its row x N / 8 +
                             its first column / 8).  FO_ERR_UNSUPPORTED when
                             an output holds 2^28 or more vectors */
} fo_table;               /* R = 1 for FO_LAYOUT_TILE, else n_dest */

/* Copy table `which` into out[0 .. capacity); *length = its full length.
 * FO_ERR_ARG if capacity is too small (length is still set).  After
 * fo_plan_route the routing-dependent tables (UNIT, PART_*, DEST_UNITS) live
 * on the device: the first call afterwards synchronises the device and
 * downloads them (FO_ERR_CUDA if that fails). */
fo_status fo_plan_table(const fo_plan* plan, int32_t which, int32_t* out,
                        int64_t capacity, int64_t* length);

/* Launch settings of the consumer and reorder kernels ([P1] 五: the
 * communication side runs beside the GEMM and moves each group once it is
 * signalled).
 *  consumer_ctas, reorder_ctas: grid sizes (<= 0: the defaults, measured
 *      beside the GEMM: consumer 4 CTAs per SM for SUM / RS, 1 per SM for
 *      COPY / A2A, 3 per SM for fo_consume_reorder (its direct variant: 1
 *      per SM for A2A); reorder 3 per SM).
 *  overlap: non-zero (default) launches the consumer as a programmatic
 *      dependent launch: issued on the GEMM's stream right after
 *      fo_signaled_gemm, it starts as soon as every GEMM CTA is resident and
 *      runs alongside the GEMM.  The consumer then also publishes when each
 *      group is fully written, and fo_reorder_back issued right after it is
 *      in turn its programmatic dependent: it starts once every consumer CTA
 *      is resident and moves each group as soon as that group is consumed.
 *      Zero launches both as ordinary kernels (the consumer starts after the
 *      GEMM has finished, the reorder after the consumer: the serial
 *      baseline). */
fo_status fo_plan_set_launch(fo_plan* plan, int32_t consumer_ctas,
                             int32_t reorder_ctas, int32_t overlap);

/* Pacing of fo_consume_reorder beside the GEMM (overlap on).  While the GEMM
 * still runs, only consumer CTAs 0 .. ctas_during_gemm-1 take work; the
 * others first wait (bounded, like every flag wait) for the last group's
 * flag -- the GEMM's end -- and then take whatever is left, from the first
 * group on.  A consumer that moves less data while the GEMM runs competes
 * less with it for HBM and SM time, and catches up once it has finished.
 * 0 (default) or a value of at least the grid: every CTA works from the
 * first flag on.  With FO_CONSUMER_RESERVED and its default grid (below)
 * pacing is off.  The results do not depend on it. */
fo_status fo_plan_set_pacing(fo_plan* plan, int32_t ctas_during_gemm);

/* Where the consumer's CTAs run beside the GEMM.  [P1] 四、实时调优, offline
 * stage: the communication kernel occupies some SMs, and the GEMM's wave
 * count is taken over the SMs left to it (tiles / (SMs - communication
 * SMs)); here the plan's wave width W plays that role.
 *  FO_CONSUMER_SHARED (default): consumer CTAs may share an SM with a CTA
 *      of the signaled GEMM.
 *  FO_CONSUMER_RESERVED: fo_consume_group, fo_consume_reorder and
 *      fo_consume_group_noalloc request (unused) dynamic shared memory that
 *      does not fit beside a GEMM CTA, so while the GEMM runs their CTAs
 *      run only on the SMs it leaves free: the device's SM count minus
 *      min(W, tiles).  Their default grid is then as many CTAs as those
 *      SMs hold at once (the kernel's occupancy with that shared memory), so
 *      none waits for an SM; a grid set with fo_plan_set_launch still wins.
 * The results do not depend on the placement.  FO_ERR_ARG for an unknown
 * value; FO_ERR_UNSUPPORTED for FO_CONSUMER_RESERVED when the GEMM leaves
 * no SM free, or when the shared memory needed is above the default
 * dynamic limit (48 KB); FO_ERR_CUDA when the device cannot be queried. */
typedef enum {
  FO_CONSUMER_SHARED = 0,
  FO_CONSUMER_RESERVED = 1
} fo_consumer_placement;
fo_status fo_plan_set_consumer_placement(fo_plan* plan, fo_consumer_placement placement);

/* How fo_signaled_gemm maps tiles onto CTAs.  Either way W CTAs take the
 * launch slots c, c + W, ... (wave = slot / W) and every tile gets the same
 * epilogue; only the MMA differs.
 *  FO_GEMM_SINGLE: one CTA per tile, tcgen05.mma with M = 128.
 *  FO_GEMM_PAIRS:  CTAs 2p and 2p+1 form a cluster; their tiles at slots
 *      2i and 2i+1 must be vertically adjacent (same expert and columns,
 *      rows 128 apart: W even, an even tile count and even band heights),
 *      and one tcgen05.mma.cta_group::2 (M = 256) computes both, each CTA
 *      staging its own A rows and half of B.
 *      The device must also hold all W CTAs as pairs at once (a pair needs
 *      both SMs of a TPC; with partly disabled TPCs that can be fewer than
 *      the SM count), or the waves would not run side by side.
 *  FO_GEMM_AUTO (default): pairs when the plan and the device allow them. */
typedef enum { FO_GEMM_AUTO = 0, FO_GEMM_SINGLE = 1, FO_GEMM_PAIRS = 2 } fo_gemm_variant;

/* Select the variant.  *pairable (may be NULL): whether pairs are possible
 * for this plan on this device; *pair_capacity (may be NULL): how many CTAs
 * the device holds at once as pairs of the pair kernel.  FO_ERR_UNSUPPORTED
 * if FO_GEMM_PAIRS is asked when pairs are not possible. */
fo_status fo_plan_set_gemm(fo_plan* plan, fo_gemm_variant variant, int32_t* pairable,
                           int32_t* pair_capacity);

/* Last-wave split.  When the last wave holds n <= W / 2 tiles (e.g. 68 of
 * 148), n CTAs would idle through it; instead each of its tiles is computed
 * by two CTAs over halves of K: CTA c < n (the tile's own CTA) takes the
 * first half, CTA c + n the second and hands its fp32 partial sums over
 * through a workspace in the plan (128 x tile_n x 4 bytes per tile); the
 * owner adds them and stores, counts and signals the tile as usual.  Waves,
 * groups, tables and the counting table do not change; only the order of
 * the fp32 additions of those tiles does.  Enabled by default when the
 * shape allows it and W does not exceed the device's SM count (an owner
 * waits for its helper, so every CTA must be resident at once).
 * *split_tiles (may be NULL): how many tiles are split (0 when disabled or
 * not possible). */
fo_status fo_plan_set_split(fo_plan* plan, int32_t enable, int32_t* split_tiles);

/* Timelines ([P2] Figure 3 records each tile's completion time with
 * globaltimer to show the wave pattern).  Device uint64 buffers owned by the
 * caller, kept alive while tracing; NULL stops that trace.
 *  stamps [tiles + W + 2 * split tiles]: every GEMM launch writes
 *      stamps[slot] = %globaltimer (ns) when the tile at that launch slot has
 *      been stored and counted, stamps[tiles + c] = the start time of CTA c,
 *      and for the i-th split tile of the last wave (fo_plan_set_split)
 *      stamps[tiles + W + 2i] = when its helper handed its partial sums over
 *      and stamps[tiles + W + 2i + 1] = when its owner's half was computed.
 *  consumer_stamps [2P + 4 * consumer CTAs], zeroed by the caller before
 *      the consume call (fo_consume_group or fo_consume_reorder): [j] = when
 *      group j's last chunk was processed; [P + j] = when group j's last
 *      reorder item was done (fo_consume_reorder only); then per CTA c,
 *      [2P + 4c ..]: SM id, start time, end time, chunks processed. */
fo_status fo_plan_set_trace(fo_plan* plan, uint64_t* stamps, uint64_t* consumer_stamps);

/* Sticky status word of the plan's GEMM and reorder launches (calls with
 * no status argument): FO_OK, or FO_ERR_TIMEOUT if one of their bounded
 * waits on their own copies ran out.  Synchronises the device; clears the
 * word when `clear` is non-zero. */
fo_status fo_plan_device_status(const fo_plan* plan, int32_t* kernel_status,
                                int32_t clear);

void fo_plan_destroy(fo_plan* plan);

/* Counting table initialisation ([P1] 一 "实现方法: 组级 Tile 计数": the table
 * starts at [0, ..., 0]): cudaMemsetAsync of count_table[0 .. P) on the
 * stream the GEMM will run on.  count_table: device int32[P].  Optional:
 * fo_signaled_gemm resets the table itself; this call is for callers that
 * want it cleared earlier (to read it before the next launch). */
fo_status fo_counting_table_init(const fo_plan* plan, int32_t* count_table,
                                 void* cuda_stream);

/* The signaled GEMM ([P1] 五 "扩展主循环"/"Epilogue 集成", [P2] Figure 5):
 * one persistent kernel of W CTAs computes every tile of C = A . B
 * (tcgen05 tensor cores, fp32 accumulation in tensor memory); as each tile
 * finishes, its epilogue writes the tile's rows, rounded to bf16, to their
 * units in C_reordered (the pre-communication reorder), then adds 1 to
 * count_table[j] of the tile's group j, and the tile that makes it reach
 * |G_j| stores `epoch` into flags[j] (release at GPU scope, after every
 * store of the group is visible).
 *  A:  device, M x K bf16 row-major.
 *  B:  host array of n_experts (1 for a plain GEMM) device pointers, each
 *      K x N bf16 row-major.
 *  C_reordered: device, M * N bf16 (M * N / tile_n units).
 *  count_table: device int32[P].  The kernel resets it to [0, ..., 0]
 *      itself (CTA 0, before any tile is counted), so the caller need not
 *      (fo_counting_table_init does the same as a separate memset); it ends
 *      equal to |G_j|.
 *  flags: device uint32[P].  CTA 0 clears them with the counting table,
 *      before any consumer launched after this call can start.  count_table
 *      and flags may both be NULL: the GEMM then signals nothing.
 *  epoch: the value this iteration's flags take.  A new one per iteration
 *      is the simplest; a step captured in a CUDA graph may replay with the
 *      same one (the flags are cleared at every launch, and the kernels'
 *      per-launch handshakes -- the counting table's reset, the split
 *      tiles' partial sums, the reorder's consumed flags -- are withdrawn
 *      by each launch when it has used them).
 * Requires K % 64 == 0 and a device with compute capability 10.3. */
fo_status fo_signaled_gemm(const fo_plan* plan, const void* A,
                           const void* const* B, void* C_reordered,
                           int32_t* count_table, uint32_t* flags,
                           uint32_t epoch, void* cuda_stream);

/* The communication stand-in ([P1] 五 "专用监控内核": a monitor kernel
 * tracking progress through atomic counters).  For group = j, or every group
 * in order when group = -1, the kernel waits until flags[j] == epoch
 * (acquire at GPU scope, __nanosleep back-off, at most spin_limit_ns per
 * group, 0 = 2 s), then processes the group's contiguous range of
 * src_reordered as `kind` says.
 *  Launch: pass the GEMM's stream to overlap (see fo_plan_set_launch).  On
 *  another stream the kernel can be scheduled before the GEMM's CTAs and
 *  hold the SMs they need; its waits then run out (FO_ERR_TIMEOUT) rather
 *  than hang, but the GEMM is delayed -- the pages' separate-stream design
 *  has this hazard, which the dependent launch removes.
 *  partials: host array of n_partials device pointers, same layout as
 *      src_reordered (SUM and RS; n_partials <= 8).
 *  dst: host array of device pointers: 1 buffer for COPY/SUM (same size as
 *      src), R buffers for RS/A2A sized by FO_TAB_DEST_UNITS.
 *  dev_status: device int32, 0 before the call; a wait that runs out sets it
 *      to FO_ERR_TIMEOUT and the kernel returns without that group's work.
 * The kernel hands work out through chunk counters in the plan's device
 * scratch; the last CTA resets them.  Consume calls on one plan that overlap
 * in time race on that scratch. */
fo_status fo_consume_group(const fo_plan* plan, int32_t group,
                           fo_consumer kind, const void* src_reordered,
                           const void* const* partials, int32_t n_partials,
                           void* const* dst, const uint32_t* flags,
                           uint32_t epoch, uint64_t spin_limit_ns,
                           int32_t* dev_status, void* cuda_stream);

/* Allocation-free variant of fo_consume_group.  The pages have no
 * counterpart to this entry point: it exists for callers that may not
 * allocate device memory when they run the overlap -- code captured into a
 * CUDA graph (no cudaMalloc during capture), serving runtimes whose memory
 * pool owns all device memory and forbids allocations on the request path,
 * and latency-critical loops that cannot wait for the allocator.
 *
 * Same arguments and results as fo_consume_group, and the same launch: a
 * programmatic dependent launch after fo_signaled_gemm with overlap on
 * (fo_plan_set_launch), also feeding an overlapped fo_reorder_back, with
 * the plan's consumer trace if one is set.  It allocates nothing: instead
 * of the plan's scratch it keeps its chunk counters in a fixed array inside
 * the library's device image, room for FO_NOALLOC_MAX_GROUPS groups (32 KB
 * on every GPU that loads the library, held until the process exits).  A
 * plan with more groups gets FO_ERR_ARG and nothing is launched.  The
 * plan's device must be the current device.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, once per device); make that first call before
 *    any stream capture.  The array is zero when the library loads and
 *    every launch leaves its counters at zero for the next one, also after
 *    a wait that ran out.
 *  - All calls share the one array: calls whose kernels overlap on the GPU
 *    (on other streams, without an ordering between them) race on it.
 *    Calls on one stream are ordered: when an earlier no-alloc consume on
 *    the same stream could still be running (no fo_signaled_gemm issued on
 *    that stream since it), the call is launched as an ordinary kernel, so
 *    it starts only after that consume has finished. */
#define FO_NOALLOC_MAX_GROUPS 4096
fo_status fo_consume_group_noalloc(const fo_plan* plan, int32_t group,
                                   fo_consumer kind, const void* src_reordered,
                                   const void* const* partials, int32_t n_partials,
                                   void* const* dst, const uint32_t* flags,
                                   uint32_t epoch, uint64_t spin_limit_ns,
                                   int32_t* dev_status, void* cuda_stream);

/* Dynamic routing ([P1] 二 (3): in an MoE layer tokens are routed to their
 * experts at run time, and the mapping table has to follow that routing).
 * The plan fixes the shape: n_experts experts of expert_rows[e] rows each
 * (each expert's capacity), so the GEMM, its tiles, waves and groups never
 * change.  This call takes a new assignment of tokens to those rows, in
 * device memory, and rebuilds every routing-dependent table on the device
 * (per-row destination, rank and output row; per-(tile, rank) bases; per-
 * (group, rank) parts) with two kernels on `stream`, so the routing never
 * goes through the host.  Later launches on the same stream use it.
 *  row_token, row_slot: device int32[M] (4-byte aligned).  Row r of the
 *      stacked expert rows holds token row_token[r], top-k slot row_slot[r];
 *      row_token[r] < 0 marks an empty row (sent nowhere).
 *  n_tokens, top_k: token ids lie in [0, n_tokens), slots in [0, top_k).
 *      They size the outputs: rank d's output of fo_reorder_back has
 *      ceil((n_tokens - d) / n_dest) * top_k rows (FO_TAB_FINAL_ROWS) and its
 *      receive buffer FO_TAB_DEST_CAPACITY units; both tables follow at once.
 *  dev_status: device int32.  A routing with a token or slot out of range,
 *      or more rows for one rank than its capacity (a (token, slot) pair
 *      given twice), sets it to FO_ERR_ARG and yields a plan that routes no
 *      row: nothing is written out of bounds.
 * Only for FO_LAYOUT_A2A_SUBTOKEN plans; FO_ERR_ARG otherwise.  Must not
 * overlap in time with a launch that reads the plan's tables. */
fo_status fo_plan_route(fo_plan* plan, const int32_t* row_token, const int32_t* row_slot,
                        int32_t n_tokens, int32_t top_k, int32_t* dev_status,
                        void* cuda_stream);

/* Post-communication reorder ([P1] 二 "通信后重排"): for the groups
 * [group_begin, group_end), move every unit from where the consumer left it
 * to its place in the final row-major layout, by the inverse mapping table.
 *  TILE:        src[0] (consumer output) -> dst[0], M x N.
 *  RS_SUBTILE:  src[k] = slice k -> dst[k], (M / R) x N; slice row
 *               h * tm + i holds global row tile_m * tm + h * k + i
 *               (h = tile_m / R).
 *  RS_ROWBLOCK: src[k] -> dst[k], (M / R) x N, rows k M/R .. (k+1) M/R - 1.
 *  A2A:         src[d] -> dst[d]: the sub-token of routed row (token t,
 *               slot q) lands in row (t / D) * top_k + q of dst[d]
 *               (top_k = 1 + the largest row_slot, or fo_plan_route's);
 *               empty rows move nowhere.
 * Issue it on the consumer's stream after fo_consume_group.  With overlap
 * on (fo_plan_set_launch) it may start while the consumer still runs and
 * waits, bounded, until the plan's last consume call has finished each
 * group it moves (a wait that runs out sets the plan's status word, see
 * fo_plan_device_status); tiles are then taken in launch order from a
 * counter in the plan's scratch, so reorder calls on one plan that overlap
 * in time race on it.  With overlap off it relies on stream order alone. */
fo_status fo_reorder_back(const fo_plan* plan, int32_t group_begin,
                          int32_t group_end, const void* const* src,
                          void* const* dst, void* cuda_stream);

/* Wave-group tuning ([P1] 四、实时调优, Algorithm 1).  The offline inputs are
 * the GEMM's duration (gemm_us, e.g. measured with fo_signaled_gemm) and the
 * communication latency curve: n_points >= 2 samples (curve_bytes[i],
 * curve_us[i]) of latency against message size, distinct sizes, any order;
 * between samples the curve is linear, below the smallest sample it is that
 * sample's latency, above the largest it follows the last segment's slope.
 * A group's data size is its tile count (the last wave may be partial)
 * times tile_m * tile_n * 2 bytes; its compute time is gemm_us / T per
 * wave.  The predicted latency of a partition is E_P, with
 *   E_i = max(compute end of groups 1..i, E_{i-1}) + curve(bytes of G_i).
 * desc: the shape fields as for fo_plan_groups (host_only may be set). */

/* Predicted latency (us) of the partition in desc->group_waves. */
fo_status fo_predict_partition(const fo_plan_desc* desc, double gemm_us,
                               const double* curve_bytes, const double* curve_us,
                               int32_t n_points, double* predicted_us);

/* The partition with the smallest predicted latency over all 2^(T-1)
 * candidates, found exactly by a dynamic program over group boundaries in
 * O(T^2) (the pages enumerate the candidates).  Writes the waves per group
 * to group_waves[0 .. *n_groups) (capacity >= T always suffices; FO_ERR_ARG
 * if capacity is too small, *n_groups still set) and the prediction to
 * *predicted_us (may be NULL). */
fo_status fo_tune_partition(const fo_plan_desc* desc, double gemm_us,
                            const double* curve_bytes, const double* curve_us,
                            int32_t n_points, int32_t* group_waves, int32_t capacity,
                            int32_t* n_groups, double* predicted_us);

/* The same two calls with the interference of one GPU, where the GEMM and
 * the consumer share memory and SMs and each slows the other while both run
 * (the pages' model has them on separate hardware; this is a reading for
 * one GPU, not the pages'):
 *  gemm_slowdown (sigma > 0): while a communication runs, the GEMM advances
 *      at 1 / sigma of its rate (gemm_us / T per wave alone);
 *  comm_slowdown (rho > 0): while the GEMM runs, a communication advances at
 *      1 / rho of the curve's rate.
 * A group's communication starts once its waves are computed and the
 * previous one has ended; the schedule is simulated event by event.
 * sigma = rho = 1 gives fo_predict_partition / fo_tune_partition exactly.
 * With other factors the search is exhaustive (all 2^(T-1) candidates, the
 * first on ties) up to T = 20 waves; beyond it, a local search: single cuts
 * toggled while the prediction falls, from the best of the exact plain
 * optimum, the finest partition and one wave then groups of two.  Factors
 * that are not finite and positive are FO_ERR_ARG. */
fo_status fo_predict_partition_ex(const fo_plan_desc* desc, double gemm_us,
                                  const double* curve_bytes, const double* curve_us,
                                  int32_t n_points, double gemm_slowdown,
                                  double comm_slowdown, double* predicted_us);
fo_status fo_tune_partition_ex(const fo_plan_desc* desc, double gemm_us,
                               const double* curve_bytes, const double* curve_us,
                               int32_t n_points, double gemm_slowdown, double comm_slowdown,
                               int32_t* group_waves, int32_t capacity, int32_t* n_groups,
                               double* predicted_us);

/* Element-wise epilogue fused into the post-communication pass ([P1] 五
 * "Epilogue 集成": ReLU, SiLU and bias addition usually run in the GEMM's
 * epilogue; FlashOverlap fuses the post-communication reorder with them).
 * y = act(x + bias[col]): x and bias are bf16, the addition and the
 * activation fp32, one rounding to bf16 (nearest even); RELU keeps v when
 * v > 0 (else 0), SILU is v / (1 + exp(-v)).  bias: device bf16[N] or NULL
 * (16-byte aligned), indexed by the output column. */
typedef enum { FO_ACT_NONE = 0, FO_ACT_RELU = 1, FO_ACT_SILU = 2 } fo_activation;

/* fo_reorder_back with the element-wise epilogue applied to every moved
 * value (fo_reorder_back is this call with bias = NULL, act = NONE). */
fo_status fo_reorder_back_fused(const fo_plan* plan, int32_t group_begin, int32_t group_end,
                                const void* const* src, void* const* dst, const void* bias,
                                fo_activation act, void* cuda_stream);

/* fo_consume_group and fo_reorder_back_fused in one persistent kernel, for
 * the same results in both sets of buffers: comm_dst receives what
 * fo_consume_group writes to dst, final_dst what fo_reorder_back_fused
 * writes to dst.  Every group is moved to its final layout while the GEMM
 * still computes later groups ([P1] 五: the post-communication reorder fused
 * with the element-wise epilogue to save a launch):
 * a CTA that has written a chunk of units to comm_dst reads them back from
 * there (still in L2) and stores them to final_dst at once, so a group is
 * final one chunk after its flag rises.  No CTA waits for another.
 *  comm_dst: as fo_consume_group's dst, or NULL for the direct variant: the
 *      communication buffers are then neither written nor read, and each
 *      consumed unit (the same copy or the same fp32 sum, in the same
 *      order) is stored straight to its final place.  final_dst is
 *      bit-identical either way; the direct variant moves fewer bytes
 *      (SUM with n partials: (n + 2) x C rather than (n + 4) x C; COPY and
 *      A2A: 2 x C rather than 4 x C, for C the output's bytes).
 *      Each unit's place comes from FO_TAB_UNIT_PLACE (one table load).
 *      FO_ERR_UNSUPPORTED if an output holds 2^28 or more 16-byte vectors
 *      (4 GiB), which that table cannot name.
 * Layouts: TILE (COPY, SUM), RS (RS), A2A (A2A).  Uses the plan's scratch;
 * calls that overlap in time on one plan race on it. */
fo_status fo_consume_reorder(const fo_plan* plan, int32_t group, fo_consumer kind,
                             const void* src_reordered, const void* const* partials,
                             int32_t n_partials, void* const* comm_dst, void* const* final_dst,
                             const void* bias, fo_activation act, const uint32_t* flags,
                             uint32_t epoch, uint64_t spin_limit_ns, int32_t* dev_status,
                             void* cuda_stream);

/* The AllGather after a ReduceScatter, with the row exchange and the
 * element-wise epilogue in one pass ([P1] 二 (2): the gathered rows are put
 * in order by a block-cyclic permutation that needs no mapping table and
 * fuses with element-wise operations).  RS layouts only.
 *  slices: host array of R device pointers, slice k as fo_reorder_back
 *      leaves it ((M / R) x N, row-major).
 *  out: device M x N row-major.  RS_SUBTILE: out row tile_m * tm + h * k + i
 *      = slice k row h * tm + i (h = tile_m / R); RS_ROWBLOCK: out row
 *      k * M/R + rho = slice k row rho.  On one GPU every slice is local, so
 *      the gather is this copy. */
fo_status fo_allgather_rows(const fo_plan* plan, const void* const* slices, void* out,
                            const void* bias, fo_activation act, void* cuda_stream);

const char* fo_status_string(fo_status status);

#ifdef __cplusplus
}
#endif

#endif /* FO_H */
