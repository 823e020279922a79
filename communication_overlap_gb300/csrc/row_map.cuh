// Inverse mapping of one tile row and the fused element-wise epilogue,
// shared by the post-communication reorder and the fused consumer+reorder.
//
// Page: "FlashOverlap: 信号驱动计算通信重叠论文详解" -- 二、重排机制 (the inverse
// mapping table restores the layout after communication; Figure 6's tile,
// subtile and sub-token patterns) and 五、CUTLASS 扩展实现 "Epilogue 集成"
// (element-wise operations fused with the post-communication reorder).
#pragma once

#include "device_common.cuh"

namespace fo {

// Device tables the inverse mapping reads.
struct RowMap {
  const TileInfo* tile;
  const int32_t* part_start;
  const int32_t* part_dst;
  const int32_t* dest_base;
  const int32_t* row_dest;
  const int32_t* row_rank;
  const int32_t* final_row;
  int32_t layout, R, h, rows_per;
};

inline RowMap make_row_map(const fo_plan* p) {
  RowMap m{};
  m.tile = p->dev.tile;
  m.part_start = p->dev.part_start;
  m.part_dst = p->dev.part_dst;
  m.dest_base = p->dev.dest_base;
  m.row_dest = p->dev.row_dest;
  m.row_rank = p->dev.row_rank;
  m.final_row = p->dev.final_row;
  m.layout = p->layout;
  m.R = p->R;
  m.h = kTileM / p->R;
  m.rows_per = p->M / p->R;
  return m;
}

// Row r of the tile at slot s: the unit's place in the consumer's buffer k
// (src_unit) and the row it belongs to in output k (dst_row).  k = -1 (and
// nothing else set) for an All-to-All row that holds no token.
__device__ __forceinline__ void map_row(const RowMap& a, const TileInfo& ti, int32_t s, int32_t r,
                                        int* k_out, int32_t* src_unit, int32_t* dst_row) {
  int k = 0;
  if (a.layout == FO_LAYOUT_TILE) {
    *src_unit = ti.unit_base + r;
    *dst_row = ti.row0 + r;
  } else {
    int32_t u;
    if (a.layout == FO_LAYOUT_RS_SUBTILE) {
      k = r / a.h;
      const int32_t i = r - k * a.h;
      u = ti.unit_base + k * ti.sub_stride + i;
      *dst_row = (ti.row0 / kTileM) * a.h + i;
    } else if (a.layout == FO_LAYOUT_RS_ROWBLOCK) {
      k = ti.dest;
      u = ti.unit_base + r;
      *dst_row = ti.row0 + r - k * a.rows_per;
    } else {  // FO_LAYOUT_A2A_SUBTOKEN
      const int32_t rho = ti.row0 + r;
      k = a.row_dest[rho];
      if (k < 0) {
        *k_out = -1;
        return;
      }
      u = a.dest_base[s * a.R + k] + a.row_rank[rho];
      *dst_row = a.final_row[rho];
    }
    const int32_t jk = ti.group * a.R + k;
    *src_unit = a.part_dst[jk] + (u - a.part_start[jk]);
  }
  *k_out = k;
}

// The fused element-wise epilogue: act(x + bias) in fp32, rounded once to
// bf16 (nearest even).  ReLU keeps v only when v > 0; SiLU is v / (1 + e^-v).
__device__ __forceinline__ float epilogue_op(float v, float b, int act) {
  v = __fadd_rn(v, b);
  if (act == FO_ACT_RELU) v = v > 0.0f ? v : 0.0f;
  else if (act == FO_ACT_SILU) v = v / (1.0f + expf(-v));
  return v;
}

// Eight bf16 values of columns col .. col+7 through the epilogue.
__device__ __forceinline__ uint4 epilogue8(uint4 x, const uint16_t* bias, int32_t col, int act) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float b0 = 0.0f, b1 = 0.0f;
    if (bias != nullptr) {
      b0 = __uint_as_float(uint32_t(bias[col + 2 * i]) << 16);
      b1 = __uint_as_float(uint32_t(bias[col + 2 * i + 1]) << 16);
    }
    o[i] = pack_bf16x2(epilogue_op(bf16lo(w[i]), b0, act), epilogue_op(bf16hi(w[i]), b1, act));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace fo
