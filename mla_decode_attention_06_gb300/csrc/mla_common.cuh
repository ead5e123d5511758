// Shared definitions of the MLA decode CUDA library (device side and host side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla_decode.h"

namespace mla {

constexpr int kTileKeys = 64;      // keys per decode tile
constexpr int kMaxHeads = 128;     // heads per query token (one MMA M tile)
constexpr int kDeviceCheckFailed = 1;
constexpr int kDeviceTimeout = 2;

// Per query token: which request it belongs to and the key range it attends.
// Dense: [lo, hi) are logical key positions; sparse: [lo, hi) are index slots.
// Keys are processed in tiles of kTileKeys aligned to logical position 0, so
// the token covers tiles [tile_first, tile_first + ntiles); across all tokens
// its tiles occupy the global tile interval [tile_start, tile_start + ntiles).
//
// When a call folds the query tokens of a request in pairs (two consecutive
// tokens of one request share every cache tile they read), the first token of
// a pair leads: [lo, hi) and its tiles cover the union of both tokens' key
// ranges and ntok = 2; the second token follows: no tiles of its own (ntiles =
// 0, ntok = 0).  [mlo, mhi) is always the token's own key range (its mask).
struct TokenPlan {
  int32_t b;
  int32_t lo, hi;
  int32_t tile_first;
  int32_t tile_start;
  int32_t ntiles;
  int32_t part_first, part_last;   // the KV partitions holding its first / last tile
  int32_t mlo, mhi;                // the token's own key range
  int32_t ntok;                    // tokens walked with these tiles: 1, 2 (a pair's first) or 0
  int32_t pad;
};

struct PlanHeader {
  int32_t total_tiles;
  int32_t status;   // device-side check / timeout bits
  int32_t pad[62];
};

// Key source of a call: a dense paged cache or a list of physical rows.
struct KeySource {
  const int32_t* block_table;  // dense: [B, bt_stride]
  int32_t bt_stride;
  const uint32_t* cache_lens;  // dense: [B]
  const int32_t* indices;      // sparse: [B, idx_stride]
  int32_t idx_stride;
  const int32_t* topk_lengths; // sparse: [B] or NULL
  int32_t page_size;
  int32_t num_pages;
};

// Byte offsets of the workspace sections:
//   header     PlanHeader (total tiles, status word)
//   plan       TokenPlan [T]
//   counters   int [T, 4]: per split token, partitions that claimed it / wrote their
//              partial, each per cluster rank
//   bounds     int [2K + 1]: first global tile of each KV partition, then the total,
//              then the token holding each partition's first tile
//   q_full     bf16 [T, 128, L+R]: absorbed queries, rows h >= H zero
//   o_lat      bf16 [T, H, L]: normalised latent outputs
//   lse        fp32 [T, H]
//   part_o     fp32 [K, 2 * NI, H, L]: partials of the first / last segment of each
//              partition, NI token slots each (2 when tokens are folded in pairs)
//   part_lse   fp32 [K, 2 * NI, 2, H]: their log-sum-exp, one copy per latent half
struct WorkspaceLayout {
  size_t header, plan, counters, bounds, q_full, o_lat, lse, part_o, part_lse, total;
};

// Host-side: the layout for T tokens, K KV partitions and NI token slots per partial.
inline WorkspaceLayout workspace_layout(const mla_dims_t& d, int T, int K, int NI = 1) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  WorkspaceLayout w{};
  size_t o = 0;
  w.header = o;  o = up(o + sizeof(PlanHeader));
  w.plan = o;    o = up(o + sizeof(TokenPlan) * (size_t)(T > 0 ? T : 1));
  w.counters = o; o = up(o + sizeof(int) * 4 * (size_t)(T > 0 ? T : 1));
  w.bounds = o;  o = up(o + sizeof(int) * (2 * (size_t)K + 1));
  w.q_full = o;  o = up(o + (size_t)T * kMaxHeads * (d.kv_lora_rank + d.qk_rope) * 2);
  w.o_lat = o;   o = up(o + (size_t)T * d.num_heads * d.kv_lora_rank * 2);
  w.lse = o;     o = up(o + (size_t)T * d.num_heads * 4);
  w.part_o = o;  o = up(o + (size_t)K * 2 * NI * d.num_heads * d.kv_lora_rank * 4);
  w.part_lse = o; o = up(o + (size_t)K * 2 * NI * 2 * d.num_heads * 4);   // [K, slot, latent half, H]
  w.total = o;
  return w;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// OCP E4M3FN code -> float through the hardware fp8 -> half conversion (exact).
__device__ __forceinline__ float e4m3_to_f32(uint8_t code) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(h));
}

// Partition bounds when the plan balances by cost: a token costs
// kTileCost per tile plus kSegmentCost for the segment it starts (reading out
// and writing its output or partial, switching the query: about 2.5 tiles of
// decode time).  Balancing applies when every partition gets at least
// kMinPartitionCost, which keeps consecutive bounds at least two tiles apart.
constexpr int kTileCost = 8;
constexpr int kSegmentCost = 20;
constexpr int kMinPartitionCost = 40;

// Token whose global tile interval contains tile g (tokens with no tiles are skipped).
__device__ __forceinline__ int token_of_tile(const TokenPlan* plan, int T, int g) {
  int lo = 0, hi = T - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (plan[mid].tile_start <= g) lo = mid; else hi = mid - 1;
  }
  while (lo < T && plan[lo].ntiles == 0) ++lo;   // zero-length tokens share tile_start
  return lo;
}

}  // namespace mla
