// Per-token key ranges, the global 64-key tile numbering and the bounds of
// the decode's KV partitions (the on-device counterpart of the packed dispatch
// metadata `scalar_args_buf` and of `num_partitions_in` on the
// generic_flare_mla_decode_kv_cache_ragged page).  Run by one thread block
// inside the first kernel of a call.
#pragma once
#include <math_constants.h>

#include "mla_common.cuh"

namespace mla {

struct PlanInputs {
  const uint32_t* offsets;   // [B+1]
  int B, T;
  KeySource ks;
  int mask, window;
  TokenPlan* plan;           // [T]
  PlanHeader* hdr;
  int* counters;             // [T, 4] split-token claim / written counters, zeroed here
  int* bounds;               // [2K + 1] partition bounds, then each partition's first token, written here
  int K;                     // KV partitions
  __nv_bfloat16* o_lat;      // [T, H, L]: zeroed for tokens without keys
  float* lse_ws;             // [T, H]:    -inf for tokens without keys
  int H, L;
  bool fold;                 // pair consecutive tokens of a request (they share tiles)
};

// Key range [lo, hi) of the query at position pos of request b with cache_len len.
__device__ __forceinline__ void plan_key_range(int mask, int window, int len, int pos, int& lo, int& hi) {
  if (mask == MLA_MASK_NULL) { lo = 0; hi = len; }
  else if (mask == MLA_MASK_CAUSAL) { lo = 0; hi = pos + 1; }
  else { hi = pos + 1; lo = max(0, hi - window); }
}

// Whole block (blockDim.x a multiple of 32, <= 1024).  Each thread owns a
// contiguous run of tokens and counts their tiles; a block-wide exclusive scan
// numbers the tiles globally.
__device__ __forceinline__ void plan_block(const PlanInputs& in) {
  __shared__ int warp_sums[32];
  __shared__ int any_bad;
  const int tid = threadIdx.x, nthr = blockDim.x;
  if (tid == 0) {
    any_bad = 0;
    atomicExch(&in.hdr->status, 0);   // the plan runs first in every call
    in.hdr->pad[0] = 0;               // time-out record
    in.hdr->pad[1] = 0;
  }
  __syncthreads();
  const int per = (in.T + nthr - 1) / nthr;
  const int t0 = min(in.T, tid * per), t1 = min(in.T, t0 + per);
  const KeySource& ks = in.ks;
  int my_tiles = 0;
  bool bad = false;
  for (int t = t0; t < t1; ++t) {
    // request of token t: last b with offsets[b] <= t (one query per request is
    // the common case, so try b = t before searching)
    int b = min(t, in.B - 1);
    if (!((int)in.offsets[b] <= t && t < (int)in.offsets[b + 1])) {
      int lo_b = 0, hi_b = in.B - 1;
      while (lo_b < hi_b) {
        const int mid = (lo_b + hi_b + 1) >> 1;
        if ((int)in.offsets[mid] <= t) lo_b = mid; else hi_b = mid - 1;
      }
      b = lo_b;
    }
    const int qb = (int)in.offsets[b], qe = (int)in.offsets[b + 1];
    int lo = 0, hi = 0;
    int ulo = 0, uhi = 0;   // the tiles walked: the token's own range, or its pair's union
    int ntok = 1;
    bool ok = qb <= t && t < qe && (int)in.offsets[in.B] == in.T;
    const bool follower = in.fold && ((t - qb) & 1);
    const bool paired = in.fold && !follower && t + 1 < qe;
    if (ks.indices) {
      int cnt = ks.topk_lengths ? ks.topk_lengths[b] : ks.idx_stride;
      if (cnt < 0) { cnt = 0; ok = false; }
      hi = min(cnt, ks.idx_stride);
      ulo = lo;
      uhi = hi;                          // a request's tokens share its index list
    } else {
      const int len = (int)ks.cache_lens[b];
      const int pos = len - (qe - qb) + (t - qb);
      if (len > ks.bt_stride * ks.page_size || pos < 0) ok = false;
      plan_key_range(in.mask, in.window, len, pos, lo, hi);
      ulo = lo;
      uhi = hi;
      if (paired) {
        int lo2, hi2;
        plan_key_range(in.mask, in.window, len, pos + 1, lo2, hi2);
        if (hi2 > lo2) {
          if (uhi > ulo) { ulo = min(ulo, lo2); uhi = max(uhi, hi2); }
          else { ulo = lo2; uhi = hi2; }
        }
      }
    }
    if (!ok) { lo = hi = ulo = uhi = 0; bad = true; }
    if (paired) ntok = 2;
    if (follower) { ulo = uhi = 0; ntok = 0; }
    TokenPlan p;
    p.b = b;
    p.lo = ulo;
    p.hi = uhi;
    p.mlo = lo;
    p.mhi = hi;
    p.ntok = ntok;
    p.pad = 0;
    p.tile_first = uhi > ulo ? ulo / kTileKeys : 0;
    p.ntiles = uhi > ulo ? (uhi + kTileKeys - 1) / kTileKeys - p.tile_first : 0;
    p.tile_start = my_tiles;   // local for now
    p.part_first = p.part_last = 0;
    in.plan[t] = p;
    my_tiles += p.ntiles;
  }
  if (bad) any_bad = 1;

  const int lane = tid & 31, wid = tid >> 5;
  int incl = my_tiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = lane < (nthr >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    warp_sums[lane] = v;   // inclusive warp totals
  }
  __syncthreads();
  const int base = (wid > 0 ? warp_sums[wid - 1] : 0) + incl - my_tiles;
  const int total = warp_sums[(nthr >> 5) - 1];
  for (int t = t0; t < t1; ++t) in.plan[t].tile_start += base;
  for (int i = tid; i < 4 * in.T; i += nthr) in.counters[i] = 0;
  if (tid == nthr - 1) in.hdr->total_tiles = total;

  // KV partition bounds: equal cost (tiles plus a charge per token) when every
  // partition gets at least kMinPartitionCost, else equal tile counts.  A bound
  // that falls in a token's charge goes to its first tile, one that falls in
  // its tiles to the tile it reaches.
  const int K = in.K;
  long long my_cost = 0;
  for (int t = t0; t < t1; ++t) {
    const int n = in.plan[t].ntiles;
    my_cost += (long long)kTileCost * n + (n > 0 ? kSegmentCost : 0);
  }
  long long cincl = my_cost;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, cincl, o);
    if (lane >= o) cincl += v;
  }
  __shared__ long long cost_sums[32];
  if (lane == 31) cost_sums[wid] = cincl;
  __syncthreads();
  if (wid == 0) {
    long long v = lane < (nthr >> 5) ? cost_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    cost_sums[lane] = v;
  }
  __syncthreads();
  const long long ctot = cost_sums[(nthr >> 5) - 1];
  // Each thread sets the bounds that fall inside its own tokens, with the token
  // that holds each partition's first tile, and each token's first and last
  // partition: no search over global memory.
  const bool balanced = K > 1 && ctot >= (long long)kMinPartitionCost * K;
  const int q = K > 0 ? (total + K - 1) / K : 0;   // tiles per partition when not balanced
  int* first_token = in.bounds + K + 1;
  long long c0 = (wid > 0 ? cost_sums[wid - 1] : 0) + cincl - my_cost;
  for (int t = t0; t < t1; ++t) {
    TokenPlan& p = in.plan[t];
    if (p.ntiles == 0) continue;
    const int n = p.ntiles;
    const long long c1 = c0 + (long long)kTileCost * n + kSegmentCost;
    if (balanced) {
      // bounds k with c0 <= ctot * k / K < c1: past the token's charge, to the
      // tile the cost reaches (at most its last tile, so the token holds it)
      for (int k = (int)(c0 * K / ctot); k < K; ++k) {
        const long long bk = ctot * k / K;
        if (bk >= c1) break;
        if (bk < c0) continue;
        const long long rel = bk - c0 - kSegmentCost;
        const int into = rel <= 0 ? 0 : (int)min((long long)(n - 1), (rel + kTileCost - 1) / kTileCost);
        in.bounds[k] = p.tile_start + into;
        first_token[k] = t;
      }
      // tile j of the token lies in the last partition whose bound is at or
      // before it: the last k with ctot * k / K <= x(j), where x(j) is the cost
      // up to tile j (the whole token for its last tile)
      auto part_at = [&](int j) {
        const long long x = j == n - 1 ? c1 - 1 : c0 + kSegmentCost + (long long)kTileCost * j;
        return (int)min((long long)(K - 1), ((x + 1) * K - 1) / ctot);
      };
      p.part_first = part_at(0);
      p.part_last = part_at(n - 1);
    } else {
      for (int k = (p.tile_start + q - 1) / q; k < K && (long long)k * q < p.tile_start + n; ++k) {
        in.bounds[k] = k * q;
        first_token[k] = t;
      }
      p.part_first = min(K - 1, p.tile_start / q);
      p.part_last = min(K - 1, (p.tile_start + n - 1) / q);
    }
    c0 = c1;
  }
  // partitions past the last tile (tile counts below K) are empty
  for (int k = tid; k < K; k += nthr)
    if (!balanced && (long long)k * q >= total) {
      in.bounds[k] = total;
      first_token[k] = 0;
    }
  if (tid == 0) in.bounds[K] = total;
  __syncthreads();
  // tokens with no key: zero latent output and lse = -inf (the decode never visits
  // them); each thread clears its own tokens.  A pair's second token is written by
  // the decode unless the pair walks no tile.
  for (int t = t0; t < t1; ++t) {
    const TokenPlan& p = in.plan[t];
    if (p.ntiles != 0) continue;
    if (p.ntok == 0 && t > 0 && in.plan[t - 1].ntiles != 0 && in.plan[t - 1].ntok == 2) continue;
    uint4* o = reinterpret_cast<uint4*>(in.o_lat + (size_t)t * in.H * in.L);
    for (int i = 0; i < in.H * in.L / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
    for (int i = 0; i < in.H; ++i) in.lse_ws[(size_t)t * in.H + i] = -CUDART_INF_F;
  }
  __syncthreads();
  if (tid == 0 && any_bad) atomicOr(&in.hdr->status, kDeviceCheckFailed);
}

}  // namespace mla
