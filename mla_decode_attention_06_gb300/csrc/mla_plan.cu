// K0: per-token key ranges and the global tile numbering that the decode
// partitions split evenly (the on-device counterpart of the packed dispatch
// metadata `scalar_args_buf` and of `num_partitions_in` on the
// generic_flare_mla_decode_kv_cache_ragged page).
#include "mla_kernels.cuh"

namespace mla {

// One block of 1024 threads.  Each thread owns a contiguous run of tokens,
// counts their tiles, and a block-wide exclusive scan numbers them globally.
__global__ void __launch_bounds__(1024) plan_kernel(const uint32_t* __restrict__ offsets, int B, int T,
                                                    KeySource ks, int mask, int window,
                                                    TokenPlan* __restrict__ plan,
                                                    PlanHeader* __restrict__ hdr) {
  __shared__ int warp_sums[32];
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  __syncthreads();
  const int per = (T + blockDim.x - 1) / blockDim.x;
  const int t0 = min(T, tid * per), t1 = min(T, t0 + per);

  int my_tiles = 0;
  for (int t = t0; t < t1; ++t) {
    // request of token t: last b with offsets[b] <= t
    int lo_b = 0, hi_b = B - 1;
    while (lo_b < hi_b) {
      int mid = (lo_b + hi_b + 1) >> 1;
      if ((int)offsets[mid] <= t) lo_b = mid; else hi_b = mid - 1;
    }
    const int b = lo_b;
    const int qb = (int)offsets[b], qe = (int)offsets[b + 1];
    int lo = 0, hi = 0;
    bool ok = qb <= t && t < qe && (int)offsets[B] == T;
    if (ks.indices) {
      int cnt = ks.topk_lengths ? ks.topk_lengths[b] : ks.idx_stride;
      if (cnt < 0) { cnt = 0; ok = false; }
      hi = min(cnt, ks.idx_stride);
    } else {
      const int len = (int)ks.cache_lens[b];
      const int qlen = qe - qb;
      const int pos = len - qlen + (t - qb);
      if (len > ks.bt_stride * ks.page_size || pos < 0) ok = false;
      if (mask == MLA_MASK_NULL) { lo = 0; hi = len; }
      else if (mask == MLA_MASK_CAUSAL) { lo = 0; hi = pos + 1; }
      else { hi = pos + 1; lo = max(0, hi - window); }
    }
    if (!ok) { lo = 0; hi = 0; bad = 1; }
    TokenPlan p;
    p.b = b;
    p.lo = lo;
    p.hi = hi;
    p.tile_first = hi > lo ? lo / kTileKeys : 0;
    p.ntiles = hi > lo ? (hi + kTileKeys - 1) / kTileKeys - p.tile_first : 0;
    p.tile_start = my_tiles;   // local for now
    p.pad[0] = p.pad[1] = 0;
    plan[t] = p;
    my_tiles += p.ntiles;
  }

  // block-wide exclusive scan of my_tiles
  const int lane = tid & 31, wid = tid >> 5;
  int incl = my_tiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    warp_sums[lane] = v;   // inclusive warp totals
  }
  __syncthreads();
  const int base = (wid > 0 ? warp_sums[wid - 1] : 0) + incl - my_tiles;
  for (int t = t0; t < t1; ++t) plan[t].tile_start += base;
  if (tid == blockDim.x - 1) hdr->total_tiles = base + my_tiles;
  __syncthreads();
  // the planner runs first in every call, so it (re)sets the status word
  if (tid == 0) hdr->status = bad ? kDeviceCheckFailed : 0;
}

cudaError_t launch_plan(const uint32_t* offsets, int B, int T, const KeySource& ks, int mask,
                        int window, TokenPlan* plan, PlanHeader* hdr, cudaStream_t s) {
  plan_kernel<<<1, 1024, 0, s>>>(offsets, B, T, ks, mask, window, plan, hdr);
  return cudaGetLastError();
}

}  // namespace mla
