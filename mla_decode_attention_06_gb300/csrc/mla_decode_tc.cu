// K2 (tensor-core version): split-KV MLA decode on tcgen05 with TMEM accumulators.
//
// Work split: partition k of K owns the global 64-key tiles [bounds[k],
// bounds[k+1]), which the plan sets for equal cost (tiles plus a charge per
// token it starts); it walks them as segments, one per query token it
// touches, and writes either the finished latent output (segment = whole
// token) or a partial (o_p, lse_p) that the last partition to claim the token
// merges.  These are the split-KV partitions behind num_partitions_in on the
// generic_flare_mla_decode_kv_cache_ragged page.
//
// With 128 heads sharing every cached row, scores S = Q . K^T (M = 128 heads,
// N = 64 keys, K = 576) and the update O += P . C (M = 128, N = 512, K = 64) are
// dense contractions.  O for 128 heads x 512 latent columns in fp32 would fill all
// 512 TMEM columns, so one partition runs on a cluster of two CTAs that split
// the latent columns of O: CTA r owns columns [256r, 256r + 256).  Scores are
// not split: every cache tile is multicast by TMA into both CTAs (each CTA
// issues half of the boxes), and both compute the full S for the tile with the
// same instructions on the same bits, hence the same S, the same online softmax
// and the same P; each then applies P to its own half of the latent columns.
// Nothing is exchanged between the two CTAs but the tiles and the "stage free"
// signals (tcgen05.commit multicast to both CTAs' empty barriers).
//
// The absorbed query (576 columns per head) is split between TMEM and shared
// memory: latent columns [0, 256) sit in TMEM as the A operand of
// tcgen05.mma (bf16 pairs), latent [256, 512) and the rope columns in
// 128B-swizzled shared memory.  TMEM: O (256) | S, two 64-column buffers |
// Q latent (128).  Narrow latents (64) run the same code on one CTA.
//
// Warp roles (224 threads; 352 with the converter warps of an e4m3 cache):
//   warp 0      TMA producer: the query's shared-memory part once per segment,
//               cache tiles through the page table into a kStages-deep ring,
//               and an L2 prefetch of the tile two ahead.
//   warp 1      TMEM owner and QK issuer (one thread); its other lanes zero
//               cache rows outside the key range before the MMAs read them
//               (0 * NaN would poison P . C).
//   warps 2-5   softmax: thread = head row = TMEM lane.  Writes the query's
//               TMEM part, reads S, masks, keeps running max / sum in the log2
//               domain, writes P (bf16 pairs) back into TMEM where the P . C
//               MMA takes it as its A operand, rescales O only when the running
//               max grows by more than 2^8, and writes the segment's output.
//   warps 6-9   (e4m3 cache) widen the tile's codes x row scale into bf16.
//   last warp   P . C issuer (one thread), so a ready P never waits behind a QK.
// Every wait is bounded in time; a timeout sets a status bit and the kernel
// unwinds without hanging.
#include <math_constants.h>

#include <mutex>

#include "mla_kernels.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace tc {

using namespace sm100;

constexpr int kMaxStages = 4;

// How cache rows reach shared memory.
enum LoadMode : int {
  kLoadDense = 0,   // bf16 pool through the page table, TMA tiles multicast to the cluster
  kLoadFp8 = 1,     // e4m3 pool through the page table: TMA bytes (multicast), widened by converter warps
  kLoadSparse = 2,  // bf16 pool rows named by an index list, TMA gather4: each CTA gathers half
                    // of a tile's boxes and multicasts them to both CTAs of the cluster
};
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows by > 2^8
// The producer reads the page-table entries of the tile this many ahead of the one it
// loads and prefetches that tile's boxes into L2.
constexpr int kPrefetchAhead = 2;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct Smem {   // control block after the stage ring
  uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t kv_conv[kMaxStages];  // e4m3 rows widened (kLoadFp8)
  uint64_t kv_conv_a[kMaxStages];  // ... their first raw box (latent [0, RW)), when NRH > 1
  uint64_t row_mask[kMaxStages];
  uint64_t q_full, q_empty;
  uint64_t qa_full, qa_done;     // query latent [0, QT) staged in shared memory / moved into TMEM
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_free;
  uint64_t conv_sync;            // converters: every code read before the overlapping rows are written
  uint64_t fix_bar, fix_done;    // softmax: partial written / claim outcome published
  uint64_t mrg_full[2], mrg_done[2];   // merge: a half partial landed in its buffer / was read
  uint64_t bye;                  // the other CTAs are done touching this CTA's shared memory
  // kLoadSparse: physical row of each tile row; kLoadFp8: each tile row's scale (fp32
  // bits), copied in with the tile
  alignas(16) int32_t rowid[kMaxStages][64];
  uint32_t tmem_base;
  int abort;
  int fix_last;   // this CTA merges the split token it just finished (it claimed it last)
};

template <int kLatentPerCta, int kCluster, int kMode>
struct Cfg {
  static constexpr int CL = kCluster;
  // A cluster of four folds two query tokens of a request: CTA r takes token slot
  // r / 2 and latent half r % 2; every cache tile is multicast to all four.
  static constexpr int NHALF = CL == 4 ? 2 : CL;    // latent slices of O in the cluster
  static constexpr int NSLOT = CL == 4 ? 2 : 1;     // query tokens walked together
  static constexpr int kMcMask = (1 << CL) - 1;     // every CTA of the cluster
  static constexpr int LC = kLatentPerCta;          // latent columns of O owned by one CTA
  static constexpr int L = LC * NHALF;              // latent width
  static constexpr int NLB = L / 64;                // 64-column latent boxes per cached row
  static constexpr int kBox = 64 * 128;             // one 128B-swizzled box: 64 rows x 128 B
  static constexpr int kStageBytes = (NLB + 1) * kBox;   // latent boxes + one rope box
  static constexpr int kStages = CL >= 2 ? 2 : kMaxStages;
  static constexpr int QT = L < 256 ? L : 256;      // latent columns of the query held in TMEM
  static constexpr int NQS = (L - QT) / 64;         // latent boxes of the query in shared memory
  static constexpr int kQBox = 128 * 128;           // 128 rows x 128 B
  static constexpr int kQBytes = (NQS + 1) * kQBox; // + the rope box
  static constexpr int kSCol = LC;                  // two 64-column S buffers after O
  static constexpr int kQCol = LC + 128;            // query latent [0, QT) as bf16 pairs
  static constexpr int kTmemCols = (kQCol + QT / 2) <= 256 ? 256 : 512;
  static constexpr int RW = L < 256 ? L : 256;      // e4m3 bytes per raw box row
  static constexpr int NRH = L / RW;                // raw boxes per cached row
  static constexpr int kRawOff = NLB >= 8 ? 4 * kBox : 0;   // codes land where the last latent boxes go
  static constexpr int kConvThreads = 64 * NRH;                // warps 6.. (kLoadFp8): one per row and raw box
  static constexpr int kPvWarp = kMode == kLoadFp8 ? 6 + kConvThreads / 32 : 6;   // the P . C issuer
  static constexpr int kThreads = 32 * (kPvWarp + 1);
  static constexpr int kRegionBytes = kQBytes + kStages * kStageBytes;   // query buffer + stage ring
  static constexpr int kMrgHalf = (LC / 2) * kMaxHeads * 4;               // merge: one half partial slice
  static constexpr int kStgBytes = kMaxHeads * (LC * 2 + 16);             // merge: staged output rows
  static constexpr int kSmem = 1024 + kRegionBytes + (int)sizeof(Smem);
  static_assert(LC % 64 == 0 && (CL == 1 || CL == 2 || CL == 4), "latent slice");
  static_assert(kQCol + QT / 2 <= 512, "TMEM columns");
  static_assert(kStgBytes + 2 * kMrgHalf <= kRegionBytes, "merge buffers in the idle region");
  static_assert(kMode != kLoadFp8 || NRH % CL == 0, "raw boxes split over the cluster");
  static_assert(kMode != kLoadFp8 || NRH == 1 || QT == RW, "raw box 0 is the QK's TMEM-operand part");
  static_assert(QT / 64 <= NQS + 1, "the query staging fits the query buffer");
  static_assert(kSmem <= 232448, "shared memory");
};

struct Maps {
  CUtensorMap kv_lat;    // bf16 latent boxes (dense: page rows, sparse: 1 row) / e4m3 bytes (kLoadFp8)
  CUtensorMap kv_rope;   // bf16 rope box
  CUtensorMap q;         // absorbed queries [T * 128, L + R], 64-column boxes
};

// Walks the segments of partition k (tiles [g0, g1)): calls f(si, t, plan, first_tile, end_tile,
// is_first_segment, next_t) where next_t is the token of the following segment
// (-1 if none).  Consecutive segments belong to consecutive tokens, so the plan
// entry of token t + 1 is loaded when segment t starts and is ready at the
// boundary; only a token without keys in between (they share tile_start) falls
// back to the search.
template <class F>
__device__ __forceinline__ void for_each_segment(const DecodeArgs& a, int k, int g0, int g1, F&& f) {
  int g = g0;
  int si = 0;
  int t = g0 < g1 ? a.bounds[a.K + 1 + k] : 0;   // the token holding tile g0, recorded by the plan
  while (g < g1) {
    if (t < 0 || t >= a.T) {   // a plan that does not cover g: report, never loop
      atomicOr(&a.hdr_mut->status, kDeviceCheckFailed);
      return;
    }
    const TokenPlan tp = a.plan[t];
    const TokenPlan tn = t + 1 < a.T ? a.plan[t + 1] : TokenPlan{};
    const int ia = g - tp.tile_start;
    const int ie = min(g1, tp.tile_start + tp.ntiles) - tp.tile_start;
    if (ia < 0 || ie <= ia) {
      atomicOr(&a.hdr_mut->status, kDeviceCheckFailed);
      return;
    }
    const int g_next = tp.tile_start + ie;
    int next_t = -1;
    if (g_next < g1) next_t = (t + 1 < a.T && tn.ntiles > 0) ? t + 1 : token_of_tile(a.plan, a.T, g_next);
    f(si, t, tp, ia, ie, g == g0, next_t);
    g = g_next;
    t = next_t;
    ++si;
  }
}

__device__ __forceinline__ bool aborted(const Smem* cs) {
  return *reinterpret_cast<const volatile int*>(&cs->abort) != 0;
}

// First time-out of a call: barrier offset in shared memory, thread and block.
__device__ __forceinline__ void record_timeout(uint64_t* bar, PlanHeader* hdr) {
  const int code = (int)(0x80000000u | ((uint32_t)threadIdx.x << 18) | (smem_u32(bar) & 0x3FFFFu));
  if (atomicCAS(&hdr->pad[0], 0, code) == 0) hdr->pad[1] = (int)blockIdx.x;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Smem* cs, PlanHeader* hdr) {
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  record_timeout(bar, hdr);
  atomicOr(&hdr->status, kDeviceTimeout);
  *reinterpret_cast<volatile int*>(&cs->abort) = 1;
  return false;
}

// Bounded wait until the counter that other CTAs increment reaches `target`.
__device__ __forceinline__ bool wait_count(const int* ctr, int target, uint64_t limit_ns) {
  if (*reinterpret_cast<const volatile int*>(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(32);
    if (*reinterpret_cast<const volatile int*>(ctr) >= target) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool wait_cluster_or_abort(uint64_t* bar, uint32_t parity, Smem* cs,
                                                      PlanHeader* hdr) {
  if (mbar_wait<true>(bar, parity, kWaitLimitNs)) return true;
  record_timeout(bar, hdr);
  atomicOr(&hdr->status, kDeviceTimeout);
  *reinterpret_cast<volatile int*>(&cs->abort) = 1;
  return false;
}

// Four rows (y0..y3) of one box column range into four consecutive smem rows.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y0, int y1,
                                            int y2, int y3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
      "%5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3)
      : "memory");
}

// The same four rows delivered to every CTA of the cluster in `cta_mask`.
__device__ __forceinline__ void tma_gather4_mc(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y0, int y1,
                                               int y2, int y3, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "h"(cta_mask)
      : "memory");
}

// Two e4m3 codes times a row scale, rounded to a bf16 pair (low half = first code):
// the codes widen exactly (through f16), one packed fp32 multiply (round to
// nearest, per lane as two scalar ones) scales both, one conversion rounds both.
__device__ __forceinline__ uint32_t e4m3x2_scaled_bf16x2(uint16_t two, float scale) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  float x, y;
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %4};\n\tmul.rn.f32x2 d, a, b;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(x), "=f"(y)
      : "f"(f.x), "f"(f.y), "f"(scale));
  const __nv_bfloat162 b = __floats2bfloat162_rn(x, y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Two floats rounded to a bf16 pair (low half = lo) in one conversion.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Partials of split tokens are stored interleaved, [partition, slot, L / 4, H]
// float4: a warp's 32 head rows of one 4-column chunk are 512 contiguous bytes,
// and one CTA's latent half of one partial is a single contiguous block.  A
// partition has 2 * ns slots: its first and its last segment, each with ns token
// slots (two when tokens are folded in pairs); slot = segment slot * ns + token slot.
__device__ __forceinline__ size_t part_index(int k, int slot, int c, int row, int L, int H, int ns) {
  return ((size_t)(k * 2 * ns + slot) * (L / 4) + c) * H + row;
}

// The merge of merge_in_tmem (below) with per-thread loads instead of bulk
// copies, every partial read from global memory: the e4m3 instance merges an
// earlier segment's token this way (measured faster there; the bf16 instances
// use merge_in_tmem with no partial in TMEM).  Same operations in the same
// order, so the bits are the same.
__device__ __noinline__ void merge_split_token(const DecodeArgs& a, int t, const TokenPlan& tp, int kf, int kl,
                                               int slot_kf, uint32_t rank, int row, int lat_x0, int LC, int ns,
                                               int ts) {
  const int H = a.d.num_heads, L = a.d.kv_lora_rank;
  const float4* __restrict__ part_o = reinterpret_cast<const float4*>(a.part_o);
  const float* __restrict__ part_lse = a.part_lse;
  auto slot_of = [&](int k) { return (k == kf ? slot_kf : 0) * ns + ts; };
  auto lse_of = [&](int k) { return __ldcg(part_lse + ((size_t)(k * 2 * ns + slot_of(k)) * 2 + rank) * H + row); };
  float mx = -CUDART_INF_F;
  for (int k = kf; k <= kl; ++k) mx = fmaxf(mx, lse_of(k));
  float sum = 0.f;
  if (mx != -CUDART_INF_F)
    for (int k = kf; k <= kl; ++k) sum += __expf(lse_of(k) - mx);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  for (int col0 = 0; col0 < LC; col0 += 32) {
    float4 acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mx != -CUDART_INF_F) {
      for (int k = kf; k <= kl; ++k) {
        const float w = __expf(lse_of(k) - mx) * inv;
        const int c0 = (lat_x0 + col0) / 4;
        float4 u[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) u[i] = __ldcg(part_o + part_index(k, slot_of(k), c0 + i, row, L, H, ns));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[i].x = fmaf(w, u[i].x, acc[i].x);
          acc[i].y = fmaf(w, u[i].y, acc[i].y);
          acc[i].z = fmaf(w, u[i].z, acc[i].z);
          acc[i].w = fmaf(w, u[i].w, acc[i].w);
        }
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(a.o_lat + ((size_t)t * H + row) * L + lat_x0 + col0);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      dst[i] = make_uint4(pack_bf16(acc[2 * i].x, acc[2 * i].y), pack_bf16(acc[2 * i].z, acc[2 * i].w),
                          pack_bf16(acc[2 * i + 1].x, acc[2 * i + 1].y), pack_bf16(acc[2 * i + 1].z, acc[2 * i + 1].w));
  }
  if (rank == 0) a.lse_ws[(size_t)t * H + row] = mx != -CUDART_INF_F ? mx + __logf(sum) : -CUDART_INF_F;
}

// Warp-uniform forms: every lane waits, then the warp votes, so lanes never
// diverge around warp-collective instructions (tcgen05.ld/st, shuffles, votes).
__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, Smem* cs, PlanHeader* hdr) {
  const bool ok = wait_or_abort(bar, parity, cs, hdr);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool wwait_cluster(uint64_t* bar, uint32_t parity, Smem* cs, PlanHeader* hdr) {
  const bool ok = wait_cluster_or_abort(bar, parity, cs, hdr);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool waborted(const Smem* cs) { return __any_sync(0xffffffffu, aborted(cs)); }

// Log-sum-exp merge of one split token's partials for head `row`, latent
// columns [lat_x0, lat_x0 + LC):  lse = ln sum_p e^{lse_p},
// o = sum_p e^{lse_p - lse} o_p.  Partitions with an empty key set carry
// lse_p = -inf and drop out.  Partition kf holds the token in slot 1 (its last
// segment) if the token began inside its range, every other partition in slot 0.
// Run by the last partition to claim the token, after its own final segment,
// when the query buffer and stage ring are idle.  If the token is that final
// segment's (k in [kf, kl]), O in TMEM still holds this CTA's own partial
// (unnormalised; 1 / row sum = inv); otherwise (k = -1: a token of the CTA's
// first segment) every partial is in global memory.  Each partial's slice
// (one contiguous block of the interleaved layout) comes in as two halves of
// LC / 2 columns by bulk copy, double-buffered at the end of the idle region,
// the first two issued before the weights are known.  acc = sum over
// partitions, in order, of fmaf(w_p, o_p, acc) from zero, whichever partition
// merges, so the bits do not depend on it.  acc lives in TMEM at `tacc` (the S
// and query columns, idle after the last QK).  Each thread stages its own bf16
// output row at the start of the region (rows padded by 16 bytes) and writes it
// with one bulk copy.  Warp-uniform; false on a time-out.
template <int LC>
__device__ __noinline__ bool merge_in_tmem(const DecodeArgs& a, Smem* cs, int t, const TokenPlan& tp, int k, int kf,
                                           int kl, int slot_kf, uint32_t rank, int row, int lat_x0, uint32_t trow,
                                           uint32_t tacc, float lse_own, float inv, uint8_t* stg, uint8_t* hb,
                                           int& nmrg, int ns, int ts) {
  constexpr int LH = LC / 2;                            // columns per half slice
  constexpr uint32_t kHalf = (uint32_t)LH * kMaxHeads * 4;
  constexpr int kStgStride = LC * 2 + 16;               // bytes per staged row
  const int H = a.d.num_heads, L = a.d.kv_lora_rank;
  PlanHeader* hdr = a.hdr_mut;
  const bool live = row < H;
  auto slot_of = [&](int kk) { return (kk == kf ? slot_kf : 0) * ns + ts; };
  auto lse_ptr = [&](int kk) { return a.part_lse + ((size_t)(kk * 2 * ns + slot_of(kk)) * 2 + rank) * H + row; };
  const int np = kl - kf + 1;
  const bool own = k >= kf && k <= kl;                  // this CTA's partial is in TMEM (O)
  const int nj = 2 * (np - (own ? 1 : 0));              // half slices to bring in
  const uint32_t half_bytes = (uint32_t)(LH * H * 4);
  auto issue = [&](int j) {                             // thread row 0: bring in half slice j
    const int g = nmrg + j, b = g & 1;
    if (g >= 2 && !wait_or_abort(&cs->mrg_done[b], ((g - 2) >> 1) & 1, cs, hdr)) return false;
    int p = kf + (j >> 1);
    if (own && p >= k) ++p;
    mbar_arrive_expect_tx(&cs->mrg_full[b], half_bytes);
    bulk_copy_g2s(hb + b * kHalf,
                  reinterpret_cast<const float4*>(a.part_o) +
                      part_index(p, slot_of(p), lat_x0 / 4 + (j & 1) * (LH / 4), 0, L, H, ns),
                  half_bytes, &cs->mrg_full[b]);
    return true;
  };
  bool ok = true;
  if (row == 0) {
    fence_proxy_async_global();
    if (nj > 0) ok = issue(0);
    if (ok && nj > 1) ok = issue(1);
  }
  if (!__all_sync(0xffffffffu, ok)) return false;
  // max, then sum over p in order of e^(lse_p - max); up to eight partitions'
  // log-sum-exps are loaded once, eight at a time
  float lv0[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int kk = kf + j;
    lv0[j] = kk > kl ? -CUDART_INF_F : (kk == k ? lse_own : __ldcg(lse_ptr(kk)));
  }
  auto lse_at = [&](int kk) {
    if (kk - kf < 8) {
      float v = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 8; ++j) v = (kk - kf == j) ? lv0[j] : v;
      return v;
    }
    return kk == k ? lse_own : __ldcg(lse_ptr(kk));
  };
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < 8; ++j) mx = fmaxf(mx, lv0[j]);
  for (int kk = kf + 8; kk <= kl; ++kk) mx = fmaxf(mx, lse_at(kk));
  float sum = 0.f;
  if (mx != -CUDART_INF_F) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < np) sum += __expf(lv0[j] - mx);
    for (int kk = kf + 8; kk <= kl; ++kk) sum += __expf(lse_at(kk) - mx);
  }
  const float inv_sum = sum > 0.f ? 1.f / sum : 0.f;
  int j = 0;
  for (int kk = kf; kk <= kl; ++kk) {
    const float w = mx != -CUDART_INF_F ? __expf(lse_at(kk) - mx) * inv_sum : 0.f;
    const bool first = kk == kf;
    if (kk == k) {
      // 32 columns per step, every load of the step in flight before one wait
#pragma unroll 1
      for (int col = 0; col < LC; col += 32) {
        uint32_t u[32], acc[32];
        tmem_ld32(trow + col, u);
        if (!first) tmem_ld32(tacc + col, acc);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          acc[i] = __float_as_uint(fmaf(w, __uint_as_float(u[i]) * inv, first ? 0.f : __uint_as_float(acc[i])));
        tmem_st32(tacc + col, acc);
      }
      tmem_st_wait();
      continue;
    }
    for (int h = 0; h < 2; ++h, ++j) {
      const int g = nmrg + j, b = g & 1;
      if (!wwait(&cs->mrg_full[b], (g >> 1) & 1, cs, hdr)) return false;
      const float4* sp = reinterpret_cast<const float4*>(hb + b * kHalf);
#pragma unroll 1
      for (int col = 0; col < LH; col += 32) {
        uint32_t acc[32];
        const uint32_t tc = tacc + h * LH + col;
        if (!first) tmem_ld32(tc, acc);
        float4 x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = live ? sp[(col / 4 + i) * H + row] : make_float4(0.f, 0.f, 0.f, 0.f);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float v[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[4 * i + e] = __float_as_uint(fmaf(w, v[e], first ? 0.f : __uint_as_float(acc[4 * i + e])));
        }
        tmem_st32(tc, acc);
      }
      tmem_st_wait();
      mbar_arrive(&cs->mrg_done[b]);
      if (row == 0 && j + 2 < nj) ok = issue(j + 2);
      if (!__all_sync(0xffffffffu, ok)) return false;
    }
  }
  nmrg += nj;
  // the merged row as bf16 in this thread's staging row, then one bulk copy
  uint8_t* srow = stg + (size_t)row * kStgStride;
#pragma unroll 1
  for (int col = 0; col < LC; col += 32) {
    uint32_t r[32];
    tmem_ld32(tacc + col, r);
    tmem_ld_wait();
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] = pack_bf16(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
    uint4* d = reinterpret_cast<uint4*>(srow + col * 2);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  }
  if (live) {
    fence_proxy_async_smem();
    bulk_copy_s2g(a.o_lat + ((size_t)t * H + row) * L + lat_x0, srow, LC * 2);
    bulk_commit();
    if (rank == 0) a.lse_ws[(size_t)t * H + row] = mx != -CUDART_INF_F ? mx + __logf(sum) : -CUDART_INF_F;
    bulk_wait_all();
  }
  return true;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


template <int LC, int CL, int MODE>
__global__ void __launch_bounds__(Cfg<LC, CL, MODE>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ Maps maps, const DecodeArgs a) {
  using C = Cfg<LC, CL, MODE>;
  constexpr int S = C::kStages;
  constexpr int L = C::L;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = sm;                                  // query latent [QT, L) boxes, then the rope box
  uint8_t* sStage = sQ + C::kQBytes;                 // S stages of NLB latent boxes + 1 rope box
  Smem* cs = reinterpret_cast<Smem*>(sStage + S * C::kStageBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = CL >= 2 ? cluster_ctarank() : 0u;   // rank in the cluster
  // latent half of O this CTA owns, and its query token slot (folded pairs); both
  // compile-time known where the cluster walks one token
  const uint32_t rank = C::NSLOT > 1 ? crank % C::NHALF : crank;
  const int tslot = C::NSLOT > 1 ? (int)(crank / C::NHALF) : 0;
  const int k = blockIdx.x / CL;
  PlanHeader* hdr = a.hdr_mut;
  const int H = a.d.num_heads;
  const int KQ = L + a.d.qk_rope;
  const int lat_x0 = (int)rank * LC;
  // cache rope columns: they start at L in a bf16 row, at byte L (bf16 column L / 2) in an e4m3 row
  const int rope_x0 = MODE == kLoadFp8 ? L / 2 : L;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&cs->kv_full[s], 1);
      mbar_init(&cs->kv_empty[s], CL);   // one tcgen05.commit from each CTA of the cluster
      mbar_init(&cs->kv_conv[s], C::kConvThreads);
      mbar_init(&cs->kv_conv_a[s], C::kConvThreads);
    }
    mbar_init(&cs->q_full, 1 + 128);     // producer (TMA bytes) + every softmax thread (TMEM part)
    mbar_init(&cs->q_empty, 1);
    mbar_init(&cs->qa_full, 1);
    mbar_init(&cs->qa_done, 128);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&cs->s_full[b], 1);
      mbar_init(&cs->p_full[b], 128);
      mbar_init(&cs->pv_done[b], 1);
    }
    mbar_init(&cs->o_free, 128);
    mbar_init(&cs->conv_sync, C::kConvThreads);
    mbar_init(&cs->fix_bar, 128);
    mbar_init(&cs->fix_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&cs->mrg_full[i], 1);
      mbar_init(&cs->mrg_done[i], 128);
    }
    mbar_init(&cs->bye, CL > 1 ? CL - 1 : 1);   // one arrival from every other CTA
    cs->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&cs->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&maps.kv_lat);
    prefetch_tensormap(&maps.kv_rope);
    prefetch_tensormap(&maps.q);
  }
  tc_fence_before();
  // both CTAs' barriers are initialised before either multicasts into the other
  if (CL >= 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cs->tmem_base;
  // the W_uv kernel may start its prologue now; the plan and q_full of the
  // absorb kernel must be complete before anything below reads them
  griddep_launch_dependents();
  griddep_wait();

  const int g0 = a.bounds[k], g1 = a.bounds[k + 1];
  const int ps = a.ks.page_size;
  const int rows_per_load = ps < kTileKeys ? ps : kTileKeys;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    auto load_box = [&](void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
      if (CL >= 2) tma_load_2d_mc(dst, map, bar, x, y, (uint16_t)C::kMcMask);
      else tma_load_2d(dst, map, bar, x, y);
    };
    int c = 0;
    bool bad = false;
    for_each_segment(a, k, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool, int next_t) {
      const int tq = tslot < tp.ntok ? t + tslot : t;   // this CTA's query token (slot 0's when none)
      bool q_pending = true;   // the query's shared-memory part goes right after the first tile
      // The next segment's absorbed query is read at this segment's end; it goes
      // into L2 a few tiles before that (earlier, the cache stream evicts it again).
      const int q_prefetch_at = ie - 4 > ia ? ie - 4 : ia;
      constexpr int kOwn = MODE == kLoadFp8 ? C::NRH / CL : C::NLB / CL;   // this CTA's boxes per load
      const int nloads = kTileKeys / rows_per_load;
      const uint64_t lmask = rows_per_load == 64 ? ~0ull : ((1ull << rows_per_load) - 1);
      // rows j and j + 32 of tile `it`: which key / slot, and is it live?  fetch
      // only reads the page-table entries (or indices) so that several tiles'
      // reads can be in flight at once; finish checks and decodes them.
      auto fetch = [&](int it, int (&raw)[2]) {
        const int key0 = (tp.tile_first + it) * kTileKeys;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int key = key0 + lane + 32 * h;
          raw[h] = 0;
          if (key >= tp.lo && key < tp.hi)
            raw[h] = MODE == kLoadSparse ? a.ks.indices[(size_t)tp.b * a.ks.idx_stride + key]
                                         : a.ks.block_table[(size_t)tp.b * a.ks.bt_stride + key / ps];
        }
      };
      auto finish = [&](int it, const int (&raw)[2], bool (&v)[2], int (&rid)[2], int (&pg)[2]) {
        const int key0 = (tp.tile_first + it) * kTileKeys;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int key = key0 + lane + 32 * h;
          bool ok = key >= tp.lo && key < tp.hi;
          rid[h] = 0;
          pg[h] = 0;
          if (ok) {
            if (MODE == kLoadSparse) {
              const int idx = raw[h];
              if (idx >= 0 && idx < a.ks.num_pages * ps) {
                rid[h] = idx;
              } else {
                ok = false;
                if (idx != -1) bad = true;
              }
            } else {
              const int page = raw[h];
              if (page < 0 || page >= a.ks.num_pages) { ok = false; bad = true; }
              else { pg[h] = page; rid[h] = page * ps + key % ps; }
            }
          }
          v[h] = ok;
        }
      };
      auto lookup = [&](int it, bool (&v)[2], int (&rid)[2], int (&pg)[2]) {
        int raw[2];
        fetch(it, raw);
        finish(it, raw, v, rid, pg);
      };
      // the pool row of load p of a tile, from the lane that looked up its first live row
      auto load_row = [&](int it, int p, uint64_t pm, const int (&pg)[2]) {
        const int r0 = p * rows_per_load;
        const int fr = r0 + __ffsll((long long)pm) - 1;
        const int pa = __shfl_sync(0xffffffffu, pg[0], fr & 31);
        const int pb = __shfl_sync(0xffffffffu, pg[1], fr & 31);
        const int page = fr < 32 ? pa : pb;
        return page * ps + ((tp.tile_first + it) * kTileKeys + r0) % ps;
      };
      // L2 prefetch of this CTA's boxes of tile `it` (paged modes): its load, issued
      // when a stage frees up, then reads L2 instead of waiting on HBM
      auto prefetch_from = [&](int it, const bool (&v)[2], const int (&pg)[2]) {
        if (MODE == kLoadSparse || it >= ie) return;
        const uint64_t mask = (uint64_t)__ballot_sync(0xffffffffu, v[0]) |
                              ((uint64_t)__ballot_sync(0xffffffffu, v[1]) << 32);
        for (int p = 0; p < nloads; ++p) {
          const uint64_t pm = (mask >> (p * rows_per_load)) & lmask;
          if (!pm) continue;
          const int y = load_row(it, p, pm, pg);
          if (lane < kOwn) {
            if (MODE == kLoadFp8) tma_prefetch_2d(&maps.kv_lat, ((int)crank * kOwn + lane) * C::RW, y);
            else tma_prefetch_2d(&maps.kv_lat, 64 * ((int)crank * kOwn + lane), y);
          } else if (lane == kOwn && crank == 0) {
            tma_prefetch_2d(&maps.kv_rope, rope_x0, y);
          }
        }
      };
      auto issue_qa = [&]() {   // the query's TMEM part (latent [0, QT)) into the staging buffer
        if (lane == 0) {
          mbar_arrive_expect_tx(&cs->qa_full, (C::QT / 64) * C::kQBox);
          for (int i = 0; i < C::QT / 64; ++i)
            tma_load_2d(sQ + i * C::kQBox, &maps.q, &cs->qa_full, 64 * i, tq * kMaxHeads);
        }
        __syncwarp();
      };
      // the partition's first query goes out before any page-table read: the
      // first QK waits on it, not on the cache
      const bool qa_sent = si == 0;
      if (qa_sent) issue_qa();
      if (si > 0 && MODE != kLoadSparse && ia + 1 < ie) {
        // a later segment waits for a free stage first: bring its second tile
        // into L2 meanwhile
        bool v1[2];
        int rid1[2], pg1[2];
        lookup(ia + 1, v1, rid1, pg1);
        prefetch_from(ia + 1, v1, pg1);
      }
      for (int it = ia; it < ie; ++it, ++c) {
        if (waborted(cs)) return;
        const int s = c % S;
        if (lane == 0 && it == q_prefetch_at && next_t >= 0 && next_t + tslot < a.T)
          bulk_prefetch_l2(a.q_full + (size_t)(next_t + tslot) * kMaxHeads * KQ, (uint32_t)(kMaxHeads * KQ * 2));
        if (it == q_prefetch_at && next_t < 0 && ie < tp.ntiles) {
          // the partition's last segment ends inside its token: if this partition
          // finishes the token last it merges the later partitions' partials
          // (written long ago, by their first segments); bring this CTA's slices
          // of them into L2 now (one lane per partition)
          const int kl = tp.part_last;
          const int L4 = L / 4, Hh = a.d.num_heads;
          constexpr int NS = C::NSLOT;
          for (int kk = k + 1 + lane; kk <= kl; kk += 32) {
            bulk_prefetch_l2(reinterpret_cast<const float4*>(a.part_o) + ((size_t)(kk * 2 * NS + tslot) * L4 + lat_x0 / 4) * Hh,
                             (uint32_t)(LC * Hh * 4));
            bulk_prefetch_l2(a.part_lse + (size_t)(kk * 2 * NS + tslot) * 2 * Hh, (uint32_t)(2 * Hh * 4));
          }
        }
        // global reads of this tile and (bf16 pool) of the one two ahead, for its
        // L2 prefetch, issued together before the wait for the stage so their
        // latency overlaps it.  The e4m3 kernel, short of registers, reads the
        // tile two ahead after issuing this one's loads instead.
        int raw[2], raw2[2];
        fetch(it, raw);
        const bool pf = MODE == kLoadDense && it + kPrefetchAhead < ie;
        if (pf) fetch(it + kPrefetchAhead, raw2);
        bool v[2], v2[2];
        int rid[2], pg[2], rid2[2], pg2[2];
        if (MODE != kLoadDense) finish(it, raw, v, rid, pg);
        // stage s is free in both CTAs once both have committed their P . C of its last tile
        if (c >= S && !wwait(&cs->kv_empty[s], ((c / S) & 1) ^ 1, cs, hdr)) return;
        if (MODE == kLoadDense) finish(it, raw, v, rid, pg);
        if (pf) finish(it + kPrefetchAhead, raw2, v2, rid2, pg2);
        if (MODE == kLoadSparse) {
          cs->rowid[s][lane] = rid[0];
          cs->rowid[s][lane + 32] = rid[1];
        }
        const uint64_t mask = (uint64_t)__ballot_sync(0xffffffffu, v[0]) |
                              ((uint64_t)__ballot_sync(0xffffffffu, v[1]) << 32);
        uint8_t* st = sStage + s * C::kStageBytes;
        uint8_t* st_rope = st + C::NLB * C::kBox;
        if (MODE == kLoadSparse) {
          // every row is fetched (row 0 stands in for a dead slot; its P . C part is zeroed);
          // each CTA gathers half of the boxes and multicasts them to both
          if (lane == 0) {
            cs->row_mask[s] = mask;
            mbar_arrive_expect_tx(&cs->kv_full[s], 64 * (C::NLB + 1) * 128);
          }
          __syncwarp();
          if (lane < 16) {
            // this CTA's share of the boxes (both CTAs see the same rows), multicast
            const int r0 = 4 * lane;
            const int y0 = cs->rowid[s][r0], y1 = cs->rowid[s][r0 + 1];
            const int y2 = cs->rowid[s][r0 + 2], y3 = cs->rowid[s][r0 + 3];
            constexpr int kOwnBoxes = C::NLB / CL;
#pragma unroll
            for (int j = 0; j < kOwnBoxes; ++j) {
              const int i = (int)crank * kOwnBoxes + j;
              if (CL >= 2)
                tma_gather4_mc(st + i * C::kBox + r0 * 128, &maps.kv_lat, &cs->kv_full[s], 64 * i, y0, y1, y2, y3,
                               (uint16_t)C::kMcMask);
              else
                tma_gather4(st + i * C::kBox + r0 * 128, &maps.kv_lat, &cs->kv_full[s], 64 * i, y0, y1, y2, y3);
            }
            if (crank == 0) {
              if (CL >= 2)
                tma_gather4_mc(st_rope + r0 * 128, &maps.kv_rope, &cs->kv_full[s], rope_x0, y0, y1, y2, y3,
                               (uint16_t)C::kMcMask);
              else
                tma_gather4(st_rope + r0 * 128, &maps.kv_rope, &cs->kv_full[s], rope_x0, y0, y1, y2, y3);
            }
          }
        } else {
          // pages of this tile that hold at least one live row; both CTAs count the
          // same bytes, most of which the other CTAs' multicasts deliver (an e4m3 row's
          // 4-byte scale each CTA copies for itself)
          const uint32_t row_bytes = (MODE == kLoadFp8 ? L + 4 : C::NLB * 128) + 128;
          uint32_t live_rows = 0;
          for (int p = 0; p < nloads; ++p)
            if ((mask >> (p * rows_per_load)) & lmask) live_rows += rows_per_load;
          if (lane == 0) {
            cs->row_mask[s] = mask;
            mbar_arrive_expect_tx(&cs->kv_full[s], live_rows * row_bytes);
          }
          __syncwarp();
          for (int p = 0; p < nloads; ++p) {
            const uint64_t pm = (mask >> (p * rows_per_load)) & lmask;
            if (!pm) continue;
            const int r0 = p * rows_per_load;
            const int y = load_row(it, p, pm, pg);
            // one box per lane: this CTA's share of the latent (or raw e4m3) boxes, then the rope box (rank 0)
            if (lane < kOwn) {
              if (MODE == kLoadFp8) {
                const int h = (int)crank * kOwn + lane;
                load_box(st + C::kRawOff + h * 64 * C::RW + r0 * C::RW, &maps.kv_lat, &cs->kv_full[s], h * C::RW, y);
              } else {
                const int i = (int)crank * kOwn + lane;
                load_box(st + i * C::kBox + r0 * 128, &maps.kv_lat, &cs->kv_full[s], 64 * i, y);
              }
            } else if (lane == kOwn && crank == 0) {
              load_box(st_rope + r0 * 128, &maps.kv_rope, &cs->kv_full[s], rope_x0, y);
            } else if (MODE == kLoadFp8 && lane == kOwn + 1) {
              // the load's row scales: rows y .. y + rows_per_load - 1 are consecutive
              // (one page), y a multiple of 8, so the copy is 16-byte aligned
              bulk_copy_g2s(&cs->rowid[s][r0], a.kv_scales + y, (uint32_t)rows_per_load * 4, &cs->kv_full[s]);
            }
          }
          if (pf) {
            prefetch_from(it + kPrefetchAhead, v2, pg2);
          } else if (MODE == kLoadFp8 && it + kPrefetchAhead < ie) {
            lookup(it + kPrefetchAhead, v2, rid2, pg2);
            prefetch_from(it + kPrefetchAhead, v2, pg2);
          }
        }
        __syncwarp();
        if (q_pending) {
          // The previous segment's last QK has read the query buffers.  The query's
          // TMEM part (latent [0, QT)) comes in through the shared-memory buffer
          // first: TMA, then the softmax threads copy their rows into TMEM; then
          // the buffer takes the shared-memory part (latent [QT, L) and rope).
          if (!qa_sent) {
            if (!wwait(&cs->q_empty, (si - 1) & 1, cs, hdr)) return;
            issue_qa();
          }
          if (!wwait(&cs->qa_done, si & 1, cs, hdr)) return;
          if (lane == 0) {
            mbar_arrive_expect_tx(&cs->q_full, C::kQBytes);
            for (int i = 0; i < C::NQS; ++i)
              tma_load_2d(sQ + i * C::kQBox, &maps.q, &cs->q_full, C::QT + 64 * i, tq * kMaxHeads);
            tma_load_2d(sQ + C::NQS * C::kQBox, &maps.q, &cs->q_full, L, tq * kMaxHeads);
          }
          __syncwarp();
          q_pending = false;
        }
      }
    });
    if (bad) atomicOr(&hdr->status, kDeviceCheckFailed);
    // no TMA write of ours still in flight, and (cluster) no commit of the peer
    // still to arrive on our barriers, when the CTA leaves
    if (lane == 0) {
      for (int j = c - S; j < c; ++j) {
        if (j < 0) continue;
        mbar_wait(&cs->kv_full[j % S], (j / S) & 1, kWaitLimitNs);
        if (CL >= 2) mbar_wait(&cs->kv_empty[j % S], (j / S) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- QK issuer
    // QK of tile c as soon as its rows have landed.  The S buffer of tile c held
    // P of tile c - 2, which the P . C warp reads: wait for that MMA to complete.
    // The MMA queue is shallow, so the 36 MMAs are issued back to back.
    const uint32_t idesc_qk = idesc_bf16_f32(128, 64, false, false);
    // K-major operand descriptors of the query boxes and of stage 0; the start
    // address field is advanced by (byte offset >> 4) for every other operand
    const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 1024, kLayoutSw128);
    const uint64_t dk0 = smem_desc(smem_u32(sStage), 16, 1024, kLayoutSw128);
    int cq = 0, nseg = 0;
    for_each_segment(a, k, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool, int) {
      nseg = si + 1;
      if (waborted(cs)) return;
      // the query's TMEM part is in place before its shared-memory part lands
      // (that load reuses the staging buffer): the segment's first QK issues its
      // TMEM-operand MMAs in between
      if (!wwait(&cs->qa_done, si & 1, cs, hdr)) return;
      bool q_smem = false;
      for (int it = ia; it < ie; ++it, ++cq) {
        if (waborted(cs)) return;
        const int s = cq % S, b = cq & 1;
        const uint32_t par = (cq / S) & 1;
        if (cq >= 2 && !wwait(&cs->pv_done[b], ((cq - 2) >> 1) & 1, cs, hdr)) return;
        if (!wwait(MODE != kLoadFp8 ? &cs->kv_full[s] : C::NRH > 1 ? &cs->kv_conv_a[s] : &cs->kv_conv[s], par, cs,
                   hdr))
          return;
        const uint64_t mask = cs->row_mask[s];
        if (MODE != kLoadFp8 && mask != ~0ull) {
          // Rows outside the key range may hold anything (NaN included).  Their
          // scores are dropped by the row mask, not by value, so only this CTA's
          // P . C boxes need them zeroed (P = 0 times NaN would poison O): one
          // row per step, one 16-byte chunk of its 4 x 128 bytes per lane.
          uint8_t* vb = sStage + s * C::kStageBytes + (lat_x0 / 64) * C::kBox;
          constexpr int kVChunks = (LC / 64) * 8;
          uint64_t dead = ~mask;
          while (dead) {
            const int row = __ffsll((long long)dead) - 1;
            dead &= dead - 1;
            for (int ch = lane; ch < kVChunks; ch += 32)
              *reinterpret_cast<uint4*>(vb + (ch >> 3) * C::kBox + row * 128 + (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        const uint64_t dk = dk0 + (uint64_t)((s * C::kStageBytes) >> 4);
        const uint32_t sd = tmem + C::kSCol + 64 * b;
        // latent [0, QT): A = query in TMEM; then latent [QT, L) and the rope
        // (64 columns; past qk_rope both sides read the TMA zero fill) with A =
        // query boxes in shared memory.  The MMA queue is shallow, so the issue
        // runs back to back; the box loops stay rolled to keep the code small.
        if (lane == 0) {
#pragma unroll 1
          for (int j = 0; j < C::QT / 64; ++j) {
            const uint64_t dkj = dk + (uint64_t)((j * C::kBox) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ts(sd, tmem + C::kQCol + 8 * (4 * j + kk), dkj + (uint64_t)((kk * 32) >> 4), idesc_qk,
                     (j > 0 || kk > 0) ? 1u : 0u);
          }
        }
        if (!q_smem) {
          __syncwarp();
          if (!wwait(&cs->q_full, si & 1, cs, hdr)) return;
          tc_fence_after();
          q_smem = true;
        }
        if (MODE == kLoadFp8 && C::NRH > 1) {
          // the rest of the tile's latent columns and the dead rows' rope zeros
          __syncwarp();
          if (!wwait(&cs->kv_conv[s], par, cs, hdr)) return;
          tc_fence_after();
        }
        if (lane == 0) {
#pragma unroll 1
          for (int i = 0; i <= C::NQS; ++i) {
            // box i of the query buffer pairs with cache box QT / 64 + i (the rope box after the latent ones)
            const uint64_t dqi = dq0 + (uint64_t)((i * C::kQBox) >> 4);
            const uint64_t dki = dk + (uint64_t)(((C::QT / 64 + i) * C::kBox) >> 4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(sd, dqi + (uint64_t)((kk * 32) >> 4), dki + (uint64_t)((kk * 32) >> 4), idesc_qk, 1u);
          }
          mma_commit(&cs->s_full[b]);
          // the segment's last QK: its query buffers may be refilled once it completes
          if (it + 1 == ie) mma_commit(&cs->q_empty);
        }
        __syncwarp();
      }
    });
    // the last commit lands on this CTA's barrier before the CTA leaves
    if (lane == 0 && nseg > 0) mbar_wait(&cs->q_empty, (nseg - 1) & 1, kWaitLimitNs);
    __syncwarp();
  } else if (warp == C::kPvWarp) {
    // ------------------------------------------------------------- P . C issuer
    // O += P . C for tile c as soon as its P is in TMEM (and, for a segment's
    // first tile, the previous segment's O has been read); the commit frees the
    // stage in both CTAs of the cluster.
    const uint32_t idesc_pv = idesc_bf16_f32(128, LC, false, true);
    const uint64_t dv0 = smem_desc(smem_u32(sStage) + (lat_x0 / 64) * C::kBox, C::kBox, 1024, kLayoutSw128);
    int cp = 0;
    for_each_segment(a, k, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool, int) {
      for (int it = ia; it < ie; ++it, ++cp) {
        if (waborted(cs)) return;
        const int b = cp & 1;
        if (!wwait(&cs->p_full[b], (cp >> 1) & 1, cs, hdr)) return;
        if (it == ia && si > 0 && !wwait(&cs->o_free, (si - 1) & 1, cs, hdr)) return;
        tc_fence_after();
        if (lane == 0) {
          // B = this CTA's latent boxes of the stage, keys along K (MN-major)
          const uint64_t dv = dv0 + (uint64_t)(((cp % S) * C::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ts(tmem, tmem + C::kSCol + 64 * b + 8 * kk, dv + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                   (it == ia && kk == 0) ? 0u : 1u);
          if (CL >= 2) mma_commit_mc(&cs->kv_empty[cp % S], (uint16_t)C::kMcMask);
          else mma_commit(&cs->kv_empty[cp % S]);
          mma_commit(&cs->pv_done[b]);
        }
        __syncwarp();
      }
    });
  } else if (MODE == kLoadFp8 && warp >= 6) {
    // ------------------------------------------------------------- e4m3 converters
    // Tile row crow = ci % 64 is widened by NRH threads, thread hh = ci / 64 taking
    // the hh-th RW / NRH bytes of each raw box: e4m3 code x row scale -> bf16 in the
    // 128B-swizzled latent boxes, raw box p after raw box p - 1; dead rows become
    // zeros (latent and rope).  The codes sit where the last raw box's latent boxes
    // go (L = 512: boxes 4-7; L = 64: box 0), so the last pass writes only after
    // every thread has read its codes; earlier passes write boxes that hold none.
    // A pass holds only its part of the row in registers.  The row scales come
    // into shared memory with the tile (the producer copies them asynchronously).
    const int ci = tid - 192, crow = ci & 63, hh = ci >> 6;
    constexpr int kPart = C::RW / C::NRH;          // bytes of a raw box row per thread
    constexpr int kChunks = kPart / 16;
    static_assert(kChunks >= 1 && (kChunks & (kChunks - 1)) == 0, "chunks per part: a power of two");
    int c = 0;
    for_each_segment(a, k, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool, int) {
      for (int it = ia; it < ie; ++it, ++c) {
        if (waborted(cs)) return;
        const int s = c % S;
        if (!wwait(&cs->kv_full[s], (c / S) & 1, cs, hdr)) return;
        uint8_t* st = sStage + s * C::kStageBytes;
        const bool live = (cs->row_mask[s] >> crow) & 1ull;
        const float sc = live ? __int_as_float(cs->rowid[s][crow]) : 0.f;
#pragma unroll 1
        for (int p = 0; p < C::NRH; ++p) {
          // raw[q] holds 16-byte chunk (q + crow) mod kChunks of this thread's part: rows
          // are RW bytes apart, so the rotation puts eight neighbouring rows' reads on
          // eight different banks (in order they would all hit the same ones)
          uint4 raw[kChunks];
          const uint8_t* src = st + C::kRawOff + p * 64 * C::RW + crow * C::RW + hh * kPart;
#pragma unroll
          for (int q = 0; q < kChunks; ++q)
            raw[q] = *reinterpret_cast<const uint4*>(src + ((q + crow) & (kChunks - 1)) * 16);
          if (p == C::NRH - 1) {
            mbar_arrive(&cs->conv_sync);
            if (!wwait(&cs->conv_sync, c & 1, cs, hdr)) return;
          }
          // chunk q's 16 widened columns go to two 16-byte slots of the swizzled box row
          auto put = [&](int q, const uint32_t (&o)[8]) {
            const int col = p * C::RW + hh * kPart + 16 * ((q + crow) & (kChunks - 1));   // its first column
            uint8_t* box = st + (col >> 6) * C::kBox + crow * 128;
            const int ch = (col & 63) >> 3;          // 16-byte chunk within the 128-byte row
            *reinterpret_cast<uint4*>(box + (((ch) ^ (crow & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(box + (((ch + 1) ^ (crow & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          };
          if (live) {
#pragma unroll
            for (int q = 0; q < kChunks; ++q) {
              const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
              uint32_t o[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                o[2 * i] = e4m3x2_scaled_bf16x2((uint16_t)(w[i] & 0xffff), sc);
                o[2 * i + 1] = e4m3x2_scaled_bf16x2((uint16_t)(w[i] >> 16), sc);
              }
              put(q, o);
            }
          } else {
            // a dead row (only in a token's ragged tiles) becomes zeros
            const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
            for (int q = 0; q < kChunks; ++q) put(q, z);
          }
          if (C::NRH > 1 && p == 0) {
            // latent [0, RW) is in place: the QK's TMEM-operand part may start
            fence_proxy_async_smem();
            mbar_arrive(&cs->kv_conv_a[s]);
          }
        }
        if (!live && hh == 0) {
          uint4* rr = reinterpret_cast<uint4*>(st + C::NLB * C::kBox + crow * 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) rr[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        mbar_arrive(&cs->kv_conv[s]);
      }
    });
  } else {
    // ------------------------------------------------------------- softmax
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    const float sl2 = a.scale * 1.4426950408889634f;
    // segment si's query, latent [0, QT), from the staging buffer (128 rows x 128 B
    // per 64 columns, 128B-swizzled) into this head's TMEM row as bf16 pairs
    // (low half = even column); then the buffer is released to the producer
    auto copy_q = [&](int si_q) -> bool {
      if (!wwait(&cs->qa_full, si_q & 1, cs, hdr)) return false;
#pragma unroll 1
      for (int i = 0; i < C::QT / 64; ++i) {
        const uint8_t* rowp = sQ + i * C::kQBox + row * 128;
        uint32_t w[32];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + ((ch ^ (row & 7)) << 4));
          w[4 * ch] = v.x;
          w[4 * ch + 1] = v.y;
          w[4 * ch + 2] = v.z;
          w[4 * ch + 3] = v.w;
        }
        tmem_st32(trow + C::kQCol + 32 * i, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&cs->qa_done);
      mbar_arrive(&cs->q_full);
      return true;
    };
    int c = 0;
    int nfix = 0;   // split-token segments ended (phase of fix_done)
    int nbar = 0;   // split-token partials published (phase of fix_bar)
    int pend_t = -1, pend_claim = -1;   // a split token of an earlier segment, its claim (row 0)
    TokenPlan pend_tp{};
    int nmrg = 0;   // half partials brought in by bulk copy (buffer and phase of mrg_full / mrg_done)
    bool q_ready = false;   // the coming segment's query is already in TMEM
    for_each_segment(a, k, g0, g1, [&](int si, int t0, const TokenPlan& tp, int ia, int ie, bool is_first_seg,
                                     int next_t) {
      if (waborted(cs)) return;
      // this CTA's query token: slot tslot of a folded pair; a slot the pair does
      // not fill repeats slot 0's work without writing anything
      const bool shadow = C::NSLOT > 1 && tslot >= (tp.ntok > 1 ? tp.ntok : 1);
      const int t = shadow ? t0 : t0 + tslot;
      int mlo = tp.lo, mhi = tp.hi;
      if constexpr (C::NSLOT > 1) {
        mlo = tslot == 0 ? tp.mlo : a.plan[t].mlo;
        mhi = tslot == 0 ? tp.mhi : a.plan[t].mhi;
      }
      // a folded token may attend fewer keys than the tiles of its pair cover
      const bool own_mask = C::NSLOT > 1 && (mlo > tp.lo || mhi < tp.hi);
      if (!q_ready && !copy_q(si)) return;
      q_ready = false;
      float m = -CUDART_INF_F, l = 0.f;
      int last_c = -1;
      for (int it = ia; it < ie; ++it, ++c) {
        if (waborted(cs)) return;
        const int s = c % S, b = c & 1;
        if (!wwait(&cs->kv_full[s], (c / S) & 1, cs, hdr)) return;   // row mask visibility
        uint64_t mask = cs->row_mask[s];
        if (own_mask) {
          // keys of the tile outside this token's own range do not count
          const int key0 = (tp.tile_first + it) * kTileKeys;
          const int a0 = mlo - key0, a1 = mhi - key0;
          const uint64_t above = a0 <= 0 ? ~0ull : (a0 >= 64 ? 0ull : ~0ull << a0);
          const uint64_t below = a1 >= 64 ? ~0ull : (a1 <= 0 ? 0ull : (1ull << a1) - 1);
          mask &= above & below;
        }
        if (!wwait(&cs->s_full[b], (c >> 1) & 1, cs, hdr)) return;
        tc_fence_after();
        // S row (64 fp32) for this thread's head; both halves of the load in flight at once
        uint32_t sr[64];
        tmem_ld32(trow + C::kSCol + 64 * b, *reinterpret_cast<uint32_t(*)[32]>(sr));
        tmem_ld32(trow + C::kSCol + 64 * b + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
        tmem_ld_wait();
        float sv[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) sv[j] = __uint_as_float(sr[j]);
        // row max of the scaled scores (log2 domain); dead keys do not count.
        // Eight independent chains, then a tree, keep the dependency depth short;
        // full tiles (the common case) skip the mask tests.
        const bool all_live = mask == ~0ull;
        float mx;
        {
          const bool up = sl2 >= 0.f;   // the max of s * scale is the min of s when scale < 0
          float r8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) r8[i] = sv[i];
          if (all_live) {
            if (up) {
#pragma unroll
              for (int j = 8; j < 64; ++j) r8[j & 7] = fmaxf(r8[j & 7], sv[j]);
            } else {
#pragma unroll
              for (int j = 8; j < 64; ++j) r8[j & 7] = fminf(r8[j & 7], sv[j]);
            }
          } else {
            const float fill = up ? -CUDART_INF_F : CUDART_INF_F;
#pragma unroll
            for (int i = 0; i < 8; ++i) r8[i] = ((mask >> i) & 1ull) ? sv[i] : fill;
#pragma unroll
            for (int j = 8; j < 64; ++j) {
              const float x = ((mask >> j) & 1ull) ? sv[j] : fill;
              r8[j & 7] = up ? fmaxf(r8[j & 7], x) : fminf(r8[j & 7], x);
            }
          }
#pragma unroll
          for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) r8[i] = up ? fmaxf(r8[i], r8[i + w]) : fminf(r8[i], r8[i + w]);
          mx = r8[0] == (up ? -CUDART_INF_F : CUDART_INF_F) ? -CUDART_INF_F : r8[0] * sl2;
        }
        // Lazy rescale: a row moves its reference max only when the new max is
        // more than 2^8 above it.  tcgen05.ld/st are warp-collective, so when any
        // row of the warp needs O rescaled the whole warp runs the loop (alpha = 1
        // for the others).
        const bool want = m != -CUDART_INF_F && mx > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, want)) {
          const float alpha = want ? ex2(m - mx) : 1.f;
          if (!wwait(&cs->pv_done[(c - 1) & 1], ((c - 1) >> 1) & 1, cs, hdr)) return;
          tc_fence_after();
#pragma unroll 1
          for (int col = 0; col < LC; col += 32) {
            uint32_t r[32];
            tmem_ld32(trow + col, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(trow + col, r);
          }
          tmem_st_wait();
          if (want) {
            l *= alpha;
            m = mx;
          }
        }
        if (m == -CUDART_INF_F) m = mx;   // first live key of the segment: O is still empty
        // P = 2^(scale * log2(e) * s - m) as bf16 pairs over the S columns in TMEM
        uint32_t pk[32];
        float ps4[4] = {0.f, 0.f, 0.f, 0.f};
        const float neg_m = -m;
        if (all_live) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float p0 = ex2(fmaf(sv[2 * j], sl2, neg_m));
            const float p1 = ex2(fmaf(sv[2 * j + 1], sl2, neg_m));
            ps4[j & 3] += p0 + p1;
            pk[j] = pack_bf16(p0, p1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float p0 = ex2(fmaf(sv[2 * j], sl2, neg_m));
            float p1 = ex2(fmaf(sv[2 * j + 1], sl2, neg_m));
            p0 = ((mask >> (2 * j)) & 1ull) ? p0 : 0.f;
            p1 = ((mask >> (2 * j + 1)) & 1ull) ? p1 : 0.f;
            ps4[j & 3] += p0 + p1;
            pk[j] = pack_bf16(p0, p1);
          }
        }
        l += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
        tmem_st32(trow + C::kSCol + 64 * b, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&cs->p_full[b]);
        last_c = c;
      }
      if (last_c < 0) return;
      // ------------------------------------------------------------- epilogue
      // the next segment's query goes into TMEM as soon as this segment's last QK
      // is done, so the next QKs overlap this segment's last P . C and output
      if (next_t >= 0 && next_t < a.T) {
        if (!copy_q(si + 1)) return;
        q_ready = true;
      }
      const bool complete = ia == 0 && ie == tp.ntiles;
      const bool final_seg = tp.tile_start + ie >= g1;   // the partition's last segment
      constexpr int NS = C::NSLOT;
      const int kf = tp.part_first, kl = tp.part_last;
      // partition kf holds the token in its second slot if the token began inside its range
      const int slot_kf = complete ? 0 : (tp.tile_start != a.bounds[kf] ? 1 : 0);
      // Split token: every partition (per cluster rank) claims it once; the last
      // to claim merges all partitions' partials into o_lat / lse once the
      // partials are counted as written.  A partition's final segment claims
      // before its last P . C completes, so that if it merges, its own partial
      // never leaves TMEM.  An earlier segment (at most one: the partition's
      // first) writes its partial, counts it and claims without waiting for the
      // outcome; it is decided after the partition's final segment.  A claimer
      // that does not merge depends on nothing outside its CTA from its claim to
      // its written count, so a merger's wait ends.
      const bool early_claim = !complete && final_seg && !shadow;
      int claim = 0;
      if (early_claim && row == 0) claim = atomicAdd(&a.counters[4 * t + rank], 1);
      if (!wwait(&cs->pv_done[last_c & 1], (last_c >> 1) & 1, cs, hdr)) return;
      tc_fence_after();
      // row 0 of a merger: wait for the other partitions' written partials
      auto await_written = [&]() {
        if (wait_count(&a.counters[4 * t + 2 + rank], kl - kf, kWaitLimitNs)) {
          __threadfence();
          return true;
        }
        record_timeout(&cs->fix_done, hdr);
        atomicOr(&hdr->status, kDeviceTimeout);
        *reinterpret_cast<volatile int*>(&cs->abort) = 1;
        return false;
      };
      bool merger = false;
      if (early_claim) {
        if (row == 0) {
          cs->fix_last = claim == kl - kf && await_written();
          mbar_arrive(&cs->fix_done);
        }
        if (!wwait(&cs->fix_done, nfix & 1, cs, hdr) || waborted(cs)) return;
        ++nfix;
        merger = cs->fix_last;
      }
      const int slot = (is_first_seg ? 0 : 1) * NS + tslot;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
      const bool live = row < H && !shadow;
      if (!merger) {
#pragma unroll 1
        for (int col = 0; col < LC; col += 32) {
          uint32_t r[32];
          tmem_ld32(trow + col, r);
          tmem_ld_wait();
          if (!live) continue;
          if (complete) {
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[i] = pack_bf16(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(a.o_lat + ((size_t)t * H + row) * L + lat_x0 + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          } else {
            float4* po = reinterpret_cast<float4*>(a.part_o);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              po[part_index(k, slot, (lat_x0 + col) / 4 + i, row, L, H, NS)] =
                  make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                              __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
          }
        }
        if (live) {
          if (complete) {
            if (rank == 0) a.lse_ws[(size_t)t * H + row] = lse;
          } else {
            a.part_lse[((size_t)(k * 2 * NS + slot) * 2 + rank) * H + row] = lse;
          }
        }
      }
      // O has been read: the next segment's first P . C may overwrite it
      tc_fence_before();
      mbar_arrive(&cs->o_free);
      if (complete || shadow) return;
      if (merger) {
        // the partition's final segment: O in TMEM still holds this CTA's own
        // partial and the query buffer and stage ring are idle
        if (!merge_in_tmem<LC>(a, cs, t, tp, k, kf, kl, slot_kf, rank, row, lat_x0, trow, trow + C::kSCol, lse, inv, sQ,
                               sQ + C::kRegionBytes - 2 * C::kMrgHalf, nmrg, NS, tslot))
          return;
        if (row == 0) {
          a.counters[4 * t + rank] = 0;
          a.counters[4 * t + 2 + rank] = 0;
        }
        return;
      }
      // publish the partial: the barrier orders the 128 threads' rows before
      // thread row 0, whose release increment covers them all
      mbar_arrive(&cs->fix_bar);
      if (row == 0 && wait_or_abort(&cs->fix_bar, nbar & 1, cs, hdr)) {
        red_add_release_gpu(&a.counters[4 * t + 2 + rank], 1);
        if (!early_claim) pend_claim = atomicAdd(&a.counters[4 * t + rank], 1);
      }
      ++nbar;
      if (!early_claim) {
        // only a token's last partition holds it in an earlier segment, its first
        if (pend_t >= 0 && row == 0) atomicOr(&hdr->status, kDeviceCheckFailed);
        pend_t = t;
        pend_tp = tp;
      }
      __syncwarp();
    });
    if (pend_t >= 0) {
      // the earlier segment's claim: the last claimer merges once all partials,
      // its own included, are counted as written; every partial is in global
      // memory (this CTA's own rows were written by these same threads)
      const int kf = pend_tp.part_first, kl = pend_tp.part_last;
      const int slot_kf = pend_tp.tile_start != a.bounds[kf] ? 1 : 0;
      if (row == 0) {
        bool last = pend_claim == kl - kf;
        if (last) {
          last = wait_count(&a.counters[4 * pend_t + 2 + rank], kl - kf + 1, kWaitLimitNs);
          if (last) {
            __threadfence();
          } else {
            record_timeout(&cs->fix_done, hdr);
            atomicOr(&hdr->status, kDeviceTimeout);
            *reinterpret_cast<volatile int*>(&cs->abort) = 1;
          }
        }
        cs->fix_last = last;
        mbar_arrive(&cs->fix_done);
      }
      if (wwait(&cs->fix_done, nfix & 1, cs, hdr) && !waborted(cs) && cs->fix_last) {
        // the final segment is done: query buffer, stage ring and TMEM S / query
        // columns are idle; no partial of this token is in TMEM
        // (a time-out inside has set the abort flag; the threads go on to the teardown)
        bool merged = true;
        if constexpr (MODE == kLoadFp8) {
          if (row < H) merge_split_token(a, pend_t, pend_tp, kf, kl, slot_kf, rank, row, lat_x0, LC, C::NSLOT, tslot);
        } else {
          merged = merge_in_tmem<LC>(a, cs, pend_t, pend_tp, -1, kf, kl, slot_kf, rank, row, lat_x0, trow,
                                     trow + C::kSCol, 0.f, 0.f, sQ, sQ + C::kRegionBytes - 2 * C::kMrgHalf, nmrg,
                                     C::NSLOT, tslot);
        }
        if (merged && row == 0) {
          a.counters[4 * pend_t + rank] = 0;
          a.counters[4 * pend_t + 2 + rank] = 0;
        }
      }
    }
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (CL >= 2 && tid == 32) {
    // Tell the other CTAs this CTA is done, and wait (bounded) until they have all
    // said the same before this CTA's shared memory goes away.  Everything they send
    // into this CTA (multicast tiles, multicast stage commits) has been awaited on
    // this CTA's own barriers already, so the signal needs no release ordering (a
    // release at cluster scope here stalled for tens of microseconds).
    for (uint32_t r = 0; r < (uint32_t)CL; ++r)
      if (r != crank) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&cs->bye), r));
    if (!mbar_poll_cluster(&cs->bye, 0, kWaitLimitNs)) {
      record_timeout(&cs->bye, hdr);
      atomicOr(&hdr->status, kDeviceTimeout);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Failure-detection self-test: one thread waits, through the same bounded wait
// the decode uses, on an mbarrier that nothing ever arrives on.  No copy, MMA or
// peer CTA is in flight, so giving up after `limit_ns` leaves nothing behind; the
// time-out is recorded in the header exactly as a decode wait records it.
__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(PlanHeader* hdr, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) {
    record_timeout(&bar, hdr);
    atomicOr(&hdr->status, kDeviceTimeout);
  }
}

// ----------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
               uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor maps of a launch depend only on these; consecutive calls on the
// same buffers (the serving loop) reuse the last encoding.
struct MapKey {
  int device;
  const void* kv_pool;
  const void* q_full;
  int L, R, ps, num_pages, T;
  bool operator==(const MapKey& o) const {
    return device == o.device && kv_pool == o.kv_pool && q_full == o.q_full && L == o.L && R == o.R && ps == o.ps &&
           num_pages == o.num_pages && T == o.T;
  }
};

}  // namespace tc

cudaError_t ensure_smem_limit(const void* func, int bytes) {
  // (kernel, device) pairs whose limit is already raised; a handful of kernels
  struct Entry {
    const void* func;
    int device, bytes;
  };
  static std::mutex mu;
  static Entry done[64];
  static int n = 0;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < n; ++i) {
    if (done[i].func == func && done[i].device == device) {
      if (done[i].bytes >= bytes) return cudaSuccess;
      slot = i;
    }
  }
  // the limit counts dynamic bytes only (static shared memory comes on top), so
  // it is raised to exactly what this launch needs, and again if a later one needs more
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (slot >= 0) done[slot].bytes = bytes;
  else if (n < 64) done[n++] = Entry{func, device, bytes};
  return cudaSuccess;
}

namespace tc {

template <int LC, int CL, int MODE>
cudaError_t launch(const DecodeArgs& a, cudaStream_t s) {
  using C = Cfg<LC, CL, MODE>;
  constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int L = a.d.kv_lora_rank, R = a.d.qk_rope, KQ = L + R, ps = a.d.page_size;
  const uint32_t rows = MODE == kLoadSparse ? 1u : (uint32_t)(ps < kTileKeys ? ps : kTileKeys);
  const uint64_t pool_rows = (uint64_t)a.d.num_pages * ps;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return cudaErrorInvalidDevice;
  const MapKey key{device, a.kv_pool, a.q_full, L, R, ps, a.d.num_pages, a.T};
  static std::mutex cache_mu;
  static bool cache_valid = false;
  static MapKey cache_key;
  static Maps cache_maps;
  Maps maps;
  bool hit;
  {
    std::lock_guard<std::mutex> lock(cache_mu);
    hit = cache_valid && cache_key == key;
    if (hit) maps = cache_maps;
  }
  if (!hit) {
    bool ok;
    if (MODE == kLoadFp8) {
      const uint64_t rb = (uint64_t)L + 2 * R;   // bytes per cached row
      ok = encode_2d(&maps.kv_lat, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.kv_pool, rb, pool_rows, rb, C::RW, rows,
                     CU_TENSOR_MAP_SWIZZLE_NONE) &&
           encode_2d(&maps.kv_rope, kBF16, a.kv_pool, rb / 2, pool_rows, rb, 64, rows, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
      ok = encode_2d(&maps.kv_lat, kBF16, a.kv_pool, KQ, pool_rows, (uint64_t)KQ * 2, 64, rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
      maps.kv_rope = maps.kv_lat;   // the rope box is one more 64-column box of the same rows
    }
    ok = ok && encode_2d(&maps.q, kBF16, a.q_full, KQ, (uint64_t)a.T * kMaxHeads, (uint64_t)KQ * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lock(cache_mu);
    cache_key = key;
    cache_maps = maps;
    cache_valid = true;
  }
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(decode_tc_kernel<LC, CL, MODE>), C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.K * CL);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap with the absorb kernel's tail
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<LC, CL, MODE>, maps, a);
}

// Clusters of this instance that the device holds at once (its shared memory, its
// cluster size): the default partition count, so that no partition waits for a
// second wave.  Cached per device.
template <int LC, int CL, int MODE>
int max_active_clusters() {
  using C = Cfg<LC, CL, MODE>;
  static std::mutex mu;
  static int cached[64] = {};
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[device] > 0) return cached[device];
  if (ensure_smem_limit(reinterpret_cast<const void*>(decode_tc_kernel<LC, CL, MODE>), C::kSmem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CL * 256);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<LC, CL, MODE>, &cfg) != cudaSuccess) {
    cudaGetLastError();   // a failed query leaves no error behind
    return 0;
  }
  cached[device] = n;
  return n;
}

template <int MODE>
cudaError_t launch_mode(const DecodeArgs& a, cudaStream_t s) {
  if (a.d.kv_lora_rank == 512) {
    if constexpr (MODE != kLoadFp8) {
      if (a.fold) return launch<256, 4, MODE>(a, s);
    }
    return launch<256, 2, MODE>(a, s);
  }
  return launch<64, 1, MODE>(a, s);
}

}  // namespace tc

// Shapes with a tensor-core instance: (L, R) = (512, 64) on a 2-CTA cluster,
// and L = 64 with R <= 32 on one CTA; qk_nope and v_head multiples of 8, v_head <= 512;
// dense pages of 8..64 tokens or a multiple of 64.
int decode_default_partitions(const mla_dims_t& d, bool fold, bool fp8_cache, bool sparse) {
  if (d.kv_lora_rank != 512) {
    if (sparse) return tc::max_active_clusters<64, 1, tc::kLoadSparse>();
    if (fp8_cache) return tc::max_active_clusters<64, 1, tc::kLoadFp8>();
    return tc::max_active_clusters<64, 1, tc::kLoadDense>();
  }
  if (fold && !fp8_cache) {
    if (sparse) return tc::max_active_clusters<256, 4, tc::kLoadSparse>();
    return tc::max_active_clusters<256, 4, tc::kLoadDense>();
  }
  if (sparse) return tc::max_active_clusters<256, 2, tc::kLoadSparse>();
  if (fp8_cache) return tc::max_active_clusters<256, 2, tc::kLoadFp8>();
  return tc::max_active_clusters<256, 2, tc::kLoadDense>();
}

bool decode_fold_supported(const mla_dims_t& d, bool fp8_cache) {
  return d.kv_lora_rank == 512 && d.qk_rope == 64 && !fp8_cache;
}

bool decode_tc_supported(const mla_dims_t& d) {
  const int ps = d.page_size;
  // the weight GEMMs read q and w_uk rows through TMA (16-byte row pitch),
  // write 16-byte pieces of the output rows, and hold at most four 128-row
  // weight blocks of w_uv per CTA
  if (d.qk_nope % 8 != 0 || d.v_head < 8 || d.v_head > 512 || d.v_head % 8 != 0) return false;
  if (!(ps % kTileKeys == 0 || (kTileKeys % ps == 0 && ps >= 8))) return false;
  if (d.kv_lora_rank == 512 && d.qk_rope == 64) return true;
  if (d.kv_lora_rank == 64 && d.qk_rope <= 32 && d.qk_rope % 8 == 0) return true;
  return false;
}

cudaError_t launch_wait_selftest(PlanHeader* hdr, uint64_t limit_ns, cudaStream_t s) {
  tc::wait_selftest_kernel<<<1, 32, 0, s>>>(hdr, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  if (a.ks.indices) return tc::launch_mode<tc::kLoadSparse>(a, s);
  if (a.kv_fmt == KVFmt::kE4M3) return tc::launch_mode<tc::kLoadFp8>(a, s);
  return tc::launch_mode<tc::kLoadDense>(a, s);
}

}  // namespace mla
