// K2 (tensor-core version): split-KV MLA decode on tcgen05 with TMEM accumulators.
//
// Work split: partition k of K owns the global 64-key tiles [k*Q, (k+1)*Q)
// (Q = ceil(total/K)); it walks them as segments, one per query token it
// touches, and writes either the finished latent output (segment = whole
// token) or a partial (o_p, lse_p) for the combine kernel.  These are the
// split-KV partitions behind num_partitions_in on the
// generic_flare_mla_decode_kv_cache_ragged page.
//
// One partition runs on a cluster of kCluster CTAs (2 for the 512-wide latent,
// 1 for narrow latents).  With 128 heads sharing every cached row, scores
// S = Q . K^T (M = 128 heads, N = 64 keys, K = 576) and the update
// O += P . C (M = 128, N = 512, K = 64) are dense contractions.  O for 128
// heads x 512 latent columns in fp32 fills all 512 TMEM columns, so the two
// CTAs of a cluster split the latent columns: CTA r owns latent columns
// [256r, 256r + 256) and rope columns [512 + 32r, 512 + 32r + 32).  Each loads
// only its 288-column slice of every cached row (TMA, 128B / 64B swizzle),
// computes a partial S over that slice, and the two partial S tiles are
// exchanged through distributed shared memory; both CTAs then hold the same
// S = S_0 + S_1 (fp32 addition is commutative, so bit-identical), run the same
// online softmax, and each applies P to its own 256 latent columns.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: query slice once per segment, cache tiles
//               through the page table into a kStages-deep ring.
//   warp 1      TMEM owner and MMA issuer (one thread); its other lanes zero
//               cache rows outside the key range before the MMAs read them
//               (0 * NaN would poison P . C).
//   warps 2-5   softmax: thread = head row = TMEM lane.  Reads S, exchanges
//               partial S, masks, keeps running max / sum in the log2
//               domain, writes P (bf16 pairs) back into TMEM where the PV MMA
//               takes it as its A operand, rescales O only when the running
//               max grows by more than 2^8, and writes the segment's output.
// Every wait is bounded in time; a timeout sets a status bit and the kernel
// unwinds without hanging.
#include <math_constants.h>

#include "mla_kernels.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace tc {

using namespace sm100;

constexpr int kStages = 3;

// How cache rows reach shared memory.
enum LoadMode : int {
  kLoadDense = 0,   // bf16 pool through the page table, TMA tiles
  kLoadFp8 = 1,     // e4m3 pool through the page table: TMA bytes, widened in place by converter warps
  kLoadSparse = 2,  // bf16 pool rows named by an index list, TMA gather4
};
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows by > 2^8
constexpr uint64_t kWaitLimitNs = 1000000000ull;

template <int kLatentPerCta, int kCluster, int kMode>
struct Cfg {
  static constexpr int kThreads = kMode == kLoadFp8 ? 256 : 192;   // + 2 converter warps for e4m3
  static constexpr int LC = kLatentPerCta;          // latent columns owned by one CTA
  static constexpr int NLB = LC / 64;               // 64-column (128 B) latent boxes
  static constexpr int RC = 32;                     // rope box columns (64 B)
  static constexpr int kLatBoxKv = 64 * 128;        // 64 rows x 128 B
  static constexpr int kRopeBoxKv = 64 * 64;        // 64 rows x 64 B
  static constexpr int kStageBytes = NLB * kLatBoxKv + kRopeBoxKv;
  static constexpr int kLatBoxQ = 128 * 128;
  static constexpr int kQBytes = NLB * kLatBoxQ + 128 * 64;
  static constexpr int kXBytes = kCluster == 2 ? 128 * 64 * 4 : 0;
  static constexpr int kTmemCols = (LC + 128) <= 256 ? 256 : 512;
  static constexpr int kSCol = LC;                  // S buffers after O
  static constexpr int kSmem = 1024 + kQBytes + kStages * kStageBytes + kXBytes + 1024;
  static_assert(LC % 64 == 0 && LC <= 256, "latent slice");
};

struct Smem {   // control block at the end of dynamic shared memory
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_free;
  uint64_t x_full, x_empty;
  uint64_t kv_conv[kStages];     // e4m3 rows widened (kLoadFp8)
  uint64_t conv_sync;            // converters: every row read before any is overwritten
  uint64_t fix_bar, fix_done;    // softmax: partial written / merge decision published
  uint64_t bye;                  // the peer CTA is done touching this CTA's shared memory
  uint64_t row_mask[kStages];
  int32_t rowid[kStages][64];    // physical row of each tile row (kLoadFp8, kLoadSparse)
  uint32_t tmem_base;
  int abort;
  int fix_last;   // this CTA merges the split token it just finished
};

struct Maps {
  CUtensorMap kv_lat;    // bf16 latent boxes (kLoadDense: ps rows, kLoadSparse: 1 row) / e4m3 bytes (kLoadFp8)
  CUtensorMap kv_rope;   // bf16 rope box
  CUtensorMap q_lat, q_rope;
};

// Walks the segments of partition k: calls f(t, plan, first_tile, end_tile, g_first).
template <class F>
__device__ __forceinline__ void for_each_segment(const DecodeArgs& a, int g0, int g1, F&& f) {
  int g = g0;
  int si = 0;
  while (g < g1) {
    const int t = token_of_tile(a.plan, a.T, g);
    if (t < 0 || t >= a.T) {   // a plan that does not cover g: report, never loop
      atomicOr(&a.hdr_mut->status, kDeviceCheckFailed);
      return;
    }
    const TokenPlan tp = a.plan[t];
    const int ia = g - tp.tile_start;
    const int ie = min(g1, tp.tile_start + tp.ntiles) - tp.tile_start;
    if (ia < 0 || ie <= ia) {
      atomicOr(&a.hdr_mut->status, kDeviceCheckFailed);
      return;
    }
    f(si, t, tp, ia, ie, g == g0);
    g = tp.tile_start + ie;
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

// Two e4m3 codes times a row scale, rounded to a bf16 pair (low half = first code).
__device__ __forceinline__ uint32_t e4m3x2_scaled_bf16x2(uint16_t two, float scale) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
  return *reinterpret_cast<const uint32_t*>(&b);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Log-sum-exp merge of one split token's partials for head `row`, latent
// columns [lat_x0, lat_x0 + LC):  lse = ln sum_p e^{lse_p},
// o = sum_p e^{lse_p - lse} o_p.  Partitions with an empty key set carry
// lse_p = -inf and drop out.  Partition k holds the token in slot 0 (its
// first segment) unless the token began inside partition kf's range.
__device__ __noinline__ void merge_split_token(const DecodeArgs& a, int t, const TokenPlan& tp, int kf, int kl,
                                               int Qt, uint32_t rank, int row, int lat_x0, int LC) {
  const int H = a.d.num_heads, L = a.d.kv_lora_rank;
  auto slot_of = [&](int k) { return (k == kf && tp.tile_start != k * Qt) ? 1 : 0; };
  float mx = -CUDART_INF_F;
  for (int k = kf; k <= kl; ++k)
    mx = fmaxf(mx, __ldcg(a.part_lse + ((size_t)(k * 2 + slot_of(k)) * 2 + rank) * H + row));
  float sum = 0.f;
  if (mx != -CUDART_INF_F)
    for (int k = kf; k <= kl; ++k)
      sum += __expf(__ldcg(a.part_lse + ((size_t)(k * 2 + slot_of(k)) * 2 + rank) * H + row) - mx);
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  for (int col = 0; col < LC; col += 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (mx != -CUDART_INF_F) {
      for (int k = kf; k <= kl; ++k) {
        const size_t src = (size_t)(k * 2 + slot_of(k)) * H + row;
        const float w = __expf(__ldcg(a.part_lse + ((size_t)(k * 2 + slot_of(k)) * 2 + rank) * H + row) - mx) * inv;
        const float4* p = reinterpret_cast<const float4*>(a.part_o + src * L + lat_x0 + col);
        const float4 u = __ldcg(p), v = __ldcg(p + 1);
        acc[0] += w * u.x; acc[1] += w * u.y; acc[2] += w * u.z; acc[3] += w * u.w;
        acc[4] += w * v.x; acc[5] += w * v.y; acc[6] += w * v.z; acc[7] += w * v.w;
      }
    }
    uint4 o;
    o.x = pack_bf16(acc[0], acc[1]);
    o.y = pack_bf16(acc[2], acc[3]);
    o.z = pack_bf16(acc[4], acc[5]);
    o.w = pack_bf16(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(a.o_lat + ((size_t)t * H + row) * L + lat_x0 + col) = o;
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

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


template <int LC, int CL, int MODE>
__global__ void __launch_bounds__(Cfg<LC, CL, MODE>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ Maps maps, const DecodeArgs a) {
  using C = Cfg<LC, CL, MODE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = sm;
  uint8_t* sStage = sQ + C::kQBytes;
  float* sX = reinterpret_cast<float*>(sStage + kStages * C::kStageBytes);
  Smem* cs = reinterpret_cast<Smem*>(reinterpret_cast<uint8_t*>(sX) + C::kXBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = CL == 2 ? cluster_ctarank() : 0u;
  const uint32_t peer = rank ^ 1u;
  const int k = blockIdx.x / CL;
  PlanHeader* hdr = a.hdr_mut;
  const int L = a.d.kv_lora_rank, H = a.d.num_heads;
  const int lat_x0 = (int)rank * LC;
  // this CTA's rope columns: in the absorbed query row they start at L; in the
  // cache they start at L too, except in the e4m3 pool's bf16 view (L / 2)
  const int q_rope_x0 = L + (int)rank * (a.d.qk_rope / CL);
  const int rope_x0 = (MODE == kLoadFp8 ? L / 2 : L) + (int)rank * (a.d.qk_rope / CL);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&cs->kv_full[s], 1);
      mbar_init(&cs->kv_empty[s], 1);
      mbar_init(&cs->kv_conv[s], 64);
    }
    mbar_init(&cs->q_full, 1);
    mbar_init(&cs->q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&cs->s_full[b], 1);
      mbar_init(&cs->p_full[b], 128);
      mbar_init(&cs->pv_done[b], 1);
    }
    mbar_init(&cs->o_free, 128);
    mbar_init(&cs->x_full, 1);   // expect_tx by row 0 + 32 KB of st.async from the peer
    mbar_init(&cs->x_empty, 128);
    mbar_init(&cs->conv_sync, 64);
    mbar_init(&cs->fix_bar, 128);
    mbar_init(&cs->fix_done, 1);
    mbar_init(&cs->bye, 1);
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
    prefetch_tensormap(&maps.q_lat);
    prefetch_tensormap(&maps.q_rope);
  }
  tc_fence_before();
  if (CL == 2) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cs->tmem_base;
  // the W_uv kernel may start its prologue now; the plan and q_full of the
  // absorb kernel must be complete before anything below reads them
  griddep_launch_dependents();
  griddep_wait();

  const int total = a.hdr->total_tiles;
  const int g0 = partition_begin(k, a.K, total), g1 = partition_begin(k + 1, a.K, total);
  const int ps = a.ks.page_size;
  const int rows_per_load = ps < kTileKeys ? ps : kTileKeys;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    int c = 0;
    bool bad = false;
    for_each_segment(a, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool) {
      if (waborted(cs)) return;
      if (si > 0 && !wwait(&cs->q_empty, (si - 1) & 1, cs, hdr)) return;
      if (lane == 0) {
        mbar_arrive_expect_tx(&cs->q_full, C::kQBytes);
        for (int i = 0; i < C::NLB; ++i)
          tma_load_2d(sQ + i * C::kLatBoxQ, &maps.q_lat, &cs->q_full, lat_x0 + 64 * i, t * kMaxHeads);
        tma_load_2d(sQ + C::NLB * C::kLatBoxQ, &maps.q_rope, &cs->q_full, q_rope_x0, t * kMaxHeads);
      }
      for (int it = ia; it < ie; ++it, ++c) {
        if (waborted(cs)) return;
        const int s = c % kStages;
        if (c >= kStages && !wwait(&cs->kv_empty[s], ((c / kStages) & 1) ^ 1, cs, hdr)) return;
        const int key0 = (tp.tile_first + it) * kTileKeys;
        // rows j and j + 32 of this tile: which key / slot, and is it live?
        bool v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int key = key0 + lane + 32 * h;
          bool ok = key >= tp.lo && key < tp.hi;
          int rid = 0;
          if (ok) {
            if (MODE == kLoadSparse) {
              const int idx = a.ks.indices[(size_t)tp.b * a.ks.idx_stride + key];
              if (idx >= 0 && idx < a.ks.num_pages * ps) {
                rid = idx;
              } else {
                ok = false;
                if (idx != -1) bad = true;
              }
            } else {
              const int page = a.ks.block_table[(size_t)tp.b * a.ks.bt_stride + key / ps];
              if (page < 0 || page >= a.ks.num_pages) { ok = false; bad = true; }
              else rid = page * ps + key % ps;
            }
          }
          v[h] = ok;
          if (MODE != kLoadDense) cs->rowid[s][lane + 32 * h] = rid;
        }
        const uint64_t mask = (uint64_t)__ballot_sync(0xffffffffu, v[0]) |
                              ((uint64_t)__ballot_sync(0xffffffffu, v[1]) << 32);
        uint8_t* st = sStage + s * C::kStageBytes;
        uint8_t* st_rope = st + C::NLB * C::kLatBoxKv;
        if (MODE == kLoadSparse) {
          // every row is fetched (row 0 stands in for a dead slot and is zeroed before use)
          if (lane == 0) {
            cs->row_mask[s] = mask;
            mbar_arrive_expect_tx(&cs->kv_full[s], 64 * (C::NLB * 128 + 64));
          }
          __syncwarp();
          if (lane < 16) {
            const int r0 = 4 * lane;
            const int y0 = cs->rowid[s][r0], y1 = cs->rowid[s][r0 + 1];
            const int y2 = cs->rowid[s][r0 + 2], y3 = cs->rowid[s][r0 + 3];
#pragma unroll
            for (int i = 0; i < C::NLB; ++i)
              tma_gather4(st + i * C::kLatBoxKv + r0 * 128, &maps.kv_lat, &cs->kv_full[s], lat_x0 + 64 * i, y0, y1, y2, y3);
            tma_gather4(st_rope + r0 * 64, &maps.kv_rope, &cs->kv_full[s], rope_x0, y0, y1, y2, y3);
          }
        } else if (lane == 0) {
          cs->row_mask[s] = mask;
          // pages of this tile that hold at least one live row
          const int nloads = kTileKeys / rows_per_load;
          const uint32_t row_bytes = MODE == kLoadFp8 ? (LC + 64) : (C::NLB * 128 + 64);
          uint32_t bytes = 0;
          for (int p = 0; p < nloads; ++p) {
            const uint64_t pm = (rows_per_load == 64) ? mask : ((mask >> (p * rows_per_load)) & ((1ull << rows_per_load) - 1));
            if (pm) bytes += rows_per_load * row_bytes;
          }
          mbar_arrive_expect_tx(&cs->kv_full[s], bytes);
          for (int p = 0; p < nloads; ++p) {
            const uint64_t pm = (rows_per_load == 64) ? mask : ((mask >> (p * rows_per_load)) & ((1ull << rows_per_load) - 1));
            if (!pm) continue;
            const int kp = key0 + p * rows_per_load;
            const int page = a.ks.block_table[(size_t)tp.b * a.ks.bt_stride + kp / ps];
            const int y = page * ps + kp % ps;
            const int r0 = p * rows_per_load;
            if (MODE == kLoadFp8) {
              // raw e4m3 rows (LC bytes each) at the start of the stage, widened later
              tma_load_2d(st + r0 * LC, &maps.kv_lat, &cs->kv_full[s], lat_x0, y);
            } else {
              for (int i = 0; i < C::NLB; ++i)
                tma_load_2d(st + i * C::kLatBoxKv + r0 * 128, &maps.kv_lat, &cs->kv_full[s], lat_x0 + 64 * i, y);
            }
            tma_load_2d(st_rope + r0 * 64, &maps.kv_rope, &cs->kv_full[s], rope_x0, y);
          }
        }
        __syncwarp();
      }
    });
    if (bad) atomicOr(&hdr->status, kDeviceCheckFailed);
    // make sure no TMA write is still in flight when the CTA leaves
    if (lane == 0) {
      for (int j = c - kStages; j < c; ++j) {
        if (j < 0) continue;
        mbar_wait(&cs->kv_full[j % kStages], (j / kStages) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    const uint32_t idesc_qk = idesc_bf16_f32(128, 64, false, false);
    const uint32_t idesc_pv = idesc_bf16_f32(128, LC, false, true);
    const uint32_t sQa = smem_u32(sQ);
    const uint32_t sSa = smem_u32(sStage);
    int c = 0;
    int prev_s = -1, prev_b = -1, prev_c = -1;
    bool first_pv_of_seg = true;
    int seg_of_prev = -1;
    auto issue_pv = [&](int si) {
      // P(prev) is in TMEM, O is free for the segment's first PV
      if (!wwait(&cs->p_full[prev_b], (prev_c / 2) & 1, cs, hdr)) return false;
      if (first_pv_of_seg && si > 0 && !wwait(&cs->o_free, (si - 1) & 1, cs, hdr)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t st = sSa + prev_s * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bd = smem_desc(st + kk * 2048, C::kLatBoxKv, 1024, kLayoutSw128);
          mma_ts(tmem, tmem + C::kSCol + 64 * prev_b + 8 * kk, bd, idesc_pv,
                 (first_pv_of_seg && kk == 0) ? 0u : 1u);
        }
        mma_commit(&cs->kv_empty[prev_s]);
        mma_commit(&cs->pv_done[prev_b]);
      }
      __syncwarp();
      first_pv_of_seg = false;
      return true;
    };
    for_each_segment(a, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool) {
      if (waborted(cs)) return;
      if (!wwait(&cs->q_full, si & 1, cs, hdr)) return;
      first_pv_of_seg = true;
      for (int it = ia; it < ie; ++it, ++c) {
        if (waborted(cs)) return;
        const int s = c % kStages, b = c & 1;
        if (MODE == kLoadFp8) {
          if (!wwait(&cs->kv_conv[s], (c / kStages) & 1, cs, hdr)) return;
        } else if (!wwait(&cs->kv_full[s], (c / kStages) & 1, cs, hdr)) {
          return;
        }
        const uint64_t mask = cs->row_mask[s];
        if (MODE != kLoadFp8 && mask != ~0ull) {
          // zero rows outside the key range in every box of the stage
          uint8_t* st = sStage + s * C::kStageBytes;
          const int chunks_per_row = C::NLB * 8 + 4;   // 16-byte chunks
          for (int i = lane; i < 64 * chunks_per_row; i += 32) {
            const int row = i / chunks_per_row, ch = i % chunks_per_row;
            if ((mask >> row) & 1ull) continue;
            uint8_t* dst = ch < C::NLB * 8 ? st + (ch >> 3) * C::kLatBoxKv + row * 128 + (ch & 7) * 16
                                           : st + C::NLB * C::kLatBoxKv + row * 64 + (ch - C::NLB * 8) * 16;
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t st = sSa + s * C::kStageBytes;
          int j = 0;
#pragma unroll
          for (int i = 0; i < C::NLB; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk, ++j) {
              const uint64_t ad = smem_desc(sQa + i * C::kLatBoxQ + kk * 32, 16, 1024, kLayoutSw128);
              const uint64_t bd = smem_desc(st + i * C::kLatBoxKv + kk * 32, 16, 1024, kLayoutSw128);
              mma_ss(tmem + C::kSCol + 64 * b, ad, bd, idesc_qk, j > 0 ? 1u : 0u);
            }
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t ad = smem_desc(sQa + C::NLB * C::kLatBoxQ + kk * 32, 16, 512, kLayoutSw64);
            const uint64_t bd = smem_desc(st + C::NLB * C::kLatBoxKv + kk * 32, 16, 512, kLayoutSw64);
            mma_ss(tmem + C::kSCol + 64 * b, ad, bd, idesc_qk, 1u);
          }
          mma_commit(&cs->s_full[b]);
        }
        __syncwarp();
        if (prev_c >= 0 && seg_of_prev == si && !issue_pv(si)) return;
        prev_s = s;
        prev_b = b;
        prev_c = c;
        seg_of_prev = si;
      }
      if (prev_c >= 0 && !issue_pv(si)) return;
      prev_c = -1;
      if (lane == 0) mma_commit(&cs->q_empty);
      __syncwarp();
    });
  } else if (MODE == kLoadFp8 && warp >= 6) {
    // ------------------------------------------------------------- e4m3 converters
    // thread ci widens tile row ci: LC e4m3 codes x row scale -> bf16 in the
    // 128B-swizzled latent boxes; dead rows become zeros (latent and rope).
    const int ci = tid - 192;
    int c = 0;
    for_each_segment(a, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool) {
      for (int it = ia; it < ie; ++it, ++c) {
        if (waborted(cs)) return;
        const int s = c % kStages;
        if (!wwait(&cs->kv_full[s], (c / kStages) & 1, cs, hdr)) return;
        uint8_t* st = sStage + s * C::kStageBytes;
        const bool live = (cs->row_mask[s] >> ci) & 1ull;
        const float sc = live ? a.kv_scales[cs->rowid[s][ci]] : 0.f;
        uint4 raw[LC / 16];
#pragma unroll
        for (int q = 0; q < LC / 16; ++q) raw[q] = *reinterpret_cast<const uint4*>(st + ci * LC + q * 16);
        // all rows are read before any is overwritten (the codes live where the bf16 rows go)
        mbar_arrive(&cs->conv_sync);
        if (!wwait(&cs->conv_sync, c & 1, cs, hdr)) return;
#pragma unroll
        for (int q = 0; q < LC / 16; ++q) {
          const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            o[2 * i] = live ? e4m3x2_scaled_bf16x2((uint16_t)(w[i] & 0xffff), sc) : 0u;
            o[2 * i + 1] = live ? e4m3x2_scaled_bf16x2((uint16_t)(w[i] >> 16), sc) : 0u;
          }
          const int col = 16 * q;                  // first latent column of this chunk pair
          uint8_t* box = st + (col >> 6) * C::kLatBoxKv + ci * 128;
          const int ch = (col & 63) >> 3;          // 16-byte chunk within the 128-byte row
          *reinterpret_cast<uint4*>(box + (((ch) ^ (ci & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(box + (((ch + 1) ^ (ci & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        if (!live) {
          uint4* rr = reinterpret_cast<uint4*>(st + C::NLB * C::kLatBoxKv + ci * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) rr[i] = make_uint4(0, 0, 0, 0);
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
    uint32_t peer_x = 0, peer_xfull = 0, peer_xempty = 0;
    if (CL == 2) {
      peer_x = mapa_shared(smem_u32(sX), peer);
      peer_xfull = mapa_shared(smem_u32(&cs->x_full), peer);
      peer_xempty = mapa_shared(smem_u32(&cs->x_empty), peer);
    }
    int c = 0;
    int nfix = 0;   // split-token merges attempted (phase of fix_bar / fix_done)
    for_each_segment(a, g0, g1, [&](int si, int t, const TokenPlan& tp, int ia, int ie, bool is_first_seg) {
      if (waborted(cs)) return;
      float m = -CUDART_INF_F, l = 0.f;
      int last_c = -1;
      for (int it = ia; it < ie; ++it, ++c) {
        if (waborted(cs)) return;
        const int s = c % kStages, b = c & 1;
        if (!wwait(&cs->kv_full[s], (c / kStages) & 1, cs, hdr)) return;   // row mask visibility
        const uint64_t mask = cs->row_mask[s];
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
        if (CL == 2) {
          // my partial S goes to the peer with asynchronous stores that count bytes on
          // the peer's x_full; the peer's partial arrives in mine the same way
          if (c > 0 && !wwait_cluster(&cs->x_empty, (c - 1) & 1, cs, hdr)) return;
          if (row == 0) mbar_arrive_expect_tx(&cs->x_full, 128 * 64 * 4);
          const uint32_t dst = peer_x + (uint32_t)(row * 256);
#pragma unroll
          for (int ch = 0; ch < 16; ++ch)
            st_async_v4(dst + (uint32_t)((ch ^ (row & 15)) * 16), sr[4 * ch], sr[4 * ch + 1], sr[4 * ch + 2],
                        sr[4 * ch + 3], peer_xfull);
          if (!wwait_cluster(&cs->x_full, c & 1, cs, hdr)) return;
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) {
            const float4 pv = *reinterpret_cast<const float4*>(sX + row * 64 + (ch ^ (row & 15)) * 4);
            sv[4 * ch] += pv.x;
            sv[4 * ch + 1] += pv.y;
            sv[4 * ch + 2] += pv.z;
            sv[4 * ch + 3] += pv.w;
          }
          mbar_arrive_cluster(peer_xempty);
        }
        // row max of the scaled scores (log2 domain); dead keys do not count
        const bool all_live = mask == ~0ull;
        float mx;
        if (sl2 >= 0.f) {
          float r = -CUDART_INF_F;
#pragma unroll
          for (int j = 0; j < 64; ++j) r = fmaxf(r, (all_live || ((mask >> j) & 1ull)) ? sv[j] : -CUDART_INF_F);
          mx = r == -CUDART_INF_F ? r : r * sl2;
        } else {
          float r = CUDART_INF_F;
#pragma unroll
          for (int j = 0; j < 64; ++j) r = fminf(r, (all_live || ((mask >> j) & 1ull)) ? sv[j] : CUDART_INF_F);
          mx = r == CUDART_INF_F ? -CUDART_INF_F : r * sl2;
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
        float psum = 0.f;
        const float neg_m = -m;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float p0 = ex2(fmaf(sv[2 * j], sl2, neg_m));
          float p1 = ex2(fmaf(sv[2 * j + 1], sl2, neg_m));
          if (!all_live) {
            p0 = ((mask >> (2 * j)) & 1ull) ? p0 : 0.f;
            p1 = ((mask >> (2 * j + 1)) & 1ull) ? p1 : 0.f;
          }
          psum += p0 + p1;
          pk[j] = pack_bf16(p0, p1);
        }
        l += psum;
        tmem_st32(trow + C::kSCol + 64 * b, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&cs->p_full[b]);
        last_c = c;
      }
      if (last_c < 0) return;
      // ------------------------------------------------------------- epilogue
      if (!wwait(&cs->pv_done[last_c & 1], (last_c >> 1) & 1, cs, hdr)) return;
      tc_fence_after();
      const bool complete = ia == 0 && ie == tp.ntiles;
      const int slot = is_first_seg ? 0 : 1;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
      const bool live = row < H;
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
          float4* dst = reinterpret_cast<float4*>(a.part_o + ((size_t)(k * 2 + slot) * H + row) * L + lat_x0 + col);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                 __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
        }
      }
      // O has been read: the next segment's first P . C may overwrite it
      tc_fence_before();
      mbar_arrive(&cs->o_free);
      if (live) {
        if (complete) {
          if (rank == 0) a.lse_ws[(size_t)t * H + row] = lse;
        } else {
          a.part_lse[((size_t)(k * 2 + slot) * 2 + rank) * H + row] = lse;
        }
      }
      if (!complete) {
        // split token: the partition that finishes it last (per cluster rank)
        // merges every partition's partial into o_lat / lse
        __threadfence();
        mbar_arrive(&cs->fix_bar);
        const int Qt = (total + a.K - 1) / a.K;
        const int kf = tp.tile_start / Qt, kl = (tp.tile_start + tp.ntiles - 1) / Qt;
        bool ok0 = true;
        if (row == 0) {
          ok0 = wait_or_abort(&cs->fix_bar, nfix & 1, cs, hdr);
          if (ok0) {
            const int prev = atomicAdd(&a.counters[2 * t + rank], 1);
            cs->fix_last = prev == kl - kf;
            mbar_arrive(&cs->fix_done);
          }
        }
        const bool ok1 = wait_or_abort(&cs->fix_done, nfix & 1, cs, hdr);
        if (!__all_sync(0xffffffffu, ok0 && ok1)) return;
        ++nfix;
        if (cs->fix_last) {
          __threadfence();
          if (live) merge_split_token(a, t, tp, kf, kl, Qt, rank, row, lat_x0, LC);
          if (row == 0) a.counters[2 * t + rank] = 0;
        }
      }
    });
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (CL == 2 && tid == 0) {
    // every remote store / arrive of this CTA is issued; tell the peer, and wait
    // (bounded) until the peer says the same before this CTA's memory goes away
    mbar_arrive_cluster(mapa_shared(smem_u32(&cs->bye), peer));
    if (!mbar_wait<true>(&cs->bye, 0, kWaitLimitNs)) {
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

template <int LC, int CL, int MODE>
cudaError_t launch(const DecodeArgs& a, cudaStream_t s) {
  using C = Cfg<LC, CL, MODE>;
  constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int L = a.d.kv_lora_rank, R = a.d.qk_rope, KQ = L + R, ps = a.d.page_size;
  const uint32_t rows = MODE == kLoadSparse ? 1u : (uint32_t)(ps < kTileKeys ? ps : kTileKeys);
  const uint64_t pool_rows = (uint64_t)a.d.num_pages * ps;
  Maps maps;
  bool ok;
  if (MODE == kLoadFp8) {
    const uint64_t rb = (uint64_t)L + 2 * R;   // bytes per cached row
    ok = encode_2d(&maps.kv_lat, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.kv_pool, rb, pool_rows, rb, LC, rows,
                   CU_TENSOR_MAP_SWIZZLE_NONE) &&
         encode_2d(&maps.kv_rope, kBF16, a.kv_pool, rb / 2, pool_rows, rb, 32, rows, CU_TENSOR_MAP_SWIZZLE_64B);
  } else {
    ok = encode_2d(&maps.kv_lat, kBF16, a.kv_pool, KQ, pool_rows, (uint64_t)KQ * 2, 64, rows,
                   CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_2d(&maps.kv_rope, kBF16, a.kv_pool, KQ, pool_rows, (uint64_t)KQ * 2, 32, rows,
                   CU_TENSOR_MAP_SWIZZLE_64B);
  }
  ok = ok &&
       encode_2d(&maps.q_lat, kBF16, a.q_full, KQ, (uint64_t)a.T * kMaxHeads, (uint64_t)KQ * 2, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B) &&
       encode_2d(&maps.q_rope, kBF16, a.q_full, KQ, (uint64_t)a.T * kMaxHeads, (uint64_t)KQ * 2, 32, 128,
                 CU_TENSOR_MAP_SWIZZLE_64B);
  if (!ok) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<LC, CL, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmem);
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

template <int MODE>
cudaError_t launch_mode(const DecodeArgs& a, cudaStream_t s) {
  if (a.d.kv_lora_rank == 512) return launch<256, 2, MODE>(a, s);
  return launch<64, 1, MODE>(a, s);
}

}  // namespace tc

// Shapes with a tensor-core instance: (L, R) = (512, 64) on a 2-CTA cluster,
// and L = 64 with R <= 32 on one CTA; dense pages of 8..64 tokens or a
// multiple of 64.
bool decode_tc_supported(const mla_dims_t& d) {
  const int ps = d.page_size;
  if (!(ps % kTileKeys == 0 || (kTileKeys % ps == 0 && ps >= 8))) return false;
  if (d.kv_lora_rank == 512 && d.qk_rope == 64) return true;
  if (d.kv_lora_rank == 64 && d.qk_rope <= 32 && d.qk_rope % 8 == 0) return true;
  return false;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  if (a.ks.indices) return tc::launch_mode<tc::kLoadSparse>(a, s);
  if (a.kv_fmt == KVFmt::kE4M3) return tc::launch_mode<tc::kLoadFp8>(a, s);
  return tc::launch_mode<tc::kLoadDense>(a, s);
}

}  // namespace mla
