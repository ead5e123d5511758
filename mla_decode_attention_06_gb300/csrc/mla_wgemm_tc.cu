// K1 and K3 on tcgen05: the two per-head weight GEMMs of the absorbed MLA
// decode (mla_decode_branch_fp8 page: "q_nope_proj = q_nope_t @ w_uk" and
// "output = raw_output_t @ w_uv"; w_uk [num_heads, kv_latent_dim,
// qk_nope_head_dim], w_uv [num_heads, v_head_dim, kv_latent_dim]).
//
// Both have the shape  D[m, t] = sum_k W[h, m, k] * X[t, h, k]  per head h:
//   absorb (K1): W = w_uk, m = latent column l, k = nope column, X = q
//                -> written as bf16 into q_full[t, h, l]; CTAs of the first
//                   m block also copy q_rope into q_full[t, h, L:L+R].
//   W_uv   (K3): W = w_uv, m = v column, k = latent column, X = o_lat
//                -> written as bf16 into out[t, h, v] (and lse copied out).
// One CTA owns one head (or half of its rows, when they split evenly into
// 128-row blocks: two CTAs per head, two per SM) and up to 128 tokens: MB
// blocks of 128 weight rows (M <= 512), N = tokens, K streamed in 64-column
// steps.  A step loads the MB weight boxes and one activation box; the ring is
// as deep as shared memory allows (the absorb holds all of K = 128, W_uv all
// of K = 512 in 8 stages), so every load of the CTA is in flight at once and
// one wave of CTAs covers the GEMM.  The weights are read once per
// token block, which is what bounds these kernels (HBM): 16.8 MB per weight at
// the DeepSeek-V3 shapes.
//
// FP8 weights: e4m3 codes are widened to bf16 (exactly: every e4m3 value is a
// bf16 value) in shared memory, and the 128 x 128 block scale is applied in
// the epilogue; because the scale changes every 128 columns of k, each
// 128-wide k block accumulates into its own TMEM columns and the epilogue sums
// scale_b * D_b.
#include <algorithm>
#include <mutex>

#include "mla_kernels.cuh"
#include "mla_plan.cuh"
#include "sm100_ptx.cuh"

namespace mla {
namespace wg {

using namespace sm100;

constexpr int kThreads = 128;
constexpr int kMaxStages = 8;
constexpr int kMaxMB = 4;                  // 128-row weight blocks per CTA (M <= 512)
constexpr int kMaxTokens = 128;            // tokens per CTA (MMA N)
constexpr int kStageBudget = 220 * 1024;   // shared memory for the ring
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kABytes = 128 * 128;         // 128 rows x 64 bf16
constexpr int kA8Bytes = 128 * 64;         // 128 rows x 64 e4m3

struct Maps {
  CUtensorMap w;   // bf16 [H*M rows, K cols] (128B swizzle) or e4m3 [H*M, K] (no swizzle)
  CUtensorMap x;   // bf16 3-D {Kx cols, H, T} (128B swizzle)
};

struct Args {
  int mode;            // 0 absorb, 1 W_uv
  int H, T, M, K;      // heads, tokens, weight rows per head, contraction length
  int TN;              // tokens per CTA (multiple of 16, <= 128)
  int MB, S;           // weight row blocks per CTA, ring stages
  int MC;              // CTAs per head: CTA mc of head h owns row blocks [mc * MB, mc * MB + MB)
  const float* wscale; // e4m3 block scales [H, ceil(M/128), ceil(K/128)]
  // absorb
  __nv_bfloat16* q_full; int KQ, L, R, N; const __nv_bfloat16* q;
  // W_uv
  __nv_bfloat16* out; int V; const float* lse_ws; float* lse_out;
  PlanHeader* hdr;
  PlanInputs pin;      // absorb: block (0, H * MC, 0) plans the call
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, PlanHeader* hdr) {
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  atomicOr(&hdr->status, kDeviceTimeout);
  return false;
}
// The k loop's issuing thread spins instead (a suspended waiter can wake well
// after the phase completes).
__device__ __forceinline__ bool spin_bar(uint64_t* bar, uint32_t parity, PlanHeader* hdr) {
  if (mbar_spin(bar, parity, kWaitLimitNs)) return true;
  atomicOr(&hdr->status, kDeviceTimeout);
  return false;
}

// e4m3 byte pair -> bf16x2 through the exact fp8 -> half conversion.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f.x)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f.y)) << 16);
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) wgemm_kernel(const __grid_constant__ Maps maps, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int TN = a.TN, MB = a.MB, S = a.S;
  const int kBBytes = TN * 128;
  // stage: MB bf16 weight boxes | activation box | (e4m3) MB raw weight boxes
  const int stage_smem = MB * kABytes + kBBytes + (kFp8 ? MB * kA8Bytes : 0);
  const uint32_t stage_tx = MB * (kFp8 ? kA8Bytes : kABytes) + kBBytes;
  // the ring, reused by the epilogue as a [MB][TN][128] bf16 staging tile
  const int ring_bytes = max(S * stage_smem, MB * TN * 128 * 2);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + ring_bytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* done = empty + kMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  auto w_box = [&](int s, int i) { return sm + s * stage_smem + i * kABytes; };
  auto x_box = [&](int s) { return sm + s * stage_smem + MB * kABytes; };
  auto w8_box = [&](int s, int i) { return sm + s * stage_smem + MB * kABytes + kBBytes + i * kA8Bytes; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y / a.MC, mb0 = (blockIdx.y % a.MC) * MB, t0 = blockIdx.z * TN;
  // absorb: one block of its own plans the call, beside the GEMM blocks (the
  // decode reads the plan after this grid completes)
  if (a.mode == 0 && (int)blockIdx.y == a.H * a.MC) {
    if (blockIdx.z == 0) plan_block(a.pin);
    return;
  }
  const int nkb = (a.K + 63) / 64;                 // 64-wide k steps
  const int nacc = kFp8 ? (a.K + 127) / 128 : 1;   // accumulators per weight block
  const int ncols_needed = MB * nacc * TN;
  const uint32_t tcols = ncols_needed <= 32 ? 32 : ncols_needed <= 64 ? 64 : ncols_needed <= 128 ? 128
                         : ncols_needed <= 256 ? 256 : 512;

  auto load_w = [&](int kb) {
    const int s = kb % S;
    for (int i = 0; i < MB; ++i)
      tma_load_2d(kFp8 ? w8_box(s, i) : w_box(s, i), &maps.w, &full[s], kb * 64, h * a.M + 128 * (mb0 + i));
  };
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    fence_mbar_init();
    // the weights depend neither on the previous kernel nor on TMEM: they start
    // streaming before the allocation and the block-wide sync
    for (int kb = 0; kb < nkb && kb < S; ++kb) {
      mbar_arrive_expect_tx(&full[kb], stage_tx);
      load_w(kb);
    }
    prefetch_tensormap(&maps.x);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto load_x = [&](int kb) {
    const int s = kb % S;
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            smem_u32(x_box(s))),
        "l"(reinterpret_cast<uint64_t>(&maps.x)), "r"(smem_u32(&full[s])), "r"(kb * 64), "r"(h), "r"(t0)
        : "memory");
  };
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");   // q (absorb) / o_lat, lse of the decode (W_uv)
  if (tid == 0)
    for (int kb = 0; kb < nkb && kb < S; ++kb) load_x(kb);
  // W_uv: the log-sum-exp rows go out while the MMAs run (not thread 0's warp
  // when one thread runs the k loop)
  if (a.mode == 1 && a.lse_out && mb0 == 0 && (kFp8 || warp > 0)) {
    const int first = kFp8 ? tid : tid - 32, stride = kFp8 ? kThreads : kThreads - 32;
    for (int j = first; j < TN; j += stride)
      if (t0 + j < a.T) a.lse_out[(size_t)(t0 + j) * a.H + h] = a.lse_ws[(size_t)(t0 + j) * a.H + h];
  }

  const uint32_t idesc = idesc_bf16_f32(128, TN, false, false);
  // MMAs of k step kb (stage s) into the accumulators, and the stage's refill
  auto issue = [&](int kb, int s) -> bool {
    const int acc = kFp8 ? (kb >> 1) : 0;
    const bool first_in_acc = kFp8 ? ((kb & 1) == 0) : (kb == 0);
    const uint64_t bd0 = smem_desc(smem_u32(x_box(s)), 16, 1024, kLayoutSw128);
    for (int i = 0; i < MB; ++i) {
      const uint64_t ad0 = smem_desc(smem_u32(w_box(s, i)), 16, 1024, kLayoutSw128);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(tmem + (i * nacc + acc) * TN, ad0 + (uint64_t)(kk * 2), bd0 + (uint64_t)(kk * 2), idesc,
               (first_in_acc && kk == 0) ? 0u : 1u);
    }
    mma_commit(&empty[s]);
    if (kb + S < nkb) {
      // the stage is refilled once the MMAs above have read it
      if (!spin_bar(&empty[s], (kb / S) & 1, a.hdr)) return false;
      mbar_arrive_expect_tx(&full[s], stage_tx);
      load_w(kb + S);
      load_x(kb + S);
    }
    return true;
  };
  // absorb: the rope columns of q go to q_full unchanged (independent of the
  // GEMM, so done while the MMAs run), 16 bytes at a time with every load of a
  // thread issued before its stores (q and q_full may not alias, but the
  // compiler cannot know that); absent heads are zero rows
  auto copy_rope = [&](int first, int stride) {
    const int cpr = a.R / 8;   // 16-byte chunks per (token, head) row
    constexpr int kBatch = 8;
    for (int i0 = first; i0 < TN * cpr; i0 += stride * kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * stride, t = t0 + i / cpr;
        if (i < TN * cpr && t < a.T)
          v[j] = __ldg(reinterpret_cast<const uint4*>(a.q + ((size_t)t * a.H + h) * (a.N + a.R) + a.N) + i % cpr);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j * stride, t = t0 + i / cpr;
        if (i < TN * cpr && t < a.T)
          reinterpret_cast<uint4*>(a.q_full + ((size_t)t * kMaxHeads + h) * a.KQ + a.L)[i % cpr] = v[j];
      }
    }
    if (h == 0 && a.H < kMaxHeads) {
      const int per = (kMaxHeads - a.H) * a.KQ;
      for (int i = first; i < TN * per; i += stride) {
        const int t = t0 + i / per;
        if (t < a.T) a.q_full[((size_t)t * kMaxHeads + a.H) * a.KQ + i % per] = __float2bfloat16_rn(0.f);
      }
    }
  };
  bool ok = true;
  if (!kFp8) {
    // one thread runs the whole k loop; the others only wait for the result
    if (a.mode == 0 && mb0 == 0 && warp > 0) copy_rope(tid - 32, kThreads - 32);
    if (tid == 0) {
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % S;
        ok = spin_bar(&full[s], (kb / S) & 1, a.hdr);
        if (!ok) break;
        tc_fence_after();
        ok = issue(kb, s);
      }
    }
  } else {
    if (a.mode == 0 && mb0 == 0) copy_rope(tid, kThreads);
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % S;
      // every thread waits; the CTA proceeds only if all saw the stage arrive
      if (!__syncthreads_and(wait_bar(&full[s], (kb / S) & 1, a.hdr))) {
        ok = false;
        break;
      }
      // widen row `tid` of each e4m3 box into the 128B-swizzled bf16 layout; a
      // thread takes its row's eight 8-byte pieces in a rotated order (rows are 64
      // bytes apart: in order, a half warp's reads would share two banks)
      for (int i = 0; i < MB; ++i) {
        const uint8_t* src = w8_box(s, i) + tid * 64;
        uint8_t* dst = w_box(s, i) + tid * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const int ch = (c8 + tid) & 7;
          const uint2 raw = *reinterpret_cast<const uint2*>(src + ch * 8);
          uint4 v;
          v.x = e4m3x2_to_bf16x2((uint16_t)(raw.x & 0xffff));
          v.y = e4m3x2_to_bf16x2((uint16_t)(raw.x >> 16));
          v.z = e4m3x2_to_bf16x2((uint16_t)(raw.y & 0xffff));
          v.w = e4m3x2_to_bf16x2((uint16_t)(raw.y >> 16));
          *reinterpret_cast<uint4*>(dst + ((ch ^ (tid & 7)) * 16)) = v;
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      tc_fence_after();
      bool issued_ok = true;
      if (tid == 0) issued_ok = issue(kb, s);
      if (!__syncthreads_and(issued_ok)) {
        ok = false;
        break;
      }
    }
  }
  if (tid == 0) mma_commit(done);
  __syncwarp();
  const bool fin = wait_bar(done, 0, a.hdr);
  ok = __syncthreads_and(ok) && fin;
  tc_fence_after();

  // ------------------------------------------------------------------ epilogue
  // D (TMEM lane = weight row m, column = token) goes through shared memory
  // (the ring is idle now) as [block][token][128 rows] bf16, then out as
  // 16-byte pieces of the contiguous output rows.
  const int row = 32 * warp + lane;    // weight row within a block = TMEM lane
  const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
  __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(sm);
  for (int i = 0; i < MB; ++i) {
    float sc[4] = {1.f, 1.f, 1.f, 1.f};
    if (kFp8) {
      const int nmb = (a.M + 127) / 128;
      for (int b = 0; b < nacc && b < 4; ++b) sc[b] = a.wscale[((size_t)h * nmb + mb0 + i) * nacc + b];
    }
    for (int j0 = 0; j0 < TN; j0 += 32) {
      // 32 token columns of every accumulator in flight before one wait
      float v[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = 0.f;
      for (int b = 0; b < nacc; ++b) {
        uint32_t r[32];
        if (j0 + 32 <= TN) {
          tmem_ld32(trow + (i * nacc + b) * TN + j0, r);
        } else {
          tmem_ld16(trow + (i * nacc + b) * TN + j0, *reinterpret_cast<uint32_t(*)[16]>(r));
#pragma unroll
          for (int q = 16; q < 32; ++q) r[q] = 0u;
        }
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] += sc[b] * __uint_as_float(r[q]);
      }
#pragma unroll
      for (int q = 0; q < 32; ++q)
        if (j0 + q < TN) stg[((size_t)i * TN + j0 + q) * 128 + row] = __float2bfloat16_rn(v[q]);
    }
  }
  __syncthreads();
  if (ok) {
    // output row of (token t, block i): 128 weight rows (fewer in the last
    // block) as 16 pieces of 16 bytes; 8 rows of 16 threads per pass
    const int piece = tid & 15;
    const int ntok = min(TN, a.T - t0);
    for (int i = 0; i < MB; ++i) {
      const int m = 128 * (mb0 + i) + 8 * piece;
      if (m >= a.M) continue;
      const __nv_bfloat16* src = stg + (size_t)i * TN * 128 + 8 * piece;
      __nv_bfloat16* dst = a.mode == 0 ? a.q_full + ((size_t)t0 * kMaxHeads + h) * a.KQ + m
                                       : a.out + ((size_t)t0 * a.H + h) * a.V + m;
      const size_t dst_pitch = a.mode == 0 ? (size_t)kMaxHeads * a.KQ : (size_t)a.H * a.V;
      for (int tt = tid >> 4; tt < ntok; tt += kThreads / 16)
        *reinterpret_cast<uint4*>(dst + tt * dst_pitch) = *reinterpret_cast<const uint4*>(src + tt * 128);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

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

cudaError_t launch(const Args& a0, WFmt wf, const void* w, const void* x, int Kx, cudaStream_t s) {
  Args a = a0;
  EncodeTiledFn fn = encode_fn();
  if (!fn || a.T == 0) return a.T == 0 ? cudaSuccess : cudaErrorInvalidValue;
  a.TN = a.T >= kMaxTokens ? kMaxTokens : ((a.T + 15) / 16) * 16;
  a.MB = (a.M + 127) / 128;
  if (a.MB > kMaxMB) return cudaErrorInvalidValue;
  // two CTAs per head when the row blocks split evenly: twice the CTAs (two
  // fit on an SM), half the weight bytes and output rows each
  a.MC = a.MB % 2 == 0 ? 2 : 1;
  a.MB /= a.MC;
  {
    // TMEM: MB weight blocks x (e4m3: one accumulator per 128-wide k block) x TN columns
    const int nacc = wf == WFmt::kE4M3 ? (a.K + 127) / 128 : 1;
    while (a.TN > 16 && a.MB * nacc * a.TN > 512) a.TN -= 16;
    if (a.MB * nacc * a.TN > 512) return cudaErrorInvalidValue;
  }
  const int stage_smem = a.MB * kABytes + a.TN * 128 + (wf == WFmt::kE4M3 ? a.MB * kA8Bytes : 0);
  {
    const int nkb = (a.K + 63) / 64;
    int st = kStageBudget / stage_smem;
    if (st > kMaxStages) st = kMaxStages;
    if (st > nkb) st = nkb;
    a.S = st < 1 ? 1 : st;
  }
  // the two GEMMs of a call (absorb, W_uv) keep their last tensor maps: the
  // serving loop calls them on the same buffers every layer call
  struct Key {
    int device, mode, T, TN, Kx, K, H, M;
    bool f8;
    const void *w, *x;
    bool operator==(const Key& o) const {
      return device == o.device && mode == o.mode && T == o.T && TN == o.TN && Kx == o.Kx && K == o.K && H == o.H &&
             M == o.M && f8 == o.f8 && w == o.w && x == o.x;
    }
  };
  static std::mutex cache_mu;
  static bool cache_valid[2] = {false, false};
  static Key cache_key[2];
  static Maps cache_maps[2];
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return cudaErrorInvalidDevice;
  const Key key{device, a.mode, a.T, a.TN, Kx, a.K, a.H, a.M, wf == WFmt::kE4M3, w, x};
  Maps maps;
  bool hit;
  {
    std::lock_guard<std::mutex> lock(cache_mu);
    hit = cache_valid[a.mode] && cache_key[a.mode] == key;
    if (hit) maps = cache_maps[a.mode];
  }
  if (!hit) {
  {
    const bool f8 = wf == WFmt::kE4M3;
    cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.H * a.M};
    cuuint64_t strides[1] = {(cuuint64_t)a.K * (f8 ? 1 : 2)};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    if (fn(&maps.w, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w),
           dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           f8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)Kx, (cuuint64_t)a.H, (cuuint64_t)a.T};
    cuuint64_t strides[2] = {(cuuint64_t)Kx * 2, (cuuint64_t)a.H * Kx * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)a.TN};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
    std::lock_guard<std::mutex> lock(cache_mu);
    cache_key[a.mode] = key;
    cache_maps[a.mode] = maps;
    cache_valid[a.mode] = true;
  }
  const bool f8 = wf == WFmt::kE4M3;
  const size_t ring_bytes = std::max((size_t)a.S * stage_smem, (size_t)a.MB * a.TN * 128 * 2);
  const size_t smem = 1024 + ring_bytes + (2 * kMaxStages + 2) * 8;
  if (smem > 232448) return cudaErrorInvalidValue;
  dim3 grid(1, a.H * a.MC + (a.mode == 0 ? 1 : 0), (a.T + a.TN - 1) / a.TN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // W_uv overlaps the decode's tail
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.mode == 1 ? 1 : 0;
  cudaError_t e;
  if (f8) {
    e = ensure_smem_limit(reinterpret_cast<const void*>(wgemm_kernel<true>), (int)smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, wgemm_kernel<true>, maps, a);
  } else {
    e = ensure_smem_limit(reinterpret_cast<const void*>(wgemm_kernel<false>), (int)smem);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, wgemm_kernel<false>, maps, a);
  }
  return e;
}

}  // namespace wg

cudaError_t launch_absorb_tc(const mla_dims_t& d, int T, const __nv_bfloat16* q, WFmt wf, const void* w_uk,
                             const float* w_uk_scale, __nv_bfloat16* q_full, PlanHeader* hdr,
                             const PlanInputs& plan, cudaStream_t s) {
  wg::Args a{};
  a.mode = 0;
  a.H = d.num_heads;
  a.T = T;
  a.M = d.kv_lora_rank;
  a.K = d.qk_nope;
  a.wscale = w_uk_scale;
  a.q_full = q_full;
  a.KQ = d.kv_lora_rank + d.qk_rope;
  a.L = d.kv_lora_rank;
  a.R = d.qk_rope;
  a.N = d.qk_nope;
  a.q = q;
  a.hdr = hdr;
  a.pin = plan;
  return wg::launch(a, wf, w_uk, q, d.qk_nope + d.qk_rope, s);
}

cudaError_t launch_uv_tc(const mla_dims_t& d, int T, const __nv_bfloat16* o_lat, WFmt wf, const void* w_uv,
                         const float* w_uv_scale, const float* lse_ws, __nv_bfloat16* out, float* lse_out,
                         PlanHeader* hdr, cudaStream_t s) {
  wg::Args a{};
  a.mode = 1;
  a.H = d.num_heads;
  a.T = T;
  a.M = d.v_head;
  a.K = d.kv_lora_rank;
  a.wscale = w_uv_scale;
  a.out = out;
  a.V = d.v_head;
  a.lse_ws = lse_ws;
  a.lse_out = lse_out;
  a.hdr = hdr;
  return wg::launch(a, wf, w_uv, o_lat, d.kv_lora_rank, s);
}

}  // namespace mla
