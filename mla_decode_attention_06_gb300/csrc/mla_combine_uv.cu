// K3: log-sum-exp combine of the split-KV partials, then the W_uv projection
// back to v_head (mla_decode_branch_fp8 page: "output = raw_output_t @ w_uv",
// w_uv [num_heads, v_head_dim, kv_latent_dim]).
//
// Combine of the partitions p that cover one (token, head):
//   lse = ln sum_p exp(lse_p),   o = sum_p exp(lse_p - lse) * o_p
// Partitions whose key set was empty carry lse_p = -inf and drop out.
#include <math_constants.h>

#include "mla_kernels.cuh"

namespace mla {

constexpr int kUvTokens = 8;
constexpr int kUvThreads = 256;

template <WFmt WF>
__device__ __forceinline__ float wuv_elem(const void* w, const float* ws, int V, int L, int h, int v,
                                          int l) {
  const size_t idx = ((size_t)h * V + v) * L + l;
  if constexpr (WF == WFmt::kBF16) {
    return bf16_to_f32(((const uint16_t*)w)[idx]);
  } else {
    const int nv = (V + 127) >> 7, nl = (L + 127) >> 7;
    return e4m3_to_f32(((const uint8_t*)w)[idx]) * ws[((size_t)h * nv + (v >> 7)) * nl + (l >> 7)];
  }
}

// grid (H, ceil(T / 8)).
template <WFmt WF>
__global__ void __launch_bounds__(kUvThreads) combine_uv_kernel(DecodeArgs a, const void* __restrict__ w_uv,
                                                                const float* __restrict__ w_uv_scale,
                                                                __nv_bfloat16* __restrict__ out,
                                                                float* __restrict__ lse_out) {
  extern __shared__ float so[];   // [8][L]
  __shared__ int s_kf[kUvTokens], s_kl[kUvTokens], s_mode[kUvTokens];
  __shared__ float s_mx[kUvTokens], s_inv[kUvTokens], s_lse[kUvTokens];
  const int H = a.d.num_heads, L = a.d.kv_lora_rank, V = a.d.v_head;
  const int h = blockIdx.x, t0 = blockIdx.y * kUvTokens;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int total = a.hdr->total_tiles;
  const int Q = (total + a.K - 1) / a.K;
  // partial slot of partition k for a token whose first global tile is `start`:
  // its first partition kf holds it as the last segment (slot 1) unless the
  // token starts exactly at the partition's start.
  auto src_of = [&](int k, int kf, int start) {
    const int slot = (k == kf && start != k * Q) ? 1 : 0;
    return (k * 2 + slot) * H + h;
  };

  // warp tt classifies token tt: 0 = no keys, 1 = complete in o_lat, 2 = merge partials
  if (warp < kUvTokens) {
    const int tt = warp, t = t0 + tt;
    int mode = 0, kf = 0, kl = -1;
    float mx = -CUDART_INF_F, lse = -CUDART_INF_F, sum = 0.f;
    if (t < a.T) {
      const TokenPlan tp = a.plan[t];
      if (tp.ntiles > 0) {
        kf = tp.tile_start / Q;
        kl = (tp.tile_start + tp.ntiles - 1) / Q;
        if (kf == kl) {
          mode = 1;
          lse = a.lse_ws[(size_t)t * H + h];
        } else {
          for (int k = kf + lane; k <= kl; k += 32) mx = fmaxf(mx, a.part_lse[src_of(k, kf, tp.tile_start)]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (mx != -CUDART_INF_F) {
            for (int k = kf + lane; k <= kl; k += 32) sum += expf(a.part_lse[src_of(k, kf, tp.tile_start)] - mx);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            mode = 2;
            lse = mx + logf(sum);
          }
        }
        if (lane == 0) s_kf[tt] = tp.tile_start;   // reused below as the token's first tile
      }
    }
    if (lane == 0) {
      s_mode[tt] = mode;
      s_kl[tt] = kl;
      s_mx[tt] = mx;
      s_inv[tt] = sum > 0.f ? 1.f / sum : 0.f;
      s_lse[tt] = lse;
      if (mode != 2) s_kf[tt] = 0;
    }
  }
  __syncthreads();
  for (int i = tid; i < kUvTokens * L; i += kUvThreads) {
    const int tt = i / L, l = i % L, t = t0 + tt;
    float v = 0.f;
    const int mode = s_mode[tt];
    if (mode == 1) {
      v = __bfloat162float(a.o_lat[((size_t)t * H + h) * L + l]);
    } else if (mode == 2) {
      const int start = s_kf[tt], kf = start / Q, kl = s_kl[tt];
      const float mx = s_mx[tt], inv = s_inv[tt];
      for (int k = kf; k <= kl; ++k) {
        const int src = src_of(k, kf, start);
        v += expf(a.part_lse[src] - mx) * inv * a.part_o[(size_t)src * L + l];
      }
    }
    so[i] = v;
  }
  __syncthreads();
  for (int v = warp; v < V; v += kUvThreads / 32) {
    float acc[kUvTokens];
#pragma unroll
    for (int tt = 0; tt < kUvTokens; ++tt) acc[tt] = 0.f;
    for (int l = lane; l < L; l += 32) {
      const float w = wuv_elem<WF>(w_uv, w_uv_scale, V, L, h, v, l);
#pragma unroll
      for (int tt = 0; tt < kUvTokens; ++tt) acc[tt] += w * so[tt * L + l];
    }
#pragma unroll
    for (int tt = 0; tt < kUvTokens; ++tt) {
      float x = acc[tt];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      const int t = t0 + tt;
      if (lane == 0 && t < a.T) out[((size_t)t * H + h) * V + v] = __float2bfloat16_rn(x);
    }
  }
  if (lse_out && tid < kUvTokens && t0 + tid < a.T) lse_out[(size_t)(t0 + tid) * H + h] = s_lse[tid];
}

cudaError_t launch_combine_uv(const DecodeArgs& a, WFmt wf, const void* w_uv,
                              const float* w_uv_scale, __nv_bfloat16* out, float* lse_out,
                              cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  dim3 grid(a.d.num_heads, (a.T + kUvTokens - 1) / kUvTokens);
  const size_t smem = sizeof(float) * kUvTokens * a.d.kv_lora_rank;
  if (wf == WFmt::kBF16)
    combine_uv_kernel<WFmt::kBF16><<<grid, kUvThreads, smem, s>>>(a, w_uv, w_uv_scale, out, lse_out);
  else
    combine_uv_kernel<WFmt::kE4M3><<<grid, kUvThreads, smem, s>>>(a, w_uv, w_uv_scale, out, lse_out);
  return cudaGetLastError();
}

}  // namespace mla
