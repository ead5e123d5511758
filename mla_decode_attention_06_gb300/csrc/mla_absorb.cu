// K1: the W_uk absorb.  q_lat[t,h,:] = w_uk[h] . q_nope[t,h,:], concatenated
// with q_rope into the 576-wide (L + R) query row the decode consumes
// (mla_decode_branch_fp8 page: "q_nope_proj = q_nope_t @ w_uk" and
// "q_full = concat(q_nope_proj, q_rope, axis=2)").
//
// The query rows are stored 128 per token ([T, 128, L+R] bf16, rows h >= H
// zero) so the decode reads one full M = 128 tile per token.
#include "mla_kernels.cuh"

namespace mla {

constexpr int kAbsorbTokens = 8;    // tokens per block
constexpr int kAbsorbThreads = 256;

template <WFmt WF>
__device__ __forceinline__ float w_elem(const void* w, const float* ws, int A, int Bd, int h, int i,
                                        int j) {
  const size_t idx = ((size_t)h * A + i) * Bd + j;
  if constexpr (WF == WFmt::kBF16) {
    return bf16_to_f32(((const uint16_t*)w)[idx]);
  } else {
    const int na = (A + 127) >> 7, nb = (Bd + 127) >> 7;
    return e4m3_to_f32(((const uint8_t*)w)[idx]) * ws[((size_t)h * na + (i >> 7)) * nb + (j >> 7)];
  }
}

// grid (H, ceil(T / 8)); one warp produces one latent row l for 8 tokens at a time.
template <WFmt WF>
__global__ void __launch_bounds__(kAbsorbThreads) absorb_kernel(mla_dims_t d, int T,
                                                                const uint16_t* __restrict__ q,
                                                                const void* __restrict__ w_uk,
                                                                const float* __restrict__ w_uk_scale,
                                                                uint16_t* __restrict__ q_full) {
  extern __shared__ float sq[];   // [8][N]
  const int H = d.num_heads, N = d.qk_nope, R = d.qk_rope, L = d.kv_lora_rank, KQ = L + R;
  const int h = blockIdx.x, t0 = blockIdx.y * kAbsorbTokens;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kAbsorbTokens * N; i += kAbsorbThreads) {
    const int tt = i / N, n = i % N, t = t0 + tt;
    sq[i] = t < T ? bf16_to_f32(q[((size_t)t * H + h) * (N + R) + n]) : 0.f;
  }
  __syncthreads();
  for (int l = warp; l < L; l += kAbsorbThreads / 32) {
    float acc[kAbsorbTokens];
#pragma unroll
    for (int tt = 0; tt < kAbsorbTokens; ++tt) acc[tt] = 0.f;
    for (int n = lane; n < N; n += 32) {
      const float w = w_elem<WF>(w_uk, w_uk_scale, L, N, h, l, n);
#pragma unroll
      for (int tt = 0; tt < kAbsorbTokens; ++tt) acc[tt] += w * sq[tt * N + n];
    }
#pragma unroll
    for (int tt = 0; tt < kAbsorbTokens; ++tt) {
      float v = acc[tt];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      const int t = t0 + tt;
      if (lane == 0 && t < T)
        q_full[((size_t)t * kMaxHeads + h) * KQ + l] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  }
  // rope columns are copied unchanged
  for (int i = tid; i < kAbsorbTokens * R; i += kAbsorbThreads) {
    const int tt = i / R, r = i % R, t = t0 + tt;
    if (t < T) q_full[((size_t)t * kMaxHeads + h) * KQ + L + r] = q[((size_t)t * H + h) * (N + R) + N + r];
  }
  // rows of absent heads are zero
  if (h == 0) {
    for (int i = tid; i < kAbsorbTokens * (kMaxHeads - H) * KQ; i += kAbsorbThreads) {
      const int per = (kMaxHeads - H) * KQ;
      const int tt = i / per, rem = i % per, t = t0 + tt;
      if (t < T) q_full[((size_t)t * kMaxHeads + H) * KQ + rem] = 0;
    }
  }
}

cudaError_t launch_absorb(const mla_dims_t& d, int T, const __nv_bfloat16* q, WFmt wf,
                          const void* w_uk, const float* w_uk_scale, __nv_bfloat16* q_full,
                          cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 grid(d.num_heads, (T + kAbsorbTokens - 1) / kAbsorbTokens);
  const size_t smem = sizeof(float) * kAbsorbTokens * d.qk_nope;
  if (wf == WFmt::kBF16)
    absorb_kernel<WFmt::kBF16><<<grid, kAbsorbThreads, smem, s>>>(
        d, T, (const uint16_t*)q, w_uk, w_uk_scale, (uint16_t*)q_full);
  else
    absorb_kernel<WFmt::kE4M3><<<grid, kAbsorbThreads, smem, s>>>(
        d, T, (const uint16_t*)q, w_uk, w_uk_scale, (uint16_t*)q_full);
  return cudaGetLastError();
}

}  // namespace mla
