// K2 (CUDA-core version): split-KV MLA decode over 64-key tiles.
//
// Partition k of K owns the global tiles [k*Q, (k+1)*Q), Q = ceil(total/K)
// (the split-KV partitions of num_partitions_in on the
// generic_flare_mla_decode_kv_cache_ragged page).  A block handles 16 heads of
// one partition; it walks the partition's segments (one per query token it
// touches), keeps a running max / sum per head (online softmax) and either
// writes the normalised latent output (the token lies wholly inside the
// partition) or a partial (o_p, lse_p) for the combine step.
#include <math_constants.h>

#include "mla_kernels.cuh"

namespace mla {

constexpr int kSimtHeads = 16;
constexpr int kSimtThreads = 256;
constexpr int kSimtMaxL16 = 32;   // L / 16 <= 32, so L <= 512

template <KVFmt KF>
__global__ void __launch_bounds__(kSimtThreads) decode_simt_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int H = a.d.num_heads, L = a.d.kv_lora_rank, R = a.d.qk_rope, KQ = L + R;
  const int TS = KQ + 2;   // padded tile row (bf16) to spread banks
  float* sQ = reinterpret_cast<float*>(smem);          // [16][KQ]
  float* sP = sQ + kSimtHeads * KQ;                    // [16][64]
  int* sRow = reinterpret_cast<int*>(sP + kSimtHeads * kTileKeys);   // [64]
  uint16_t* sT = reinterpret_cast<uint16_t*>(sRow + kTileKeys);      // [64][TS]

  const int k = blockIdx.x, hg = blockIdx.y;
  const int tid = threadIdx.x, hh = tid >> 4, l16 = tid & 15;
  const int h = hg * kSimtHeads + hh;
  const int total = a.hdr->total_tiles;
  const int g0 = partition_begin(k, a.K, total), g1 = partition_begin(k + 1, a.K, total);
  if (g0 >= g1) return;
  const int nl = L >> 4;
  const int ps = a.ks.page_size;
  const float sl2 = a.scale * 1.4426950408889634f;   // scores in the log2 domain
  bool bad = false;

  int g = g0;
  int t = token_of_tile(a.plan, a.T, g);
  while (g < g1) {
    const TokenPlan tp = a.plan[t];
    const int seg_a = g - tp.tile_start;
    const int seg_e = min(g1, tp.tile_start + tp.ntiles) - tp.tile_start;
    const bool complete = seg_a == 0 && seg_e == tp.ntiles;
    const int slot = (g == g0) ? 0 : 1;

    __syncthreads();
    for (int i = tid; i < kSimtHeads * KQ; i += kSimtThreads) {
      const int r = i / KQ, c = i % KQ, hr = hg * kSimtHeads + r;
      sQ[i] = hr < H ? __bfloat162float(a.q_full[((size_t)t * kMaxHeads + hr) * KQ + c]) : 0.f;
    }
    float m = -CUDART_INF_F, lsum = 0.f;
    float o[kSimtMaxL16];
#pragma unroll
    for (int i = 0; i < kSimtMaxL16; ++i) o[i] = 0.f;

    for (int it = seg_a; it < seg_e; ++it) {
      const int key0 = (tp.tile_first + it) * kTileKeys;
      __syncthreads();
      if (tid < kTileKeys) {
        const int key = key0 + tid;
        int row = -1;
        if (key >= tp.lo && key < tp.hi) {
          if (a.ks.indices) {
            const int idx = a.ks.indices[(size_t)tp.b * a.ks.idx_stride + key];
            if (idx >= 0 && idx < a.ks.num_pages * ps) row = idx;
            else if (idx != -1) bad = true;
          } else {
            const int page = a.ks.block_table[(size_t)tp.b * a.ks.bt_stride + key / ps];
            if (page >= 0 && page < a.ks.num_pages) row = page * ps + key % ps;
            else bad = true;
          }
        }
        sRow[tid] = row;
      }
      __syncthreads();
      const int half = KQ >> 1;
      for (int i = tid; i < kTileKeys * half; i += kSimtThreads) {
        const int j = i / half, c2 = i % half;
        const int row = sRow[j];
        uint32_t v = 0;
        if (row >= 0) {
          if constexpr (KF == KVFmt::kBF16) {
            v = reinterpret_cast<const uint32_t*>(
                static_cast<const uint16_t*>(a.kv_pool) + (size_t)row * KQ)[c2];
          } else {
            const uint8_t* rp = static_cast<const uint8_t*>(a.kv_pool) + (size_t)row * (L + 2 * R);
            const int c = 2 * c2;
            if (c < L) {
              const float sc = a.kv_scales[row];
              const float x0 = e4m3_to_f32(rp[c]) * sc, x1 = e4m3_to_f32(rp[c + 1]) * sc;
              v = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
                  ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
            } else {
              v = *reinterpret_cast<const uint32_t*>(rp + L + 2 * (c - L));
            }
          }
        }
        reinterpret_cast<uint32_t*>(sT + (size_t)j * TS)[c2] = v;
      }
      __syncthreads();

      // scores of head hh for keys j = l16 + 16 r
      float s[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int j = l16 + 16 * r;
        const float* qr = sQ + hh * KQ;
        const uint32_t* kr = reinterpret_cast<const uint32_t*>(sT + (size_t)j * TS);
        float acc = 0.f;
        for (int c2 = 0; c2 < half; ++c2) {
          const uint32_t kv = kr[c2];
          acc += qr[2 * c2] * bf16_to_f32((uint16_t)(kv & 0xffff)) +
                 qr[2 * c2 + 1] * bf16_to_f32((uint16_t)(kv >> 16));
        }
        s[r] = sRow[j] >= 0 ? acc * sl2 : -CUDART_INF_F;
      }
      float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off, 16));
      const float m_new = fmaxf(m, mx);
      float alpha = 1.f, psum = 0.f;
      if (m_new != -CUDART_INF_F) {
        alpha = (m == -CUDART_INF_F) ? 0.f : exp2f(m - m_new);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float p = (s[r] == -CUDART_INF_F) ? 0.f : exp2f(s[r] - m_new);
          sP[hh * kTileKeys + l16 + 16 * r] = p;
          psum += p;
        }
      } else {
#pragma unroll
        for (int r = 0; r < 4; ++r) sP[hh * kTileKeys + l16 + 16 * r] = 0.f;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off, 16);
      lsum = lsum * alpha + psum;
      m = m_new;
      __syncwarp();
#pragma unroll
      for (int i = 0; i < kSimtMaxL16; ++i) {
        if (i < nl) {
          float acc = o[i] * alpha;
          const int col = l16 + 16 * i;
          for (int j = 0; j < kTileKeys; ++j) acc += sP[hh * kTileKeys + j] * bf16_to_f32(sT[(size_t)j * TS + col]);
          o[i] = acc;
        }
      }
    }

    if (h < H) {
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const float lse = lsum > 0.f ? (m + log2f(lsum)) * 0.6931471805599453f : -CUDART_INF_F;
      if (complete) {
#pragma unroll
        for (int i = 0; i < kSimtMaxL16; ++i)
          if (i < nl) a.o_lat[((size_t)t * H + h) * L + l16 + 16 * i] = __float2bfloat16_rn(o[i] * inv);
        if (l16 == 0) a.lse_ws[(size_t)t * H + h] = lse;
      } else {
        const size_t base = ((size_t)(k * 2 + slot) * H + h);
#pragma unroll
        for (int i = 0; i < kSimtMaxL16; ++i)
          if (i < nl) a.part_o[base * L + l16 + 16 * i] = o[i] * inv;
        if (l16 == 0) a.part_lse[base] = lse;
      }
    }
    g = tp.tile_start + seg_e;
    if (g < g1) t = token_of_tile(a.plan, a.T, g);
  }
  if (bad) atomicOr(&a.hdr_mut->status, kDeviceCheckFailed);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const int KQ = a.d.kv_lora_rank + a.d.qk_rope;
  const size_t smem = sizeof(float) * kSimtHeads * KQ + sizeof(float) * kSimtHeads * kTileKeys +
                      sizeof(int) * kTileKeys + 2 * (size_t)kTileKeys * (KQ + 2);
  dim3 grid(a.K, (a.d.num_heads + kSimtHeads - 1) / kSimtHeads);
  cudaError_t e;
  if (a.kv_fmt == KVFmt::kBF16) {
    e = cudaFuncSetAttribute(decode_simt_kernel<KVFmt::kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    decode_simt_kernel<KVFmt::kBF16><<<grid, kSimtThreads, smem, s>>>(a);
  } else {
    e = cudaFuncSetAttribute(decode_simt_kernel<KVFmt::kE4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    decode_simt_kernel<KVFmt::kE4M3><<<grid, kSimtThreads, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace mla
