// The fused branch prologue of the mla_decode_branch_fp8 page (description:
// "Apply RoPE to the query and the key cache (in-place)", "Apply RMSNorm to
// the non-rope portion of the key cache (in-place)"; Args freqs_cis,
// kv_norm_gamma, epsilon), run before the absorb of a decode step.
//
// For query token t of request b at position pos = cache_len - qlen + i:
//   - every head's rope values (x[2i], x[2i+1]) turn by freqs_cis[pos] (the
//     table holds interleaved (cos, sin) pairs): (x0 c - x1 s, x0 s + x1 c);
//   - the cache row at position pos of request b (the row this step wrote) gets
//     RMSNorm of its latent part, c / sqrt(mean(c^2) + eps) * gamma, and the
//     same rotation of its rope part;
//   - nothing else changes.
// Every result is the bf16 (nearest, ties to even) of the expression's value:
//   - rotations: the two products of bf16 values are exact in fp32 and their
//     difference / sum is formed exactly as an fp32 pair (TwoSum), which is
//     rounded to bf16 once, looking at the low part only at a halfway point; the
//     result is the exactly rounded value of x0 c - x1 s (x0 s + x1 c), as a
//     double-precision evaluation gives it;
//   - RMSNorm: the mean square, 1 / sqrt(mean + eps) and the two products are
//     double precision; the mean square is summed by a tree and 1 / sqrt comes
//     from the double-precision rsqrt (both within a few units of the last place
//     of the in-order, correctly rounded evaluation, far below the bf16 rounding
//     step), the products rounded on their own, the result rounded once to bf16.
//
// A token's heads are shared by G blocks (blockIdx.y = 0 .. G-1, G chosen so the
// grid fills the SMs' resident block slots in one wave); block 0 of each token
// also normalises the cache row.
// Each thread loads a batch of its rotation pairs before it stores any (the
// compiler cannot tell that q and the tables do not overlap, so a loop that
// loads, turns and stores one pair at a time waits out a global-memory round
// trip per pair).
#include <cstdio>

#include "mla_kernels.cuh"

namespace mla {
namespace pro {

constexpr int kThreads = 256;
constexpr int kBatch = 16;   // rotation pairs a thread loads before it stores
constexpr int kMaxLatent = 512;

struct Args {
  int H, N, R, L, ps, num_pages, B, T, max_seq_len, bt_stride;
  double eps;
  __nv_bfloat16* q;                 // [T, H, N+R], rope part turned in place
  __nv_bfloat16* pool;              // [num_pages * ps, L+R], the query tokens' rows rewritten
  const uint32_t* offsets;          // [B+1]
  const uint32_t* cache_lens;       // [B]
  const int32_t* block_table;       // [B, bt_stride]
  const __nv_bfloat16* freqs;       // [max_seq_len, R]
  const __nv_bfloat16* gamma;       // [L]
  PlanHeader* hdr;                  // status word
};

__device__ __forceinline__ double bf(const __nv_bfloat16 v) {
  return (double)__uint_as_float(((uint32_t)__bfloat16_as_ushort(v)) << 16);
}

// Double -> bf16 bits, rounded once to nearest with ties to even (8 significant
// bits), written from the binary formats: a normal bf16 result keeps the top 7
// stored mantissa bits of the double, rounded on the 45 dropped bits; below the
// smallest normal bf16 (2^-126) the quantum is fixed at 2^-133.
__device__ __forceinline__ uint16_t round_bf16(double x) {
  const unsigned long long u = (unsigned long long)__double_as_longlong(x);
  const uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
  const unsigned long long mag = u & 0x7FFFFFFFFFFFFFFFull;
  if (mag > 0x7FF0000000000000ull) return 0x7FC0;                 // NaN
  const int e = (int)(mag >> 52) - 1023;                            // unbiased exponent
  if (mag == 0) return sign;
  if (e < -126) {
    // subnormal bf16 range: k = nearest-even integer of |x| / 2^-133 (exact scaling)
    const double k = rint(fabs(x) * 0x1p133);                       // rint: nearest, ties to even
    return (uint16_t)(sign | (uint16_t)k);                          // k <= 128 lands on the smallest normal
  }
  const unsigned long long half = 1ull << 44, keep = ~((1ull << 45) - 1);
  const unsigned long long lsb = (mag >> 45) & 1ull;
  const unsigned long long r = (mag + half - 1 + lsb) & keep;      // nearest, ties to even
  const int er = (int)(r >> 52) - 1023;
  if (er > 127) return (uint16_t)(sign | 0x7F80u);                   // overflow to infinity
  // r has 8 significant bits and a bf16 exponent: re-bias into the 16-bit format
  const uint32_t bexp = (uint32_t)(er + 127);
  const uint32_t bman = (uint32_t)((r >> 45) & 0x7Fu);
  return (uint16_t)(sign | (bexp << 7) | bman);
}

__device__ __forceinline__ float bff(const __nv_bfloat16 v) {
  return __uint_as_float(((uint32_t)__bfloat16_as_ushort(v)) << 16);
}

// bf16 bits of the exact sum hi + lo, where (hi, lo) is a TwoSum pair (hi = fl(hi + lo),
// |lo| at most half an fp32 ulp of hi): nearest, ties to even.  Only when hi lies
// exactly halfway between two bf16 values does lo decide the direction.
__device__ __forceinline__ uint16_t round_bf16_pair(float hi, float lo) {
  const uint32_t u = __float_as_uint(hi);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;                // NaN
  const uint32_t sign = u & 0x80000000u, mag = u & 0x7FFFFFFFu;
  const uint32_t rem = mag & 0xFFFFu, base = mag >> 16;
  bool up;
  if (rem != 0x8000u) {
    up = rem > 0x8000u;
  } else {
    const float away = sign ? -lo : lo;                                 // lo along hi's direction
    up = away > 0.f || (away == 0.f && (base & 1u));
  }
  return (uint16_t)((sign >> 16) | (base + (up ? 1u : 0u)));
}

// (a + b) as an exact pair: hi = fl(a + b), lo = the rounding error (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float& hi, float& lo) {
  hi = __fadd_rn(a, b);
  const float z = __fsub_rn(hi, a);
  lo = __fadd_rn(__fsub_rn(a, __fsub_rn(hi, z)), __fsub_rn(b, z));
}

// bf16 pair (low half first) as two floats.
__device__ __forceinline__ void bf2(uint32_t v, float& lo, float& hi) {
  lo = __uint_as_float(v << 16);
  hi = __uint_as_float(v & 0xFFFF0000u);
}

// (x0, x1) turned by (c, s), as bf16 bits: the products of bf16 values are
// exact in fp32.
__device__ __forceinline__ void rotate(float x0, float x1, float c, float s, uint16_t& y0, uint16_t& y1) {
  float h0, l0, h1, l1;
  two_sum(__fmul_rn(x0, c), -__fmul_rn(x1, s), h0, l0);
  two_sum(__fmul_rn(x0, s), __fmul_rn(x1, c), h1, l1);
  y0 = round_bf16_pair(h0, l0);
  y1 = round_bf16_pair(h1, l1);
}

__global__ void __launch_bounds__(kThreads) prologue_kernel(const Args a) {
  __shared__ double s_inv;
  __shared__ double s_part[kThreads / 32];
  __shared__ long long s_req[4];   // b, first token, end token, cache length of the token's request
  const int t = blockIdx.x, tid = threadIdx.x;
  const bool row_block = blockIdx.y == 0;   // this block also normalises the cache row
  // gamma does not depend on anything: its loads go out first
  constexpr int kLatPerThread = kMaxLatent / kThreads;
  double g[kLatPerThread];
#pragma unroll
  for (int j = 0; j < kLatPerThread; ++j) {
    const int l = tid + j * kThreads;
    g[j] = row_block && l < a.L ? bf(a.gamma[l]) : 0.0;
  }
  // this block's heads [h0, h1) of the query's rope part: pair i = (head h0 + i / (R/2),
  // pair i % (R/2)), at an even element offset (4-byte aligned, checked by the entry point)
  const int half = a.R / 2;
  const int h0 = (int)((long long)blockIdx.y * a.H / gridDim.y), h1 = (int)((long long)(blockIdx.y + 1) * a.H / gridDim.y);
  const int npairs = (h1 - h0) * half;
  auto qpair = [&](int i) {
    return reinterpret_cast<uint32_t*>(a.q + ((size_t)t * a.H + h0 + i / half) * (a.N + a.R) + a.N + 2 * (i % half));
  };
  // the first batch of pairs needs no request: its loads go out before the lookup
  uint32_t xw[kBatch];
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    const int i = tid + j * kThreads;
    xw[j] = i < npairs ? *qpair(i) : 0u;
  }
  // the token's request: the b with offsets[b] <= t < offsets[b + 1], found by every
  // thread testing its own b (one round trip instead of a search's log2(B))
  if (tid == 0) s_req[0] = -1;
  __syncthreads();
  for (int b0 = 0; b0 < a.B; b0 += kThreads) {
    const int b = b0 + tid;
    if (b < a.B) {
      const long long qb = a.offsets[b], qe = a.offsets[b + 1];
      const long long len = a.cache_lens[b];
      if (qb <= t && t < qe) {
        s_req[0] = b;
        s_req[1] = qb;
        s_req[2] = qe;
        s_req[3] = len;
      }
    }
  }
  __syncthreads();
  const long long bq = s_req[0];
  bool ok = bq >= 0;
  const int b = ok ? (int)bq : 0;
  const long long qb = s_req[1], qe = s_req[2];
  const long long pos = ok ? s_req[3] - (qe - qb) + (t - qb) : -1;
  ok = ok && pos >= 0 && pos < a.max_seq_len && pos < (long long)a.bt_stride * a.ps;
  if (!ok) {   // skipped whole, as the decode would drop a bad page; reported
    if (tid == 0) atomicOr(&a.hdr->status, kDeviceCheckFailed);
    return;
  }
  // the page of the row (needed for the row's loads) and the rotation table go out
  // together; a bad page skips the token whole, before anything is written
  const int page = a.block_table[(size_t)b * a.bt_stride + pos / a.ps];
  const __nv_bfloat16* f = a.freqs + (size_t)pos * a.R;
  bool page_checked = false;
  for (int i0 = tid; i0 < npairs || !page_checked; i0 += kThreads * kBatch) {
    float x0[kBatch], x1[kBatch], c[kBatch], sn[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * kThreads;
      if (i < npairs) {
        bf2(i0 == tid ? xw[j] : *qpair(i), x0[j], x1[j]);
        bf2(*reinterpret_cast<const uint32_t*>(f + 2 * (i % half)), c[j], sn[j]);
      }
    }
    if (!page_checked) {
      if (page < 0 || page >= a.num_pages) {
        if (tid == 0) atomicOr(&a.hdr->status, kDeviceCheckFailed);
        return;
      }
      page_checked = true;
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = i0 + j * kThreads;
      if (i < npairs) {
        uint16_t y0, y1;
        rotate(x0[j], x1[j], c[j], sn[j], y0, y1);
        *qpair(i) = (uint32_t)y0 | ((uint32_t)y1 << 16);
      }
    }
  }
  if (!row_block) return;
  // the row: latent values and its rope pair read together; mean square summed by a tree
  __nv_bfloat16* rp = a.pool + ((size_t)page * a.ps + pos % a.ps) * (a.L + a.R);
  double v[kLatPerThread];
#pragma unroll
  for (int j = 0; j < kLatPerThread; ++j) {
    const int l = tid + j * kThreads;
    v[j] = l < a.L ? bf(rp[l]) : 0.0;
  }
  float r0 = 0.f, r1 = 0.f, rc = 0.f, rs = 0.f;
  if (tid < half) {
    r0 = bff(rp[a.L + 2 * tid]);
    r1 = bff(rp[a.L + 2 * tid + 1]);
    rc = bff(f[2 * tid]);
    rs = bff(f[2 * tid + 1]);
  }
  double part = 0.0;
#pragma unroll
  for (int j = 0; j < kLatPerThread; ++j) part = __dadd_rn(part, __dmul_rn(v[j], v[j]));
  for (int o = 16; o > 0; o >>= 1) part = __dadd_rn(part, __shfl_xor_sync(0xffffffffu, part, o));
  if ((tid & 31) == 0) s_part[tid >> 5] = part;
  __syncthreads();
  if (tid == 0) {
    double ms = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) ms = __dadd_rn(ms, s_part[w]);
    // mean: a multiply when L is a power of two (exact), else a division
    const double mean = (a.L & (a.L - 1)) == 0 ? __dmul_rn(ms, 1.0 / (double)a.L) : __ddiv_rn(ms, (double)a.L);
    s_inv = rsqrt(__dadd_rn(mean, a.eps));
  }
  __syncthreads();
  const double inv = s_inv;
#pragma unroll
  for (int j = 0; j < kLatPerThread; ++j) {
    const int l = tid + j * kThreads;
    if (l < a.L) rp[l] = __ushort_as_bfloat16(round_bf16(__dmul_rn(__dmul_rn(v[j], inv), g[j])));
  }
  if (tid < half) {
    uint16_t y0, y1;
    rotate(r0, r1, rc, rs, y0, y1);
    rp[a.L + 2 * tid] = __ushort_as_bfloat16(y0);
    rp[a.L + 2 * tid + 1] = __ushort_as_bfloat16(y1);
  }
  for (int pr = tid + kThreads; pr < half; pr += kThreads) {   // rope wider than 2 x threads
    uint16_t y0, y1;
    rotate(bff(rp[a.L + 2 * pr]), bff(rp[a.L + 2 * pr + 1]), bff(f[2 * pr]), bff(f[2 * pr + 1]), y0, y1);
    rp[a.L + 2 * pr] = __ushort_as_bfloat16(y0);
    rp[a.L + 2 * pr + 1] = __ushort_as_bfloat16(y1);
  }
}

}  // namespace pro

cudaError_t launch_prologue(const mla_dims_t& d, void* q, const uint32_t* offsets, int B, int T, void* kv_pool,
                            const int32_t* block_table, int bt_stride, const uint32_t* cache_lens,
                            const void* freqs, int max_seq_len, const void* gamma, float eps, PlanHeader* hdr,
                            cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  pro::Args a{};
  a.H = d.num_heads;
  a.N = d.qk_nope;
  a.R = d.qk_rope;
  a.L = d.kv_lora_rank;
  a.ps = d.page_size;
  a.num_pages = d.num_pages;
  a.B = B;
  a.T = T;
  a.max_seq_len = max_seq_len;
  a.bt_stride = bt_stride;
  a.eps = (double)eps;
  a.q = static_cast<__nv_bfloat16*>(q);
  a.pool = static_cast<__nv_bfloat16*>(kv_pool);
  a.offsets = offsets;
  a.cache_lens = cache_lens;
  a.block_table = block_table;
  a.freqs = static_cast<const __nv_bfloat16*>(freqs);
  a.gamma = static_cast<const __nv_bfloat16*>(gamma);
  a.hdr = hdr;
  // blocks per token: the grid fills the SMs' resident slots, at least one head each
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  // two blocks per SM are resident (registers): a single wave of at most 2 x SMs blocks
  int G = (2 * sms) / T;
  if (G > a.H) G = a.H;
  if (G > 65535) G = 65535;
  if (G < 1) G = 1;
  pro::prologue_kernel<<<dim3(T, G), pro::kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
