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
// Every value is computed in double precision from the bf16 inputs, with each
// product and sum rounded on its own (no fused multiply-add) in the order
// written above, and rounded once to bf16 (nearest, ties to even).  The mean
// square is summed in latent order by one thread.  So the results do not depend
// on the launch shape, and they are the exactly rounded values of those
// expressions.
//
// One block per query token: its threads share the token's heads and the row.
#include <cstdio>

#include "mla_kernels.cuh"

namespace mla {
namespace pro {

constexpr int kThreads = 128;
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

__device__ __forceinline__ void rotate(__nv_bfloat16* x, const __nv_bfloat16* f) {
  const double x0 = bf(x[0]), x1 = bf(x[1]), c = bf(f[0]), s = bf(f[1]);
  const uint16_t y0 = round_bf16(__dsub_rn(__dmul_rn(x0, c), __dmul_rn(x1, s)));
  const uint16_t y1 = round_bf16(__dadd_rn(__dmul_rn(x0, s), __dmul_rn(x1, c)));
  x[0] = __ushort_as_bfloat16(y0);
  x[1] = __ushort_as_bfloat16(y1);
}

__global__ void __launch_bounds__(kThreads) prologue_kernel(const Args a) {
  __shared__ double s_inv;
  __shared__ double s_lat[kMaxLatent];
  const int t = blockIdx.x, tid = threadIdx.x;
  // request of token t: the last b with offsets[b] <= t
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int)a.offsets[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const long long qb = a.offsets[b], qe = a.offsets[b + 1];
  const long long pos = (long long)a.cache_lens[b] - (qe - qb) + (t - qb);
  bool ok = qb <= t && t < qe && pos >= 0 && pos < a.max_seq_len && pos < (long long)a.bt_stride * a.ps;
  long long row = 0;
  if (ok) {
    const int page = a.block_table[(size_t)b * a.bt_stride + pos / a.ps];
    ok = page >= 0 && page < a.num_pages;
    row = (long long)page * a.ps + pos % a.ps;
  }
  if (!ok) {   // skipped whole, as the decode would drop a bad page; reported
    if (tid == 0) atomicOr(&a.hdr->status, kDeviceCheckFailed);
    return;
  }
  const __nv_bfloat16* f = a.freqs + (size_t)pos * a.R;
  // the query's rope part, every head
  for (int i = tid; i < a.H * (a.R / 2); i += kThreads) {
    const int h = i / (a.R / 2), pr = i % (a.R / 2);
    rotate(a.q + ((size_t)t * a.H + h) * (a.N + a.R) + a.N + 2 * pr, f + 2 * pr);
  }
  // the row: latent values into shared memory, mean square summed in order by one thread
  __nv_bfloat16* rp = a.pool + (size_t)row * (a.L + a.R);
  for (int l = tid; l < a.L; l += kThreads) s_lat[l] = bf(rp[l]);
  __syncthreads();
  if (tid == 0) {
    double ms = 0.0;
    for (int l = 0; l < a.L; ++l) ms = __dadd_rn(ms, __dmul_rn(s_lat[l], s_lat[l]));
    s_inv = __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(__ddiv_rn(ms, (double)a.L), a.eps)));
  }
  __syncthreads();
  const double inv = s_inv;
  for (int l = tid; l < a.L; l += kThreads)
    rp[l] = __ushort_as_bfloat16(round_bf16(__dmul_rn(__dmul_rn(s_lat[l], inv), bf(a.gamma[l]))));
  for (int pr = tid; pr < a.R / 2; pr += kThreads) rotate(rp + a.L + 2 * pr, f + 2 * pr);
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
  pro::prologue_kernel<<<T, pro::kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
