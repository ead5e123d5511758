// The FP8 indexer of the mla_indexer_ragged_float8_paged page (description: an
// FP8 product of the query with the key cache, with the query scales q_s and the
// key scales at head-size granularity, summed across heads, masked, top-k;
// Args output_indices, filled with -1 where a token has fewer keys than top_k).
// It produces the physical row lists that the sparse decode consumes.
//
// For query token t of request b, every key j of the decode's key set (causal,
// null or sliding-window over cache_lens[b], through the block table) scores
//
//   s_j = sum_h ( q_s[t,h] * k_scale[row_j] ) * ( sum_d q[t,h,d] * k[row_j,d] )
//
// and the top_k rows are returned by descending score, equal scores by
// ascending key position, NaN scores last.
//
// The result is exactly defined: an e4m3 value is a signed integer significand
// times a power of two (a multiple of 2^-9), so every product is a multiple of
// 2^-18 below 2^18 and the inner sum over d is computed exactly as a 64-bit
// integer in units of 2^-18; the head sum is then evaluated in double precision
// term by term in head order, each product and sum rounded on its own.  The
// ranking therefore does not depend on the launch shape or on accumulation
// order, and ties are broken by position, not by placement.
//
// Two kernels: scores (one block per token and 32 keys; the keys' sort keys go
// to the workspace) and selection (one block per token: radix select of the
// top_k smallest sort keys over eight 8-bit digits, then a bitonic sort of the
// chosen ones by (sort key, position)).
#include <math_constants.h>

#include <cstdio>

#include "mla_kernels.cuh"

namespace mla {
namespace idx {

constexpr int kKeysPerBlock = 32;
constexpr int kMaxIndexHeads = 128;   // heads per call (checked by the entry point)
constexpr size_t kSelectKeySmem = 160 * 1024;   // the select kernel stages up to this many key bytes
// Byte offset of the staged keys after the sort buffers (16-byte aligned).
__host__ __device__ inline size_t select_keys_offset(int sort_n) { return ((size_t)sort_n * 12 + 15) & ~(size_t)15; }

// Row pitch (ints) of the staged query and key values: D rounded up to a multiple
// of 4 (16-byte loads, rows 16-byte aligned), plus 4 more when that is a multiple
// of 8 ints (so eight consecutive rows start in eight different bank groups).
__host__ __device__ inline int padded_dims(int D) {
  const int c4 = (D + 3) / 4;
  return 4 * (c4 % 2 == 0 ? c4 + 1 : c4);
}
// Byte offset of the dot-product block after the staged values and NaN flags.
__host__ __device__ inline size_t dots_offset(int H, int D) {
  return ((((size_t)H + kKeysPerBlock) * padded_dims(D) * 4 + H + kKeysPerBlock + 15) & ~(size_t)15);
}
constexpr int kScoreThreads = 256;
constexpr int kSelectThreads = 1024;
constexpr unsigned long long kInvalidKey = ~0ull;        // a key whose page id is out of range
constexpr unsigned long long kNaNKey = ~0ull - 1ull;     // NaN scores sort after every number

struct Args {
  int H, D, ps, num_pages, B, T, mask, window, top_k, bt_stride, max_keys;
  const uint8_t* q;              // e4m3 [T, H, D]
  const float* q_s;              // [T, H]
  const uint32_t* offsets;       // [B+1]
  const uint8_t* k;              // e4m3 [num_pages * ps, D]
  const float* k_scales;         // [num_pages * ps]
  const int32_t* block_table;    // [B, bt_stride]
  const uint32_t* cache_lens;    // [B]
  unsigned long long* keys;      // workspace [T, max_keys]
  bool keys_in_smem;             // select: the launch gave room to stage max_keys keys
  int32_t* out_rows;             // [T, top_k]
  double* out_scores;            // [T, top_k] or NULL
  PlanHeader* hdr;
};

// Key range [lo, hi) of token t (positions) and its request, as the decode's mask defines it.
__device__ __forceinline__ bool token_range(const Args& a, int t, int& b, int& lo, int& hi) {
  int l = 0, r = a.B - 1;
  while (l < r) {
    const int mid = (l + r + 1) >> 1;
    if ((int)a.offsets[mid] <= t) l = mid; else r = mid - 1;
  }
  b = l;
  const int qb = (int)a.offsets[b], qe = (int)a.offsets[b + 1];
  const int len = (int)a.cache_lens[b];
  const int pos = len - (qe - qb) + (t - qb);
  lo = 0;
  hi = 0;
  if (!(qb <= t && t < qe) || pos < 0 || len > a.bt_stride * a.ps) return false;
  if (a.mask == MLA_MASK_NULL) {
    hi = len;
  } else {
    hi = pos + 1;
    if (a.mask == MLA_MASK_SLIDING_WINDOW_CAUSAL) lo = max(0, hi - a.window);
  }
  if (hi - lo > a.max_keys) return false;
  return true;
}

// e4m3 (OCP E4M3FN) code -> its value times 2^9, an integer: sig * 2^sh with the signed
// significand sig (|sig| <= 15) and sh in 0..14, so |value * 2^9| < 2^18.
__device__ __forceinline__ int e4m3_times_512(uint32_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  const int mag = (e ? (8 | m) : m) << (e ? e - 1 : 0);
  return (c & 0x80u) ? -mag : mag;
}
__device__ __forceinline__ bool e4m3_is_nan(uint32_t c) { return (c & 0x7Fu) == 0x7Fu; }

// Double -> 64-bit key whose unsigned order is descending score (NaN after every number).
__device__ __forceinline__ unsigned long long sort_key(double s) {
  if (s != s) return kNaNKey;
  if (s == 0.0) s = 0.0;   // one key for +0 and -0, which compare equal
  unsigned long long u = (unsigned long long)__double_as_longlong(s);
  u = (u >> 63) ? ~u : (u | (1ull << 63));   // ascending in s
  return ~u;                                  // descending in s
}
__device__ __forceinline__ double key_score(unsigned long long key) {
  if (key == kNaNKey) return __longlong_as_double(0x7FF8000000000000ll);
  unsigned long long u = ~key;
  u = (u >> 63) ? (u & ~(1ull << 63)) : ~u;
  return __longlong_as_double((long long)u);
}

__global__ void __launch_bounds__(kScoreThreads) scores_kernel(const Args a) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int t = blockIdx.x, j0 = blockIdx.y * kKeysPerBlock, tid = threadIdx.x;
  int b, lo, hi;
  if (!token_range(a, t, b, lo, hi)) {
    if (blockIdx.y == 0 && tid == 0) atomicOr(&a.hdr->status, kDeviceCheckFailed);
    return;
  }
  const int n = hi - lo;
  if (j0 >= n) return;
  const int nk = min(kKeysPerBlock, n - j0);
  const int HD = a.H * a.D;
  const int DP = padded_dims(a.D);                         // row pitch in ints (see padded_dims)
  int* qv = reinterpret_cast<int*>(sm);                    // [H][DP] query values x 2^9
  int* kv = qv + a.H * DP;                                 // [32][DP] key values x 2^9
  uint8_t* qnan = reinterpret_cast<uint8_t*>(kv + kKeysPerBlock * DP);   // [H]
  uint8_t* knan = qnan + a.H;                                            // [32]
  long long* dots = reinterpret_cast<long long*>(sm + dots_offset(a.H, a.D));
  __shared__ long long rows_s[kKeysPerBlock];
  __shared__ double ksc_s[kKeysPerBlock];   // the keys' row scales
  __shared__ double qs18[kMaxIndexHeads];   // q_s[h] x 2^-18, exact: the dots' unit folded in
  __shared__ int bad_s;
  if (tid == 0) bad_s = 0;
  for (int i = tid; i < a.H; i += kScoreThreads) {
    qnan[i] = 0;
    qs18[i] = __dmul_rn((double)a.q_s[(size_t)t * a.H + i], 0x1p-18);
  }
  // padding columns [D, DP) of every row hold zeros (the inner loop reads 4 at a time)
  for (int i = tid; i < (a.H + kKeysPerBlock) * (DP - a.D); i += kScoreThreads)
    qv[(i / (DP - a.D)) * DP + a.D + i % (DP - a.D)] = 0;
  if (tid < kKeysPerBlock) knan[tid] = 0;
  __syncthreads();
  // a warp per head, a lane per dimension (no division per element)
  const int wid = tid >> 5, lane = tid & 31;
  for (int h = wid; h < a.H; h += kScoreThreads / 32)
    for (int d = lane; d < a.D; d += 32) {
      const uint32_t c = a.q[(size_t)t * HD + h * a.D + d];
      qv[h * DP + d] = e4m3_times_512(c);
      if (e4m3_is_nan(c)) qnan[h] = 1;
    }
  if (tid < nk) {
    const int j = lo + j0 + tid;
    const int page = a.block_table[(size_t)b * a.bt_stride + j / a.ps];
    long long row = -1;
    if (page >= 0 && page < a.num_pages) row = (long long)page * a.ps + j % a.ps;
    else bad_s = 1;
    rows_s[tid] = row;
    ksc_s[tid] = row >= 0 ? (double)a.k_scales[row] : 0.0;
  }
  __syncthreads();
  // a warp per key, a lane per dimension
  for (int key = wid; key < kKeysPerBlock; key += kScoreThreads / 32) {
    const long long row = key < nk ? rows_s[key] : -1;
    for (int d = lane; d < a.D; d += 32) {
      const uint32_t c = row >= 0 ? a.k[(size_t)row * a.D + d] : 0u;
      kv[key * DP + d] = e4m3_times_512(c);
      if (key < nk && e4m3_is_nan(c)) knan[key] = 1;
    }
  }
  __syncthreads();
  // exact inner products in units of 2^-18 (each product below 2^36, sums in 64 bits):
  // thread (kq, hq) holds keys kq and kq + 16 and heads hq, hq + 16, ... (a 2 x H/16 block)
  {
    const int kq = tid & 15, hq = tid >> 4;
    const int nh = (a.H - hq + 15) / 16;                   // heads of this thread (<= 8)
    long long acc[2][8];
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) acc[x][y] = 0;
    const int* k0 = kv + kq * DP;
    const int* k1 = kv + (kq + 16) * DP;
    // four dimensions per step (16-byte loads; rows 16-byte aligned, zero-padded);
    // 32 x 32 -> 64-bit products, exact, summed in 64 bits
    for (int d = 0; d < a.D; d += 4) {
      const int4 x0 = *reinterpret_cast<const int4*>(k0 + d);
      const int4 x1 = *reinterpret_cast<const int4*>(k1 + d);
#pragma unroll
      for (int y = 0; y < 8; ++y) {
        if (y < nh) {
          const int4 qy = *reinterpret_cast<const int4*>(qv + (hq + 16 * y) * DP + d);
          acc[0][y] += (long long)x0.x * qy.x + (long long)x0.y * qy.y + (long long)x0.z * qy.z +
                       (long long)x0.w * qy.w;
          acc[1][y] += (long long)x1.x * qy.x + (long long)x1.y * qy.y + (long long)x1.z * qy.z +
                       (long long)x1.w * qy.w;
        }
      }
    }
    // each term of the head sum, (q_s 2^-18 ksc) dot, rounded once (both factors
    // exact), by the thread that holds the dot; the sum itself runs in head order below.
    // Rows of H + 1 doubles: the adding warp's 32 lanes (one key each) read 32 banks.
    double* terms = reinterpret_cast<double*>(dots);
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      if (y < nh) {
        const int h = hq + 16 * y;
        terms[kq * (a.H + 1) + h] = __dmul_rn(__dmul_rn(qs18[h], ksc_s[kq]), (double)acc[0][y]);
        terms[(kq + 16) * (a.H + 1) + h] = __dmul_rn(__dmul_rn(qs18[h], ksc_s[kq + 16]), (double)acc[1][y]);
      }
    }
  }
  __syncthreads();
  // head sum in head order, each product and sum rounded on its own
  if (tid < nk) {
    const long long row = rows_s[tid];
    unsigned long long key;
    if (row < 0) {
      key = kInvalidKey;
    } else {
      // (q_s ksc) (dot 2^-18) was formed as (q_s 2^-18 ksc) dot: both factors exact
      // either way, so the one rounded product is the same double
      const double* terms = reinterpret_cast<const double*>(dots);
      double s = 0.0;
      bool nan = knan[tid] != 0;
      for (int h = 0; h < a.H; ++h) {
        s = __dadd_rn(s, terms[tid * (a.H + 1) + h]);
        nan = nan || qnan[h];
      }
      if (nan) s = __longlong_as_double(0x7FF8000000000000ll);
      key = sort_key(s);
    }
    a.keys[(size_t)t * a.max_keys + j0 + tid] = key;
  }
  if (tid == 0 && bad_s) atomicOr(&a.hdr->status, kDeviceCheckFailed);
}

__global__ void __launch_bounds__(kSelectThreads) select_kernel(const Args a, int sort_n) {
  extern __shared__ __align__(16) uint8_t sm[];
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(sm);   // [sort_n] candidate keys
  int* cj = reinterpret_cast<int*>(ck + sort_n);                          // [sort_n] their positions
  // the token's keys, staged once when the launch gave room for max_keys of them
  unsigned long long* ks = reinterpret_cast<unsigned long long*>(sm + select_keys_offset(sort_n));
  __shared__ unsigned int hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_need, s_count, s_eq_base[kSelectThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x, K = a.top_k;
  int b, lo, hi;
  const bool ok = token_range(a, t, b, lo, hi);
  const int n = ok ? hi - lo : 0;
  const unsigned long long* keys = a.keys + (size_t)t * a.max_keys;
  if (a.keys_in_smem) {
    for (int i = tid; i < n; i += kSelectThreads) ks[i] = keys[i];
    __syncthreads();
    keys = ks;
  }
  unsigned long long tau = kInvalidKey;
  int need = n;   // keys equal to tau to take (all keys when n <= K)
  if (n > K) {
    // radix select of the K smallest keys, 8 bits at a time from the top
    unsigned long long prefix = 0;
    int kk = K;
    for (int digit = 7; digit >= 0; --digit) {
      const int shift = 8 * digit;
      for (int i = tid; i < 256; i += kSelectThreads) hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < n; i += kSelectThreads) {
        const unsigned long long key = keys[i];
        const bool match = digit == 7 || (key >> (shift + 8)) == (prefix >> (shift + 8));
        if (match) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      // the first bin whose running count reaches kk (bin 255 if none does): warp 0,
      // eight bins per lane, a warp scan of the lanes' sums, then the crossing lane
      if (tid < 32) {
        unsigned int h[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          h[j] = hist[8 * tid + j];
          sum += h[j];
        }
        unsigned int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += v;
        }
        const unsigned int hit = __ballot_sync(0xffffffffu, incl >= (unsigned int)kk);
        const int L = hit ? __ffs(hit) - 1 : 31;
        if (tid == L) {
          unsigned int cum = incl - sum;
          int bin = 8 * L;
          bool done = false;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (!done) {
              if (bin == 255 || cum + h[j] >= (unsigned int)kk) {
                done = true;
              } else {
                cum += h[j];
                ++bin;
              }
            }
          }
          s_prefix = prefix | ((unsigned long long)bin << shift);
          s_need = kk - (int)cum;
        }
      }
      __syncthreads();
      prefix = s_prefix;
      kk = s_need;
      __syncthreads();
    }
    tau = prefix;
    need = kk;
  }
  // collect: every key below tau, and the first `need` keys equal to tau by position
  if (tid == 0) s_count = 0;
  __syncthreads();
  const int chunk = (n + kSelectThreads - 1) / kSelectThreads;
  const int c0 = min(n, tid * chunk), c1 = min(n, c0 + chunk);
  int my_eq = 0;
  if (n > K)
    for (int i = c0; i < c1; ++i) my_eq += keys[i] == tau;
  // exclusive scan of my_eq over threads (positions are in thread order)
  const int lane = tid & 31, wid = tid >> 5;
  int incl = my_eq;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_eq_base[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = lane < kSelectThreads / 32 ? s_eq_base[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    s_eq_base[lane] = v;
  }
  __syncthreads();
  int eq_rank = (wid > 0 ? s_eq_base[wid - 1] : 0) + incl - my_eq;
  for (int i = c0; i < c1; ++i) {
    const unsigned long long key = keys[i];
    bool take;
    if (n <= K) take = true;
    else if (key < tau) take = true;
    else if (key == tau) take = eq_rank++ < need;
    else take = false;
    if (take) {
      const int slot = atomicAdd(&s_count, 1);
      ck[slot] = key;
      cj[slot] = i;
    }
  }
  __syncthreads();
  const int count = s_count;   // min(n, K)
  for (int i = count + tid; i < sort_n; i += kSelectThreads) {
    ck[i] = kInvalidKey;
    cj[i] = 0x7FFFFFFF;
  }
  __syncthreads();
  // bitonic sort of (key, position) ascending
  for (int size = 2; size <= sort_n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < sort_n; i += kSelectThreads) {
        const int pr = i ^ stride;
        if (pr > i) {
          const bool up = (i & size) == 0;
          const unsigned long long ki = ck[i], kp = ck[pr];
          const int ji = cj[i], jp = cj[pr];
          const bool gt = ki > kp || (ki == kp && ji > jp);
          if (gt == up) {
            ck[i] = kp;
            ck[pr] = ki;
            cj[i] = jp;
            cj[pr] = ji;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < K; i += kSelectThreads) {
    int32_t row = -1;
    double sc = -CUDART_INF;
    if (i < count && ck[i] != kInvalidKey) {
      const int j = lo + cj[i];
      const int page = a.block_table[(size_t)b * a.bt_stride + j / a.ps];
      row = page * a.ps + j % a.ps;
      sc = key_score(ck[i]);
    }
    a.out_rows[(size_t)t * K + i] = row;
    if (a.out_scores) a.out_scores[(size_t)t * K + i] = sc;
  }
}

}  // namespace idx

size_t indexer_workspace_bytes(int T, int max_keys) {
  return 256 + (size_t)(T > 0 ? T : 1) * (size_t)(max_keys > 0 ? max_keys : 1) * 8;
}

size_t indexer_scores_smem(int H, int D) {
  return idx::dots_offset(H, D) + (size_t)idx::kKeysPerBlock * (H + 1) * 8;
}

cudaError_t launch_indexer(int H, int D, int ps, int num_pages, int B, int T, int mask, int window, int top_k,
                           const uint8_t* q, const float* q_s, const uint32_t* offsets, const uint8_t* k,
                           const float* k_scales, const int32_t* block_table, int bt_stride,
                           const uint32_t* cache_lens, int max_keys, void* workspace, int32_t* out_rows,
                           double* out_scores, cudaStream_t s) {
  idx::Args a{};
  a.H = H;
  a.D = D;
  a.ps = ps;
  a.num_pages = num_pages;
  a.B = B;
  a.T = T;
  a.mask = mask;
  a.window = window;
  a.top_k = top_k;
  a.bt_stride = bt_stride;
  a.max_keys = max_keys;
  a.q = q;
  a.q_s = q_s;
  a.offsets = offsets;
  a.k = k;
  a.k_scales = k_scales;
  a.block_table = block_table;
  a.cache_lens = cache_lens;
  a.hdr = static_cast<PlanHeader*>(workspace);
  a.keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + 256);
  a.out_rows = out_rows;
  a.out_scores = out_scores;
  if (T == 0) return cudaSuccess;
  const size_t s1 = indexer_scores_smem(H, D);
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(idx::scores_kernel), (int)s1);
  if (e != cudaSuccess) return e;
  dim3 g1(T, (max_keys + idx::kKeysPerBlock - 1) / idx::kKeysPerBlock);
  idx::scores_kernel<<<g1, idx::kScoreThreads, s1, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  int sort_n = 1;
  while (sort_n < top_k) sort_n <<= 1;
  a.keys_in_smem = (size_t)max_keys * 8 <= idx::kSelectKeySmem;
  const size_t s2 = idx::select_keys_offset(sort_n) + (a.keys_in_smem ? (size_t)max_keys * 8 : 0);
  e = ensure_smem_limit(reinterpret_cast<const void*>(idx::select_kernel), (int)s2);
  if (e != cudaSuccess) return e;
  idx::select_kernel<<<T, idx::kSelectThreads, s2, s>>>(a, sort_n);   // a.keys_in_smem set above
  return cudaGetLastError();
}

}  // namespace mla
