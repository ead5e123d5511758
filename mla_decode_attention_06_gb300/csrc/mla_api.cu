// C ABI of libmla_decode.so: argument checks, workspace carving and the launch
// sequence  K1 W_uk absorb (+ plan) -> K2 split-KV decode (+ split merge) -> K3 W_uv.
// Nothing here allocates or synchronises unless MLA_FLAG_DEBUG_CHECKS is set.
#include <cstdio>
#include <cstring>
#include <new>

#include "mla_kernels.cuh"
#include "mla_plan.cuh"

using namespace mla;

namespace {

constexpr int kMaxSplits = 1 << 16;
constexpr int kTimedKernels = 3;
constexpr int kMaxDevices = 64;

// Event sets of the timed calls made since the last read, per device
// (created on first use, reused afterwards).
constexpr int kMaxTimedCalls = 4096;
struct EventSet {
  cudaEvent_t ev[kTimedKernels + 1];
};
struct KernelTimer {
  EventSet* sets = nullptr;
  int created = 0;
  int used = 0;      // calls recorded since the last read (saturates at kMaxTimedCalls)
  int next = 0;      // ring position
};
KernelTimer g_timer[kMaxDevices];

EventSet* next_event_set() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  KernelTimer& t = g_timer[dev];
  if (!t.sets) {
    t.sets = new (std::nothrow) EventSet[kMaxTimedCalls];
    if (!t.sets) return nullptr;
  }
  const int slot = t.next;
  if (slot >= t.created) {
    for (auto& e : t.sets[slot].ev)
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    t.created = slot + 1;
  }
  t.next = (slot + 1) % kMaxTimedCalls;
  if (t.used < kMaxTimedCalls) ++t.used;
  return &t.sets[slot];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const mla_dims_t* d) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (d->num_heads < 1 || d->qk_nope < 1 || d->qk_rope < 0 || d->kv_lora_rank < 1 || d->v_head < 1 ||
      d->page_size < 1 || d->num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (d->num_heads > kMaxHeads) return MLA_ERR_UNSUPPORTED;
  // L multiple of 16 (latent columns are split 16 per lane group), L <= 512;
  // even row widths keep every row 4-byte aligned.
  if (d->kv_lora_rank % 16 != 0 || d->kv_lora_rank > 512 || d->qk_rope % 2 != 0 || d->qk_nope % 2 != 0)
    return MLA_ERR_UNSUPPORTED;
  if ((int64_t)d->num_pages * d->page_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (!decode_tc_supported(*d)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

// Query tokens are walked in pairs (two consecutive tokens of a request share
// every cache tile they read, one tile load serving both) when the batch has at
// least two tokens per request on average, the shape has a folded instance, and
// either the caller asks for pairs or, by default, the call is sparse (its
// gathered loads bound the main loop; a dense call's tile period is set by the
// score contraction, which pairs do not shrink).
bool use_fold(const mla_dims_t* d, const mla_opts_t* o, int batch, int total_q, bool fp8_cache, bool sparse) {
  if (total_q < 2 * batch || !decode_fold_supported(*d, fp8_cache)) return false;
  if (o->flags & MLA_FLAG_FOLD_PAIRS) return true;
  if (o->flags & MLA_FLAG_PER_TOKEN) return false;
  return sparse;
}

// The partition count: the caller's, else as many partitions as the device runs at
// once for the instance the call uses (`d` given), or, for sizing the workspace, the
// SM count over the CTAs per partition, which is never below that.
int resolve_splits(const mla_opts_t* o, bool fold, int* K, const mla_dims_t* d = nullptr, bool fp8 = false,
                   bool sparse = false) {
  if (o->num_splits < 0 || o->num_splits > kMaxSplits) return MLA_ERR_INVALID_ARG;
  if (o->num_splits > 0) {
    *K = o->num_splits;
    return MLA_OK;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
  const int per = fold ? 4 : 2;   // CTAs per partition (one for narrow latents, which stay at sms / 2)
  const int bound = sms / per > 0 ? sms / per : 1;
  int n = d ? decode_default_partitions(*d, fold, fp8, sparse) : 0;
  *K = n > 0 && n <= bound ? n : bound;
  return MLA_OK;
}

int check_opts(const mla_opts_t* o) {
  if (!o) return MLA_ERR_INVALID_ARG;
  if (o->mask < MLA_MASK_NULL || o->mask > MLA_MASK_SLIDING_WINDOW_CAUSAL) return MLA_ERR_INVALID_ARG;
  if (o->mask == MLA_MASK_SLIDING_WINDOW_CAUSAL && o->window < 1) return MLA_ERR_INVALID_ARG;
  if (!(o->scale == o->scale)) return MLA_ERR_INVALID_ARG;   // NaN
  if (o->flags & ~(MLA_FLAG_DEBUG_CHECKS | MLA_FLAG_KERNEL_TIMING | MLA_FLAG_FOLD_PAIRS | MLA_FLAG_PER_TOKEN))
    return MLA_ERR_INVALID_ARG;
  if ((o->flags & MLA_FLAG_FOLD_PAIRS) && (o->flags & MLA_FLAG_PER_TOKEN)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

// Debug path: waits for the stream, then turns the status word the kernels wrote
// into the header into a status code (time-outs first, with where they happened).
int device_status(const PlanHeader* hdr, cudaStream_t stream) {
  int st_words[4] = {0, 0, 0, 0};   // status, unused, time-out record (code, block)
  if (cudaMemcpyAsync(st_words, &hdr->status, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemcpyAsync(st_words + 2, &hdr->pad[0], 2 * sizeof(int), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return MLA_ERR_CUDA;
  const int status = st_words[0];
  if (status & kDeviceTimeout) {
    std::fprintf(stderr, "mla_decode: device wait timed out (barrier smem offset 0x%x, thread %d, block %d)\n",
                 st_words[2] & 0x3FFFF, (st_words[2] >> 18) & 0x1FFF, st_words[3]);
    return MLA_ERR_TIMEOUT;
  }
  if (status & kDeviceCheckFailed) return MLA_ERR_DEVICE_CHECK;
  return MLA_OK;
}

struct CallCommon {
  const mla_dims_t* d;
  const mla_opts_t* o;
  const void* q;
  const uint32_t* offsets;
  int B, T;
  KeySource ks;
  KVFmt kv_fmt;
  const void* kv_pool;
  const float* kv_scales;
  WFmt w_fmt;
  const void *w_uk, *w_uv;
  const float *w_uk_scale, *w_uv_scale;
  void* out;
  float* lse_out;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
};

int run(const CallCommon& c) {
  int st = check_dims(c.d);
  if (st) return st;
  if ((st = check_opts(c.o))) return st;
  if (c.B < 1 || c.T < 0) return MLA_ERR_INVALID_ARG;
  if (!c.q || !c.offsets || !c.kv_pool || !c.w_uk || !c.w_uv || !c.out || !c.ws) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c.q) || !aligned16(c.kv_pool) || !aligned16(c.w_uk) || !aligned16(c.w_uv) ||
      !aligned16(c.out) || !aligned16(c.ws))
    return MLA_ERR_INVALID_ARG;
  const bool sparse = c.ks.indices != nullptr;
  const bool fold = use_fold(c.d, c.o, c.B, c.T, c.kv_fmt == KVFmt::kE4M3, sparse);
  int K = 0;
  if ((st = resolve_splits(c.o, fold, &K, c.d, c.kv_fmt == KVFmt::kE4M3, sparse))) return st;
  const WorkspaceLayout lay = workspace_layout(*c.d, c.T, K, fold ? 2 : 1);
  if (c.ws_bytes < lay.total) return MLA_ERR_WORKSPACE_TOO_SMALL;

  char* ws = static_cast<char*>(c.ws);
  PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws + lay.header);
  TokenPlan* plan = reinterpret_cast<TokenPlan*>(ws + lay.plan);
  DecodeArgs a{};
  a.d = *c.d;
  a.B = c.B;
  a.T = c.T;
  a.K = K;
  a.mask = c.o->mask;
  a.window = c.o->window;
  a.scale = c.o->scale;
  a.kv_fmt = c.kv_fmt;
  a.kv_pool = c.kv_pool;
  a.kv_scales = c.kv_scales;
  a.ks = c.ks;
  a.hdr = hdr;
  a.hdr_mut = hdr;
  a.plan = plan;
  a.q_full = reinterpret_cast<const __nv_bfloat16*>(ws + lay.q_full);
  a.o_lat = reinterpret_cast<__nv_bfloat16*>(ws + lay.o_lat);
  a.lse_ws = reinterpret_cast<float*>(ws + lay.lse);
  a.part_o = reinterpret_cast<float*>(ws + lay.part_o);
  a.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  a.counters = reinterpret_cast<int*>(ws + lay.counters);
  a.bounds = reinterpret_cast<const int*>(ws + lay.bounds);
  a.fold = fold;
  PlanInputs pin{};
  pin.offsets = c.offsets;
  pin.B = c.B;
  pin.T = c.T;
  pin.ks = c.ks;
  pin.mask = c.o->mask;
  pin.window = c.o->window;
  pin.plan = plan;
  pin.hdr = hdr;
  pin.counters = a.counters;
  pin.bounds = reinterpret_cast<int*>(ws + lay.bounds);
  pin.K = K;
  pin.o_lat = a.o_lat;
  pin.lse_ws = a.lse_ws;
  pin.H = c.d->num_heads;
  pin.L = c.d->kv_lora_rank;
  pin.fold = fold;

  EventSet* timer = nullptr;
  if (c.o->flags & MLA_FLAG_KERNEL_TIMING) {
    timer = next_event_set();
    if (!timer) return MLA_ERR_CUDA;
  }
  auto mark = [&](int i) {
    return timer ? cudaEventRecord(timer->ev[i], c.stream) : cudaSuccess;
  };
  // K1 absorb (+ plan) -> K2 split-KV decode (+ merge of split tokens) -> K3 W_uv;
  // K2 and K3 are launched as programmatic dependents of their predecessor.
  cudaError_t e = mark(0);
  if (e == cudaSuccess)
    e = launch_absorb_tc(*c.d, c.T, static_cast<const __nv_bfloat16*>(c.q), c.w_fmt, c.w_uk, c.w_uk_scale,
                         reinterpret_cast<__nv_bfloat16*>(ws + lay.q_full), hdr, pin, c.stream);
  if (e == cudaSuccess) e = mark(1);
  if (e == cudaSuccess && c.T > 0) e = launch_decode_tc(a, c.stream);
  if (e == cudaSuccess) e = mark(2);
  if (e == cudaSuccess)
    e = launch_uv_tc(*c.d, c.T, a.o_lat, c.w_fmt, c.w_uv, c.w_uv_scale, a.lse_ws, static_cast<__nv_bfloat16*>(c.out),
                     c.lse_out, hdr, c.stream);
  if (e == cudaSuccess) e = mark(3);
  if (e != cudaSuccess) {
    std::fprintf(stderr, "mla_decode: %s\n", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  if (c.o->flags & MLA_FLAG_DEBUG_CHECKS) return device_status(hdr, c.stream);
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode_workspace_size(const mla_dims_t* dims, const mla_opts_t* opts, int32_t batch, int32_t total_q,
                              size_t* bytes) {
  int st = check_dims(dims);
  if (st) return st;
  if (!opts || !bytes || batch < 1 || total_q < 0) return MLA_ERR_INVALID_ARG;
  // one size for both walks, whether or not opts asks for folded pairs; the bf16
  // shapes' size also covers an e4m3 cache (whose calls never fold)
  mla_opts_t both = *opts;
  both.flags |= MLA_FLAG_FOLD_PAIRS;
  const bool fold = use_fold(dims, &both, batch, total_q, false, false);
  int K = 0;
  if ((st = resolve_splits(opts, fold, &K))) return st;
  const size_t a = workspace_layout(*dims, total_q, K, fold ? 2 : 1).total;
  int K1 = 0;
  if ((st = resolve_splits(opts, false, &K1))) return st;
  const size_t b = workspace_layout(*dims, total_q, K1, 1).total;
  *bytes = a > b ? a : b;
  return MLA_OK;
}

int mla_decode_paged(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                     const uint32_t* input_row_offsets, int32_t batch, int32_t total_q, const void* kv_pool,
                     const int32_t* block_table, int32_t block_table_stride, const uint32_t* cache_lens,
                     const void* w_uk, const void* w_uv, void* out, float* lse_out, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (!dims || !block_table || !cache_lens || block_table_stride < 1) return MLA_ERR_INVALID_ARG;
  CallCommon c{};
  c.d = dims;
  c.o = opts;
  c.q = q;
  c.offsets = input_row_offsets;
  c.B = batch;
  c.T = total_q;
  c.ks = KeySource{block_table, block_table_stride, cache_lens, nullptr, 0, nullptr, dims->page_size,
                   dims->num_pages};
  c.kv_fmt = KVFmt::kBF16;
  c.kv_pool = kv_pool;
  c.w_fmt = WFmt::kBF16;
  c.w_uk = w_uk;
  c.w_uv = w_uv;
  c.out = out;
  c.lse_out = lse_out;
  c.ws = workspace;
  c.ws_bytes = workspace_bytes;
  c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int mla_decode_paged_fp8(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                         const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                         const void* kv_pool_fp8, const float* kv_scales, const int32_t* block_table,
                         int32_t block_table_stride, const uint32_t* cache_lens, const void* w_uk_fp8,
                         const float* w_uk_scale, const void* w_uv_fp8, const float* w_uv_scale,
                         const float* q_scale, void* out, float* lse_out, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (q_scale) return MLA_ERR_UNSUPPORTED;
  if (!dims || !block_table || !cache_lens || block_table_stride < 1 || !kv_scales || !w_uk_scale ||
      !w_uv_scale || !aligned16(kv_scales))
    return MLA_ERR_INVALID_ARG;
  CallCommon c{};
  c.d = dims;
  c.o = opts;
  c.q = q;
  c.offsets = input_row_offsets;
  c.B = batch;
  c.T = total_q;
  c.ks = KeySource{block_table, block_table_stride, cache_lens, nullptr, 0, nullptr, dims->page_size,
                   dims->num_pages};
  c.kv_fmt = KVFmt::kE4M3;
  c.kv_pool = kv_pool_fp8;
  c.kv_scales = kv_scales;
  c.w_fmt = WFmt::kE4M3;
  c.w_uk = w_uk_fp8;
  c.w_uv = w_uv_fp8;
  c.w_uk_scale = w_uk_scale;
  c.w_uv_scale = w_uv_scale;
  c.out = out;
  c.lse_out = lse_out;
  c.ws = workspace;
  c.ws_bytes = workspace_bytes;
  c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int mla_decode_sparse(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                      const uint32_t* input_row_offsets, int32_t batch, int32_t total_q, const void* kv_pool,
                      const int32_t* d_indices, int32_t indices_stride, const int32_t* topk_lengths,
                      const void* w_uk, const void* w_uv, void* out, float* lse_out, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!dims || !opts || !d_indices || indices_stride < 1) return MLA_ERR_INVALID_ARG;
  if (opts->mask != MLA_MASK_NULL) return MLA_ERR_UNSUPPORTED;
  CallCommon c{};
  c.d = dims;
  c.o = opts;
  c.q = q;
  c.offsets = input_row_offsets;
  c.B = batch;
  c.T = total_q;
  c.ks = KeySource{nullptr, 0, nullptr, d_indices, indices_stride, topk_lengths, dims->page_size,
                   dims->num_pages};
  c.kv_fmt = KVFmt::kBF16;
  c.kv_pool = kv_pool;
  c.w_fmt = WFmt::kBF16;
  c.w_uk = w_uk;
  c.w_uv = w_uv;
  c.out = out;
  c.lse_out = lse_out;
  c.ws = workspace;
  c.ws_bytes = workspace_bytes;
  c.stream = static_cast<cudaStream_t>(stream);
  return run(c);
}

int mla_decode_kernel_times(float* ms, int32_t n) {
  int dev = 0;
  if (!ms || n < 0 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  KernelTimer& t = g_timer[dev];
  const int calls = t.used;
  t.used = 0;
  if (calls == 0) return 0;
  double sum[kTimedKernels] = {};
  for (int c = 0; c < calls; ++c) {
    const int slot = (t.next - 1 - c + 2 * kMaxTimedCalls) % kMaxTimedCalls;
    EventSet& es = t.sets[slot];
    if (cudaEventSynchronize(es.ev[kTimedKernels]) != cudaSuccess) return -1;
    for (int i = 0; i < kTimedKernels; ++i) {
      float v = 0.f;
      if (cudaEventElapsedTime(&v, es.ev[i], es.ev[i + 1]) != cudaSuccess) return -1;
      sum[i] += v;
    }
  }
  for (int i = 0; i < kTimedKernels && i < n; ++i) ms[i] = (float)(sum[i] / calls);
  return calls;
}

int mla_branch_prologue(const mla_dims_t* dims, void* q, const uint32_t* input_row_offsets, int32_t batch,
                        int32_t total_q, void* kv_pool, const int32_t* block_table, int32_t block_table_stride,
                        const uint32_t* cache_lens, const void* freqs_cis, int32_t max_seq_len,
                        const void* kv_norm_gamma, float epsilon, uint32_t flags, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!dims || dims->num_heads < 1 || dims->qk_nope < 0 || dims->qk_rope < 2 || dims->qk_rope % 2 != 0 ||
      dims->kv_lora_rank < 1 || dims->kv_lora_rank > 512 || dims->page_size < 1 || dims->num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if ((int64_t)dims->num_pages * dims->page_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (batch < 1 || total_q < 0 || block_table_stride < 1 || max_seq_len < 1) return MLA_ERR_INVALID_ARG;
  if (!q || !input_row_offsets || !kv_pool || !block_table || !cache_lens || !freqs_cis || !kv_norm_gamma ||
      !workspace)
    return MLA_ERR_INVALID_ARG;
  // rotation pairs are read and written as 4-byte words
  auto aligned4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!aligned4(q) || !aligned4(kv_pool) || !aligned4(freqs_cis)) return MLA_ERR_INVALID_ARG;
  if (!(epsilon >= 0.f) || (flags & ~MLA_FLAG_DEBUG_CHECKS)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < sizeof(PlanHeader) || !aligned16(workspace)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  PlanHeader* hdr = static_cast<PlanHeader*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word is read back only in debug mode, so only then is it cleared first
  if ((flags & MLA_FLAG_DEBUG_CHECKS) && cudaMemsetAsync(hdr, 0, sizeof(PlanHeader), s) != cudaSuccess)
    return MLA_ERR_CUDA;
  const cudaError_t e = launch_prologue(*dims, q, input_row_offsets, batch, total_q, kv_pool, block_table,
                                        block_table_stride, cache_lens, freqs_cis, max_seq_len, kv_norm_gamma,
                                        epsilon, hdr, s);
  if (e != cudaSuccess) {
    std::fprintf(stderr, "mla_branch_prologue: %s\n", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  if (flags & MLA_FLAG_DEBUG_CHECKS) return device_status(hdr, s);
  return MLA_OK;
}

namespace {
constexpr int kIndexerMaxTopK = 4096;
constexpr size_t kIndexerMaxScoreSmem = 200 * 1024;

int indexer_max_keys(int32_t stride, int32_t ps, int32_t mask, int32_t window) {
  const int64_t cap = (int64_t)stride * ps;
  if (mask == MLA_MASK_SLIDING_WINDOW_CAUSAL && window < cap) return window;
  return (int)cap;
}
}  // namespace

int mla_indexer_workspace_size(int32_t total_q, int32_t block_table_stride, int32_t page_size, int32_t mask,
                               int32_t window, size_t* bytes) {
  if (!bytes || total_q < 0 || block_table_stride < 1 || page_size < 1) return MLA_ERR_INVALID_ARG;
  if ((int64_t)block_table_stride * page_size > INT32_MAX) return MLA_ERR_UNSUPPORTED;
  if (mask == MLA_MASK_SLIDING_WINDOW_CAUSAL && window < 1) return MLA_ERR_INVALID_ARG;
  *bytes = indexer_workspace_bytes(total_q, indexer_max_keys(block_table_stride, page_size, mask, window));
  return MLA_OK;
}

int mla_indexer_fp8(int32_t num_heads, int32_t head_dim, int32_t page_size, int32_t num_pages, const void* q,
                    const float* q_s, const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                    const void* k_cache, const float* k_scales, const int32_t* block_table,
                    int32_t block_table_stride, const uint32_t* cache_lens, int32_t mask, int32_t window,
                    int32_t top_k, int32_t* output_indices, double* output_scores, uint32_t flags,
                    void* workspace, size_t workspace_bytes, void* stream) {
  if (num_heads < 1 || head_dim < 1 || page_size < 1 || num_pages < 1 || batch < 1 || total_q < 0 ||
      block_table_stride < 1)
    return MLA_ERR_INVALID_ARG;
  if (mask < MLA_MASK_NULL || mask > MLA_MASK_SLIDING_WINDOW_CAUSAL) return MLA_ERR_INVALID_ARG;
  if (mask == MLA_MASK_SLIDING_WINDOW_CAUSAL && window < 1) return MLA_ERR_INVALID_ARG;
  if (top_k < 1) return MLA_ERR_INVALID_ARG;
  if (top_k > kIndexerMaxTopK) return MLA_ERR_UNSUPPORTED;
  if ((int64_t)num_pages * page_size > INT32_MAX || (int64_t)block_table_stride * page_size > INT32_MAX)
    return MLA_ERR_UNSUPPORTED;
  const size_t score_smem = indexer_scores_smem(num_heads, head_dim);
  if (num_heads > 128 || score_smem > kIndexerMaxScoreSmem) return MLA_ERR_UNSUPPORTED;
  if (!q || !q_s || !input_row_offsets || !k_cache || !k_scales || !block_table || !cache_lens ||
      !output_indices || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (flags & ~MLA_FLAG_DEBUG_CHECKS) return MLA_ERR_INVALID_ARG;
  const int max_keys = indexer_max_keys(block_table_stride, page_size, mask, window);
  if (workspace_bytes < indexer_workspace_bytes(total_q, max_keys) || !aligned16(workspace))
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  PlanHeader* hdr = static_cast<PlanHeader*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(hdr, 0, sizeof(PlanHeader), s) != cudaSuccess) return MLA_ERR_CUDA;
  const cudaError_t e =
      launch_indexer(num_heads, head_dim, page_size, num_pages, batch, total_q, mask, window, top_k,
                     static_cast<const uint8_t*>(q), q_s, input_row_offsets, static_cast<const uint8_t*>(k_cache),
                     k_scales, block_table, block_table_stride, cache_lens, max_keys, workspace, output_indices,
                     output_scores, s);
  if (e != cudaSuccess) {
    std::fprintf(stderr, "mla_indexer_fp8: %s\n", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  if (flags & MLA_FLAG_DEBUG_CHECKS) return device_status(hdr, s);
  return MLA_OK;
}

int mla_debug_wait_selftest(uint64_t limit_ns, void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes < sizeof(PlanHeader) || !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > 1000000000ull) return MLA_ERR_INVALID_ARG;
  PlanHeader* hdr = static_cast<PlanHeader*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(hdr, 0, sizeof(PlanHeader), s) != cudaSuccess) return MLA_ERR_CUDA;
  const cudaError_t e = launch_wait_selftest(hdr, limit_ns, s);
  if (e != cudaSuccess) {
    std::fprintf(stderr, "mla_decode: %s\n", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return device_status(hdr, s);
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_CHECK: return "device-side input check failed";
    case MLA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
