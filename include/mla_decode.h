/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) multi-head latent attention
 * (MLA) decode library, libmla_decode.so.
 *
 * One call computes, for every query token t of a ragged batch and every head h,
 * the absorbed MLA decode described on the Modular MAX/Mojo API pages
 * "mla_decode_branch_fp8" (fused steps: q_nope @ w_uk, concat with q_rope,
 * MLA decode, raw_output @ w_uv) and "generic_flare_mla_decode_kv_cache_ragged"
 * (Args: q, input_row_offsets, kv_collection, scale, output; Parameters:
 * mask_str, local_window_size, sparse_mla; optional d_indices, indices_stride,
 * topk_lengths):
 *
 *   q_lat[l]  = sum_n w_uk[h,l,n] q[t,h,n]                       (l < L)
 *   s_j       = scale * ( q_lat . c_kv[row_j] + q[t,h,N:N+R] . k_rope[row_j] )
 *   o         = softmax_j(s) . c_kv[rows]                          (latent, L wide)
 *   out[t,h,v]= sum_l w_uv[h,v,l] o[l]
 *   lse[t,h]  = ln sum_j exp(s_j)            (natural log of the scaled scores)
 *
 * Shapes use H = num_heads, N = qk_nope, R = qk_rope, L = kv_lora_rank,
 * V = v_head, ps = page_size, B = batch (requests), T = total query tokens.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, row-major, densely packed unless a
 *     stride argument says otherwise.  Scalars and the two structs are host memory.
 *   - The caller owns every buffer.  The library allocates nothing: scratch space
 *     is the caller's `workspace` (size from mla_decode_workspace_size).
 *     `out` and `lse_out` must not alias an input or the workspace.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and the call returns without synchronising, except when
 *     opts->flags has MLA_FLAG_DEBUG_CHECKS: then it waits for the stream and
 *     reports what the device-side checks found.
 *   - A cache row is [c_kv (L) ; k_rope (R)], the concat order of the absorbed
 *     query.  cache_lens[b] counts every cached token of request b including
 *     its query tokens: query i of a request with qlen queries sits at position
 *     pos = cache_lens[b] - qlen + i.
 *   - Masks (mask_str on the decode page): NULL attends keys j < cache_len,
 *     CAUSAL keys j <= pos, SLIDING_WINDOW_CAUSAL keys pos - window < j <= pos.
 *   - The output is fully overwritten.  A query with no key gets out = 0 and
 *     lse = -inf.
 *   - Page ids outside [0, num_pages) and sparse rows outside
 *     [0, num_pages * page_size) are never dereferenced: their keys are dropped
 *     and the device records MLA_ERR_DEVICE_CHECK (returned in debug mode).
 *   - Return value: an mla_status_t; mla_status_string() gives its text.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,        /* NULL required pointer, bad sizes, bad mask or window */
  MLA_ERR_UNSUPPORTED = 2,        /* shape without a kernel instance, H > 128, q_scale != NULL;
                                     instances: (L, R) = (512, 64), or L = 64 with R <= 32 (R % 8 == 0);
                                     N % 8 == 0; V % 8 == 0, V <= 512;
                                     page_size in {8, 16, 32, 64} or a multiple of 64 */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3,
  MLA_ERR_CUDA = 4,               /* a CUDA runtime or driver call failed */
  MLA_ERR_DEVICE_CHECK = 5,       /* debug mode: a device-side input check failed */
  MLA_ERR_TIMEOUT = 6             /* debug mode: a bounded device wait gave up */
} mla_status_t;

typedef enum {
  MLA_MASK_NULL = 0,
  MLA_MASK_CAUSAL = 1,
  MLA_MASK_SLIDING_WINDOW_CAUSAL = 2
} mla_mask_t;

#define MLA_FLAG_DEBUG_CHECKS 1u
/* Record a CUDA event pair around every kernel of the call; read the durations
 * with mla_decode_kernel_times() once the stream has finished. */
#define MLA_FLAG_KERNEL_TIMING 2u
/* Query walk.  Consecutive query tokens of a request can be walked in pairs
 * (decode page: fold_shared_index; a request's tokens share its cache rows or
 * index list): every cache tile is read once for both tokens by a cluster of
 * four CTAs.  Pairs are possible when the call has at least two query tokens
 * per request on average (total_q >= 2 * batch) and a bf16 cache with
 * (L, R) = (512, 64); otherwise every token is walked on its own.  Where
 * possible, the default folds sparse calls (whose gathered row loads bound the
 * main loop: folding halves them) and walks dense calls one token at a time
 * (their main loop is bound by each CTA's score contraction, which folding
 * does not shrink, and a cluster of four leaves SMs idle).  MLA_FLAG_FOLD_PAIRS
 * forces pairs, MLA_FLAG_PER_TOKEN forces one token at a time; setting both is
 * an invalid argument.  The two walks agree to rounding. */
#define MLA_FLAG_FOLD_PAIRS 4u
#define MLA_FLAG_PER_TOKEN 8u

/* Problem dimensions (decode page: q [.., num_heads, q_head_size];
 * mla_decode_branch_fp8 page: w_uk [num_heads, kv_latent_dim, qk_nope_head_dim],
 * w_uv [num_heads, v_head_dim, kv_latent_dim]). */
typedef struct {
  int32_t num_heads;     /* H, 1..128 */
  int32_t qk_nope;       /* N */
  int32_t qk_rope;       /* R */
  int32_t kv_lora_rank;  /* L */
  int32_t v_head;        /* V */
  int32_t page_size;     /* ps, tokens per cache page */
  int32_t num_pages;     /* pages in the pool */
} mla_dims_t;

/* Call options (decode page: mask_str, local_window_size, scale, num_partitions_in). */
typedef struct {
  int32_t mask;          /* mla_mask_t */
  int32_t window;        /* tokens, >= 1 for SLIDING_WINDOW_CAUSAL, ignored otherwise */
  float scale;           /* multiplies q.k, usually 1/sqrt(N + R) */
  int32_t num_splits;    /* KV partitions; 0 = as many as the device keeps resident at
                            once (one cluster of two CTAs each, four when query tokens
                            are walked in pairs), at most one per pair (four) of SMs,
                            from the CUDA occupancy query.  The call cuts the
                            batch's key tiles into that many partitions of about equal
                            cost (tiles plus a charge per query token started); a token
                            cut between partitions is merged in the decode kernel. */
  uint32_t flags;        /* MLA_FLAG_DEBUG_CHECKS | MLA_FLAG_KERNEL_TIMING |
                            MLA_FLAG_FOLD_PAIRS | MLA_FLAG_PER_TOKEN */
} mla_opts_t;

/* Bytes of scratch a call needs for `total_q` query tokens with these dims and
 * opts (num_splits decides the partial-result slots).  Uses the current
 * device's SM count when opts->num_splits == 0.  The size covers both query
 * walks (one token at a time and, where it applies, folded pairs) whatever
 * opts->flags says, so one workspace serves calls with either.  Writes *bytes. */
int mla_decode_workspace_size(const mla_dims_t* dims, const mla_opts_t* opts, int32_t batch,
                              int32_t total_q, size_t* bytes);

/* Dense bf16 decode over a paged cache (decode page: q, input_row_offsets,
 * kv_collection; the collection is flattened to pool + block_table + cache_lens).
 *   q                  bf16 [T, H, N+R]   (nope first, then rope)
 *   input_row_offsets  uint32 [B+1], non-decreasing, [0] = 0, [B] = T
 *   kv_pool            bf16 [num_pages, ps, L+R]
 *   block_table        int32 [B, block_table_stride]: physical page of logical page p
 *   cache_lens         uint32 [B], <= block_table_stride * ps
 *   w_uk               bf16 [H, L, N]
 *   w_uv               bf16 [H, V, L]
 *   out                bf16 [T, H, V]
 *   lse_out            float [T, H] or NULL */
int mla_decode_paged(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                     const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                     const void* kv_pool, const int32_t* block_table, int32_t block_table_stride,
                     const uint32_t* cache_lens, const void* w_uk, const void* w_uv, void* out,
                     float* lse_out, void* workspace, size_t workspace_bytes, void* stream);

/* FP8 latent cache (decode page: per_token_scale_rope_aware, "interleaved FP8+BF16";
 * indexer page: K scales at head-size granularity, i.e. one fp32 scale per row;
 * mla_decode_branch_fp8 page: w_uk_scale, w_uv_scale with block granularity).
 *   kv_pool_fp8   bytes [num_pages, ps, L + 2R]: L e4m3 (OCP E4M3FN) c_kv codes,
 *                 then R bf16 k_rope values; c_kv = code * kv_scales[row]
 *   kv_scales     float [num_pages, ps], 16-byte aligned (a page's scales are
 *                 copied into shared memory with its rows)
 *   w_uk_fp8      e4m3 [H, L, N], w_uk_scale float [H, ceil(L/128), ceil(N/128)]
 *   w_uv_fp8      e4m3 [H, V, L], w_uv_scale float [H, ceil(V/128), ceil(L/128)]
 *   q_scale       must be NULL (sigma_Q = 1, the decode page's default)
 * Other arguments as mla_decode_paged. */
int mla_decode_paged_fp8(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                         const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                         const void* kv_pool_fp8, const float* kv_scales,
                         const int32_t* block_table, int32_t block_table_stride,
                         const uint32_t* cache_lens, const void* w_uk_fp8,
                         const float* w_uk_scale, const void* w_uv_fp8, const float* w_uv_scale,
                         const float* q_scale, void* out, float* lse_out, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Sparse top-k decode (decode page: sparse_mla, d_indices, indices_stride,
 * topk_lengths; indexer page: -1 marks an unused slot).
 *   kv_pool        bf16 [num_pages, ps, L+R]
 *   d_indices      int32 [B, indices_stride]: physical pool rows (page * ps + slot)
 *                  shared by all query tokens of request b; -1 is skipped wherever
 *                  it appears; duplicates count once per occurrence
 *   topk_lengths   int32 [B] or NULL: slots k >= topk_lengths[b] are ignored
 *                  (NULL: all indices_stride slots are considered)
 * opts->mask must be MLA_MASK_NULL (no positional mask on given rows).
 * Other arguments as mla_decode_paged. */
int mla_decode_sparse(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                      const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                      const void* kv_pool, const int32_t* d_indices, int32_t indices_stride,
                      const int32_t* topk_lengths, const void* w_uk, const void* w_uv,
                      void* out, float* lse_out, void* workspace, size_t workspace_bytes,
                      void* stream);

/* Fused branch prologue (mla_decode_branch_fp8 page, description: "Apply RoPE to
 * the query and the key cache (in-place)", "Apply RMSNorm to the non-rope portion
 * of the key cache (in-place)"; Args freqs_cis, kv_norm_gamma, epsilon), run
 * before the decode call of the same step.  For query token t of request b at
 * position pos = cache_lens[b] - qlen + i:
 *   - q[t, h, N + 2i], q[t, h, N + 2i + 1] of every head turn by
 *     freqs_cis[pos, 2i] = cos, freqs_cis[pos, 2i + 1] = sin:
 *     (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos);
 *   - the cache row at position pos of request b (the row this step wrote):
 *     latent part c -> c / sqrt(mean(c^2) + epsilon) * kv_norm_gamma, rope part
 *     turned like the query's;
 *   - no other value changes.
 * Every result is the value of those expressions, evaluated in double precision,
 * rounded once to bf16, nearest with ties to even (the rotations exactly; the
 * RMSNorm within a few double-precision units of the last place, so a result
 * can differ from the correctly rounded one only when the exact value lies that
 * close to a bf16 halfway point).
 *   q              bf16 [T, H, N+R], rope part rewritten in place; 4-byte aligned
 *   kv_pool        bf16 [num_pages, ps, L+R] (L <= 512), rows rewritten in place;
 *                  4-byte aligned
 *   freqs_cis      bf16 [max_seq_len, R]: per position R/2 (cos, sin) pairs;
 *                  4-byte aligned
 *   kv_norm_gamma  bf16 [L]
 *   epsilon        >= 0
 *   flags          0 or MLA_FLAG_DEBUG_CHECKS (wait and report device checks)
 *   workspace      device memory, >= 256 bytes, 16-byte aligned (status word;
 *                  cleared and read back in debug mode only)
 * Other arguments as mla_decode_paged.  A token whose position is outside
 * [0, max_seq_len) or whose page id is outside [0, num_pages) is left unchanged
 * (query and row) and recorded: MLA_ERR_DEVICE_CHECK in debug mode. */
int mla_branch_prologue(const mla_dims_t* dims, void* q, const uint32_t* input_row_offsets, int32_t batch,
                        int32_t total_q, void* kv_pool, const int32_t* block_table, int32_t block_table_stride,
                        const uint32_t* cache_lens, const void* freqs_cis, int32_t max_seq_len,
                        const void* kv_norm_gamma, float epsilon, uint32_t flags, void* workspace,
                        size_t workspace_bytes, void* stream);

/* FP8 indexer (mla_indexer_ragged_float8_paged page: the FP8 product of the query
 * with the key cache, with the query's per-head scales q_s and the key scales at
 * head-size granularity, summed across the heads, masked, top-k; Args
 * output_indices, -1 where fewer keys exist).  It produces the row lists
 * mla_decode_sparse consumes.  For query token t of request b and every key j of
 * its key set (the decode's mask rules over cache_lens[b]):
 *   s_j = sum_h (q_s[t,h] * k_scales[row_j]) * (sum_d q[t,h,d] * k_cache[row_j,d])
 * output_indices[t, i] for i < top_k: the physical rows (page * ps + slot) of the
 * keys by descending s_j, equal scores by ascending position j, NaN scores last;
 * -1 past the number of keys.  The inner sum is exact (an e4m3 value is a multiple
 * of 2^-9, so the sum is an exact integer multiple of 2^-18) and the head sum is
 * the double-precision value of that expression evaluated in head order, each
 * product and sum rounded separately: the ranking, ties included, is exactly
 * defined.
 *   q               e4m3 (OCP E4M3FN) [T, H, D] with H = num_heads, D = head_dim
 *   q_s             float [T, H]
 *   k_cache         e4m3 [num_pages, ps, D]
 *   k_scales        float [num_pages, ps]
 *   mask, window    as mla_opts_t (NULL, CAUSAL or SLIDING_WINDOW_CAUSAL)
 *   top_k           1 .. 4096
 *   output_indices  int32 [T, top_k]
 *   output_scores   double [T, top_k] (s_j of each returned row, -inf for -1 slots) or NULL
 *   flags           0 or MLA_FLAG_DEBUG_CHECKS
 *   workspace       mla_indexer_workspace_size() bytes, 16-byte aligned
 * Other arguments as mla_decode_paged.  Keys on a page id outside [0, num_pages)
 * are never read: they come out as -1 and are recorded (MLA_ERR_DEVICE_CHECK in
 * debug mode).  num_heads > 128, or shapes whose per-block scratch exceeds the
 * limit ((H + 32)(D + 1) 4 + 256 H bytes, about 200 KB), return MLA_ERR_UNSUPPORTED. */
int mla_indexer_workspace_size(int32_t total_q, int32_t block_table_stride, int32_t page_size, int32_t mask,
                               int32_t window, size_t* bytes);
int mla_indexer_fp8(int32_t num_heads, int32_t head_dim, int32_t page_size, int32_t num_pages, const void* q,
                    const float* q_s, const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                    const void* k_cache, const float* k_scales, const int32_t* block_table,
                    int32_t block_table_stride, const uint32_t* cache_lens, int32_t mask, int32_t window,
                    int32_t top_k, int32_t* output_indices, double* output_scores, uint32_t flags,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Mean per-kernel device durations (milliseconds) over the calls on the current
 * device that set MLA_FLAG_KERNEL_TIMING since the previous read (at most the
 * last 4096), in launch order: [0] W_uk absorb (with the call's planning),
 * [1] split-KV decode (with the merge of split tokens), [2] W_uv.  Waits for
 * those calls' events and clears the record.  Writes min(n, 3) values;
 * returns the number of calls averaged, 0 if none,
 * -1 on a CUDA error.  Host-side bookkeeping only: not thread-safe. */
int mla_decode_kernel_times(float* ms, int32_t n);

/* Dense bf16 decode for callers that cannot allocate device memory (code that
 * runs where cudaMalloc is forbidden or unwanted: inside another allocator,
 * under a memory budget fixed at start-up, or in a plug-in handed only its
 * tensors).  No counterpart on the API pages: it is mla_decode_paged with the
 * workspace replaced by a 64 MiB array compiled into the library
 * (mla_decode_static_scratch_bytes() returns the size).  Arguments as
 * mla_decode_paged without workspace / workspace_bytes.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Each GPU on which this entry point's module is loaded keeps the 64 MiB
 *     until the process exits.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it; make that
 *     first call before capturing a stream into a CUDA graph.  Concurrent first
 *     calls from several host threads are safe (the lookup is serialised).
 *   - cudaDeviceReset invalidates the kept address: after resetting a device,
 *     do not call this entry point on it again in the same process.
 *   - All calls share the one array: calls that may overlap on the GPU (other
 *     streams, other host threads) race and must be serialised by the caller.
 *   - Returns MLA_ERR_WORKSPACE_TOO_SMALL, with a message on stderr, when
 *     mla_decode_workspace_size() for these arguments exceeds the array. */
size_t mla_decode_static_scratch_bytes(void);
int mla_decode_paged_static(const mla_dims_t* dims, const mla_opts_t* opts, const void* q,
                            const uint32_t* input_row_offsets, int32_t batch, int32_t total_q,
                            const void* kv_pool, const int32_t* block_table, int32_t block_table_stride,
                            const uint32_t* cache_lens, const void* w_uk, const void* w_uv, void* out,
                            float* lse_out, void* stream);

/* Self-test of the failure detection (no counterpart on the API pages).  Every
 * wait of the library's kernels is bounded in time; when one gives up, the kernel
 * records the time-out in the workspace header and unwinds instead of hanging,
 * and the debug path returns MLA_ERR_TIMEOUT.  This launches one thread that
 * waits, through that same bounded wait, on a barrier nothing arrives on (no
 * copy, MMA or other CTA involved), then reads the status back like a call with
 * MLA_FLAG_DEBUG_CHECKS.
 *   limit_ns    the wait's limit, 1 .. 1e9 nanoseconds
 *   workspace   device memory, >= 256 bytes, 16-byte aligned (its header is cleared)
 *   stream      cudaStream_t; the call synchronises it
 * Returns MLA_ERR_TIMEOUT when the time-out was detected and reported (the
 * expected outcome), MLA_ERR_INVALID_ARG for bad arguments, MLA_ERR_CUDA if a
 * CUDA call failed.  The device stays usable afterwards. */
int mla_debug_wait_selftest(uint64_t limit_ns, void* workspace, size_t workspace_bytes, void* stream);

/* Static text for a status code. */
const char* mla_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H */
