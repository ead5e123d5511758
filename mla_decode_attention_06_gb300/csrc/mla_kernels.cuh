// Launchers of the device kernels (internal to libmla_decode.so).
#pragma once
#include "mla_common.cuh"

namespace mla {

// Weight / cache element formats.
enum class WFmt { kBF16, kE4M3 };
enum class KVFmt { kBF16, kE4M3 };

struct DecodeArgs {
  mla_dims_t d;
  int B, T, K;                  // requests, query tokens, KV partitions
  int mask, window;
  float scale;
  KVFmt kv_fmt;
  const void* kv_pool;          // bf16 rows [L+R] or fp8 rows [L | 2R bytes]
  const float* kv_scales;       // fp8 row scales
  KeySource ks;
  const PlanHeader* hdr;
  PlanHeader* hdr_mut;
  const TokenPlan* plan;
  const __nv_bfloat16* q_full;  // [T, 128, L+R]
  __nv_bfloat16* o_lat;         // [T, H, L]
  float* lse_ws;                // [T, H]
  float* part_o;                // [K, 2, H, L]
  float* part_lse;              // [K, 2, 2, H]
  int* counters;                // [T, 4]
  const int* bounds;            // [2K + 1] first global tile of each partition, the total, first tokens
  bool fold;                    // query tokens walked in pairs by clusters of four CTAs
};




// Raises a kernel's dynamic shared-memory limit to `bytes` once per device (the
// driver call costs microseconds per launch otherwise).  Thread-safe.
cudaError_t ensure_smem_limit(const void* func, int bytes);

// Tensor-core decode (tcgen05): dense bf16 paged cache, shapes listed in decode_tc_supported.
bool decode_tc_supported(const mla_dims_t& d);
// Shapes with a folded (pairs of query tokens, cluster of four) decode instance.
bool decode_fold_supported(const mla_dims_t& d, bool fp8_cache);
// Partitions the device runs at once for this instance (0 if the query failed).
int decode_default_partitions(const mla_dims_t& d, bool fold, bool fp8_cache, bool sparse);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s);

// One thread waits (bounded by limit_ns) on an mbarrier nothing arrives on and
// records the time-out in *hdr as a decode wait would.
cudaError_t launch_wait_selftest(PlanHeader* hdr, uint64_t limit_ns, cudaStream_t s);

// Tensor-core weight GEMMs (K1 absorb, K3 W_uv) and the split-KV combine.
// K1: the W_uk absorb; one of its blocks also runs the plan (PlanInputs).
struct PlanInputs;
cudaError_t launch_absorb_tc(const mla_dims_t& d, int T, const __nv_bfloat16* q, WFmt wf, const void* w_uk,
                             const float* w_uk_scale, __nv_bfloat16* q_full, PlanHeader* hdr,
                             const PlanInputs& plan, cudaStream_t s);
cudaError_t launch_uv_tc(const mla_dims_t& d, int T, const __nv_bfloat16* o_lat, WFmt wf, const void* w_uv,
                         const float* w_uv_scale, const float* lse_ws, __nv_bfloat16* out, float* lse_out,
                         PlanHeader* hdr, cudaStream_t s);



// The fused branch prologue: RoPE on the query's rope part and, for each query
// token, RMSNorm + RoPE of the cache row at its position (bf16 pool), in place.
cudaError_t launch_prologue(const mla_dims_t& d, void* q, const uint32_t* offsets, int B, int T, void* kv_pool,
                            const int32_t* block_table, int bt_stride, const uint32_t* cache_lens,
                            const void* freqs, int max_seq_len, const void* gamma, float eps, PlanHeader* hdr,
                            cudaStream_t s);

// The FP8 indexer: exact scores into the workspace, then per-token top_k selection.
size_t indexer_workspace_bytes(int T, int max_keys);
// Dynamic shared memory of the scores kernel for H heads of D dimensions.
size_t indexer_scores_smem(int H, int D);
cudaError_t launch_indexer(int H, int D, int ps, int num_pages, int B, int T, int mask, int window, int top_k,
                           const uint8_t* q, const float* q_s, const uint32_t* offsets, const uint8_t* k,
                           const float* k_scales, const int32_t* block_table, int bt_stride,
                           const uint32_t* cache_lens, int max_keys, void* workspace, int32_t* out_rows,
                           double* out_scores, cudaStream_t s);

}  // namespace mla
