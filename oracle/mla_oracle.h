/*
 * fp64 CPU oracle for MLA paged decode.  TEST INFRASTRUCTURE ONLY: loaded by
 * the tests, the smoke check and the benchmark's CPU-baseline leg, never by
 * the CUDA library.  The argument meanings are described in mla_oracle.c.
 */
#ifndef MLA_ORACLE_H
#define MLA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MLA_ORACLE_MASK_NULL = 0,
  MLA_ORACLE_MASK_CAUSAL = 1,
  MLA_ORACLE_MASK_SLIDING_WINDOW_CAUSAL = 2
};

typedef struct {
  int32_t H, N, R, L, V;     /* heads, qk_nope, qk_rope, kv_lora_rank, v_head */
  int32_t page_size;
  int32_t B, T;              /* requests, query tokens */
  int32_t mask, window;
  double scale;
  int32_t kv_fp8;            /* 0: bf16 rows [L+R]; 1: [L e4m3 | R bf16] rows + row_scales */
  int32_t w_fp8;             /* 0: bf16 weights; 1: e4m3 weights + 128x128 block scales */
  const uint16_t* q;         /* bf16 bits [T, H, N+R] */
  const uint32_t* row_offsets;   /* [B+1] */
  const void* pool;          /* cache rows */
  const float* row_scales;   /* [rows] when kv_fp8 */
  const int32_t* block_table;    /* [B, block_table_stride] page ids (dense) */
  int32_t block_table_stride;
  const uint32_t* cache_lens;    /* [B] (dense) */
  const int32_t* indices;    /* [B, indices_stride] rows, -1 = skip (sparse; NULL = dense) */
  int32_t indices_stride;
  const int32_t* topk_lengths;   /* [B] or NULL */
  const void* w_uk;          /* [H, L, N] */
  const float* w_uk_scale;   /* [H, ceil(L/128), ceil(N/128)] when w_fp8 */
  const void* w_uv;          /* [H, V, L] */
  const float* w_uv_scale;   /* [H, ceil(V/128), ceil(L/128)] when w_fp8 */
  int32_t t_begin, t_end;    /* query tokens to evaluate */
} mla_oracle_args;

/* out: [T, H, V] doubles, lse: [T, H] doubles; only tokens [t_begin, t_end) are written.
 * Returns 0 on success. */
int mla_oracle_decode(const mla_oracle_args* a, double* out, double* lse);
/* FP8 indexer ("mla_indexer_ragged_float8_paged"): per query token, the top_k key
 * rows by score = sum over heads of q_s * k_scale * (q . k), e4m3 values decoded
 * exactly.  The argument meanings are described in mla_oracle.c. */
typedef struct {
  int32_t H, D;              /* indexer heads, head depth */
  int32_t page_size;
  int32_t B, T;              /* requests, query tokens */
  int32_t mask, window;      /* as for the decode */
  int32_t top_k;
  const uint8_t* q;          /* e4m3 codes [T, H, D] */
  const float* q_s;          /* [T, H] */
  const uint32_t* row_offsets;   /* [B+1] */
  const uint8_t* k;          /* e4m3 codes, cache rows [rows, D] */
  const float* k_scales;     /* [rows] */
  const int32_t* block_table;    /* [B, block_table_stride] page ids */
  int32_t block_table_stride;
  const uint32_t* cache_lens;    /* [B] */
  int32_t t_begin, t_end;    /* query tokens to evaluate */
} mla_oracle_indexer_args;

/* rows: [T, top_k] physical rows (-1 past the number of keys); scores: [T, top_k]
 * (-inf for -1 slots) or NULL.  Only tokens [t_begin, t_end) are written.
 * Returns 0 on success. */
int mla_oracle_indexer(const mla_oracle_indexer_args* a, int32_t* rows, double* scores);

/* Fused branch prologue ("mla_decode_branch_fp8"): RoPE on the query's rope part and on
 * the rope part of each query token's own cache row, RMSNorm (gamma, eps) of that row's
 * latent part, in place on bf16 data.  The argument meanings are described in
 * mla_oracle.c. */
typedef struct {
  int32_t H, N, R, L;        /* heads, qk_nope, qk_rope (even), kv_lora_rank */
  int32_t page_size;
  int32_t B, T;
  double eps;
  const uint32_t* row_offsets;   /* [B+1] */
  const uint32_t* cache_lens;    /* [B] */
  const int32_t* block_table;    /* [B, block_table_stride] */
  int32_t block_table_stride;
  const uint16_t* freqs_cis;     /* bf16 [max_seq_len, R]: (cos, sin) per rotated pair */
  int32_t max_seq_len;
  const uint16_t* gamma;         /* bf16 [L] */
} mla_oracle_prologue_args;

/* q: bf16 [T, H, N+R] and pool: bf16 rows [rows, L+R], both updated in place.
 * Returns 0 on success, 1 if a position is past max_seq_len or R is odd. */
int mla_oracle_prologue(const mla_oracle_prologue_args* a, uint16_t* q, uint16_t* pool);
uint16_t mla_oracle_round_bf16(double x);

double mla_oracle_e4m3_value(uint8_t code);
double mla_oracle_bf16_value(uint16_t bits);
int mla_oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
