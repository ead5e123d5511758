/*
 * fp64 CPU oracle for multi-head latent attention (MLA) decode over a ragged
 * batch and a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes follows the Modular MAX/Mojo API pages:
 *   - "generic_flare_mla_decode_kv_cache_ragged": decode attention over a
 *     ragged batch (Args: q [batch, heads, q_head_size], input_row_offsets,
 *     scale; Parameters: mask_str "causal" / "null" / "sliding_window_causal",
 *     local_window_size; sparse_mla with d_indices, indices_stride and
 *     topk_lengths holding physical KV rows).
 *   - "mla_decode_branch_fp8": the absorbed form.  q_nope is projected into
 *     the latent space through w_uk [heads, kv_latent_dim, qk_nope_head_dim],
 *     concatenated with q_rope, attended against the cached [c_kv ; k_rope]
 *     rows, and the latent output is projected back through
 *     w_uv [heads, v_head_dim, kv_latent_dim].  FP8 weights carry block
 *     scales (m/n/k_scale_granularity).
 *   - "mla_indexer_ragged_float8_paged": K scales at head-size granularity
 *     (one fp32 scale per cached token row); -1 marks an unused index slot.
 *
 * The oracle is the plain definition, one (query token, head) pair at a time,
 * in double precision:
 *   ql[l]   = sum_n w_uk[h,l,n] * q[t,h,n]
 *   s_j     = scale * ( sum_l ql[l] * c[row_j,l] + sum_r q[t,h,N+r] * k_rope[row_j,r] )
 *   o[l]    = sum_j exp(s_j - m) * c[row_j,l] / sum_j exp(s_j - m),   m = max_j s_j
 *   lse     = m + ln(sum_j exp(s_j - m))
 *   out[v]  = sum_l w_uv[h,v,l] * o[l]
 * An empty key set gives out = 0 and lse = -inf.
 *
 * Readings where the pages are silent:
 *   - "q_nope_t @ w_uk" contracts w_uk over its last (nope) axis; w_uv is
 *     contracted over its last (latent) axis.
 *   - a cache row is [c_kv (L) ; k_rope (R)] in the concat order of the
 *     absorbed query; cache_lens include the query tokens, so query i of a
 *     request with qlen queries sits at pos = cache_len - qlen + i.
 *   - causal keeps keys j <= pos; sliding_window_causal keeps
 *     pos - W < j <= pos; null keeps all j < cache_len.
 *   - sparse indices are physical pool rows, per request row stride
 *     indices_stride; slots k >= topk_lengths[b] are ignored, -1 is skipped
 *     wherever it appears, duplicates count as many times as they appear; a
 *     NULL topk_lengths means every slot of the stride is considered.
 *   - FP8 cache rows are [L bytes e4m3 c_kv | R bf16 k_rope]; c_kv values are
 *     code * row_scale, k_rope is not scaled.  FP8 weights are e4m3 codes
 *     times a per-head fp32 scale of the 128 x 128 block holding the element.
 *   - e4m3 is OCP E4M3FN: bias 7, no infinities, S.1111.111 is NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "mla_oracle.h"

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE binary32: widen by a 16-bit shift. */
static double bf16_value(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3FN encoding (sign, 4 exponent bits with bias
 * 7, 3 mantissa bits; exponent 0 is subnormal; only S.1111.111 is NaN). */
double mla_oracle_e4m3_value(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

double mla_oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }

/* Weight element (h, i, j) of a [H, A, Bd] matrix, bf16 or e4m3 x block scale. */
static double weight_at(const mla_oracle_args* a, const void* w, const float* wscale,
                        int A, int Bd, int h, int i, int j) {
  size_t idx = ((size_t)h * A + i) * Bd + j;
  if (a->w_fp8) {
    int na = (A + 127) / 128, nb = (Bd + 127) / 128;
    double s = (double)wscale[((size_t)h * na + i / 128) * nb + j / 128];
    return mla_oracle_e4m3_value(((const uint8_t*)w)[idx]) * s;
  }
  return bf16_value(((const uint16_t*)w)[idx]);
}

/* Decode cached row `row` into c[L] and kr[R]. */
static void load_row(const mla_oracle_args* a, int64_t row, double* c, double* kr) {
  const int L = a->L, R = a->R;
  if (a->kv_fp8) {
    const uint8_t* p = (const uint8_t*)a->pool + (size_t)row * (size_t)(L + 2 * R);
    double s = (double)a->row_scales[row];
    for (int l = 0; l < L; ++l) c[l] = mla_oracle_e4m3_value(p[l]) * s;
    for (int r = 0; r < R; ++r) {
      uint16_t bits;
      memcpy(&bits, p + L + 2 * r, 2);
      kr[r] = bf16_value(bits);
    }
  } else {
    const uint16_t* p = (const uint16_t*)a->pool + (size_t)row * (size_t)(L + R);
    for (int l = 0; l < L; ++l) c[l] = bf16_value(p[l]);
    for (int r = 0; r < R; ++r) kr[r] = bf16_value(p[L + r]);
  }
}

/* The key multiset of query token t as a list of physical rows. Returns the count. */
static int64_t key_rows(const mla_oracle_args* a, int b, int t, int64_t* rows) {
  int64_t n = 0;
  if (a->indices) {
    int64_t cnt = a->topk_lengths ? a->topk_lengths[b] : a->indices_stride;
    if (cnt > a->indices_stride) cnt = a->indices_stride;
    for (int64_t k = 0; k < cnt; ++k) {
      int32_t idx = a->indices[(size_t)b * a->indices_stride + k];
      if (idx >= 0) rows[n++] = idx;
    }
    return n;
  }
  int64_t qlen = (int64_t)a->row_offsets[b + 1] - a->row_offsets[b];
  int64_t i = t - (int64_t)a->row_offsets[b];
  int64_t len = a->cache_lens[b];
  int64_t pos = len - qlen + i;
  int64_t lo = 0, hi = len;
  if (a->mask == MLA_ORACLE_MASK_CAUSAL) {
    hi = pos + 1;
  } else if (a->mask == MLA_ORACLE_MASK_SLIDING_WINDOW_CAUSAL) {
    hi = pos + 1;
    lo = pos + 1 - a->window;
    if (lo < 0) lo = 0;
  }
  for (int64_t j = lo; j < hi; ++j) {
    int64_t page = a->block_table[(size_t)b * a->block_table_stride + j / a->page_size];
    rows[n++] = page * a->page_size + j % a->page_size;
  }
  return n;
}

static int request_of(const mla_oracle_args* a, int t) {
  int b = 0;
  while (b + 1 < a->B && (int64_t)a->row_offsets[b + 1] <= t) ++b;
  return b;
}

static int64_t max_keys(const mla_oracle_args* a) {
  int64_t m = 1;
  for (int b = 0; b < a->B; ++b) {
    int64_t k = a->indices ? a->indices_stride : (int64_t)a->cache_lens[b];
    if (k > m) m = k;
  }
  return m;
}

int mla_oracle_decode(const mla_oracle_args* a, double* out, double* lse) {
  const int H = a->H, N = a->N, R = a->R, L = a->L, V = a->V;
  const int t0 = a->t_begin, t1 = a->t_end;
  const int64_t kmax = max_keys(a);
  if (t0 < 0 || t1 > a->T || t0 > t1) return 1;
  int failed = 0;

#pragma omp parallel
  {
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * kmax);
    double* s = (double*)malloc(sizeof(double) * kmax);
    double* ql = (double*)malloc(sizeof(double) * L);
    double* o = (double*)malloc(sizeof(double) * L);
    double* c = (double*)malloc(sizeof(double) * L);
    double* kr = (double*)malloc(sizeof(double) * (R > 0 ? R : 1));
    const int ok = rows && s && ql && o && c && kr;
    if (!ok) {
#pragma omp atomic write
      failed = 1;
    }
    /* every thread reaches the work-sharing loop; one without scratch skips its share */
    {
#pragma omp for schedule(dynamic, 1)
      for (int64_t th = (int64_t)t0 * H; th < (int64_t)t1 * H; ++th) {
        if (!ok) continue;
        const int t = (int)(th / H), h = (int)(th % H);
        const int b = request_of(a, t);
        const uint16_t* qrow = a->q + ((size_t)t * H + h) * (size_t)(N + R);
        double* orow = out + ((size_t)t * H + h) * (size_t)V;
        const int64_t nk = key_rows(a, b, t, rows);

        if (nk == 0) {
          for (int v = 0; v < V; ++v) orow[v] = 0.0;
          lse[(size_t)t * H + h] = -INFINITY;
          continue;
        }
        /* absorbed query: q_nope projected through w_uk[h] */
        for (int l = 0; l < L; ++l) {
          double acc = 0.0;
          for (int n = 0; n < N; ++n)
            acc += weight_at(a, a->w_uk, a->w_uk_scale, L, N, h, l, n) * bf16_value(qrow[n]);
          ql[l] = acc;
        }
        /* scores against [c_kv ; k_rope] */
        double m = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
          load_row(a, rows[j], c, kr);
          double acc = 0.0;
          for (int l = 0; l < L; ++l) acc += ql[l] * c[l];
          for (int r = 0; r < R; ++r) acc += bf16_value(qrow[N + r]) * kr[r];
          s[j] = a->scale * acc;
          if (s[j] > m) m = s[j];
        }
        /* softmax-weighted latent output */
        double z = 0.0;
        for (int l = 0; l < L; ++l) o[l] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
          double p = exp(s[j] - m);
          z += p;
          load_row(a, rows[j], c, kr);
          for (int l = 0; l < L; ++l) o[l] += p * c[l];
        }
        for (int l = 0; l < L; ++l) o[l] /= z;
        lse[(size_t)t * H + h] = m + log(z);
        /* back to v_head through w_uv[h] */
        for (int v = 0; v < V; ++v) {
          double acc = 0.0;
          for (int l = 0; l < L; ++l) acc += weight_at(a, a->w_uv, a->w_uv_scale, V, L, h, v, l) * o[l];
          orow[v] = acc;
        }
      }
    }
    free(rows);
    free(s);
    free(ql);
    free(o);
    free(c);
    free(kr);
  }
  return failed ? 2 : 0;
}

/*
 * FP8 indexer, following the "mla_indexer_ragged_float8_paged" page: an FP8
 * product of the query with the cached keys, with the query's per-head scale
 * q_s and the key rows' scales (one per cached row, head-size granularity),
 * summed over the heads, masked, and the top_k keys returned per query token.
 *
 *   score_j = sum_h q_s[t,h] * k_scale[row_j] * sum_d q[t,h,d] * k[row_j,d]
 *
 * Readings where the page is silent:
 *   - the score is exactly that sum: no activation or extra weight per head;
 *   - the key set of query token t is the decode's (causal / null /
 *     sliding_window_causal over the request's cache_len, positions mapped to
 *     physical rows through the block table), and the returned indices are
 *     those physical rows, as the sparse decode consumes them;
 *   - the rows come in descending score, equal scores in ascending key
 *     position (so the choice does not depend on page placement), then -1
 *     for every slot past the number of keys; a NaN score sorts last.
 */
typedef struct {
  double s;
  int64_t j, row;
} idx_key;

static int idx_key_cmp(const void* pa, const void* pb) {
  const idx_key* a = (const idx_key*)pa;
  const idx_key* b = (const idx_key*)pb;
  const int na = isnan(a->s), nb = isnan(b->s);
  if (na != nb) return na ? 1 : -1;
  if (!na && a->s != b->s) return a->s > b->s ? -1 : 1;
  return a->j < b->j ? -1 : (a->j > b->j ? 1 : 0);
}

int mla_oracle_indexer(const mla_oracle_indexer_args* a, int32_t* rows, double* scores) {
  const int H = a->H, D = a->D, K = a->top_k;
  if (a->t_begin < 0 || a->t_end > a->T || a->t_begin > a->t_end || K < 1) return 1;
  int64_t kmax = 1;
  for (int b = 0; b < a->B; ++b)
    if ((int64_t)a->cache_lens[b] > kmax) kmax = a->cache_lens[b];
  int failed = 0;

#pragma omp parallel
  {
    idx_key* keys = (idx_key*)malloc(sizeof(idx_key) * kmax);
    double* qv = (double*)malloc(sizeof(double) * (size_t)H * D);
    const int ok = keys && qv;
    if (!ok) {
#pragma omp atomic write
      failed = 1;
    }
    {
#pragma omp for schedule(dynamic, 1)
      for (int t = a->t_begin; t < a->t_end; ++t) {
        if (!ok) continue;
        int b = 0;
        while (b + 1 < a->B && (int64_t)a->row_offsets[b + 1] <= t) ++b;
        const int64_t qlen = (int64_t)a->row_offsets[b + 1] - a->row_offsets[b];
        const int64_t len = a->cache_lens[b];
        const int64_t pos = len - qlen + (t - (int64_t)a->row_offsets[b]);
        int64_t lo = 0, hi = len;
        if (a->mask == MLA_ORACLE_MASK_CAUSAL) {
          hi = pos + 1;
        } else if (a->mask == MLA_ORACLE_MASK_SLIDING_WINDOW_CAUSAL) {
          hi = pos + 1;
          lo = pos + 1 - a->window;
          if (lo < 0) lo = 0;
        }
        for (int h = 0; h < H; ++h)
          for (int d = 0; d < D; ++d)
            qv[(size_t)h * D + d] = mla_oracle_e4m3_value(a->q[((size_t)t * H + h) * D + d]);
        int64_t n = 0;
        for (int64_t j = lo; j < hi; ++j) {
          const int64_t page = a->block_table[(size_t)b * a->block_table_stride + j / a->page_size];
          const int64_t row = page * a->page_size + j % a->page_size;
          const uint8_t* kr = a->k + (size_t)row * D;
          double s = 0.0;
          for (int h = 0; h < H; ++h) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qv[(size_t)h * D + d] * mla_oracle_e4m3_value(kr[d]);
            s += (double)a->q_s[(size_t)t * H + h] * (double)a->k_scales[row] * dot;
          }
          keys[n].s = s;
          keys[n].j = j;
          keys[n].row = row;
          ++n;
        }
        qsort(keys, (size_t)n, sizeof(idx_key), idx_key_cmp);
        for (int i = 0; i < K; ++i) {
          rows[(size_t)t * K + i] = i < n ? (int32_t)keys[i].row : -1;
          if (scores) scores[(size_t)t * K + i] = i < n ? keys[i].s : -INFINITY;
        }
      }
    }
    free(keys);
    free(qv);
  }
  return failed ? 2 : 0;
}

/*
 * Fused branch prologue, following the "mla_decode_branch_fp8" page: RoPE is
 * applied to the query and to the key cache in place, RMSNorm (kv_norm_gamma,
 * epsilon) to the non-rope part of the key cache in place, before the absorb.
 *
 * Readings where the page is silent:
 *   - freqs_cis [max_seq_len, R] holds, per position, R/2 rotations as
 *     interleaved (cos, sin) pairs, and the rope values pair up the same way:
 *     (x[2i], x[2i+1]) -> (x0 cos - x1 sin, x0 sin + x1 cos);
 *   - query token t of its request sits at pos = cache_len - qlen + i (as for
 *     the decode); its rope part turns by freqs_cis[pos], and so does the rope
 *     part of the cache row at position pos of its request, the row this step
 *     wrote; no other cache row changes;
 *   - RMSNorm: c / sqrt(mean(c^2) + eps) * gamma over the L latent values;
 *   - every result is computed in fp64 from the bf16 inputs and rounded once
 *     to bf16 (nearest, ties to even).
 */

/* fp64 -> bf16 bits, rounded once to nearest with ties to even (finite, normal
 * or subnormal in the bf16 range; the values here are O(1)). */
uint16_t mla_oracle_round_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  const int neg = signbit(x) != 0;
  double ax = fabs(x);
  uint16_t out;
  if (ax == 0.0) {
    out = 0;
  } else {
    int e;
    frexp(ax, &e);                      /* ax = m * 2^e, m in [0.5, 1) */
    if (e < -125) e = -125;             /* bf16 subnormals: fixed quantum 2^-133 */
    const double quantum = ldexp(1.0, e - 8);    /* 8 significant bits */
    const double k = nearbyint(ax / quantum);    /* current mode: nearest, ties to even */
    const double v = k * quantum;
    if (v >= ldexp(1.0, 128)) {
      out = 0x7F80;                     /* overflow to infinity */
    } else {
      const float f = (float)v;         /* exact: v has at most 8 significant bits */
      uint32_t u;
      memcpy(&u, &f, sizeof u);
      out = (uint16_t)(u >> 16);
    }
  }
  return (uint16_t)(out | (neg ? 0x8000 : 0));
}

int mla_oracle_prologue(const mla_oracle_prologue_args* a, uint16_t* q, uint16_t* pool) {
  const int H = a->H, N = a->N, R = a->R, L = a->L;
  if (R % 2 != 0) return 1;
  int bad = 0;
  for (int t = 0; t < a->T; ++t) {
    int b = 0;
    while (b + 1 < a->B && (int64_t)a->row_offsets[b + 1] <= t) ++b;
    const int64_t qlen = (int64_t)a->row_offsets[b + 1] - a->row_offsets[b];
    const int64_t pos = (int64_t)a->cache_lens[b] - qlen + (t - (int64_t)a->row_offsets[b]);
    if (pos < 0 || pos >= a->max_seq_len) {
      bad = 1;
      continue;
    }
    const uint16_t* f = a->freqs_cis + (size_t)pos * R;
    /* the query's rope part, every head */
    for (int h = 0; h < H; ++h) {
      uint16_t* x = q + ((size_t)t * H + h) * (size_t)(N + R) + N;
      for (int i = 0; i < R; i += 2) {
        const double x0 = bf16_value(x[i]), x1 = bf16_value(x[i + 1]);
        const double c = bf16_value(f[i]), s = bf16_value(f[i + 1]);
        x[i] = mla_oracle_round_bf16(x0 * c - x1 * s);
        x[i + 1] = mla_oracle_round_bf16(x0 * s + x1 * c);
      }
    }
    /* the cache row this token wrote */
    const int64_t page = a->block_table[(size_t)b * a->block_table_stride + pos / a->page_size];
    uint16_t* row = pool + (size_t)(page * a->page_size + pos % a->page_size) * (size_t)(L + R);
    double ms = 0.0;
    for (int l = 0; l < L; ++l) {
      const double v = bf16_value(row[l]);
      ms += v * v;
    }
    const double inv = 1.0 / sqrt(ms / L + a->eps);
    for (int l = 0; l < L; ++l) row[l] = mla_oracle_round_bf16(bf16_value(row[l]) * inv * bf16_value(a->gamma[l]));
    uint16_t* kr = row + L;
    for (int i = 0; i < R; i += 2) {
      const double x0 = bf16_value(kr[i]), x1 = bf16_value(kr[i + 1]);
      const double c = bf16_value(f[i]), s = bf16_value(f[i + 1]);
      kr[i] = mla_oracle_round_bf16(x0 * c - x1 * s);
      kr[i + 1] = mla_oracle_round_bf16(x0 * s + x1 * c);
    }
  }
  return bad;
}

int mla_oracle_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}
