/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for MLA decode attention in the
 * weight-absorbed ("no materialisation") form.  TEST INFRASTRUCTURE ONLY: it is
 * called by the test-suite, by the smoke check and by the CPU-baseline leg of
 * the benchmark, never by the product path.
 *
 * What it computes (one query row = one (b, t, h)):
 *   vLLM PR #14770 "[Attention] MLA get rid of materialization", PR
 *   description: the absorbed matrices W_Q_UK and W_UV_O are never formed;
 *   instead the query is mapped into latent space by a bmm with W_UK, attention
 *   runs over the shared latent cache, and the latent output is mapped back by a
 *   second bmm with W_UV ("sequential matmuls").
 *   "DeepSeek publica FlashMLA como codigo abierto", feature list: the latent
 *   cache is paged with 64-token blocks, values are BF16.
 *
 *   1. n = seq_len[b] - T + t + 1 keys are visible (causal inside the query
 *      block; n = seq_len[b] when T = 1).
 *   2. c_j = cache[block_table[b][j / page]][j % page][0 : d_lora + d_rope].
 *   3. ql  = [ q[b,t,h,0:d_nope] . W_UK[h]  (d_lora)  ||  q[b,t,h,d_nope:] ].
 *   4. s_j = scale * (ql . c_j);  lse = m + ln sum_j exp(s_j - m), m = max s_j;
 *      p_j = exp(s_j - lse).
 *   5. o_lat = sum_j p_j c_j[0:d_lora];  out = o_lat . W_UV[h]  (d_v).
 *
 * Every input is bf16 (uint16 bit patterns) and is widened to double exactly;
 * all arithmetic is fp64; no intermediate is rounded.  Loops follow the
 * definition above with no blocking or reordering.  OpenMP parallelises over
 * independent query rows only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "mla_oracle.h"

static double bf16_to_double(uint16_t v) {
  union { uint32_t u; float f; } x;
  x.u = ((uint32_t)v) << 16;
  return (double)x.f;
}

int mla_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Validate every block-table entry a row can touch.  Returns 0 or an error. */
static int check_inputs(const mla_oracle_dims* d, const int32_t* block_table,
                        const int32_t* seq_lens) {
  if (d->batch < 0 || d->q_len < 1 || d->num_heads < 1 || d->page_size < 1)
    return MLA_ORACLE_BAD_DIMS;
  for (int b = 0; b < d->batch; ++b) {
    int L = seq_lens[b];
    if (L < d->q_len || L > d->max_pages_per_seq * d->page_size)
      return MLA_ORACLE_BAD_SEQ_LEN;
    int npages = (L + d->page_size - 1) / d->page_size;
    for (int i = 0; i < npages; ++i) {
      int32_t pg = block_table[(int64_t)b * d->max_pages_per_seq + i];
      if (pg < 0 || pg >= d->num_pages) return MLA_ORACLE_BAD_BLOCK;
    }
  }
  return MLA_ORACLE_OK;
}

/* One query row; scratch holds ql (d_lora+d_rope) + s (seq_len) + o_lat. */
static void one_row(const mla_oracle_dims* d, int b, int t, int h,
                    const uint16_t* q, const uint16_t* cache,
                    const int32_t* block_table, const int32_t* seq_lens,
                    const uint16_t* w_uk, const uint16_t* w_uv, double scale,
                    double* scratch, double* out_row, double* lse_row,
                    double* olat_row) {
  const int dn = d->qk_nope, dr = d->qk_rope, dl = d->kv_lora, dv = d->v_head;
  const int dq = dn + dr, dc = dl + dr;
  const int T = d->q_len, H = d->num_heads, P = d->page_size;
  const int L = seq_lens[b];
  const int n = L - T + t + 1;
  double* ql = scratch;
  double* s = ql + dc;
  double* o = s + L;

  /* step 3: absorb q_nope into latent space, keep q_pe */
  const uint16_t* qr = q + (((int64_t)b * T + t) * H + h) * dq;
  const uint16_t* wk = w_uk + (int64_t)h * dn * dl;
  for (int l = 0; l < dl; ++l) {
    double acc = 0.0;
    for (int k = 0; k < dn; ++k)
      acc += bf16_to_double(qr[k]) * bf16_to_double(wk[(int64_t)k * dl + l]);
    ql[l] = acc;
  }
  for (int r = 0; r < dr; ++r) ql[dl + r] = bf16_to_double(qr[dn + r]);

  /* steps 2 and 4: gather each visible key through the block table, score */
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    int32_t pg = block_table[(int64_t)b * d->max_pages_per_seq + j / P];
    const uint16_t* cj = cache + ((int64_t)pg * P + (j % P)) * dc;
    double acc = 0.0;
    for (int k = 0; k < dc; ++k) acc += ql[k] * bf16_to_double(cj[k]);
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double sum = 0.0;
  for (int j = 0; j < n; ++j) sum += exp(s[j] - m);
  const double lse = m + log(sum);

  /* step 5: latent output, then the per-head up-projection */
  for (int l = 0; l < dl; ++l) o[l] = 0.0;
  for (int j = 0; j < n; ++j) {
    int32_t pg = block_table[(int64_t)b * d->max_pages_per_seq + j / P];
    const uint16_t* cj = cache + ((int64_t)pg * P + (j % P)) * dc;
    const double pj = exp(s[j] - lse);
    for (int l = 0; l < dl; ++l) o[l] += pj * bf16_to_double(cj[l]);
  }
  const uint16_t* wv = w_uv + (int64_t)h * dl * dv;
  for (int v = 0; v < dv; ++v) {
    double acc = 0.0;
    for (int l = 0; l < dl; ++l) acc += o[l] * bf16_to_double(wv[(int64_t)l * dv + v]);
    out_row[v] = acc;
  }
  *lse_row = lse;
  if (olat_row) memcpy(olat_row, o, sizeof(double) * dl);
}

int mla_oracle_decode(const mla_oracle_dims* d, const uint16_t* q,
                      const uint16_t* cache, const int32_t* block_table,
                      const int32_t* seq_lens, const uint16_t* w_uk,
                      const uint16_t* w_uv, double scale, int64_t n_sel,
                      const int64_t* sel, double* out, double* lse,
                      double* o_lat) {
  if (!d || !q || !cache || !block_table || !seq_lens || !w_uk || !w_uv ||
      !out || !lse)
    return MLA_ORACLE_NULL;
  int err = check_inputs(d, block_table, seq_lens);
  if (err) return err;
  const int T = d->q_len, H = d->num_heads;
  const int64_t rows = (int64_t)d->batch * T * H;
  const int64_t n = sel ? n_sel : rows;
  for (int64_t i = 0; i < n; ++i)
    if (sel && (sel[i] < 0 || sel[i] >= rows)) return MLA_ORACLE_BAD_DIMS;
  int Lmax = 0;
  for (int b = 0; b < d->batch; ++b) if (seq_lens[b] > Lmax) Lmax = seq_lens[b];
  const int64_t scratch_len = (int64_t)d->kv_lora + d->qk_rope + Lmax + d->kv_lora;
  int failed = 0;
#pragma omp parallel
  {
    double* scratch = (double*)malloc(sizeof(double) * scratch_len);
    if (!scratch) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t i = 0; i < n; ++i) {
        const int64_t r = sel ? sel[i] : i;
        const int h = (int)(r % H);
        const int t = (int)((r / H) % T);
        const int b = (int)(r / ((int64_t)H * T));
        one_row(d, b, t, h, q, cache, block_table, seq_lens, w_uk, w_uv, scale,
                scratch, out + i * d->v_head, lse + i,
                o_lat ? o_lat + i * d->kv_lora : NULL);
      }
      free(scratch);
    }
  }
  return failed ? MLA_ORACLE_NOMEM : MLA_ORACLE_OK;
}

/*
 * Split-KV partial for one query row over keys [k0, k1): the latent output
 * normalised within the range and the range's log-sum-exp.  Together with
 * mla_oracle_combine this restates the split-KV decomposition that
 * FlashAttention-style decode kernels use (FlashMLA is described as inspired by
 * FlashAttention 2 and 3): softmax over a union of key ranges equals the
 * LSE-weighted mixture of the per-range softmaxes.
 */
int mla_oracle_partial(const mla_oracle_dims* d, const uint16_t* q,
                       const uint16_t* cache, const int32_t* block_table,
                       const int32_t* seq_lens, const uint16_t* w_uk,
                       double scale, int b, int t, int h, int k0, int k1,
                       double* o_part, double* lse_part) {
  if (!d || !q || !cache || !block_table || !seq_lens || !w_uk || !o_part ||
      !lse_part)
    return MLA_ORACLE_NULL;
  int err = check_inputs(d, block_table, seq_lens);
  if (err) return err;
  const int dn = d->qk_nope, dr = d->qk_rope, dl = d->kv_lora;
  const int dq = dn + dr, dc = dl + dr, T = d->q_len, H = d->num_heads;
  const int P = d->page_size;
  if (b < 0 || b >= d->batch || t < 0 || t >= T || h < 0 || h >= H)
    return MLA_ORACLE_BAD_DIMS;
  const int n = seq_lens[b] - T + t + 1;
  if (k0 < 0 || k1 > n || k0 >= k1) return MLA_ORACLE_BAD_DIMS;
  double* ql = (double*)malloc(sizeof(double) * (dc + (k1 - k0)));
  if (!ql) return MLA_ORACLE_NOMEM;
  double* s = ql + dc;
  const uint16_t* qr = q + (((int64_t)b * T + t) * H + h) * dq;
  const uint16_t* wk = w_uk + (int64_t)h * dn * dl;
  for (int l = 0; l < dl; ++l) {
    double acc = 0.0;
    for (int k = 0; k < dn; ++k)
      acc += bf16_to_double(qr[k]) * bf16_to_double(wk[(int64_t)k * dl + l]);
    ql[l] = acc;
  }
  for (int r = 0; r < dr; ++r) ql[dl + r] = bf16_to_double(qr[dn + r]);
  double m = -INFINITY;
  for (int j = k0; j < k1; ++j) {
    int32_t pg = block_table[(int64_t)b * d->max_pages_per_seq + j / P];
    const uint16_t* cj = cache + ((int64_t)pg * P + (j % P)) * dc;
    double acc = 0.0;
    for (int k = 0; k < dc; ++k) acc += ql[k] * bf16_to_double(cj[k]);
    s[j - k0] = scale * acc;
    if (s[j - k0] > m) m = s[j - k0];
  }
  double sum = 0.0;
  for (int j = k0; j < k1; ++j) sum += exp(s[j - k0] - m);
  const double lse = m + log(sum);
  for (int l = 0; l < dl; ++l) o_part[l] = 0.0;
  for (int j = k0; j < k1; ++j) {
    int32_t pg = block_table[(int64_t)b * d->max_pages_per_seq + j / P];
    const uint16_t* cj = cache + ((int64_t)pg * P + (j % P)) * dc;
    const double pj = exp(s[j - k0] - lse);
    for (int l = 0; l < dl; ++l) o_part[l] += pj * bf16_to_double(cj[l]);
  }
  *lse_part = lse;
  free(ql);
  return MLA_ORACLE_OK;
}

/* LSE merge of n_split partials (each o normalised within its own range):
 *   lse = ln sum_s exp(lse_s);   o = sum_s exp(lse_s - lse) * o_s.          */
int mla_oracle_combine(int n_split, int dim, const double* lse_parts,
                       const double* o_parts, double* lse_out, double* o_out) {
  if (n_split < 1 || dim < 1 || !lse_parts || !o_parts || !lse_out || !o_out)
    return MLA_ORACLE_BAD_DIMS;
  double m = -INFINITY;
  for (int s = 0; s < n_split; ++s) if (lse_parts[s] > m) m = lse_parts[s];
  double sum = 0.0;
  for (int s = 0; s < n_split; ++s) sum += exp(lse_parts[s] - m);
  const double lse = m + log(sum);
  for (int k = 0; k < dim; ++k) o_out[k] = 0.0;
  for (int s = 0; s < n_split; ++s) {
    const double w = exp(lse_parts[s] - lse);
    for (int k = 0; k < dim; ++k) o_out[k] += w * o_parts[(int64_t)s * dim + k];
  }
  *lse_out = lse;
  return MLA_ORACLE_OK;
}

/* out = o_lat . W_UV[h] for one row (the second bmm on its own). */
int mla_oracle_up_project(const mla_oracle_dims* d, const uint16_t* w_uv, int h,
                          const double* o_lat, double* out_row) {
  if (!d || !w_uv || !o_lat || !out_row || h < 0 || h >= d->num_heads)
    return MLA_ORACLE_BAD_DIMS;
  const int dl = d->kv_lora, dv = d->v_head;
  const uint16_t* wv = w_uv + (int64_t)h * dl * dv;
  for (int v = 0; v < dv; ++v) {
    double acc = 0.0;
    for (int l = 0; l < dl; ++l) acc += o_lat[l] * bf16_to_double(wv[(int64_t)l * dv + v]);
    out_row[v] = acc;
  }
  return MLA_ORACLE_OK;
}
