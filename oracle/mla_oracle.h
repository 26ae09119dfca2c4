/* mla_oracle.h -- fp64 CPU oracle for weight-absorbed MLA decode.
 * Test infrastructure only (tests, smoke check, CPU baseline); the product
 * library never includes or links it. */
#ifndef MLA_ORACLE_H
#define MLA_ORACLE_H
#include <stdint.h>
#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t batch, q_len, num_heads;
  int32_t qk_nope, qk_rope, kv_lora, v_head, page_size;
  int32_t num_pages, max_pages_per_seq;
} mla_oracle_dims;

enum {
  MLA_ORACLE_OK = 0,
  MLA_ORACLE_NULL = 1,
  MLA_ORACLE_BAD_DIMS = 2,
  MLA_ORACLE_BAD_SEQ_LEN = 3,
  MLA_ORACLE_BAD_BLOCK = 4,
  MLA_ORACLE_NOMEM = 5
};

int mla_oracle_threads(void);
/* q [B,T,H,nope+rope], cache [num_pages,page,lora+rope], w_uk [H,nope,lora],
 * w_uv [H,lora,v] as bf16 bit patterns; block_table [B,max_pages], seq_lens [B].
 * sel: NULL for every row, else n_sel flat row ids ((b*T+t)*H+h).
 * out [n,v], lse [n] natural log, o_lat [n,lora] (may be NULL), n = rows or n_sel. */
int mla_oracle_decode(const mla_oracle_dims* d, const uint16_t* q,
                      const uint16_t* cache, const int32_t* block_table,
                      const int32_t* seq_lens, const uint16_t* w_uk,
                      const uint16_t* w_uv, double scale, int64_t n_sel,
                      const int64_t* sel, double* out, double* lse,
                      double* o_lat);
int mla_oracle_partial(const mla_oracle_dims* d, const uint16_t* q,
                       const uint16_t* cache, const int32_t* block_table,
                       const int32_t* seq_lens, const uint16_t* w_uk,
                       double scale, int b, int t, int h, int k0, int k1,
                       double* o_part, double* lse_part);
int mla_oracle_combine(int n_split, int dim, const double* lse_parts,
                       const double* o_parts, double* lse_out, double* o_out);
int mla_oracle_up_project(const mla_oracle_dims* d, const uint16_t* w_uv, int h,
                          const double* o_lat, double* out_row);
#ifdef __cplusplus
}
#endif
#endif
