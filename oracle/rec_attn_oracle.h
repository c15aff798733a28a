/*
 * rec_attn_oracle.h -- interface of the fp64 CPU oracle (test infrastructure only).
 * Private to oracle/: the CUDA library has its own, unrelated header.
 */
#ifndef REC_ATTN_ORACLE_H
#define REC_ATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_FP32 = 1 };
enum { ORC_SKIP = 0, ORC_PARTIAL = 1, ORC_FULL = 2 };
#define ORC_TILE 128

typedef struct {
  int32_t num_heads;
  int32_t head_dim;
  int32_t use_delay;
  int64_t delay_s;            /* delta_delay >= 0, seconds */
  int32_t window;             /* 0 = no window */
  int32_t hist_bidirectional; /* 1 = GLOBAL/HIST fully mutually visible */
  int32_t use_rope;
  double phi_min;             /* rad turned by the slowest pair over dt_max */
  double dt_max_s;            /* seconds */
  double rope_base;
  double softmax_scale;       /* <= 0 means 1/sqrt(head_dim) */
} orc_params;

/* vis(i, j) for two tokens of one request (positions are request-local). */
int orc_visible(const orc_params* p, int64_t pi, int64_t ti, int ty_i,
                int64_t pj, int64_t tj, int ty_j);
/* L x L mask of one request, row-major, 1 = visible. */
void orc_mask(const orc_params* p, int64_t L, const int64_t* t, const int8_t* ty, uint8_t* out);
/* Block [i0, i0+ni) x [j0, j0+nj) of that mask, row-major; indices >= L give 0. */
void orc_mask_block(const orc_params* p, int64_t L, const int64_t* t, const int8_t* ty,
                    int64_t i0, int64_t ni, int64_t j0, int64_t nj, uint8_t* out);
/* Exact number of visible (query, key) pairs over the batch (per head). */
uint64_t orc_visible_pairs(const orc_params* p, int32_t B, const int64_t* offsets,
                           const int64_t* t, const int8_t* ty);
/* Rotate one head vector x[0..head_dim) at absolute time t into y. */
void orc_rope(const orc_params* p, int64_t t, const double* x, double* y);
/* Attention outputs for the sorted global rows `rows` (NULL = all tokens):
 * out[n_rows][H][d], lse[n_rows][H] (natural log; -inf for a row with no
 * visible key).  q, k, v are [T][H][d] in dtype (bf16 bits or fp32).
 * Returns 0, or a negative value on invalid arguments. */
int orc_attention(const orc_params* p, int32_t B, const int64_t* offsets,
                  const int64_t* t, const int8_t* ty, int32_t dtype,
                  const void* q, const void* k, const void* v,
                  int64_t n_rows, const int64_t* rows, double* out, double* lse,
                  int32_t n_threads);
/* Fused inputs: QK-RMSNorm gains (fp64 [H][d], NULL = no norm of that side),
 * its epsilon, and sigmoid-gate pre-activations in the I/O dtype ([T][H][d],
 * NULL = no gate) for Q, K and the attention output. */
typedef struct {
  const double* q_norm_w;
  const double* k_norm_w;
  double norm_eps;
  const void* q_gate;
  const void* k_gate;
  const void* out_gate;
} orc_fused;
/* y = x / sqrt(mean(x^2) + eps) * w over one head vector of length d. */
void orc_rmsnorm(const double* x, const double* w, int d, double eps, double* y);
/* 1 / (1 + e^-x). */
double orc_sigmoid(double x);
/* orc_attention with the fused steps: q and k rows are normalised (if a gain is
 * given), gated, then rotated; outputs are gated.  f == NULL is orc_attention. */
int orc_attention_fused(const orc_params* p, int32_t B, const int64_t* offsets,
                        const int64_t* t, const int8_t* ty, int32_t dtype,
                        const void* q, const void* k, const void* v, const orc_fused* f,
                        int64_t n_rows, const int64_t* rows, double* out, double* lse,
                        int32_t n_threads);
/* Gradients of orc_attention (no fused steps) for the upstream gradient dout
 * ([T][H][d] in dtype): dq, dk, dv [T][H][d] fp64 (arrays must be offsets[0]-based
 * at 0).  Each (request, head) materialises its L x L probabilities.  Returns 0 or -1. */
int orc_attention_bwd(const orc_params* p, int32_t B, const int64_t* offsets, const int64_t* t,
                      const int8_t* ty, int32_t dtype, const void* q, const void* k, const void* v,
                      const void* dout, double* dq, double* dk, double* dv, int32_t n_threads);
/* Gradients of orc_attention_fused for the upstream gradient dout: dq, dk, dv, the
 * gate pre-activations' dq_gate, dk_gate, dout_gate ([T][H][d] fp64; zero for a gate
 * that is off) and the norm gains' dq_norm_w, dk_norm_w ([H][d], NULL to skip).
 * offsets[0] must be 0.  Returns 0 or -1. */
int orc_attention_bwd_fused(const orc_params* p, int32_t B, const int64_t* offsets, const int64_t* t,
                            const int8_t* ty, int32_t dtype, const void* q, const void* k, const void* v,
                            const orc_fused* f, const void* dout, double* dq, double* dk, double* dv,
                            double* dq_gate, double* dk_gate, double* dout_gate, double* dq_norm_w,
                            double* dk_norm_w, int32_t n_threads);
/* History compression: in request b the tokens [hist_begin[b], hist_begin[b] +
 * hist_len[b]) (time-ordered history) are replaced by sums of groups of consecutive
 * tokens; recency segment i (0 = newest) covers seg_len[i] tokens (< 0: the rest)
 * with groups of seg_group[i], the oldest group of a segment partial.  Merged tokens
 * keep time order, take the latest member time and type HIST.  x: [T][width] in dtype;
 * out_x fp64.  out arrays may be NULL (out_offsets too) to count.  Returns the total
 * output rows or -1. */
int64_t orc_compress(int32_t B, const int64_t* offsets, const int64_t* hist_begin, const int64_t* hist_len,
                     int32_t n_seg, const int64_t* seg_len, const int32_t* seg_group, int32_t dtype, int64_t width,
                     const void* x, const int64_t* t, const int8_t* ty, int64_t* out_offsets, double* out_x,
                     int64_t* out_t, int8_t* out_ty);
/* LazFormer Eq. 22 per-layer query budget N_l (round half away from zero);
 * -1 on invalid arguments. */
int64_t orc_query_keep(int64_t hist_len, int64_t n_min, int32_t layer, int32_t n_layers);
/* Rows of a pruned layer (sorted global indices): every non-user token and the last
 * `keep` user tokens of each request (keep < 0: all).  Returns the count. */
int64_t orc_kept_rows(int32_t B, const int64_t* offsets, const int8_t* ty, int64_t keep, int64_t* rows);
/* Tile classes (SKIP/PARTIAL/FULL) of every (q-tile, k-tile) pair of every
 * request, request-major then q-tile then k-tile; returns the count written.
 * cls may be NULL to query the count. */
int64_t orc_tile_classes(const orc_params* p, int32_t B, const int64_t* offsets,
                         const int64_t* t, const int8_t* ty, uint8_t* cls);

#ifdef __cplusplus
}
#endif
#endif
