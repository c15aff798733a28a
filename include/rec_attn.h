/*
 * rec_attn.h -- C-ABI of the GB300 (sm_103a) masked time-RoPE attention library.
 *
 * The library computes the forward pass of multi-head softmax attention over a
 * packed, jagged batch of request-centric token sequences
 *
 *     O_i = sum_j P_ij V_j,  P_ij = vis(i,j) exp(s_ij) / sum_j' vis(i,j') exp(s_ij'),
 *     s_ij = scale * < RoPE_t(Q_i, t_i), RoPE_t(K_j, t_j) >,
 *
 * with O_i = 0 when no key is visible.  Citations (page, section / equation):
 *   - softmax attention with an additive -inf mask: TM20K review page, section 2.1
 *     (full-attention equation); LazFormer review page, section 2.3, Eq. 19-21;
 *   - time-RoPE alpha_i(t) = t * phi_min / dt_max * base^(2i/d) on adjacent pairs of
 *     Q and K: CADET review page, section on time encoding and self-gating;
 *   - mask vis(i,j) from per-token timestamps and types: CADET delay rule
 *     M_ij = -inf if t_j > t_i - delta (section on masking the last hour), CADET
 *     candidate isolation (section on scoring hundreds of candidates in 50 ms),
 *     SORT U2U/C2U/C2C regions (section 3.1) and local attention (3.2.1), LazFormer
 *     Eq. 19-21, MTGR hybrid dynamic mask (MTGR notes on the blog index page);
 *   - packed jagged batch (one contiguous token buffer plus per-sequence start and
 *     end): CADET review page, training data engineering paragraph;
 *   - skipping fully masked blocks: CADET serving kernel and SORT section 4.1
 *     ("mask preload check").
 *
 * Mask predicate vis(i, j), for tokens i (query) and j (key) of the same request
 * (tokens of different requests never see each other; p = request-local position,
 * t = timestamp, U = {GLOBAL, HIST}):
 *   U    -> U   : hist_bidirectional ? 1 : p_j <= p_i and (window == 0 or either
 *                 token is GLOBAL or p_i - p_j < window)
 *   U    -> RT, CAND : 0
 *   RT   -> U   : 1;   RT -> RT : p_j <= p_i;   RT -> CAND : 0
 *   CAND -> U   : 1;   CAND -> RT : t_j < t_i;  CAND -> CAND : i == j
 *   use_delay   : every pair additionally needs t_j <= t_i - delay_s, except the
 *                 candidate self pair.
 * Time-RoPE: pair i (components 2i, 2i+1, i < d/2) turns by alpha_i(t) =
 * t * phi_min / dt_max_s * rope_base^(2i/d); Q_i and K_j are rotated at their own
 * timestamps (x' = x cos a - y sin a, y' = x sin a + y cos a).  The library
 * subtracts the first timestamp of each request in int64 before forming fp32
 * angles; scores depend only on time differences, so results are the same.
 *
 * Threading: functions are thread-safe for distinct plans.  All device work is
 * asynchronous on the stream passed in (a cudaStream_t given as void*; NULL =
 * legacy default stream) unless a function says it synchronizes.
 */
#ifndef REC_ATTN_H
#define REC_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define REC_ATTN_ABI_VERSION 1
#define REC_ATTN_TILE 128            /* tokens per tile (query and key side) */
#define REC_ATTN_MAX_REQUEST_LEN 262144 /* longest request a plan accepts */

typedef enum {
  REC_ATTN_OK = 0,
  REC_ATTN_ERR_INVALID_ARG = 1,   /* bad argument, detected on the host before any launch */
  REC_ATTN_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim, dtype, size) */
  REC_ATTN_ERR_CUDA = 3,          /* a CUDA runtime call failed (no GPU, launch error, ...) */
  REC_ATTN_ERR_OOM = 4,           /* device allocation failed */
  REC_ATTN_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out (device status) */
  REC_ATTN_ERR_DEVICE_INPUT = 6   /* device data out of range: type not in 0..3 or |t| >= 2^62 */
} rec_attn_status;

typedef enum { REC_ATTN_BF16 = 0, REC_ATTN_FP32 = 1 } rec_attn_dtype;

/* token types (int8 per token) */
enum { REC_ATTN_GLOBAL = 0, REC_ATTN_HIST = 1, REC_ATTN_RT = 2, REC_ATTN_CAND = 3 };

/* tile classes reported by rec_attn_tile_classes */
enum { REC_ATTN_TILE_SKIP = 0, REC_ATTN_TILE_PARTIAL = 1, REC_ATTN_TILE_FULL = 2 };

typedef struct {
  int32_t abi_version;        /* must be REC_ATTN_ABI_VERSION */
  int32_t num_heads;          /* H >= 1 */
  int32_t head_dim;           /* d: bf16 -> 64 or 128; fp32 -> 32 or 64 */
  int32_t dtype;              /* rec_attn_dtype; Q, K, V and O share it */
  int32_t use_delay;          /* 0/1: CADET delay rule */
  int64_t delay_s;            /* delta >= 0 seconds (CADET uses 3600) */
  int32_t window;             /* 0 = none; else user->user needs p_i - p_j < window */
  int32_t hist_bidirectional; /* 0/1: GLOBAL and HIST tokens fully mutually visible */
  int32_t use_rope;           /* 0/1: apply the time-RoPE to Q and K */
  double phi_min;             /* rad turned by the slowest pair over dt_max_s (1e-4) */
  double dt_max_s;            /* > 0, seconds (one year = 31536000) */
  double rope_base;           /* > 0 (6e5) */
  float softmax_scale;        /* > 0, or 0 for 1/sqrt(head_dim) */
} rec_attn_params;

typedef struct rec_attn_plan_s rec_attn_plan_t; /* opaque */

/*
 * rec_attn_plan -- validate a batch and build its attention plan.
 *
 * Arguments:
 *   params          mask / RoPE / shape parameters (copied).
 *   batch           number of requests B >= 0.
 *   offsets_host    host int64[B+1]: offsets[0] = 0, non-decreasing; request b owns
 *                   tokens [offsets[b], offsets[b+1]).  Read during the call only.
 *                   Must hold the same values as offsets_dev.
 *   offsets_dev     device int64[B+1], same values.
 *   timestamps_dev  device int64[T] seconds, T = offsets[B]; |t| < 2^62.
 *   types_dev       device int8[T], each in 0..3.
 *   stream          cudaStream_t the inputs are produced on.  The planning work (a
 *                   request-table upload and one kernel) runs on a library-owned stream
 *                   that first waits for `stream`; every later call on the plan orders
 *                   itself after that work, so a rec_attn_fwd on `stream` overlaps its
 *                   time-RoPE prologue with the planning kernel.
 *   plan_out        receives the plan.
 * The device arrays must stay valid and unchanged while the plan is used.  The
 * plan owns a device workspace (per-tile statistics, tile classes, per-query-tile
 * key-tile lists, the schedule and the rotated Q/K buffers), allocated in stream
 * order from a library-owned memory pool.  A plan depends only on the offsets,
 * timestamps, types and params, so one plan serves any number of rec_attn_fwd
 * calls (e.g. every layer of a model).
 * Errors: INVALID_ARG (bad params, offsets or NULL pointers; nothing launched),
 * UNSUPPORTED (head_dim/dtype combination, a request longer than
 * REC_ATTN_MAX_REQUEST_LEN, T >= 2^31), OOM, CUDA.  Invalid device values (types,
 * timestamps) are reported by rec_attn_device_status; the kernels never fault on
 * them.  On error *plan_out is NULL.
 */
rec_attn_status rec_attn_plan(const rec_attn_params* params, int32_t batch,
                              const int64_t* offsets_host, const int64_t* offsets_dev,
                              const int64_t* timestamps_dev, const int8_t* types_dev,
                              void* stream, rec_attn_plan_t** plan_out);

/*
 * rec_attn_plan_query_pruned -- rec_attn_plan for a layer that computes only some
 * queries (query pruning); every token stays a key.
 *
 *   keep_user_queries  -1: every query (same as rec_attn_plan).  N >= 0: in each
 *             request the computed queries are every token that is not a user token
 *             (REC_ATTN_RT, REC_ATTN_CAND) and the last N user tokens (REC_ATTN_GLOBAL,
 *             REC_ATTN_HIST) by position.  SORT review page, section 3.2.2 (Query
 *             Pruning cuts the user side, history and profile, layer by layer and never
 *             drops a candidate); LazFormer review page, Eq. 22 (the next layer keeps the
 *             most recent N_l history tokens and every target; rec_attn_query_keep gives
 *             N_l); N = 0 is target attention (only targets query the history, TM20K
 *             review page) and the candidate-only pass of M-FALCON serving.
 *
 * rec_attn_fwd on such a plan writes out (and lse) only at the computed rows; the rows
 * of pruned queries are left as they were.  Query tiles with no computed row are not
 * scheduled.  rec_attn_visible_pairs counts the pairs of computed rows only.  Tile
 * classes are those of the full mask.  Other arguments, errors and ownership as for
 * rec_attn_plan; INVALID_ARG also for keep_user_queries < -1.
 */
rec_attn_status rec_attn_plan_query_pruned(const rec_attn_params* params, int32_t keep_user_queries,
                                           int32_t batch, const int64_t* offsets_host,
                                           const int64_t* offsets_dev, const int64_t* timestamps_dev,
                                           const int8_t* types_dev, void* stream,
                                           rec_attn_plan_t** plan_out);

/*
 * rec_attn_query_keep -- LazFormer Eq. 22: user queries kept at layer `layer`
 * (1-based) of an `n_layers`-layer stack, N_l = min(hist_len, max(n_min,
 * Round[hist_len - (layer - 1) / (n_layers - 1) * (hist_len - n_min)])), Round to the
 * nearest integer with halves away from zero (computed exactly in integers).  One
 * layer keeps hist_len.  Host-only, no CUDA call.  Returns -1 for negative lengths,
 * n_layers < 1 or layer outside 1..n_layers.  (The page's defaults: 1152 compressed
 * history tokens, n_min = 128.)
 */
int64_t rec_attn_query_keep(int64_t hist_len, int64_t n_min, int32_t layer, int32_t n_layers);

/*
 * rec_attn_fwd -- attention forward for a planned batch.
 *
 *   q, k, v   device [T][H][d] row-major, contiguous, in params->dtype (bf16 bit
 *             patterns or fp32), 16-byte aligned, finite.
 *   out       device [T][H][d] in params->dtype; every row is written (rows that see
 *             no key get zeros).  May not alias q, k or v.  A 32-byte aligned out is
 *             written with 32-byte stores (whole sectors), a 16-byte aligned one with
 *             16-byte stores; the values are the same.
 *   lse       optional device float[T][H]: natural-log sum of exp(scaled scores) over
 *             visible keys, -inf for rows that see no key; NULL to skip.
 *   stream    cudaStream_t for the launches.
 * Errors: INVALID_ARG (NULL plan or pointers, misalignment, aliasing), CUDA.
 * Asynchronous: returns after enqueueing.  Launch-time anomalies inside kernels
 * (a timed-out wait) are reported by rec_attn_device_status.
 */
rec_attn_status rec_attn_fwd(rec_attn_plan_t* plan, const void* q, const void* k,
                             const void* v, void* out, float* lse, void* stream);

/*
 * Fused prologue / epilogue steps of rec_attn_fwd_fused.  Each pointer may be NULL,
 * which turns that step off; a struct of NULLs computes what rec_attn_fwd computes.
 *
 *   QK-RMSNorm (SORT review page, section 3.3.2 "Attention Gate & QK Norm"; TM20K
 *   review page, the QK Norm after the query/key projections): every query and key
 *   head vector x becomes x / sqrt(mean(x^2) + norm_eps) * w[h], w a device
 *   float[H][d] gain (q_norm_weight, k_norm_weight), 4-byte aligned.
 *
 *   Q / K sigmoid gates (CADET review page, section on time encoding and
 *   self-gating: a per-dimension coefficient in (0, 1) multiplied onto the
 *   projected Q and K): x <- x * sigmoid(g), g a device [T][H][d] array of gate
 *   pre-activations in params->dtype (q_gate, k_gate), 16-byte aligned.
 *
 *   Order on Q and K: norm, then gate, then the time-RoPE (if params->use_rope).
 *
 *   Attention output gate (SORT section 3.3.2): O <- O * sigmoid(g), g = out_gate,
 *   a device [T][H][d] array in params->dtype, 16-byte aligned, not aliasing out.
 *
 * Arithmetic is fp32; Q' and K' are rounded once to params->dtype.
 */
typedef struct {
  const float* q_norm_weight; /* [H][d] or NULL */
  const float* k_norm_weight; /* [H][d] or NULL */
  float norm_eps;             /* >= 0 (e.g. 1e-6) */
  const void* q_gate;         /* [T][H][d] or NULL */
  const void* k_gate;         /* [T][H][d] or NULL */
  const void* out_gate;       /* [T][H][d] or NULL */
} rec_attn_fused;

/*
 * rec_attn_fwd_fused -- rec_attn_fwd with the fused steps above.  Arguments, layout
 * and asynchrony as for rec_attn_fwd; `fused` is read on the host during the call.
 * When a Q/K step is on and the plan was made without the RoPE, the first such call
 * takes 2 * T * H * d elements of Q'/K' workspace from the library's memory pool on
 * `stream` (released with the plan).
 * Errors: INVALID_ARG (those of rec_attn_fwd, NULL fused, negative or non-finite
 * norm_eps, misaligned weights or gates, out_gate aliasing out), CUDA, OOM.
 */
rec_attn_status rec_attn_fwd_fused(rec_attn_plan_t* plan, const void* q, const void* k,
                                   const void* v, const rec_attn_fused* fused, void* out,
                                   float* lse, void* stream);

/*
 * rec_attn_bwd -- gradients of rec_attn_fwd with respect to q, k and v, for the
 * upstream gradient dout (training: the TM20K and LazFormer review pages train these
 * models end to end; the pages print no backward formula, so this is the derivative
 * of the forward's definition).
 *
 *   q, k, v   the forward's inputs (the time-RoPE is applied again inside).
 *   out, lse  the forward's output and log-sum-exp (lse is required here).
 *   dout      device [T][H][d] in params->dtype: dLoss/dout.
 *   dq, dk, dv  device [T][H][d] in params->dtype, written in full; they may not
 *             alias any input or each other.  All tensors 16-byte aligned; dq, dk
 *             and dv 32-byte aligned are written with 32-byte stores (same values).
 * The plan must be the forward's (same offsets, times, types, params).  On a
 * query-pruned plan (rec_attn_plan_query_pruned) the gradients are those of the
 * computed rows' outputs: pruned queries have no output, so their out and lse rows
 * are never read, their dout rows are ignored (they must still be finite: they pass
 * through the tensor cores with zero weights), their dq rows are zero and they add
 * nothing to dk and dv.
 * Supported: bf16 with head_dim 64 or 128, fp32 with
 * head_dim 32 or 64 (else UNSUPPORTED).  The first call takes workspace from the
 * library pool on `stream` (released with the plan): for bf16 the per-plan item
 * schedule (96 B per tile and head, 4 B per tile pair) and the rows' constants
 * (8 B per tile row and head); for fp32 T * H floats.  bf16: tensor cores (bf16
 * operands, fp32 accumulation; P and dS rounded to bf16 for their MMAs, as in the
 * forward's P); fp32: CUDA cores in fp32.  Gradients are rounded once to
 * params->dtype.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA, OOM.
 */
rec_attn_status rec_attn_bwd(rec_attn_plan_t* plan, const void* q, const void* k, const void* v,
                             const void* out, const float* lse, const void* dout, void* dq, void* dk,
                             void* dv, void* stream);

/*
 * rec_attn_bwd_fused -- gradients of rec_attn_fwd_fused: dq, dk, dv and those of the
 * fused steps' inputs, for the upstream gradient dout (SORT review page, section
 * 3.3.2; TM20K review page, QK Norm; CADET review page, self-gating).  The chain rule
 * runs through the output gate (dA = dout * sigmoid(c_o), dc_o = dout * out *
 * (1 - sigmoid(c_o))), the attention backward of rec_attn_bwd, the rotation, the Q/K
 * gates (dc = dg * n * sigmoid'(c)) and the QK-RMSNorm (the gains' gradients summed
 * over every token).
 *   fused    the forward's rec_attn_fused (same pointers or the same values).
 *   out, lse the forward's output (gated) and log-sum-exp; dout, dq, dk, dv as for
 *            rec_attn_bwd.
 *   grads    dq_gate, dk_gate, dout_gate: device [T][H][d] in params->dtype, required
 *            for each gate that is on; dq_norm_weight, dk_norm_weight: device float
 *            [H][d], required for each norm that is on (overwritten, not accumulated).
 * Scratch from the library pool on `stream`: one [T][H][d] array per output gate and
 * per side (Q, K) with a step on.  Supported as for rec_attn_bwd.
 * Errors: those of rec_attn_bwd; INVALID_ARG also for a missing gradient of a step that
 * is on, misaligned gates or gradients, a gradient aliasing an input.
 */
typedef struct {
  void* dq_gate;          /* [T][H][d] or NULL (q gate off) */
  void* dk_gate;          /* [T][H][d] or NULL */
  void* dout_gate;        /* [T][H][d] or NULL */
  float* dq_norm_weight;  /* [H][d] or NULL (q norm off) */
  float* dk_norm_weight;  /* [H][d] or NULL */
} rec_attn_fused_grads;
rec_attn_status rec_attn_bwd_fused(rec_attn_plan_t* plan, const void* q, const void* k, const void* v,
                                   const rec_attn_fused* fused, const void* out, const float* lse,
                                   const void* dout, void* dq, void* dk, void* dv,
                                   const rec_attn_fused_grads* grads, void* stream);

/*
 * History compression (LazFormer review page, Eq. 16-18 and Table 6; TM20K review page,
 * PATM and LPTM): in request b the history rows [hist_begin[b], hist_begin[b] +
 * hist_len[b]) (request-local, time-ordered) are replaced by sums of groups of
 * consecutive rows.  Recency segment i (i = 0 the newest) covers the next seg_len[i]
 * history rows going back in time (seg_len[i] < 0: all the rest) in groups of
 * seg_group[i] >= 1; the oldest group of a segment is the partial one.  The segments
 * must cover every history (an unbounded one does).  Output rows keep time order:
 * the rows before the history, the merged groups (oldest first; timestamp = the latest
 * member's, type REC_ATTN_HIST), the rows after it.  Examples: LazFormer "keep 1024,
 * groups of 8" is {(1024, 1), (-1, 8)}; LPTM is {(-1, 2)}; PATM's four position bands
 * are {(1000, 1), (4000, 2), (5000, 3), (-1, 4)}.  At most 8 segments.
 *
 * rec_attn_compress_lengths -- host only: out_offsets_host[0..batch] of the output.
 * rec_attn_compress -- x: device [T][width] rows in dtype (width * element size a
 *   multiple of 16 bytes, 16-byte aligned); timestamps int64 [T], types int8 [T];
 *   x_out / timestamps_out / types_out: device outputs sized by the lengths above (x_out
 *   may not overlap x).  Sums in fp32, rounded once.  offsets, hist ranges and segments
 *   are host arrays read during the call; a small request table is staged through the
 *   library pool on `stream`.  Asynchronous.
 * Errors: INVALID_ARG (negative or inconsistent ranges, uncovered history, bad segments,
 * alignment, NULL pointers), CUDA.
 */
rec_attn_status rec_attn_compress_lengths(int32_t batch, const int64_t* offsets_host,
                                          const int64_t* hist_begin_host, const int64_t* hist_len_host,
                                          int32_t n_segments, const int64_t* seg_len,
                                          const int32_t* seg_group, int64_t* out_offsets_host);
rec_attn_status rec_attn_compress(int32_t batch, const int64_t* offsets_host,
                                  const int64_t* hist_begin_host, const int64_t* hist_len_host,
                                  int32_t n_segments, const int64_t* seg_len, const int32_t* seg_group,
                                  int32_t dtype, int64_t width, const void* x, const int64_t* timestamps,
                                  const int8_t* types, void* x_out, int64_t* timestamps_out,
                                  int8_t* types_out, void* stream);

/*
 * rec_attn_fwd_compress -- rec_attn_fwd whose output is written already compressed:
 * the history compression above (same segments, hist_begin / hist_len per request, same
 * output layout, times and types) applied to the attention output O, fused into the
 * attention epilogue, so O itself never reaches memory (TM20K review page, LPTM and PATM
 * compress the history between layers; LazFormer review page, Eq. 16-18, the
 * compressed history feeds the next layer).  Each output row is the fp32 sum of its
 * group's O rows (each already normalised), rounded once to bf16.
 *   plan         a bf16 plan made by rec_attn_plan (not query-pruned: every row is
 *                needed); its offsets are the compression's request offsets.
 *   q, k, v      as for rec_attn_fwd.
 *   hist_begin_host, hist_len_host, n_segments, seg_len, seg_group: as for
 *                rec_attn_compress; every group size at most 32.
 *   x_out        device [rows_out][H][d] bf16 (rows_out from rec_attn_compress_lengths),
 *                16-byte aligned, not overlapping q, k, v; timestamps_out int64
 *                [rows_out], types_out int8 [rows_out].
 * Groups that straddle a 32-row block boundary pass their two partial sums through an
 * fp32 fix-up buffer (from the library pool on `stream`, 2 * H * d * 4 bytes per 32
 * tokens) and a second kernel; the result is deterministic.
 * Errors: INVALID_ARG (those of rec_attn_compress and rec_attn_fwd), UNSUPPORTED (fp32
 * or query-pruned plan, a group larger than 32), OOM, CUDA.  Asynchronous.
 */
rec_attn_status rec_attn_fwd_compress(rec_attn_plan_t* plan, const void* q, const void* k, const void* v,
                                      const int64_t* hist_begin_host, const int64_t* hist_len_host,
                                      int32_t n_segments, const int64_t* seg_len, const int32_t* seg_group,
                                      void* x_out, int64_t* timestamps_out, int8_t* types_out, void* stream);

/*
 * rec_attn_check_wait_timeout -- self-check of the failure detection inside the
 * pipelined kernels (the pages have no counterpart: it guards this implementation).
 * Every wait of a kernel on an mbarrier is bounded; on expiry it records
 * REC_ATTN_ERR_TIMEOUT in the status word and the CTA stops instead of hanging.  This
 * call runs the same wait on a barrier that nothing arrives at, with a limit of
 * limit_ms (1..10000), and returns the status word the kernel wrote in *status_out
 * (REC_ATTN_ERR_TIMEOUT when the mechanism works).  The device stays usable.
 * Synchronizes `stream`.  Errors: INVALID_ARG, CUDA.
 */
rec_attn_status rec_attn_check_wait_timeout(uint32_t limit_ms, int32_t* status_out, void* stream);

/*
 * rec_attn_free -- release a plan (NULL-safe).  The workspace returns to the
 * library pool in stream order on the stream of the plan's last use (after the
 * planning work), so work already enqueued there may still run; callers that used
 * other streams must synchronize them first.
 */
void rec_attn_free(rec_attn_plan_t* plan);

/*
 * rec_attn_tile_classes -- copy the plan's tile classes to host memory.
 * Order: request-major, then query tile, then key tile (n_tiles(b)^2 entries per
 * request, n_tiles(b) = ceil(len_b / 128)); values REC_ATTN_TILE_*.  SKIP: no
 * visible pair; FULL: every (query, key) pair of the tile visible and the key
 * tile complete (128 keys); PARTIAL otherwise.  Classes come from per-type bounding
 * boxes of positions and timestamps in each tile, so PARTIAL is conservative.
 * *n_needed receives the count; host_out may be NULL to query it.  Synchronizes
 * the plan's stream.  Errors: INVALID_ARG (NULL plan/n_needed, capacity too
 * small), CUDA.
 */
rec_attn_status rec_attn_tile_classes(rec_attn_plan_t* plan, uint8_t* host_out,
                                      size_t capacity, size_t* n_needed);

/*
 * rec_attn_visible_pairs -- exact number of visible (query, key) pairs of the batch
 * (per head), counted on the device.  Used for FLOP accounting (4 * d * H * pairs).
 * Synchronizes the plan's stream.  Errors: INVALID_ARG, CUDA.
 */
rec_attn_status rec_attn_visible_pairs(rec_attn_plan_t* plan, uint64_t* host_out);

/*
 * Serving with a cached history (M-FALCON, HSTU notes on the blog index page: the
 * history's keys and values are computed once per user and every micro-batch of
 * candidates is scored against them; CADET review page, scoring hundreds of
 * candidates per request within its latency budget).
 *
 * rec_attn_cache_create -- cache the rotated history keys K', the values V, times and
 * types of a batch of requests, with room for up to max_cands candidates each.
 *   params           as for rec_attn_plan (copied).
 *   batch            requests B >= 1.
 *   hist_offsets_host host int64[B+1]: history rows [offsets[b], offsets[b+1]) of
 *                    request b in the packed inputs below (offsets[0] = 0); read
 *                    during the call.  A history may be empty.
 *   hist_t_dev       device int64[Th] times; hist_types_dev device int8[Th], user-side
 *                    types (REC_ATTN_GLOBAL, REC_ATTN_HIST, REC_ATTN_RT).
 *   k_hist, v_hist   device [Th][H][d] in params->dtype, 16-byte aligned; read during
 *                    the call's stream work only (the cache keeps its own copies).
 *   max_cands        candidate slots per request (>= 1).
 *   stream           cudaStream_t of the work; cache_out receives the cache.
 * The cache owns one device buffer from the library pool: for each request
 * hist_len + max_cands rows of Q', K', V and O, their times and types, and lse.
 * Errors: INVALID_ARG (params, offsets, NULL or misaligned pointers), UNSUPPORTED
 * (a request longer than REC_ATTN_MAX_REQUEST_LEN with its slots, 2^31 rows), OOM,
 * CUDA.  On error *cache_out is NULL.
 *
 * rec_attn_cache_score -- score one micro-batch of candidates per request against
 * the cached history.  Candidate c of request b gets the attention output over
 * [history of b, c] under the mask predicate above (it sees the history rows the
 * predicate allows and itself; CAND -> CAND is self only, so the other candidates of
 * the micro-batch do not change it).
 *   cand_offsets_host host int64[B+1]: candidates [offsets[b], offsets[b+1]) belong to
 *                    request b, at most max_cands each; read during the call.
 *   cand_t_dev       device int64[Nc] candidate times (type REC_ATTN_CAND).
 *   q_cand, k_cand, v_cand device [Nc][H][d] in params->dtype, 16-byte aligned.
 *   out              device [Nc][H][d], written in full (rows that see no key: 0);
 *                    may not alias the inputs.  lse: optional device float[Nc][H].
 * The candidates are rotated against the same per-request reference time as the
 * cached history (its first row; the first candidate when the history is empty),
 * written into the cache's slots (unused slots padded), and one target-attention
 * pass runs over the cached rows.  Calls on one cache must not overlap on the GPU
 * (they share the slots).  A small table is staged through the library pool on
 * `stream`, and each call plans on the library's side stream as rec_attn_plan does.
 * Errors: INVALID_ARG (NULL cache or pointers, misalignment, aliasing, more than
 * max_cands candidates, another current device), OOM, CUDA.  Asynchronous.
 *
 * rec_attn_cache_free -- release a cache (NULL-safe).  Synchronizes the device
 * (cudaFree), so work still reading the cache completes first.
 */
typedef struct rec_attn_kv_cache_s rec_attn_kv_cache_t; /* opaque */
rec_attn_status rec_attn_cache_create(const rec_attn_params* params, int32_t batch,
                                      const int64_t* hist_offsets_host, const int64_t* hist_t_dev,
                                      const int8_t* hist_types_dev, const void* k_hist, const void* v_hist,
                                      int32_t max_cands, void* stream, rec_attn_kv_cache_t** cache_out);
rec_attn_status rec_attn_cache_score(rec_attn_kv_cache_t* cache, const int64_t* cand_offsets_host,
                                     const int64_t* cand_t_dev, const void* q_cand, const void* k_cand,
                                     const void* v_cand, void* out, float* lse, void* stream);
void rec_attn_cache_free(rec_attn_kv_cache_t* cache);

/*
 * rec_attn_applied_masks -- diagnostic copy of the visibility bits the attention
 * kernels apply, for named (query tile, key tile) pairs of a plan, so that a test can
 * hold them bit for bit against the mask predicate above (the pages' rule that masked
 * pairs get -inf, not a small constant: LazFormer review page, section 2.3, Eq. 19-21;
 * CADET delay rule; SORT section 3.1; MTGR hybrid mask).
 *
 *   n_pairs       number of pairs (>= 0).
 *   pairs_host    host int32[n_pairs][3]: (request b, query tile qt, key tile kt),
 *                 tiles numbered from 0 within request b (qt, kt < ceil(len_b / 128)).
 *   mode          0: what rec_attn_fwd's tensor-core kernel (bf16) applies: the plan's
 *                 mask-table rows where the pair has a table slot, the kernel's own row
 *                 construction otherwise;
 *                 1: the kernel's row construction for every PARTIAL pair (what a pair
 *                 beyond the table's capacity, and rec_attn_fwd_noalloc, apply);
 *                 2: the per-pair predicate of the CUDA-core kernels (fp32 path).
 *   bits_host     host uint32[n_pairs][128][4]: for query row r of the tile (request-
 *                 local position 128 qt + r), bit (c % 32) of word c / 32 is 1 when key
 *                 c of the key tile (position 128 kt + c) enters the row's softmax.  A
 *                 pair absent from the query tile's key-tile list (SKIP, or a tile of
 *                 pruned queries) is never loaded: all zero.  A FULL pair takes no mask:
 *                 all one.  Rows past the request end are zero except in FULL pairs
 *                 (computed and discarded).
 *   list_class_host  optional host uint8[n_pairs]: the class in the list entry
 *                 (REC_ATTN_TILE_*, 0xff when the pair is not listed).
 *   slot_host     optional host int32[n_pairs]: the pair's mask-table slot (-1: none).
 * Takes a temporary buffer from the library pool on the plan's stream and
 * synchronizes it.  Errors: INVALID_ARG (NULL plan or arrays, mode, a pair outside
 * the plan), OOM, CUDA.
 */
rec_attn_status rec_attn_applied_masks(rec_attn_plan_t* plan, int32_t n_pairs, const int32_t* pairs_host,
                                       int32_t mode, uint32_t* bits_host, uint8_t* list_class_host,
                                       int32_t* slot_host);

/*
 * rec_attn_device_status -- status word the plan's kernels wrote (REC_ATTN_OK,
 * REC_ATTN_ERR_DEVICE_INPUT or REC_ATTN_ERR_TIMEOUT; the first error wins).
 * Synchronizes the plan's stream.  Errors: INVALID_ARG, CUDA.
 */
rec_attn_status rec_attn_device_status(rec_attn_plan_t* plan, int32_t* status_out);

/* Kernel timings of the most recent rec_attn_fwd on a plan with timing enabled. */
typedef struct {
  float rope_ms;  /* time-RoPE prologue (0 when use_rope == 0) */
  float attn_ms;  /* attention kernel */
} rec_attn_timings;

/*
 * rec_attn_enable_timing -- from now on, rec_attn_fwd records CUDA events on its
 * stream around each kernel it launches (the events are owned by the plan).
 * Errors: INVALID_ARG (NULL plan), CUDA.
 */
rec_attn_status rec_attn_enable_timing(rec_attn_plan_t* plan);

/*
 * rec_attn_read_timings -- elapsed times of the last timed rec_attn_fwd; waits for
 * its events.  Errors: INVALID_ARG (NULL arguments, timing not enabled or no timed
 * call yet), CUDA.
 */
rec_attn_status rec_attn_read_timings(rec_attn_plan_t* plan, rec_attn_timings* out);

/*
 * rec_attn_fwd_noalloc -- plan + time-RoPE + attention in one call that allocates
 * no device memory.  The pages have no counterpart to this entry point: it exists
 * for callers that cannot call cudaMalloc, such as a process whose inference
 * runtime has reserved the GPU's memory for its own allocator and forbids other
 * allocations, or a serving loop that cannot afford cudaMalloc's latency and
 * implicit synchronisation on every request.
 *
 * Arguments mean what they mean for rec_attn_plan and rec_attn_fwd; the result is
 * the one those two calls produce.  All per-call workspace lives in one static
 * device array of REC_ATTN_NOALLOC_SCRATCH_BYTES that every GPU which loads the
 * library holds until the process exits.  A batch whose workspace does not fit
 * (request table, tile statistics and classes, key-tile lists, schedule and, with
 * the RoPE on, two rotated copies of the [T][H][d] Q/K) is rejected with
 * REC_ATTN_ERR_UNSUPPORTED before any work is enqueued; REC_ATTN_ERR_INVALID_ARG
 * as for rec_attn_plan / rec_attn_fwd.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  Every call shares the one array and leaves its contents
 * behind, so calls whose GPU work overlaps (other streams, other host threads)
 * race and must be serialised by the caller.  Device-side input errors are not
 * reported by this entry point (the plan-based API reports them).
 */
#define REC_ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
rec_attn_status rec_attn_fwd_noalloc(const rec_attn_params* params, int32_t batch,
                                     const int64_t* offsets_host, const int64_t* offsets_dev,
                                     const int64_t* timestamps_dev, const int8_t* types_dev,
                                     const void* q, const void* k, const void* v, void* out,
                                     float* lse, void* stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* rec_attn_status_string(rec_attn_status status);

#ifdef __cplusplus
}
#endif
#endif /* REC_ATTN_H */
