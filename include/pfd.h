/*
 * pfd.h -- C ABI of libpfd: sparse chunked-KV prefill and static-KV decode
 * attention for diffusion language models, on one NVIDIA GB300 (sm_103a).
 *
 * The method is the one of "Prefilling-dLLM: Predictive Prefilling for
 * Long-Context Inference in Diffusion Language Models" (technical summary):
 *   Methodology 1, "Chunked Prefill and KV Caching"   -> pfd_chunk_prefill,
 *                                                        pfd_select_chunks
 *   Methodology 2, "Two-Level Sparsity"                -> the top-B inside
 *                                                        pfd_chunk_prefill and
 *                                                        the top-K selection
 *   Methodology 3, "Decoding with Static KV Reuse" and
 *   "Attention Kernel Optimization" (split-KV, LSE merge) -> pfd_decode_attention,
 *                                                        pfd_decode_partial,
 *                                                        pfd_lse_merge
 *
 * Conventions shared by every call:
 *   - Tensors are token-major and contiguous: a [rows, heads, D] tensor keeps
 *     the D values of one (row, head) together, heads of a row together.
 *   - bf16 values are passed as raw 16-bit patterns (pfd_bf16).
 *   - Every pointer named as device memory must be CUDA device memory on the
 *     current device; the caller owns all memory.  The library allocates
 *     nothing and keeps no state between calls other than process-wide
 *     caches: the device's SM count, the TMA encoder entry point, and a
 *     bounded table of encoded TMA tensor maps keyed by (address, shape, box),
 *     so repeated calls on the same buffers do not re-encode them.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream).  The return value reports only what the host can check:
 *     invalid arguments (PFD_ERR_INVALID_ARG), shapes outside the supported
 *     set (PFD_ERR_UNSUPPORTED) and CUDA failures (PFD_ERR_CUDA).  Nothing is
 *     launched when a call returns PFD_ERR_INVALID_ARG or PFD_ERR_UNSUPPORTED,
 *     or fails to encode a TMA tensor map.  A call made of several kernels
 *     that returns PFD_ERR_CUDA from a later launch may have queued the
 *     earlier ones; its outputs are then undefined.
 *   - Errors found in device-resident data (a chunk-table entry, a selected
 *     index or a pool slot out of range) never trap: the offending item is
 *     skipped and a PFD_DEVERR_* bit is OR-ed into *dev_err when dev_err is
 *     not NULL.  The kernels wait on nothing outside their own thread block,
 *     and every internal pipeline wait is bounded (PFD_DEVERR_TIMEOUT).
 *   - PFD_DEVERR_TIMEOUT means a pipeline stage stopped making progress.  The
 *     thread block that saw it leaves its loop without draining the tensor
 *     copies and tensor-core operations it had in flight, so the outputs of
 *     that call are undefined and the CUDA context must be treated as
 *     unusable afterwards (destroy it); it only bounds how long a broken
 *     launch can occupy the GPU.
 *   - Calls are thread-safe; calls on one stream run in order.
 */
#ifndef PFD_H_
#define PFD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PFD_ABI_VERSION 2

typedef enum {
  PFD_OK = 0,
  PFD_ERR_INVALID_ARG = 1,
  PFD_ERR_UNSUPPORTED = 2,
  PFD_ERR_CUDA = 3
} pfd_status;

/* Device-side error bits (OR-ed into *dev_err). */
#define PFD_DEVERR_TABLE 1   /* chunk-table entry outside [0, pool_rows]      */
#define PFD_DEVERR_SEL 2     /* selected chunk index outside [0, table_len)   */
#define PFD_DEVERR_SLOT 4    /* slot_row[j] + B + 1 outside [0, pool_rows]    */
#define PFD_DEVERR_TIMEOUT 8 /* an internal pipeline wait ran out of budget    */
#define PFD_DEVERR_SHAPE 16  /* device cu_lq / cu_k disagree with host sizes   */
#define PFD_DEVERR_LABEL 32  /* a label outside [0, vocab)                     */

typedef uint16_t pfd_bf16; /* raw bfloat16 bits */

/* Where one chunk's cached rows live in the pool: rows row .. row+len-1. */
typedef struct {
  int32_t row;
  int32_t len;
} pfd_chunk_entry;

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* pfd_stream_t;

/* Supported shapes: head_dim D in {64, 128}; Hq a multiple of Hkv with
 * Hq / Hkv <= 128; window W <= 256 and W * (Hq / Hkv) <= 512; chunk size
 * 1 <= C <= 8192; 0 <= B <= C; at most 511 selected chunks per sequence. */

/*
 * Workspace bytes pfd_chunk_prefill needs for these sizes (device memory,
 * 256-byte aligned, contents need not be initialised).
 */
size_t pfd_chunk_prefill_workspace(int N, int C, int W, int Hq, int Hkv, int D, int B);

/*
 * Chunked prefill of one request: Methodology 1 ("Chunked Prefill and KV
 * Caching") and the intra-chunk half of Methodology 2 ("Two-Level Sparsity").
 *
 * The prefix is N chunks of C tokens; chunk j occupies rows j*(C+1) ..
 * j*(C+1)+C of q/k/v, its row j*(C+1) being the BOS row put in front of it.
 * For every chunk and query head h (KV head h / (Hq/Hkv)):
 *   out   = softmax(sm_scale * Q K^T) V over the chunk's own C+1 rows only
 *           (bidirectional, no cross-chunk keys);
 *   scores[j][t] = sum over the W window rows and all Hq heads of the
 *           window row's softmax probability of chunk row t, the softmax
 *           taken over the chunk's C+1 keys (the cumulative attention weight
 *           row t receives from the query tokens);
 *   kept_idx[j] = the B content tokens (t = 1..C, reported as t-1) with the
 *           largest fp32 score, ties to the lower index, in ascending order;
 *   pool rows slot_row[j] .. slot_row[j]+B get the K and V rows of BOS and of
 *           the kept tokens, in that order (all heads of a row together);
 *   table[j] = {slot_row[j], B+1}.
 *
 * Arguments (device memory unless stated):
 *   q            [N*(C+1), Hq, D]  bf16
 *   k, v         [N*(C+1), Hkv, D] bf16
 *   q_win        [W, Hq, D] bf16 query-window rows (may be NULL when W == 0;
 *                W == 0 gives all-zero scores and keeps t = 0..B-1)
 *   sm_scale     softmax scale; <= 0 selects 1/sqrt(D)
 *   out          [N*(C+1), Hq, D] bf16 (written)
 *   scores       [N, C+1] fp32 (written; column 0 is BOS)
 *   kept_idx     [N, B] int32 (written)
 *   pool_k/v     [pool_rows, Hkv, D] bf16 (rows of the N slots written)
 *   slot_row     [N] int32, first pool row of each chunk's slot; slots of
 *                B+1 rows must not overlap (not checked)
 *   table        [N] pfd_chunk_entry (written)
 *   dev_err      one int32, or NULL
 *   workspace    >= pfd_chunk_prefill_workspace(...) bytes
 *
 * Chunks are independent: calling this once per range of chunks, with q, k,
 * v, out, scores, kept_idx, slot_row and table offset to the range, and the
 * same q_win and pool, gives the bits of one call.  A caller may use this to
 * overlap the upload of later chunks with the prefill of earlier ones.
 */
pfd_status pfd_chunk_prefill(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                             const pfd_bf16* q_win, int N, int C, int W, int Hq, int Hkv, int D,
                             int B, float sm_scale, pfd_bf16* out, float* scores,
                             int32_t* kept_idx, pfd_bf16* pool_k, pfd_bf16* pool_v,
                             int64_t pool_rows, const int32_t* slot_row, pfd_chunk_entry* table,
                             int32_t* dev_err, void* workspace, size_t workspace_bytes,
                             pfd_stream_t stream);

/*
 * The prefill of L layers of one request in one call (Methodology 1,
 * "Chunked Prefill and KV Caching": every layer caches the KV of its chunks;
 * one pool per layer).  Layer l is exactly pfd_chunk_prefill over layer l's
 * tensors into layer l's pool; the layers run together, so each kernel
 * (chunk attention with the window statistics, window scores, top-B with
 * compaction) is launched once for all layers.
 *   q [L, N*(C+1), Hq, D], k, v [L, N*(C+1), Hkv, D] bf16 (layers stacked)
 *   q_win [L, W, Hq, D] bf16 (each layer's query-window rows)
 *   out [L, N*(C+1), Hq, D]; scores [L, N, C+1]; kept_idx [L, N, B]
 *   pool_k, pool_v [L, pool_rows, Hkv, D]: layer l's pool is rows
 *       l*pool_rows .. of the stacked buffers
 *   slot_row [N]: the slot of chunk j in every layer's pool
 *   table [L, N]: layer l's table (rows relative to layer l's pool)
 *   workspace >= pfd_chunk_prefill_layers_workspace(...) bytes
 * Limits as for pfd_chunk_prefill, with L * N * (C+1) < 2^31 rows.
 */
size_t pfd_chunk_prefill_layers_workspace(int L, int N, int C, int W, int Hq, int Hkv, int D,
                                          int B);

pfd_status pfd_chunk_prefill_layers(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                                    const pfd_bf16* q_win, int L, int N, int C, int W, int Hq,
                                    int Hkv, int D, int B, float sm_scale, pfd_bf16* out,
                                    float* scores, int32_t* kept_idx, pfd_bf16* pool_k,
                                    pfd_bf16* pool_v, int64_t pool_rows, const int32_t* slot_row,
                                    pfd_chunk_entry* table, int32_t* dev_err, void* workspace,
                                    size_t workspace_bytes, pfd_stream_t stream);

/*
 * The prefill of L requests of one shape (N, C, W, B, heads) in one call,
 * their slots in one shared pool (Methodology 1, "Chunked Prefill and KV
 * Caching": each request's chunks are processed on their own and cached;
 * Methodology 3, "Decoding with Static KV Reuse": a batch of requests decodes
 * from one pool through one chunk table).  Request l is exactly
 * pfd_chunk_prefill over request l's tensors with slot_row[l] and table[l]
 * into the shared pool; the requests run together, so each kernel is
 * launched once for the batch.
 *   q [L, N*(C+1), Hq, D], k, v [L, N*(C+1), Hkv, D] bf16 (requests stacked)
 *   q_win [L, W, Hq, D] bf16 (each request's query-window rows)
 *   out [L, N*(C+1), Hq, D]; scores [L, N, C+1]; kept_idx [L, N, B]
 *   pool_k, pool_v [pool_rows, Hkv, D]: the one pool
 *   slot_row [L, N]: first pool row of request l's chunk j; the L*N slots of
 *       B+1 rows must not overlap (not checked); a slot outside the pool
 *       raises PFD_DEVERR_SLOT and gets an empty table entry
 *   table [L, N]: rows absolute in the pool (so a batched decode reads it
 *       directly when the requests' table ranges are laid out in this order)
 *   workspace >= pfd_chunk_prefill_layers_workspace(L, N, C, W, Hq, Hkv, D,
 *       B) bytes
 * Limits as for pfd_chunk_prefill, with L * N * (C+1) < 2^31 rows.
 */
pfd_status pfd_chunk_prefill_batch(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                                   const pfd_bf16* q_win, int L, int N, int C, int W, int Hq,
                                   int Hkv, int D, int B, float sm_scale, pfd_bf16* out,
                                   float* scores, int32_t* kept_idx, pfd_bf16* pool_k,
                                   pfd_bf16* pool_v, int64_t pool_rows, const int32_t* slot_row,
                                   pfd_chunk_entry* table, int32_t* dev_err, void* workspace,
                                   size_t workspace_bytes, pfd_stream_t stream);

/*
 * pfd_chunk_prefill under the two other readings of the intra-chunk ranking
 * (Methodology 2, "Two-Level Sparsity": tokens are ranked by the cumulative
 * attention weight they receive from the query tokens).  Arguments as in
 * pfd_chunk_prefill, plus:
 *   per_kv_head  0: one ranking per chunk (scores [N, C+1], kept_idx [N, B]),
 *                   as pfd_chunk_prefill;
 *                1: one ranking per chunk and KV head: scores[j][g][t] sums
 *                   the window probabilities over the query heads of KV head
 *                   g only (scores [N, Hkv, C+1]), kept_idx [N, Hkv, B], and
 *                   KV head g's column of chunk j's pool slot holds head g's
 *                   BOS row and head g's kept rows (the slot and the table
 *                   entry are as before, so decode reads such a pool
 *                   unchanged).
 *   k_win        NULL: a window row's softmax runs over the chunk's C+1 keys
 *                   (as pfd_chunk_prefill);
 *                [W, Hkv, D] bf16 device: the window rows' own keys join
 *                   that softmax's denominator (the scores stay the
 *                   probabilities of the chunk's keys, so they sum to less
 *                   than W * Hq).  Requires W >= 1.
 * workspace >= pfd_chunk_prefill_workspace(...) bytes, as for
 * pfd_chunk_prefill.
 */
pfd_status pfd_chunk_prefill_ex(const pfd_bf16* q, const pfd_bf16* k, const pfd_bf16* v,
                                const pfd_bf16* q_win, const pfd_bf16* k_win, int N, int C, int W,
                                int Hq, int Hkv, int D, int B, float sm_scale, int per_kv_head,
                                pfd_bf16* out, float* scores, int32_t* kept_idx, pfd_bf16* pool_k,
                                pfd_bf16* pool_v, int64_t pool_rows, const int32_t* slot_row,
                                pfd_chunk_entry* table, int32_t* dev_err, void* workspace,
                                size_t workspace_bytes, pfd_stream_t stream);

/*
 * Chunk scores from the model's logits (Methodology 1, predictive scoring:
 * s_I is the negative log-likelihood of the query window given the chunk,
 * s_P the likelihood of the pseudo-labels given the chunk and the query).
 * For every chunk j and labelled row r:
 *   row_ll[j][r] = logits[j][r][labels[r]] - log(sum_v exp(logits[j][r][v]))
 *   score[j]     = sum_r row_ll[j][r]
 * i.e. the summed log-likelihood of the labels.  With the query-window
 * tokens as labels this is s_I negated (higher = more relevant, as
 * pfd_select_chunks takes it); with the pseudo-labels it is s_P.
 *   logits  [N, R, V] bf16 device (finite values)
 *   labels  [R] int32 device, shared by every chunk; a label outside
 *           [0, V) gives that row NaN and sets PFD_DEVERR_LABEL
 *   row_ll  [N, R] fp32 device (written);  score [N] fp32 device (written)
 * 1 <= N, 1 <= R, N * R < 2^31, 1 <= V < 2^31.  One pass over the logits:
 * HBM-bound.  The result does not depend on scheduling (fixed-order sums).
 */
pfd_status pfd_chunk_loglik(const pfd_bf16* logits, const int32_t* labels, int N, int R,
                            int64_t V, float* row_ll, float* score, int32_t* dev_err,
                            pfd_stream_t stream);

/*
 * Chunk selection (Methodology 1, "Selection"; Methodology 2 inter-chunk
 * sparsity): s = fl32(s_I + s_P) (one fp32 add, round to nearest even), and
 * sel = the K chunks with the largest s in rank order (s descending, ties to
 * the lower index, -0.0 == +0.0, NaN below every number).  Both scores are
 * taken as "higher = more relevant"; a caller holding a raw negative
 * log-likelihood negates it first.
 *   s_I, s_P  [N] fp32 device;  sel [K] int32 device (written);
 *   s_out     [N] fp32 device (written) or NULL.   1 <= K <= N <= 16384.
 */
pfd_status pfd_select_chunks(const float* s_I, const float* s_P, int N, int K, int32_t* sel,
                             float* s_out, pfd_stream_t stream);

/*
 * Batched form of pfd_select_chunks for several sequences whose chunks are
 * numbered consecutively in one shared chunk table: sequence b owns table
 * entries cu_n[b] .. cu_n[b+1]-1 and selects K_b = cu_k[b+1]-cu_k[b] of them.
 * sel[cu_k[b] + i] receives the table index (cu_n[b] + chunk) of its i-th
 * best chunk.  cu_n, cu_k: [batch+1] int32 device, non-decreasing.
 * max_n bounds every sequence's chunk count (<= 16384).  A sequence whose
 * device segment is malformed (no chunk, more than max_n chunks, K_b < 0 or
 * K_b > its chunk count) gets -1 in its selection slots (when 0 < K_b <=
 * max_n), which a later pfd_decode_attention reports as PFD_DEVERR_SEL.
 */
pfd_status pfd_select_chunks_batched(const float* s_I, const float* s_P, const int32_t* cu_n,
                                     const int32_t* cu_k, int batch, int max_n, int32_t* sel,
                                     float* s_out, pfd_stream_t stream);

/*
 * Number of KV splits pfd_decode_attention uses for these sizes when
 * n_splits == 0 (a plan that depends only on the arguments and the current
 * device's SM count; with no usable device, 152 SMs, a GB300's count, are
 * assumed).  cu_lq_host, cu_k_host: [batch+1] int32 host memory.
 */
int pfd_decode_plan_splits(int batch, const int32_t* cu_lq_host, const int32_t* cu_k_host,
                           int Hq, int Hkv, int D, int max_chunk_len);

/* Workspace bytes pfd_decode_attention needs (0 when one split is used). */
size_t pfd_decode_workspace(int batch, const int32_t* cu_lq_host, const int32_t* cu_k_host,
                            int Hq, int Hkv, int D, int max_chunk_len, int n_splits);

/*
 * Static-KV decode attention of one denoising step (Methodology 3,
 * "Decoding with Static KV Reuse"; "Attention Kernel Optimization").
 *
 * Sequence b has Lq_b = cu_lq[b+1]-cu_lq[b] live rows (query window +
 * response) and K_b = cu_k[b+1]-cu_k[b] selected chunks sel[cu_k[b]..].
 * For each live row and query head h (KV head h / (Hq/Hkv)):
 *   out = softmax over [ the pool rows table[c].row .. +table[c].len of every
 *         selected chunk c ; the sequence's Lq_b live rows ] of
 *         sm_scale * q . k, applied to the matching v rows (no mask);
 *   lse = natural-log log-sum-exp of the same logits.
 * The key range is cut into n_splits contiguous splits (0 = automatic); each
 * split reads its chunks in place through the table (no gather) and keeps a
 * partial softmax state: its max and denominator in fp32 and its output row
 * normalised by that denominator in bf16.  The splits are merged by a
 * log-sum-exp reduction.  The pool is only read.
 *
 * Arguments (device memory unless stated):
 *   q              [total_lq, Hq, D] bf16; k_self, v_self [total_lq, Hkv, D]
 *   cu_lq          [batch+1] int32; cu_lq_host the same values in host memory
 *   pool_k/v       [pool_rows, Hkv, D] bf16
 *   table          [table_len] pfd_chunk_entry (all chunks of all sequences)
 *   sel            [cu_k[batch]] int32 indices into table
 *   cu_k, cu_k_host [batch+1] int32 device / host
 *   max_chunk_len  upper bound of table[].len, used only to plan splits
 *   out            [total_lq, Hq, D] bf16 (written)
 *   lse            [total_lq, Hq] fp32 (written) or NULL
 *   workspace      >= pfd_decode_workspace(...) bytes (may be NULL if 0)
 */
pfd_status pfd_decode_attention(const pfd_bf16* q, const pfd_bf16* k_self,
                                const pfd_bf16* v_self, const int32_t* cu_lq,
                                const int32_t* cu_lq_host, const pfd_bf16* pool_k,
                                const pfd_bf16* pool_v, int64_t pool_rows,
                                const pfd_chunk_entry* table, int32_t table_len,
                                const int32_t* sel, const int32_t* cu_k, const int32_t* cu_k_host,
                                int batch, int Hq, int Hkv, int D, int max_chunk_len,
                                float sm_scale, int n_splits, pfd_bf16* out, float* lse,
                                int32_t* dev_err, void* workspace, size_t workspace_bytes,
                                pfd_stream_t stream);

/*
 * One device's share of a decode step split across devices ("Attention Kernel
 * Optimization": the KV dimension is partitioned, the parts are processed
 * independently and merged by a log-sum-exp reduction).
 *
 * Identical to pfd_decode_attention except for two things.  First, the
 * keys are the selected chunks sel[cu_k[b]..cu_k[b+1]) followed by the live
 * block only when self_keys == 1; with self_keys == 0 the live rows are
 * queries only.  Second, the result is that subset's partial state:
 *   part_o   [total_lq, Hq, D] bf16: softmax over the subset's keys applied
 *            to their v rows (the subset's own normalised output);
 *   part_lse [total_lq, Hq] fp32 (required): natural-log log-sum-exp of the
 *            subset's logits.  A (row, head) that sees no key at all gets
 *            part_o = 0 and part_lse = -inf.
 * A step over the whole key set is the merge (pfd_lse_merge) of partials
 * whose subsets partition it: e.g. each device passes its local selected
 * chunks, one of them (the owner of the live block) with self_keys = 1, the
 * partials are gathered, and the owner merges them.
 * workspace >= pfd_decode_partial_workspace(...) bytes (the call's own
 * internal splits).
 */
size_t pfd_decode_partial_workspace(int batch, const int32_t* cu_lq_host,
                                    const int32_t* cu_k_host, int Hq, int Hkv, int D,
                                    int max_chunk_len, int self_keys, int n_splits);

pfd_status pfd_decode_partial(const pfd_bf16* q, const pfd_bf16* k_self, const pfd_bf16* v_self,
                              const int32_t* cu_lq, const int32_t* cu_lq_host,
                              const pfd_bf16* pool_k, const pfd_bf16* pool_v, int64_t pool_rows,
                              const pfd_chunk_entry* table, int32_t table_len, const int32_t* sel,
                              const int32_t* cu_k, const int32_t* cu_k_host, int batch, int Hq,
                              int Hkv, int D, int max_chunk_len, float sm_scale, int self_keys,
                              int n_splits, pfd_bf16* part_o, float* part_lse, int32_t* dev_err,
                              void* workspace, size_t workspace_bytes, pfd_stream_t stream);

/*
 * Log-sum-exp merge of n_parts partial states from any source ("Attention
 * Kernel Optimization"), for every (row, head) of rows x Hq:
 *   M = max_s part_lse[s],  w_s = exp(part_lse[s] - M),
 *   out = sum_s w_s part_o[s] / sum_s w_s,  lse = M + ln(sum_s w_s).
 * A part with part_lse = -inf has weight 0; if every part has, out = 0 and
 * lse = -inf.
 *   part_o   [n_parts, rows, Hq, D] bf16 device (8-byte aligned)
 *   part_lse [n_parts, rows, Hq] fp32 device
 *   out      [rows, Hq, D] bf16 device (written);  lse [rows, Hq] fp32 or NULL
 * 1 <= n_parts <= 64; D in {64, 128}.
 */
pfd_status pfd_lse_merge(const pfd_bf16* part_o, const float* part_lse, int n_parts, int rows,
                         int Hq, int D, pfd_bf16* out, float* lse, pfd_stream_t stream);

/*
 * Dynamic chunk reselection.  The pages list static selection (no
 * reselection during decoding) as a limitation of the method; this is the
 * reading taken here.  At a reselection step the live rows score every chunk
 * of their sequence by the attention mass its cached rows receive at that
 * step's normaliser:
 *   mass[c] = (1 / (Lq_b * Hq)) * sum over the sequence's live rows r, query
 *             heads h and the rows t of chunk c's slot of
 *             exp(sm_scale * q[r][h] . k_pool[t][h / (Hq/Hkv)] - lse[r][h])
 * with lse the step's decode log-sum-exp (pfd_decode_attention's lse
 * output).  For a selected chunk this is its share of the step's attention;
 * for the others, the share they would take at the same normaliser.
 * Sequence b's chunks are table entries cu_n_host[b] .. cu_n_host[b+1]-1;
 * mass is written at the same indices.
 *   q            [total_lq, Hq, D] bf16 live rows (the step's queries)
 *   cu_lq        [batch+1] int32 device; cu_lq_host, cu_n_host [batch+1] host
 *   pool_k       [pool_rows, Hkv, D] bf16; table [table_len]
 *   lse          [total_lq, Hq] fp32 device
 *   mass         [table_len] fp32 device (written for the listed chunks; a
 *                sequence with no live rows, Lq_b = 0, has no mass and its
 *                entries are left as they were)
 *   workspace    >= pfd_chunk_mass_workspace(...) bytes
 * batch <= 64.  QK on the tensor cores over every chunk's slot (no PV);
 * fixed-order sums, so repeated calls give the same bits.
 */
size_t pfd_chunk_mass_workspace(int batch, const int32_t* cu_lq_host, const int32_t* cu_n_host,
                                int Hq, int Hkv);

pfd_status pfd_chunk_mass(const pfd_bf16* q, const int32_t* cu_lq, const int32_t* cu_lq_host,
                          const pfd_bf16* pool_k, int64_t pool_rows, const pfd_chunk_entry* table,
                          int32_t table_len, const int32_t* cu_n_host, const float* lse, int batch,
                          int Hq, int Hkv, int D, float sm_scale, float* mass, int32_t* dev_err,
                          void* workspace, size_t workspace_bytes, pfd_stream_t stream);

/*
 * The new selection: for every chunk s'[c] = fl32(s[c] + fl32(lambda *
 * mass[c])) (two fp32 roundings, nearest even), then the top-K of s' per
 * sequence with pfd_select_chunks_batched's rules and layout (sel holds
 * table indices in rank order; s_out [..] receives s', or NULL).  s is the
 * static score fl32(s_I + s_P) (pfd_select_chunks's s_out).  lambda >= 0;
 * lambda = 0 gives the static selection.
 */
pfd_status pfd_reselect_chunks(const float* s, const float* mass, float lambda,
                               const int32_t* cu_n, const int32_t* cu_k, int batch, int max_n,
                               int32_t* sel, float* s_out, pfd_stream_t stream);

/* Bytes of the static device scratch used by
 * pfd_decode_attention_static_scratch (per device). */
#define PFD_DECODE_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * pfd_decode_attention without a workspace argument.  The pages describe no
 * such call: it is a library convenience for callers that cannot allocate
 * device memory when they call (a host program that links only this library
 * and holds no device allocator; a hook inside another runtime that owns and
 * accounts every device byte and forbids allocation there).
 *
 * The split-KV partials go to one statically allocated device buffer of
 * PFD_DECODE_STATIC_SCRATCH_BYTES per device instead of caller workspace;
 * nothing is allocated.  Every call looks up the current device's copy of
 * the buffer (cudaGetSymbolAddress, with that device current); nothing is
 * cached, so calls after a device reset need no special care.  The first
 * call on a device may make the CUDA runtime load this library's device code
 * there; make it before any stream capture begins.  Every call on a device
 * shares the buffer, so calls whose work overlaps on the GPU (streams with
 * no ordering between them) race and give undefined results; calls on one
 * stream run in order and are safe.
 *
 * With n_splits == 0 the call uses the split count pfd_decode_plan_splits
 * reports, lowered to the largest count whose partials fit the buffer (one
 * split needs no scratch, so every size runs).  An explicit n_splits whose
 * partials need more than PFD_DECODE_STATIC_SCRATCH_BYTES
 * (pfd_decode_workspace(...) reports the need) returns PFD_ERR_UNSUPPORTED
 * with nothing launched.  Arguments, results and device-side errors are
 * otherwise those of pfd_decode_attention; PFD_ERR_CUDA is returned when the
 * buffer's address cannot be found on the current device.
 */
pfd_status pfd_decode_attention_static_scratch(
    const pfd_bf16* q, const pfd_bf16* k_self, const pfd_bf16* v_self, const int32_t* cu_lq,
    const int32_t* cu_lq_host, const pfd_bf16* pool_k, const pfd_bf16* pool_v, int64_t pool_rows,
    const pfd_chunk_entry* table, int32_t table_len, const int32_t* sel, const int32_t* cu_k,
    const int32_t* cu_k_host, int batch, int Hq, int Hkv, int D, int max_chunk_len,
    float sm_scale, int n_splits, pfd_bf16* out, float* lse, int32_t* dev_err,
    pfd_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char* pfd_status_string(pfd_status status);

/* PFD_ABI_VERSION of the loaded library. */
int pfd_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PFD_H_ */
