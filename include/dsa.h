/*
 * dsa.h -- C ABI of the DSA sparse-attention hot path on GB300 (sm_103a).
 *
 * The path has three stages over a block-paged KV cache:
 *   1. indexer score  -- "Day-0 Adaptation of Trillion-Parameter MoE Models on
 *      Domestic GPUs", section 3 (1) Index Selection: a lightweight similarity
 *      score of every cached position against the query;
 *   2. top-K          -- same passage (the K best positions found block by
 *      block, then combined across blocks), with the deterministic tie rule of
 *      "Day-0 Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
 *      Accelerators", section 4 (equal scores: the lower position wins);
 *   3. sparse attention -- first page, section 3 (3): exact softmax attention
 *      over the selected positions only, with separate decode (memory-bound)
 *      and prefill (compute-bound) paths.
 * The cache layout follows first page, section 3 (2): pages of `block_size`
 * consecutive positions stored contiguously, an index table jumping between
 * pages.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    never allocates, frees or keeps a pointer after a call returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and launches kernels only: no host synchronisation, no
 *    allocation, so the calls may be captured into a CUDA graph.
 *  - Tensors are dense and row-major in the shapes written next to them, except
 *    the KV pools, whose rows are `*_row_stride` elements apart.
 *  - Return value: DSA_OK, or a negative DSA_ERR_* code for errors the host can
 *    see (bad pointer, shape, dtype or workspace).  Then nothing was launched
 *    and the message is in dsa_last_error_string().
 *  - Errors that depend on device data (a block-table entry outside
 *    [0, num_blocks), an index past its sequence, a bounded wait that ran out)
 *    never trap: the offending position or row is skipped (score -inf, row left
 *    out of the softmax) and a DSA_STATUS_* bit is OR-ed into the status word
 *    at the start of the call's workspace; dsa_get_status() reads it.
 *  - Workspaces: query the size with the matching dsa_*_workspace_size(), pass a
 *    caller-owned device buffer of at least that size, 256-byte aligned and
 *    ZERO-FILLED before its first use.  The library leaves it in a reusable
 *    state after every call (counters return to zero; the status word is sticky
 *    until read with clear=1).  Calls that share a workspace must not overlap
 *    on the GPU (issue them on one stream, or order the streams).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* = cudaStream_t */

/* host-visible return codes */
#define DSA_OK 0
#define DSA_ERR_INVALID (-1)     /* null pointer, bad shape, K, stride or layout */
#define DSA_ERR_UNSUPPORTED (-2) /* no kernel for this dtype / head count / dims */
#define DSA_ERR_WORKSPACE (-3)   /* workspace missing, misaligned or too small */
#define DSA_ERR_CUDA (-4)        /* a CUDA call failed; see dsa_last_error_string() */
#define DSA_ERR_TIMEOUT (-5)     /* reported by dsa_get_status() users, see below */

/* device status bits (dsa_get_status) */
#define DSA_STATUS_BAD_BLOCK 0x1  /* block-table entry outside [0, num_blocks) */
#define DSA_STATUS_BAD_INDEX 0x2  /* selected index >= its sequence length */
#define DSA_STATUS_BAD_LENGTH 0x4 /* seq_len > max_blocks_per_seq*block_size, or > ld */
#define DSA_STATUS_TIMEOUT 0x8    /* a bounded device wait gave up */

/* element types */
#define DSA_BF16 0     /* bfloat16 */
#define DSA_FP8_E4M3 1 /* OCP FP8 E4M3 ("fn": no infinities) */

/*
 * Paged cache layout ("Day-0 Adaptation of Trillion-Parameter MoE Models on
 * Domestic GPUs", section 3 (2)).  Logical position p of sequence b is stored
 * in physical row  block_table[b][p / block_size] * block_size + p % block_size
 * of every pool (KV pool, indexer-key pool).  Unused table entries may hold
 * any value; they are never read.
 */
typedef struct dsa_paged_layout {
  int32_t block_size;          /* positions per page, 1..1024 (64 in the workloads) */
  int32_t num_blocks;          /* pages in each pool (NB) */
  int32_t max_blocks_per_seq;  /* row length of block_table */
  int32_t batch;               /* number of sequences B */
  int32_t max_seq_len;         /* host-known bound: every seq_lens[b] <= max_seq_len */
  int32_t reserved_;           /* set to 0 */
  const int32_t* block_table;  /* device [batch][max_blocks_per_seq] */
  const int32_t* seq_lens;     /* device [batch]: cached positions L_b (query included) */
} dsa_paged_layout;

/* ---------------------------------------------------------------------------
 * Stage 1: indexer score.
 * Source: "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
 * section 3 (1) (each cached position scored by its similarity to the
 * query through low-dimensional keys), read as
 *     scores[r][p] = sum_h w[r][h] * max(0, sum_d q_idx[r][h][d] * k_idx[p][d])
 * for every position p the query may see: p <= q_pos[r] and p < L_b (causal,
 * the current position included).  Entries of the row past the last eligible
 * position are not part of the result and may be left untouched.
 * Accumulation is fp32; with integer-valued q_idx/k_idx/w
 * (the pages' workloads) the scores are exact integers below 2^24.
 *
 *  layout      paged layout; only block_table/seq_lens rows of the queried
 *              sequences are read
 *  q_idx       [Nq][H_i][D_i] of `dtype` -- indexer queries
 *  w           [Nq][H_i] fp32 -- head weights
 *  kidx_pool   [num_blocks][block_size][D_i] of `dtype` -- indexer keys
 *  dtype       DSA_BF16 or DSA_FP8_E4M3 (q_idx and kidx_pool share it)
 *  H_i, D_i    indexer heads (1..128) and dim (32, 64 or 128)
 *  q_seq       [Nq] sequence of each query, or NULL: query r is sequence r
 *  q_pos       [Nq] absolute position of each query, or NULL: L_b - 1 (decode)
 *  scores      [Nq][ld] fp32 output; ld >= eligible positions of every row
 *  ws          workspace of dsa_index_score_workspace_size() bytes
 * Errors: DSA_ERR_INVALID for null pointers, Nq < 0, ld < 1 or a bad layout;
 * DSA_ERR_UNSUPPORTED for other H_i/D_i/dtype and for Nq > 65535 (call in
 * chunks of queries).  Device: out-of-range block ids give -inf scores and
 * DSA_STATUS_BAD_BLOCK.
 */
size_t dsa_index_score_workspace_size(int Nq, int H_i, int D_i, int64_t ld);
int dsa_index_score(const dsa_paged_layout* layout, const void* q_idx, const float* w,
                    const void* kidx_pool, int dtype, int H_i, int D_i,
                    const int32_t* q_seq, const int32_t* q_pos, int Nq, float* scores,
                    int64_t ld, void* ws, size_t ws_bytes, dsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Stage 1, prefill form: all Nq queries belong to sequence `seq` and query r
 * sits at position q_pos[r] (q_pos NULL: position r).  Same scores as
 * dsa_index_score with q_seq[r] = seq.  Source: "Day-0 Adaptation of
 * Trillion-Parameter MoE Models on Domestic GPUs", section 3 (3): the prefill
 * stage processes the whole prompt at once and is compute-intensive, so the
 * queries share every key tile (a dense causal contraction on tensor cores).
 * Errors as for dsa_index_score; seq must be in [0, batch).
 */
size_t dsa_index_score_prefill_workspace_size(int Nq, int H_i, int D_i, int64_t ld);
int dsa_index_score_prefill(const dsa_paged_layout* layout, int seq, const void* q_idx,
                            const float* w, const void* kidx_pool, int dtype, int H_i, int D_i,
                            const int32_t* q_pos, int Nq, float* scores, int64_t ld, void* ws,
                            size_t ws_bytes, dsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Stage 2: top-K selection.
 * Source: "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
 * section 3 (1) (selection done per block of positions and then combined
 * over the blocks, with no sort of the whole row); tie rule from "Day-0
 * Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
 * Accelerators", section 4: among equal scores the lower position wins.
 * For row r, among positions 0..n_eligible[r]-1, keep the min(K, n) positions
 * with the largest score (scores compared as values: -0.0 ties +0.0), write
 * them to idx[r] in ascending position order and pad with -1.
 *
 *  scores      [Nq][ld] fp32 (finite or -inf; NaN ranks below every value)
 *  n_eligible  [Nq] int32, each in [0, ld] (larger values are clamped to ld
 *              and flagged DSA_STATUS_BAD_LENGTH)
 *  K           1..65536
 *  idx         [Nq][K] int32 output
 *  ws          workspace of dsa_topk_workspace_size() bytes
 */
size_t dsa_topk_workspace_size(int Nq, int64_t ld, int K);
int dsa_topk(const float* scores, int64_t ld, const int32_t* n_eligible, int Nq, int K,
             int32_t* idx, void* ws, size_t ws_bytes, dsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * dsa_topk_noalloc: the selection of dsa_topk (same arguments and results,
 * minus the workspace) for callers that cannot allocate device memory: code
 * given a stream but no allocator by the framework that owns the GPU's
 * memory, real-time threads that must not wait on allocator locks, and
 * deployments whose device memory is fully divided up in advance.  The pages
 * have no counterpart; this is a deployment convenience.
 *  Scratch: one fixed array of DSA_TOPK_NOALLOC_SCRATCH_BYTES inside the
 *    library, present on every GPU that loads it until the process exits.  No
 *    call allocates or frees device memory.
 *  First call on a device: looks up the array's device address (once per
 *    device, with that device current) and keeps it for the life of the
 *    process.  Make that first call before any stream capture.  A
 *    cudaDeviceReset() of that device invalidates the kept address: do not
 *    reset a device between calls of this function in one process.
 *  Limit: a problem whose scratch would exceed the array
 *    (dsa_topk_workspace_size() > DSA_TOPK_NOALLOC_SCRATCH_BYTES) is rejected
 *    with DSA_ERR_WORKSPACE and a message; nothing is launched.
 *  Sharing: every call uses the same array.  Calls that overlap on the GPU
 *    (unordered streams, several host threads) race and corrupt each other's
 *    results; order them on one stream.  The status word is cleared at the
 *    start of each call and cannot be read back.
 */
#define DSA_TOPK_NOALLOC_SCRATCH_BYTES (8u << 20)
int dsa_topk_noalloc(const float* scores, int64_t ld, const int32_t* n_eligible, int Nq, int K,
                     int32_t* idx, dsa_stream_t stream);
/* The size of that fixed array as this build of the library has it
 * (DSA_TOPK_NOALLOC_SCRATCH_BYTES), for callers that load the library at run
 * time and cannot see the header's define. */
size_t dsa_topk_noalloc_scratch_bytes(void);

/* ---------------------------------------------------------------------------
 * Stage 3a: sparse attention, decode (one query per sequence).
 * Source: "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
 * section 3 (3) (decode: one token per step, memory-bandwidth-bound) and the
 * execution chain of "Day-0 Adaptation of Ultra-Large-Scale MoE Models on
 * Heterogeneous AI Accelerators", section 4 (cache gather + sparse attention).
 * For sequence b and head h, over the selected positions j (idx[b][*] >= 0),
 * whose rows are gathered through the block table:
 *     z_j = sm_scale * q[b][h] . K_j,   out[b][h] = sum_j softmax(z)_j V_j,
 *     lse[b][h] = log sum_j exp(z_j)
 * One shared K/V head (multi-query); fp32 accumulation and softmax.
 *
 *  q            [B][Hq][Dqk] bf16
 *  k_pool       physical rows of Dqk bf16, k_row_stride elements apart
 *  v_pool       physical rows of Dv bf16, v_row_stride elements apart; may be
 *               k_pool itself (latent cache: V = first Dv dims of the K row)
 *  Hq           1..64 query heads; Dqk, Dv multiples of 8 (>= 8), Dv <= 512,
 *               Hq * Dqk * 2 + 4 * (Dqk + Dv) <= 200 KB (q of one query held in
 *               shared memory); B (Nq for prefill) <= 65535.  Other shapes
 *               return DSA_ERR_UNSUPPORTED.
 *  idx          [B][K] int32 positions from dsa_topk (-1 = padding, skipped)
 *  out          [B][Hq][Dv] bf16 output (0 for a row with no selected position)
 *  lse          [B][Hq] fp32 output, or NULL (-inf for an empty row)
 *  ws           workspace of dsa_sparse_attn_decode_workspace_size() bytes
 * Device errors: an index >= L_b or a bad block id skips that row and sets
 * DSA_STATUS_BAD_INDEX / DSA_STATUS_BAD_BLOCK.
 */
size_t dsa_sparse_attn_decode_workspace_size(int B, int Hq, int Dqk, int Dv, int K);
int dsa_sparse_attn_decode(const dsa_paged_layout* layout, const void* q, const void* k_pool,
                           int64_t k_row_stride, const void* v_pool, int64_t v_row_stride,
                           int Hq, int Dqk, int Dv, const int32_t* idx, int K, float sm_scale,
                           void* out, float* lse, void* ws, size_t ws_bytes,
                           dsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Stage 3b: sparse attention, prefill (many queries, each with its own
 * selected set).  Source: "Day-0 Adaptation of Trillion-Parameter MoE Models
 * on Domestic GPUs", section 3 (3) (prefill: whole prompt at once,
 * compute-intensive).  Same arithmetic as stage 3a for each query r of
 * sequence q_seq[r]:
 *  q            [Nq][Hq][Dqk] bf16
 *  q_seq        [Nq] int32 sequence of each query, or NULL: all in sequence 0
 *  q_pos        [Nq] int32 absolute position of each query, or NULL.  When
 *               given, only the first min(K, q_pos+1) entries of idx[r] are
 *               read and an index > q_pos (non-causal) is skipped and flagged
 *               DSA_STATUS_BAD_INDEX
 *  idx          [Nq][K] int32
 *  out          [Nq][Hq][Dv] bf16, lse [Nq][Hq] fp32 or NULL
 *  ws           workspace of dsa_sparse_attn_prefill_workspace_size() bytes
 * Other arguments and errors as for stage 3a.
 */
size_t dsa_sparse_attn_prefill_workspace_size(int Nq, int Hq, int Dqk, int Dv, int K);
int dsa_sparse_attn_prefill(const dsa_paged_layout* layout, const void* q, const void* k_pool,
                            int64_t k_row_stride, const void* v_pool, int64_t v_row_stride,
                            int Hq, int Dqk, int Dv, const int32_t* q_seq,
                            const int32_t* q_pos, int Nq, const int32_t* idx, int K,
                            float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes,
                            dsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Cache write: store new rows into the paged caches -- a whole prompt after
 * prefill, the appended token at each decode step.  Source: "Day-0
 * Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
 * Accelerators", section 4: the KV cache is written in the block layout, and
 * the layout written during prefill must match exactly the gather addresses
 * read during decode.  Row i goes to position pos[i] of sequence seq[i], i.e.
 * physical row block_table[seq][pos / block_size] * block_size
 * + pos % block_size -- the same mapping every gather above uses.
 *
 *  layout      paged layout (seq_lens is read only by the append form)
 *  seq, pos    [N] int32 sequence and position of each new row; both NULL:
 *              the append form of a decode step, row i goes to position
 *              seq_lens[i] - 1 of sequence i (N <= batch; seq_lens already
 *              counts the new token)
 *  kv_new      [N][row_elems] bf16 rows (K, or the latent K/V row), or NULL
 *  row_elems   bf16 elements per row, a multiple of 8
 *  kv_pool     physical rows of row_elems bf16, kv_row_stride elements apart
 *              (a multiple of 8, >= row_elems)
 *  kidx_new    [N][D_i] indexer-key rows of kidx_dtype, or NULL
 *  kidx_pool   [num_blocks][block_size][D_i] of kidx_dtype
 *  ws          workspace of dsa_cache_write_workspace_size() bytes
 * Pointers 16-byte aligned.  Rows of the same physical row written twice in
 * one call (a caller error the call does not detect): each 16-byte piece of
 * that row holds the piece of one of them, which one unspecified, so the row
 * may mix them.
 * Errors: DSA_ERR_INVALID for null pointers, N < 0, bad sizes, strides or
 * alignment.  Device: a sequence outside [0, batch), a position outside the
 * block table or a block id outside [0, num_blocks) skips that row and sets
 * DSA_STATUS_BAD_BLOCK.
 */
size_t dsa_cache_write_workspace_size(void);
int dsa_cache_write(const dsa_paged_layout* layout, const int32_t* seq, const int32_t* pos, int N,
                    const void* kv_new, int row_elems, void* kv_pool, int64_t kv_row_stride,
                    const void* kidx_new, int D_i, int kidx_dtype, void* kidx_pool, void* ws,
                    size_t ws_bytes, dsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Whole steps: one call for one decode step or one prefill (chunk), each the
 * cache write followed by the three stages on `stream` (no host
 * synchronisation in between).  Source: "Day-0 Adaptation of
 * Trillion-Parameter MoE Models on Domestic GPUs", section 3 (3): decode
 * indexing is incremental -- the indexer keys of earlier positions stay in
 * the cache and a step only adds the new position's row before scoring --
 * and prefill handles a whole prompt at once; "Day-0 Adaptation of
 * Ultra-Large-Scale MoE Models on Heterogeneous AI Accelerators", section 4:
 * index selection, KV cache write, then gather + sparse attention.
 *
 * dsa_decode_step: layout->seq_lens[b] already counts sequence b's new token.
 *  k_new       [B][Dqk] bf16 new K rows (the latent row for a latent cache),
 *              written at position seq_lens[b] - 1 of k_pool (rows
 *              k_row_stride elements apart)
 *  v_new       [B][Dv] bf16 new V rows into v_pool, or NULL when v_pool is
 *              k_pool and V is the first Dv dims of the K row
 *  kidx_new    [B][D_i] new indexer-key rows of idx_dtype into kidx_pool
 *  q_idx, w, q as for dsa_index_score / dsa_sparse_attn_decode (query b is
 *              sequence b at its newest position)
 *  scores      [B][ld], idx [B][K], out [B][Hq][Dv], lse [B][Hq] or NULL
 *  ws          dsa_decode_step_workspace_size(...) bytes; the step's status
 *              word (all stages OR into it) is at offset 0
 * dsa_prefill_step: the Nq queries of sequence `seq` at positions q_pos
 * (device [Nq]); their new rows (k_new/v_new/kidx_new, [Nq][...]) are written
 * at those positions first, so a prompt (or a chunk of one after an existing
 * prefix) is cached and attended in one call; n_eligible [Nq] = q_pos + 1.
 * Errors: those of the calls the step makes, with nothing after the first
 * failing call launched.
 */
size_t dsa_decode_step_workspace_size(int B, int H_i, int D_i, int64_t ld, int Hq, int Dqk,
                                      int Dv, int K);
int dsa_decode_step(const dsa_paged_layout* layout, const void* k_new, void* k_pool,
                    int64_t k_row_stride, const void* v_new, void* v_pool, int64_t v_row_stride,
                    const void* kidx_new, void* kidx_pool, int idx_dtype, const void* q_idx,
                    const float* w, int H_i, int D_i, const void* q, int Hq, int Dqk, int Dv,
                    int K, float sm_scale, float* scores, int64_t ld, int32_t* idx, void* out,
                    float* lse, void* ws, size_t ws_bytes, dsa_stream_t stream);
size_t dsa_prefill_step_workspace_size(int Nq, int H_i, int D_i, int64_t ld, int Hq, int Dqk,
                                       int Dv, int K);
int dsa_prefill_step(const dsa_paged_layout* layout, int seq, const int32_t* q_pos,
                     const int32_t* n_eligible, int Nq, const void* k_new, void* k_pool,
                     int64_t k_row_stride, const void* v_new, void* v_pool, int64_t v_row_stride,
                     const void* kidx_new, void* kidx_pool, int idx_dtype, const void* q_idx,
                     const float* w, int H_i, int D_i, const void* q, int Hq, int Dqk, int Dv,
                     int K, float sm_scale, float* scores, int64_t ld, int32_t* idx, void* out,
                     float* lse, void* ws, size_t ws_bytes, dsa_stream_t stream);

/* dsa_prefill_step_chunked — "Day-0 Adaptation of Trillion-Parameter MoE Models
 * on Domestic GPUs", section 3 (3): the prefill stage fuses index selection and
 * exact attention into large-granularity operators.  The same work as
 * dsa_prefill_step (cache write, indexer score, top-K, attention; same
 * arguments and results), without the [Nq][ld] score matrix: the queries are
 * scored and selected `chunk` rows at a time, and a chunk's scores live in one
 * scratch region of the workspace that the next chunk overwrites.  The score
 * memory is chunk x ld x 4 bytes instead of Nq x ld x 4 (a 16384-token prompt:
 * 48 MB instead of 1 GB), and with the default chunk it stays in L2 between the
 * indexer that writes it and the top-K that reads it, so the scores make no
 * round trip through HBM.
 *  ld          row length of the scratch (>= the largest n_eligible)
 *  chunk       queries per chunk; 0: the largest multiple of 16 whose scores
 *              fit 48 MB (at least 16)
 *  idx, out, lse, ws: as for dsa_prefill_step; ws =
 *              dsa_prefill_step_chunked_workspace_size(...) bytes, for the same
 *              chunk argument
 * Errors: those of dsa_prefill_step; chunk < 0 is DSA_ERR_INVALID.
 */
size_t dsa_prefill_step_chunked_workspace_size(int Nq, int H_i, int D_i, int64_t ld, int Hq,
                                               int Dqk, int Dv, int K, int chunk);
int dsa_prefill_step_chunked(const dsa_paged_layout* layout, int seq, const int32_t* q_pos,
                             const int32_t* n_eligible, int Nq, const void* k_new, void* k_pool,
                             int64_t k_row_stride, const void* v_new, void* v_pool,
                             int64_t v_row_stride, const void* kidx_new, void* kidx_pool,
                             int idx_dtype, const void* q_idx, const float* w, int H_i, int D_i,
                             const void* q, int Hq, int Dqk, int Dv, int K, float sm_scale,
                             int64_t ld, int chunk, int32_t* idx, void* out, float* lse, void* ws,
                             size_t ws_bytes, dsa_stream_t stream);

/* ---------------------------------------------------------------------------
 * Block-level bounds for incremental decode indexing — "Day-0 Adaptation of
 * Trillion-Parameter MoE Models on Domestic GPUs", section 3 (3): decode-time
 * index selection reuses the index structure of earlier steps and computes
 * only what is needed.  The structure is a bound pool beside the indexer-key
 * pool: for every page, per key dimension d, the largest and the smallest key
 * over the page's cached positions, as key codes:
 *   kbound_pool [NB][2][D_i] in the keys' dtype (row 0 maxima, row 1 minima).
 * dsa_index_bounds_update: recompute the bounds of the pages holding the rows
 *   (seq[i], pos[i]), i < N — call it after dsa_cache_write with the same
 *   seq/pos (after a decode step's append: one page per sequence) — or, with
 *   seq = pos = NULL, of every page slot below each sequence's length.  The
 *   layout's seq_lens must include the rows written.  ws: the status word
 *   (dsa_index_bounds_update_workspace_size() bytes); a page id outside
 *   [0, NB) is skipped and flags DSA_STATUS_BAD_BLOCK.
 * dsa_index_score_bounded: the decode form of dsa_index_score (query b is the
 *   query of sequence b, every cached position eligible, B = layout->batch,
 *   scores [B][ld]) that leaves out 128-position tiles whose scores cannot
 *   reach the top-K of size K: the bounds give each tile an upper bound of
 *   its scores; the ceil(K/128) + 1 tiles with the largest bounds are scored
 *   first, and every other tile whose bound is below the K-th largest of
 *   those scores is left out — its scores are -inf, its keys are not read.
 *   Every other score equals dsa_index_score's, so dsa_topk over the row
 *   selects exactly what it selects over the full row.  Pays off only where
 *   pages differ in their keys (on keys drawn independently per position
 *   every bound covers the row's largest score and nothing is left out).
 *   ws: dsa_index_score_bounded_workspace_size(B, H_i, D_i, ld, K) bytes.
 *   B <= 65535 (DSA_ERR_UNSUPPORTED otherwise, nothing launched).
 * dsa_index_bounded_stats: after the work queued on `stream` (this call
 *   synchronises it), the tiles the last dsa_index_score_bounded call on ws
 *   left out and the tiles it bounded.
 */
size_t dsa_index_bounds_update_workspace_size(void);
int dsa_index_bounds_update(const dsa_paged_layout* layout, const int32_t* seq,
                            const int32_t* pos, int N, const void* kidx_pool, int D_i,
                            int idx_dtype, void* kbound_pool, void* ws, size_t ws_bytes,
                            dsa_stream_t stream);
size_t dsa_index_score_bounded_workspace_size(int B, int H_i, int D_i, int64_t ld, int K);
int dsa_index_score_bounded(const dsa_paged_layout* layout, const void* q_idx, const float* w,
                            const void* kidx_pool, int idx_dtype, int H_i, int D_i,
                            const void* kbound_pool, int K, float* scores, int64_t ld, void* ws,
                            size_t ws_bytes, dsa_stream_t stream);
int dsa_index_bounded_stats(void* ws, dsa_stream_t stream, uint64_t* tiles_skipped,
                            uint64_t* tiles_bounded);

/* ---------------------------------------------------------------------------
 * Utilities (no counterpart on the pages).
 * dsa_get_status: copy the status word of a workspace to *status (host), after
 *   the work queued on `stream` so far has finished (this call synchronises the
 *   stream); clear != 0 resets it to 0.  Returns DSA_OK or DSA_ERR_*.
 * dsa_last_error_string: message of the last failing call on this host thread.
 * dsa_launch_count: kernels this library has launched in this process.
 * dsa_version: 10000*major + 100*minor + patch.
 * dsa_selftest_bounded_wait: one bounded mbarrier wait of the kind every
 *   pipelined kernel uses (one thread of one CTA).  expire != 0: nothing
 *   arrives, the wait gives up after limit_ns (1 us .. 1 s) and
 *   DSA_STATUS_TIMEOUT is OR-ed into the status word of ws (>= 256 bytes);
 *   expire == 0: the barrier completes first and nothing is recorded.  For
 *   testing the give-up path without a hang; the context stays usable.
 */
int dsa_get_status(void* ws, dsa_stream_t stream, int32_t* status, int clear);
const char* dsa_last_error_string(void);
uint64_t dsa_launch_count(void);
int dsa_version(void);
int dsa_selftest_bounded_wait(int expire, uint64_t limit_ns, void* ws, size_t ws_bytes,
                              dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
