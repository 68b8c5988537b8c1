/*
 * mla_prefill.h -- C ABI of a GB300 (sm_103a) library for ragged-batch
 * Multi-head Latent Attention (MLA) prefill over a paged latent KV cache.
 *
 * The path has four stages, each an entry point below, plus a fused entry
 * point that runs 1 to 4, and the step in front of it that writes
 * the new tokens' latent rows into the paged cache:
 *   0. mla_latent_cache_write -- RMSNorm + RoPE + paged store
 *                                ("mla_prefill_decode_graph_bf16", Args:
 *                                 freqs_cis, kv_norm_gamma, epsilon)
 *   1. mla_prefill_plan       -- chunk plan      ("mla_prefill_plan" page)
 *   2. mla_gather_latent      -- paged gather    ("mla_prefill_decode_graph_bf16",
 *                                                 Parameters: kv_input_fn)
 *   3. mla_upproject          -- K/V projection  ("mla_prefill_decode_graph_bf16",
 *                                                 Args: w_k, w_uv)
 *   4. mla_prefill_attention  -- causal attention with LSE merge across chunks
 *                                                ("flare_mla_prefill_dispatch")
 *   2'. mla_chunk_cache_rows, 3'. mla_upproject_paged,
 *   4'. mla_prefill_attention_paged -- a table of where each buffer row lives
 *       in the paged cache, and stages 3 and 4 reading the latent and k_rope
 *       rows there in place instead of from stage 2's buffers.  Same results;
 *       on GB300 they run slower than stage 2 plus 3 and 4 (the projection
 *       re-reads each latent row once per head tile), so the fused entry
 *       point does not use them.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     stated otherwise.  The library allocates no memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronises.  A host return of
 *     MLA_OK means the work was enqueued.  The kernels of the plan, gather,
 *     projection, attention and decode entry points are programmatic
 *     dependent launches: each may start launching while the kernel before
 *     it on the stream finishes, and waits for that kernel to complete before
 *     it touches memory, so stream order is unchanged.
 *   - Tensors are dense row-major with the leading dimensions written in the
 *     comments.  Integer tables are uint32/int32 as on the pages.
 *   - Geometry is fixed by the pages: q_depth 192 = 128 nope + 64 rope,
 *     cache_depth 576 = 512 latent + 64 rope, v_depth 128, kv_num_heads 1.
 *   - Element types (`dtype`): MLA_BF16 (bfloat16) or MLA_E4M3
 *     (float8_e4m3fn).  Attention output is always bfloat16.
 *   - Problems found on the device (plan overflow, bad offsets, bad page ids,
 *     a pipeline wait that timed out) are written to the caller's
 *     `int32_t* d_status` (first error wins; kernels never clear it; the
 *     fused entry point clears it first).  `d_status` may be NULL.
 *   - Every kernel that finds MLA_DEV_TIMEOUT already in *d_status when it
 *     starts does no work and returns, so one timeout stops the rest of the
 *     enqueued pipeline on that status word instead of letting it run on
 *     partial results.  Outputs of such calls are left untouched.
 *   - fp8 scales are descales: real value = stored value * scale.
 */
#ifndef MLA_PREFILL_H
#define MLA_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mla_status_t;
typedef void* mla_stream_t; /* cudaStream_t */

/* Host return codes. */
enum {
  MLA_OK = 0,
  MLA_ERR_ARG = -1,       /* null or misaligned (16 B) pointer, or a bad size */
  MLA_ERR_GEOMETRY = -2,  /* head count / layout outside what the kernels support */
  MLA_ERR_DTYPE = -3,     /* dtype not MLA_BF16 or MLA_E4M3 */
  MLA_ERR_LAUNCH = -4,    /* the CUDA runtime refused a launch or a tensor map */
  MLA_ERR_WORKSPACE = -5  /* workspace missing or smaller than mla_prefill_workspace_bytes */
};

/* Device status codes written to *d_status. */
enum {
  MLA_DEV_OK = 0,
  MLA_DEV_TOO_MANY_CHUNKS = 1, /* the plan needs more than max_chunks rows (truncated) */
  MLA_DEV_BAD_OFFSETS = 2,     /* input_row_offsets[0] != 0, decreasing, or total >= 2^31 */
  MLA_DEV_BAD_PAGE = 3,        /* a page-table entry is negative or >= num_pages */
  MLA_DEV_TIMEOUT = 4          /* a pipeline wait exceeded its limit; the kernel drained and exited */
};

enum { MLA_BF16 = 0, MLA_E4M3 = 1 };

/* Human-readable text for a host or device status code (static storage).
 * Utility of this library; no counterpart on the pages. */
const char* mla_status_string(int32_t code);

/* ABI version of this header.  Utility of this library; no counterpart on the
 * pages. */
int32_t mla_abi_version(void);
#define MLA_ABI_VERSION 2

/*
 * Which attention kernel mla_prefill_attention / mla_prefill launch for
 * `dtype`: "pair" (bf16 on two-SM clusters) or "e4m3" (the e4m3 form of the
 * same kernel).  There is one kernel per dtype and no fallback: a device that
 * cannot keep a two-CTA cluster of it resident gets MLA_ERR_LAUNCH from the
 * call.  Static storage; NULL for an unknown dtype.  The pages have no
 * counterpart: this is an introspection call.
 */
const char* mla_attention_kernel(int32_t dtype);

/*
 * Self-test of the failure detection the kernels rely on (the pages have
 * no counterpart to it).  Launches one cluster of `cluster_size` (1 or 2) CTAs that
 * wait on barriers nothing ever arrives at.  With one CTA it waits
 * `limit_ns`; with two, CTA 1 waits `limit_ns` and CTA 0 the library's full
 * limit (2 s), and CTA 0 must return as soon as CTA 1 gives up, through the
 * abort flag a timed-out wait raises in every CTA of its cluster.  Every wait
 * of every kernel in this library is bounded the same way.
 *
 * d_status:      int32, receives MLA_DEV_TIMEOUT
 * d_elapsed_ns:  int64 [cluster_size], 8-byte aligned: how long each CTA
 *                waited (-1 if its barrier completed, which cannot happen)
 * limit_ns:      1000 .. 2e9
 * Errors: host MLA_ERR_ARG for null or misaligned pointers or sizes out of
 * range; MLA_ERR_LAUNCH if the launch fails.
 */
mla_status_t mla_selftest_bounded_wait(int32_t* d_status, int64_t* d_elapsed_ns, int64_t limit_ns,
                                       int32_t cluster_size, mla_stream_t stream);

/*
 * 0. Latent-cache write.  Follows "mla_prefill_decode_graph_bf16" (Args:
 * freqs_cis -- precomputed RoPE values [max_seq_len, qk_rope_head_dim];
 * kv_norm_gamma -- RMSNorm weights [kv_lora_rank]; epsilon; kv_collection;
 * Parameters: kv_input_fn, the [tot_seq_len, 576] latent rows).  The step in
 * front of the prefill path: it puts the new tokens into the paged cache that
 * mla_gather_latent reads.
 *
 * New token i of sequence b (row input_row_offsets[b] + i of kv_latent and q)
 * sits at context position p = cache_lengths[b] + i.  Its latent row is 512
 * c_kv values followed by 64 k_rope values:
 *   c_kv'   = c_kv / sqrt(mean(c_kv^2) + epsilon) * kv_norm_gamma
 *   k_rope' = k_rope rotated by freqs_cis[p]
 * where a rotation treats the 64 values and the 64-value freqs_cis row as 32
 * complex numbers stored as interleaved (real, imaginary) pairs and multiplies
 * them.  The row [c_kv' | k_rope'] times kv_inv_scale, rounded to the cache's
 * type (nearest even; e4m3 saturates at +-448), is stored at page
 * page_table[b][p / page_size], slot p % page_size.  If q is not NULL, the
 * rope part (values 128..191) of every head of q[row] is rotated in place by
 * freqs_cis[p] and rounded to bf16; the nope part is left untouched.
 *
 * kv_cache:       [num_pages][page_size][576], bf16 or e4m3 (dtype), written
 * q:              [total_q_tokens][H][192] bf16, rotated in place, or NULL
 * kv_latent:      [total_q_tokens][576] bf16, the new tokens' latent rows
 * kv_norm_gamma:  [512] float32
 * freqs_cis:      [max_seq_len][64] float32
 * input_row_offsets [B+1], cache_lengths [B], page_table [B][max_pages_per_seq]
 *                 as in mla_prefill_plan and mla_gather_latent
 * kv_inv_scale:   1 for bf16; for e4m3 the reciprocal of the cache's descale
 * Pointers to kv_cache, q, kv_latent, kv_norm_gamma and freqs_cis must be
 * 16-byte aligned.  Errors: host MLA_ERR_DTYPE for another cache dtype,
 * MLA_ERR_ARG for null or misaligned pointers, B < 1, total_q_tokens < 0,
 * H < 1 with q given, page_size, num_pages, max_pages_per_seq or max_seq_len
 * < 1, epsilon < 0 or kv_inv_scale <= 0.  Device MLA_DEV_BAD_OFFSETS for a
 * token outside every sequence or a position >= max_seq_len (that token is
 * skipped), MLA_DEV_BAD_PAGE for a missing page (its cache row is not
 * written; its q is still rotated).
 */
mla_status_t mla_latent_cache_write(void* kv_cache, void* q, const void* kv_latent,
                                    const float* kv_norm_gamma, const float* freqs_cis,
                                    const uint32_t* input_row_offsets,
                                    const uint32_t* cache_lengths, const int32_t* page_table,
                                    int32_t num_pages, int32_t page_size,
                                    int32_t max_pages_per_seq, int32_t batch_size,
                                    int32_t num_heads, int32_t total_q_tokens,
                                    int32_t max_seq_len, float epsilon, float kv_inv_scale,
                                    int32_t dtype, int32_t* d_status, mla_stream_t stream);

/*
 * 1. Chunk plan.  Follows "mla_prefill_plan" (Args: buffer_row_offsets,
 * cache_offsets, buffer_lengths, input_row_offsets, k_cache, buffer_token_size).
 *
 * Every sequence b has cache_lengths[b] cached tokens and
 * input_row_offsets[b+1] - input_row_offsets[b] new tokens; its context is
 * L_b = cached + new tokens, cached first.  All contexts are laid end to end in
 * batch order and cut into consecutive chunks of buffer_token_size rows.  For
 * chunk c (0 <= c < max_chunks):
 *   buffer_row_offsets[c][b]  first buffer row of sequence b (b <= B; [c][B] = rows used)
 *   cache_offsets[c][b]       first context position of sequence b in the chunk
 *                             (L_b once b is finished, 0 before it starts)
 *   buffer_lengths[c]         rows used, or -1 if the chunk is unused.
 *
 * buffer_row_offsets: [max_chunks][B+1] uint32, output
 * cache_offsets:      [max_chunks][B]   uint32, output
 * buffer_lengths:     [max_chunks]      int32,  output
 * input_row_offsets:  [B+1] uint32 cumulative new-token offsets, starting at 0
 * cache_lengths:      [B]   uint32 cached tokens per sequence (the page's k_cache lengths)
 * Errors: host MLA_ERR_ARG for null pointers, B < 0, max_chunks < 1 or
 * buffer_token_size == 0.  Device MLA_DEV_TOO_MANY_CHUNKS when more than
 * max_chunks chunks are needed (the first max_chunks rows are still written),
 * MLA_DEV_BAD_OFFSETS for malformed offsets (tables then unspecified).
 */
mla_status_t mla_prefill_plan(uint32_t* buffer_row_offsets, uint32_t* cache_offsets,
                              int32_t* buffer_lengths, const uint32_t* input_row_offsets,
                              const uint32_t* cache_lengths, int32_t batch_size,
                              int32_t max_chunks, uint32_t buffer_token_size, int32_t* d_status,
                              mla_stream_t stream);

/*
 * 2. Latent gather.  Follows "mla_prefill_decode_graph_bf16" (Parameters:
 * kv_input_fn, the loader of KV latents [tot_seq_len, cache_head_dim]) and the
 * k_rope operand of "flare_mla_prefill_dispatch" (Parameters: k_rope_t;
 * Args: cache_offsets).
 *
 * For chunk `chunk` of the plan, every sequence b and t < n_cb (its rows in the
 * chunk): buffer row buffer_row_offsets[chunk][b] + t receives the cache token
 * at context position p = cache_offsets[chunk][b] + t of sequence b, stored in
 * page page_table[b][p / page_size] at slot p % page_size.  Elements 0..511 of
 * the 576-wide cache row go to c_kv_buf, 512..575 to k_rope_buf.  Bit copy.
 * Buffer rows at and beyond buffer_lengths[chunk] are not written.  A chunk
 * with buffer_lengths[chunk] == -1 does nothing.
 *
 * c_kv_buf:    [buffer_token_size][512] dtype, output
 * k_rope_buf:  [buffer_token_size][64]  dtype, output
 * kv_cache:    [num_pages][page_size][576] dtype
 * page_table:  [B][max_pages_per_seq] int32 physical page ids
 * buffer_row_offsets, cache_offsets, buffer_lengths: the plan tables (all chunks)
 * Errors: host MLA_ERR_ARG / MLA_ERR_DTYPE; device MLA_DEV_BAD_PAGE for a page id
 * outside [0, num_pages) or a position beyond max_pages_per_seq pages (row skipped).
 */
mla_status_t mla_gather_latent(void* c_kv_buf, void* k_rope_buf, const void* kv_cache,
                               const int32_t* page_table, int32_t num_pages, int32_t page_size,
                               int32_t max_pages_per_seq, const uint32_t* buffer_row_offsets,
                               const uint32_t* cache_offsets, const int32_t* buffer_lengths,
                               int32_t chunk, int32_t batch_size, uint32_t buffer_token_size,
                               int32_t dtype, int32_t* d_status, mla_stream_t stream);

/*
 * 3. Up-projection.  Follows "mla_prefill_decode_graph_bf16" (Args: w_k
 * [num_heads * qk_nope_head_dim, kv_latent_dim]; w_uv [num_heads, v_head_dim,
 * kv_latent_dim]).
 *
 * For rows r < n (n = buffer_lengths[chunk], or buffer_token_size when
 * buffer_lengths is NULL) and head h:
 *   k_nope[r][h][:] = s * c_kv_buf[r][:] . w_k[h*128 + :][:]^T
 *   v[r][h][:]      = s * c_kv_buf[r][:] . w_uv[h][:][:]^T
 * with s = ckv_scale * w_scale * kv_out_inv_scale, fp32 accumulation, rounded
 * to the storage dtype (nearest even; e4m3 saturates at +-448).  Rows from n
 * up to the next multiple of 128 (within buffer_token_size) are written as 0.
 *
 * k_nope:     [buffer_token_size][num_heads][128] dtype, output
 * v:          [buffer_token_size][num_heads][128] output: bf16 for MLA_BF16; for
 *             MLA_E4M3, f16 holding the e4m3-rounded values (exactly the e4m3
 *             result, stored 2 bytes wide so that the attention's P*V runs on
 *             f16 operands with no widening; the pages have no counterpart for
 *             this storage choice)
 * c_kv_buf:   [buffer_token_size][512] dtype
 * w_k:        [num_heads*128][512] dtype;  w_uv: [num_heads][128][512] dtype
 * Errors: host MLA_ERR_ARG / MLA_ERR_DTYPE / MLA_ERR_GEOMETRY (num_heads < 1),
 * MLA_ERR_LAUNCH; device MLA_DEV_TIMEOUT (d_status may be NULL).
 */
mla_status_t mla_upproject(void* k_nope, void* v, const void* c_kv_buf, const void* w_k,
                           const void* w_uv, const int32_t* buffer_lengths, int32_t chunk,
                           uint32_t buffer_token_size, int32_t num_heads, int32_t dtype,
                           float ckv_scale, float w_scale, float kv_out_inv_scale,
                           int32_t* d_status, mla_stream_t stream);

/*
 * 2'. Cache-row table of every plan chunk: where in the paged cache each
 * buffer row lives ("mla_prefill_decode_graph_bf16", Args: buffer_row_offsets,
 * cache_offsets, and the kv_collection's pages; "flare_mla_prefill_dispatch",
 * Args: cache_offsets, the start of a chunk's keys in the paged k_rope).  It is
 * the lookup mla_gather_latent does, kept as 4 bytes per row instead of the
 * row itself, so that stages 3' and 4' read the rows in place.
 *
 * cache_rows: [max_chunks][buffer_token_size] int32 output.  For chunk c and
 *             buffer row r < buffer_lengths[c] of sequence b
 *             (buffer_row_offsets[c][b] <= r < buffer_row_offsets[c][b+1]),
 *             position j = cache_offsets[c][b] + r - buffer_row_offsets[c][b]:
 *             cache_rows[c][r] = page_table[b][j / page_size] * page_size +
 *             j % page_size, the row's index in the cache seen as
 *             [num_pages * page_size][576].  Rows at or past buffer_lengths[c]
 *             (and every row of an unused chunk) are 0.
 * Other arguments as in mla_gather_latent, for all chunks at once.
 * Errors: host MLA_ERR_ARG (null pointers, sizes < 1, num_pages * page_size
 * >= 2^31, max_chunks > 65535), MLA_ERR_LAUNCH; device MLA_DEV_BAD_PAGE (a
 * position outside the page table or a page id outside [0, num_pages): that
 * row's entry is 0), MLA_DEV_TIMEOUT seen on entry (no work).
 */
mla_status_t mla_chunk_cache_rows(int32_t* cache_rows, const int32_t* page_table,
                                  int32_t num_pages, int32_t page_size, int32_t max_pages_per_seq,
                                  const uint32_t* buffer_row_offsets, const uint32_t* cache_offsets,
                                  const int32_t* buffer_lengths, int32_t max_chunks,
                                  int32_t batch_size, uint32_t buffer_token_size, int32_t* d_status,
                                  mla_stream_t stream);

/*
 * 3'. Up-projection of one plan chunk with the c_kv rows read straight from
 * the paged cache ("mla_prefill_decode_graph_bf16", Args: w_k, w_uv, and the
 * kv_collection the prefill branch reads the chunk's latent rows from).  The
 * result equals mla_gather_latent followed by mla_upproject, without the c_kv
 * buffer in between.
 *
 * Arguments as in mla_upproject, with c_kv_buf replaced by
 * kv_cache:       the cache as [num_cache_rows][576] dtype
 * cache_rows:     the chunk's [buffer_token_size] row of mla_chunk_cache_rows
 *                 (buffer row r is cache row cache_rows[r])
 * num_cache_rows: num_pages * page_size; an entry outside [0, num_cache_rows)
 *                 is reported (MLA_DEV_BAD_PAGE) and read as row 0.
 * buffer_lengths is required here.
 */
mla_status_t mla_upproject_paged(void* k_nope, void* v, const void* kv_cache,
                                 const int32_t* cache_rows, int32_t num_cache_rows,
                                 const int32_t* buffer_lengths, int32_t chunk,
                                 uint32_t buffer_token_size, const void* w_k, const void* w_uv,
                                 int32_t num_heads, int32_t dtype, float ckv_scale, float w_scale,
                                 float kv_out_inv_scale, int32_t* d_status, mla_stream_t stream);

/*
 * 4. Prefill attention for one plan chunk.  Follows "flare_mla_prefill_dispatch"
 * (Args: output [total_q_tokens, num_heads, v_depth]; q [total_q_tokens,
 * num_heads, q_depth]; k, v (ragged K nope and V); k_rope [cache_len, 1,
 * q_depth - depth]; valid_length (cumulative row offsets); max_prompt_len;
 * scale; cache_offsets) with the causal mask of mla_prefill_decode_graph_bf16
 * (Parameters: mask_str).
 *
 * New token i of sequence b sits at context position P = cache_lengths[b] + i.
 * The chunk's keys of sequence b are buffer rows r in [buffer_row_offsets
 * [chunk][b], buffer_row_offsets[chunk][b+1]) at positions j = cache_offsets
 * [chunk][b] + (r - buffer_row_offsets[chunk][b]); key r is visible iff j <= P.
 * Score = scale * q_scale * k_scale * (q[t][h][0:128] . k_nope[r][h] +
 * q[t][h][128:192] . k_rope[r]); the chunk's softmax-weighted V (times v_scale)
 * and log-sum-exp (natural log) are merged with the running fp32 result in
 * o_acc / lse_acc.  In the chunk that holds position P the merged result is
 * written to out (bf16) and lse; in earlier chunks it is kept in o_acc/lse_acc.
 * Rows whose position lies before the chunk are left untouched.
 *
 * out:      [total_q_tokens][num_heads][128] bf16, output
 * lse:      [total_q_tokens][num_heads] fp32 output, or NULL
 * o_acc:    [total_q_tokens][num_heads][128] fp32 scratch, lse_acc [total_q_tokens]
 *           [num_heads] fp32 scratch; both may be NULL only when max_chunks == 1.
 *           They carry state from one chunk's call to the next.
 * q:        [total_q_tokens][num_heads][192] dtype (128 nope, then 64 rope)
 * k_nope:   [buffer_token_size][num_heads][128] dtype; k_rope: [buffer_token_size][64]
 * v:        [buffer_token_size][num_heads][128] bf16, or f16 for MLA_E4M3 (the
 *           e4m3-rounded values mla_upproject writes)
 * Rows of k_nope/k_rope beyond a sequence's keys are read but masked; rows of v
 * beyond them are never used.
 * max_prompt_len: largest new-token count of any sequence (sizes the grid).
 * Errors: host MLA_ERR_ARG / MLA_ERR_DTYPE / MLA_ERR_GEOMETRY, MLA_ERR_LAUNCH.
 * Device:
 *   MLA_DEV_TIMEOUT          a pipeline wait ran out; rows not yet stored keep
 *                            whatever out held before.
 *   MLA_DEV_TOO_MANY_CHUNKS  a row needs merge state but o_acc / lse_acc are
 *                            NULL (more than one chunk holds its keys, or the
 *                            plan was truncated at max_chunks); that row of
 *                            out is not written.
 *   MLA_DEV_BAD_OFFSETS      input_row_offsets[b+1] > total_q_tokens: sequence
 *                            b is left out (its rows of out are not written).
 */
mla_status_t mla_prefill_attention(void* out, float* lse, float* o_acc, float* lse_acc,
                                   const void* q, const void* k_nope, const void* v,
                                   const void* k_rope, const uint32_t* input_row_offsets,
                                   const uint32_t* cache_lengths,
                                   const uint32_t* buffer_row_offsets,
                                   const uint32_t* cache_offsets, const int32_t* buffer_lengths,
                                   int32_t chunk, int32_t max_chunks, int32_t batch_size,
                                   int32_t num_heads, int32_t max_prompt_len,
                                   int32_t total_q_tokens, uint32_t buffer_token_size,
                                   float scale, float q_scale, float k_scale, float v_scale,
                                   int32_t dtype, int32_t* d_status, mla_stream_t stream);

/*
 * 4'. Prefill attention for one plan chunk with k_rope read straight from the
 * paged cache, as "flare_mla_prefill_dispatch" does (Parameters: k_rope_t is a
 * KVCacheMHAOperand; Args: k_rope with shape [cache_len, 1, 64] and
 * cache_offsets, the per-sequence start of the chunk in the cache).  No
 * k_rope buffer is needed, so mla_gather_latent need not write one.
 *
 * Same arguments, results and errors as mla_prefill_attention, except that
 * k_rope is replaced by
 * kv_cache:       the cache as [num_cache_rows][576] dtype; columns 512..575
 *                 are k_rope
 * cache_rows:     the chunk's [buffer_token_size] row of mla_chunk_cache_rows:
 *                 key r (a buffer row) is cache row cache_rows[r]
 * num_cache_rows: num_pages * page_size.
 * k_nope and v stay buffer rows.  Device errors add MLA_DEV_BAD_PAGE: a key's
 * entry is outside [0, num_cache_rows) (its score is then meaningless).
 */
mla_status_t mla_prefill_attention_paged(void* out, float* lse, float* o_acc, float* lse_acc,
                                         const void* q, const void* k_nope, const void* v,
                                         const void* kv_cache, const int32_t* cache_rows,
                                         int32_t num_cache_rows,
                                         const uint32_t* input_row_offsets,
                                         const uint32_t* cache_lengths,
                                         const uint32_t* buffer_row_offsets,
                                         const uint32_t* cache_offsets,
                                         const int32_t* buffer_lengths, int32_t chunk,
                                         int32_t max_chunks, int32_t batch_size,
                                         int32_t num_heads, int32_t max_prompt_len,
                                         int32_t total_q_tokens, uint32_t buffer_token_size,
                                         float scale, float q_scale, float k_scale,
                                         float v_scale, int32_t dtype, int32_t* d_status,
                                         mla_stream_t stream);

/*
 * Prefill attention for one plan chunk without caller scratch.  The pages have
 * no counterpart to this entry point.
 *
 * Same arguments and results as mla_prefill_attention, minus o_acc and lse_acc:
 * the fp32 state carried from one chunk's call to the next lives in a fixed
 * array inside this library (MLA_NOALLOC_MAX_ROWS rows of 129 floats, about
 * 16.9 MB, held on every GPU that loads the library until the process exits).
 * It exists for callers that cannot allocate device memory: code running
 * inside a host framework that owns the whole device memory pool and offers no
 * allocator, and loops that must not call cudaMalloc because it synchronises
 * the device.  This function allocates nothing and calls no allocating routine.
 *
 * - total_q_tokens * num_heads must be <= MLA_NOALLOC_MAX_ROWS; larger calls
 *   return MLA_ERR_WORKSPACE (use mla_prefill_attention with caller scratch).
 * - Every call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress), so the address stays right after a
 *   cudaDeviceReset.  The first call on a device may load the library's
 *   device code there; make that first call before any stream capture.
 *   Failure of the lookup returns MLA_ERR_LAUNCH.
 * - All calls share the one array and it keeps the last call's contents.  A
 *   multi-chunk sequence of calls (chunk 0, 1, ...) relies on that; calls from
 *   different sequences that overlap on the GPU (other streams, other threads)
 *   race on the array.  Nothing in it needs to start at zero.
 */
#define MLA_NOALLOC_MAX_ROWS 32768
mla_status_t mla_prefill_attention_noalloc(void* out, float* lse, const void* q,
                                           const void* k_nope, const void* v, const void* k_rope,
                                           const uint32_t* input_row_offsets,
                                           const uint32_t* cache_lengths,
                                           const uint32_t* buffer_row_offsets,
                                           const uint32_t* cache_offsets,
                                           const int32_t* buffer_lengths, int32_t chunk,
                                           int32_t max_chunks, int32_t batch_size,
                                           int32_t num_heads, int32_t max_prompt_len,
                                           int32_t total_q_tokens, uint32_t buffer_token_size,
                                           float scale, float q_scale, float k_scale,
                                           float v_scale, int32_t dtype, int32_t* d_status,
                                           mla_stream_t stream);

/*
 * Workspace bytes needed by mla_prefill for these sizes (plan tables, the
 * chunk's latent, k_rope, K and V buffers, and the fp32 merge state when
 * max_chunks > 1).  The buffers follow "mla_prefill_decode_graph_bf16" (Args:
 * buffer_row_offsets, cache_offsets, buffer_length) and
 * "flare_mla_prefill_dispatch" (Args: k, v, k_rope); the pages size none of
 * them, so this call has no counterpart there.  Host only; returns 0 for
 * invalid sizes (B < 0, H < 1, total_q_tokens < 0, max_chunks < 1,
 * buffer_token_size == 0) or an unknown dtype.
 */
size_t mla_prefill_workspace_bytes(int32_t batch_size, int32_t num_heads,
                                   int32_t total_q_tokens, int32_t max_chunks,
                                   uint32_t buffer_token_size, int32_t dtype);

/*
 * Fused path: plan, then for every chunk c < max_chunks gather, up-project and
 * attend, all enqueued on `stream` with no host synchronisation (chunks the
 * plan leaves unused exit on the device).  Follows the prefill branch of
 * "mla_prefill_decode_graph_bf16" with the tables of "mla_prefill_plan".
 * Errors add MLA_ERR_ARG for num_pages * page_size >= 2^31.
 *
 * out [total_q_tokens][num_heads][128] bf16 output; lse [total_q_tokens]
 * [num_heads] fp32 output or NULL.  Inputs as in the stage entry points.  For
 * e4m3, K and V are stored in e4m3 in the cache's descale domain (out scale
 * 1/ckv_scale), so the attention uses k_scale = v_scale = ckv_scale.
 * workspace: device memory of at least mla_prefill_workspace_bytes(...) bytes,
 * 256-byte aligned.  *d_status is cleared first.
 */
mla_status_t mla_prefill(void* out, float* lse, const void* q, const uint32_t* input_row_offsets,
                         const uint32_t* cache_lengths, const void* kv_cache,
                         const int32_t* page_table, int32_t num_pages, int32_t page_size,
                         int32_t max_pages_per_seq, const void* w_k, const void* w_uv,
                         int32_t batch_size, int32_t num_heads, int32_t total_q_tokens,
                         int32_t max_prompt_len, uint32_t buffer_token_size, int32_t max_chunks,
                         float scale, float q_scale, float ckv_scale, float w_scale,
                         int32_t dtype, void* workspace, size_t workspace_bytes,
                         int32_t* d_status, mla_stream_t stream);

/*
 * Partitions per sequence the library uses for mla_decode when num_partitions
 * is 0 (size the workspace with it).  It cuts every sequence's keys into
 * pieces of about the same size -- between 256 and 2048 keys, chosen from the
 * batch's sizes for about one item per SM pair of the GPU -- so that
 * short and long sequences make items of equal cost; this returns the most
 * pieces a sequence can get.  max_keys: max_seq_len for dense decode (the
 * longest context, new tokens included), the list stride for sparse decode.
 * Follows "mla_prefill_decode_graph_bf16" (Args: num_partitions_in, the
 * caller's override; max_seq_len).  Host only; 1 for invalid sizes.
 */
int32_t mla_decode_partitions(int32_t batch_size, int32_t num_heads, int32_t max_new_tokens,
                              int32_t max_keys);

/*
 * Workspace bytes mla_decode needs: the 576-wide query rows (bf16), every
 * partition's latent result (bf16) and LSE (fp32), and the merged bf16 latent
 * result.
 * The decode branch of "mla_prefill_decode_graph_bf16" (Args: w_uk, w_uv,
 * num_partitions_in) sizes no buffer, so this call has no counterpart on the
 * pages.  Host only; 0 for invalid sizes.
 */
size_t mla_decode_workspace_bytes(int32_t num_heads, int32_t total_q_tokens, int32_t num_partitions);

/*
 * Decode attention in the absorbed form.  Follows the decode branch of
 * "mla_prefill_decode_graph_bf16" (Args: q [tot_seq_len, num_heads, 192];
 * w_uk [num_heads, kv_latent_dim, qk_nope_head_dim], projecting each head's
 * nope query into latent space; w_uv [num_heads, v_head_dim, kv_latent_dim],
 * projecting the result back; scale; num_partitions_in; and the sparse form:
 * d_indices, indices_stride, topk_lengths, attn_sink_ptr).
 *
 * New token i of sequence b is row t = input_row_offsets[b] + i of q and out.
 * For head h:
 *   q_lat = w_uk[h] . q[t][h][0:128]                          (512 values)
 *   s_j   = scale * (q_lat . c_kv_j + q[t][h][128:192] . k_rope_j)
 *   out[t][h] = w_uv[h] . sum_j softmax(s)_j c_kv_j           (128 values)
 * over keys j, each a 576-wide cache row (c_kv = values 0..511, k_rope =
 * 512..575):
 *   - dense (d_indices NULL): context positions 0 .. cache_lengths[b] + i of
 *     sequence b, read from page page_table[b][j / page_size], slot
 *     j % page_size (the cache holds the new tokens' rows too);
 *   - sparse (d_indices given): the physical cache rows d_indices[b *
 *     indices_stride + e] (row = page * page_size + slot) for e <
 *     topk_lengths[b] (indices_stride when topk_lengths is NULL), the same
 *     list for every token of sequence b, no causal limit.
 * With attn_sink given, sink = attn_sink[b] is one more logit in every
 * softmax of sequence b with no value row: out is scaled by
 * e^LSE / (e^LSE + e^sink) and lse includes it.  The keys are split into
 * ranges whose partial results merge by LSE; the result does not depend on
 * the split beyond rounding.
 * num_partitions > 0 splits every sequence into that many ranges; 0 lets the
 * library pick ranges of equal size (mla_decode_partitions).
 * q_lat and the merged latent result are rounded to bf16 for the tensor-core
 * projections, and each partition's normalised latent result is stored as
 * bf16; scores, softmax, LSE and the merge arithmetic run in fp32.
 *
 * out:      [total_q_tokens][num_heads][128] bf16, output
 * lse:      [total_q_tokens][num_heads] fp32 output (natural log), or NULL
 * q:        [total_q_tokens][num_heads][192] bf16
 * kv_cache: [num_pages][page_size][576] bf16
 * w_uk [num_heads][512][128], w_uv [num_heads][128][512] bf16
 * input_row_offsets [B+1], cache_lengths [B], page_table [B][max_pages_per_seq]
 * max_new_tokens: largest new-token count of any sequence (sizes the grid)
 * max_seq_len: largest context (cached + new tokens) of any sequence; bounds
 *            the partitions when num_partitions is 0
 * workspace: device memory of at least mla_decode_workspace_bytes(num_heads,
 *            total_q_tokens, num_partitions or mla_decode_partitions(...)),
 *            256-byte aligned.
 * Errors: host MLA_ERR_DTYPE (bf16 only: the page's graph is bf16),
 * MLA_ERR_GEOMETRY, MLA_ERR_ARG (null or misaligned pointers, bad sizes),
 * MLA_ERR_WORKSPACE, MLA_ERR_LAUNCH.  Device MLA_DEV_BAD_OFFSETS
 * (input_row_offsets[b+1] > total_q_tokens: sequence b left out),
 * MLA_DEV_BAD_PAGE (a page id or sparse row out of range: those keys read
 * zeros or row 0, and the result of their rows is not meaningful),
 * MLA_DEV_TIMEOUT.
 */
mla_status_t mla_decode(void* out, float* lse, const void* q, const uint32_t* input_row_offsets,
                        const uint32_t* cache_lengths, const void* kv_cache, const int32_t* page_table,
                        int32_t num_pages, int32_t page_size, int32_t max_pages_per_seq,
                        const void* w_uk, const void* w_uv, int32_t batch_size, int32_t num_heads,
                        int32_t total_q_tokens, int32_t max_new_tokens, int32_t max_seq_len,
                        int32_t num_partitions, float scale, const int32_t* d_indices,
                        int32_t indices_stride,
                        const int32_t* topk_lengths, const float* attn_sink, int32_t dtype,
                        void* workspace, size_t workspace_bytes, int32_t* d_status,
                        mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_PREFILL_H */
