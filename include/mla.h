/*
 * mla.h - C ABI of the B300 (sm_103a) Multi-head Latent Attention decode library.
 *
 * The method (DeepSeek-V2, as explained on the "DeepSeek-V2" explainer page,
 * Part B Steps 5-8, and the DeepSeek-V2 paper breakdown, "How It Works"):
 * every cached token keeps only a 512-number latent c (Step 5, eq. 9) and one
 * 64-number rotated RoPE key k^R shared by all heads (Step 7), i.e. a
 * 576-number row per token per layer (Step 8).  The per-head key k = W^UK c
 * is never built: the query is moved into latent space instead (Step 6,
 * "absorbing" W^UK), all 128 heads score against the same latent rows, the
 * content and RoPE scores add inside the softmax (Step 7), and W^UV is
 * applied to the latent attention output afterwards (Step 6: the values are
 * never materialised either).
 *
 * Fixed shapes: H = 128 heads, d_c = 512 latent, d_r = 64 RoPE, d_h = 128 per
 * head, row width D = 576, page = 64 tokens.  Element types: bf16 tensors are
 * passed as `void*` holding IEEE bfloat16 bit patterns; lse is float32.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *    row-major, 16-byte aligned.  The library allocates no device memory.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work; they return before the GPU has run it.
 *  - Host-side argument checks happen before anything is enqueued; on a
 *    failure the call returns the error code and launches nothing.
 *  - Faults found on the device (a block-table entry outside [0, num_pages),
 *    a sequence length outside [0, max_pages*64], a wait that timed out) never
 *    trap: the kernel records a bit in the library's device status word,
 *    clamps or skips the offending access, and finishes.  Read the word with
 *    mla_get_device_status().
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, so CUDA callers can pass their stream directly. */
typedef struct CUstream_st *mla_stream_t;

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,   /* null pointer, negative or zero size where one is required */
    MLA_ERR_SHAPE = 2,         /* sizes outside the supported range */
    MLA_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned */
    MLA_ERR_WORKSPACE = 4,     /* workspace null or smaller than mla_decode_workspace_size() */
    MLA_ERR_UNSUPPORTED = 5,   /* heads != 128, or the current device is not sm_103 */
    MLA_ERR_CUDA = 6,          /* a CUDA runtime/driver call failed while enqueuing */
    MLA_ERR_DEVICE_FAULT = 7   /* a device-side guard tripped (see mla_get_device_status) */
} mla_status_t;

/* Bits of the device status word. */
#define MLA_DEV_BAD_BLOCK_TABLE 0x1u  /* a block-table entry outside [0, num_pages) was read */
#define MLA_DEV_BAD_SEQ_LEN     0x2u  /* a sequence length outside [0, max_pages * 64], or (cache
                                         write) a new token's position negative or past the
                                         block table */
#define MLA_DEV_WAIT_TIMEOUT    0x4u  /* an on-chip wait gave up (kernel bailed out) */
#define MLA_DEV_PLAN_OVERFLOW   0x8u  /* the split plan did not fit the workspace */
#define MLA_DEV_SELECT_OVERFLOW 0x10u /* the top-k selection counted more than k picks (an internal
                                         inconsistency; the extra picks are dropped, never written) */

/*
 * mla_absorb_q - move the content query into latent space (explainer Step 6,
 * the 2-d toy example and "absorbing one matrix into another"), and append the
 * decoupled RoPE query unchanged (Step 7):
 *     q_abs[n,h,0:512]   = W_UK[h]^T q_nope[n,h,:]      (fp32 accumulate, bf16 out)
 *     q_abs[n,h,512:576] = q_rope[n,h,:]
 *
 * q_nope  [n_tokens, n_heads, 128] bf16
 * q_rope  [n_tokens, n_heads, 64]  bf16
 * w_uk    [n_heads, 128, 512]      bf16, W_UK[h] maps a latent c to the key k = W_UK[h] c
 * q_abs   [n_tokens, n_heads, 576] bf16 (output)
 * n_heads must be 128; 1 <= n_tokens <= 65536.
 */
mla_status_t mla_absorb_q(const void *q_nope, const void *q_rope, const void *w_uk, void *q_abs,
                          int n_tokens, int n_heads, mla_stream_t stream);

/*
 * mla_decode_workspace_size - bytes of device workspace mla_decode needs for
 * this batch.  num_splits is the value that will be passed to mla_decode
 * (0 = automatic split-KV plan).  Returns 0 for invalid sizes.
 */
size_t mla_decode_workspace_size(int batch, int q_len, int num_splits);

/*
 * mla_decode - weight-absorbed MLA attention over a paged latent cache
 * (explainer Steps 6-8).  For every sequence b, query token t and head h:
 *     s_j   = scale * q_abs[b,t,h,:] . row_j          (576-wide: content + RoPE, Step 7)
 *     o_lat = sum_j softmax(s)_j * row_j[0:512]        (latent output, Step 6)
 *     lse   = log sum_j exp(s_j)                       (natural log)
 * over the visible tokens j of sequence b, where row_j =
 * kv_pool[block_table[b, j / 64], j % 64, :].
 *
 * q_abs        [batch, q_len, n_heads, 576] bf16 (from mla_absorb_q, or given)
 * kv_pool      [num_pages, 64, 576] bf16; row = [c (512) | k^R (64)]
 * block_table  [batch, max_pages] int32, device; entries past ceil(L_b/64) are not read
 * seq_lens     [batch] int32, device; L_b = cached tokens of sequence b (never read
 *              on the host; the q_len new tokens are included when causal)
 * scale        softmax scale (1/sqrt(192) for DeepSeek-V2 shapes)
 * causal       0: every query sees all L_b tokens.  1: query t sees tokens
 *              0 .. L_b - q_len + t (the new tokens are the last q_len rows).
 * num_splits   0 = automatic split-KV plan from the sequence lengths and SM count;
 *              k > 0 forces k splits per (sequence, query token) (testing/tuning).
 * o_lat        [batch, q_len, n_heads, 512] bf16 (output)
 * lse          [batch, q_len, n_heads] float32 (output); a query with no
 *              visible token gets o_lat = 0 and lse = -inf.
 * workspace    device scratch of at least mla_decode_workspace_size() bytes,
 *              owned by the caller; must not be shared by calls that overlap.
 * Limits: n_heads == 128; 1 <= batch; 1 <= q_len <= 64; batch * q_len <= 65536;
 *         max_pages >= 1; num_pages >= 1.
 */
mla_status_t mla_decode(const void *q_abs, const void *kv_pool, const int32_t *block_table,
                        const int32_t *seq_lens, int batch, int q_len, int n_heads, int num_pages,
                        int max_pages, float scale, int causal, int num_splits, void *o_lat,
                        float *lse, void *workspace, size_t workspace_bytes, mla_stream_t stream);

/* Size of the library-owned scratch used by mla_decode_static_scratch (64 MiB). */
#define MLA_STATIC_SCRATCH_BYTES (64u << 20)

/*
 * mla_decode_static_scratch - mla_decode for callers that cannot allocate device
 * memory.  The paper has no counterpart to this call; it exists for integration only.
 *
 * Some callers have no way to obtain device memory: a plug-in running inside a host
 * application that owns every device allocation and hands plug-ins no allocator, or a
 * serving loop whose rule is "no cudaMalloc after start-up" because an allocation can
 * synchronise the device and stall the requests in flight.  This call takes the same
 * arguments as mla_decode minus the workspace, and uses instead a fixed scratch array
 * of MLA_STATIC_SCRATCH_BYTES that the library keeps in device memory.  Every GPU that
 * loads the library holds that array until the process exits.  The call allocates
 * nothing itself.
 *
 * Limit: requests whose mla_decode_workspace_size(batch, q_len, num_splits) exceeds
 * MLA_STATIC_SCRATCH_BYTES are rejected with MLA_ERR_WORKSPACE before anything is
 * enqueued.  With the automatic plan (num_splits = 0) that admits batch * q_len up to 90.
 *
 * First call per device: it looks up the device address of the array (with that
 * device current), once; make that first call before any stream capture begins.
 *
 * Sharing: all calls on a device use the same array, which keeps whatever the previous
 * call left there.  Nothing in it needs to start at zero (the planning kernel rewrites
 * every field the later kernels read), but calls whose GPU execution overlaps -- two
 * streams, or two host threads on one device -- race on the array and corrupt each
 * other's results.  Keep them ordered: one stream, or synchronise between them.
 */
mla_status_t mla_decode_static_scratch(const void *q_abs, const void *kv_pool, const int32_t *block_table,
                                       const int32_t *seq_lens, int batch, int q_len, int n_heads,
                                       int num_pages, int max_pages, float scale, int causal, int num_splits,
                                       void *o_lat, float *lse, mla_stream_t stream);

/*
 * mla_combine - merge attention results computed over disjoint token sets
 * (the split-KV reduction of mla_decode, exposed for callers that split a
 * sequence themselves, e.g. across devices):
 *     lse[m] = log sum_r exp(lse_parts[r,m]);  o[m,:] = sum_r exp(lse_parts[r,m] - lse[m]) o_parts[r,m,:]
 * o_parts [n_parts, rows, 512] float32, lse_parts [n_parts, rows] float32,
 * o_out [rows, 512] bf16, lse_out [rows] float32.  Parts with lse = -inf
 * carry no weight; a row whose parts are all -inf gets o = 0, lse = -inf.
 */
mla_status_t mla_combine(const float *o_parts, const float *lse_parts, int n_parts, int rows,
                         void *o_out, float *lse_out, mla_stream_t stream);

/*
 * mla_up_proj - regenerate the per-head output from the latent attention output
 * (explainer Step 5: values v = W^UV c; Step 6: applied after attention):
 *     out[n,h,:] = W_UV[h] o_lat[n,h,:]          (fp32 accumulate, bf16 out)
 * o_lat [n_tokens, n_heads, 512] bf16, w_uv [n_heads, 128, 512] bf16,
 * out [n_tokens, n_heads, 128] bf16.  n_heads must be 128; 1 <= n_tokens <= 65536.
 */
mla_status_t mla_up_proj(const void *o_lat, const void *w_uv, void *out, int n_tokens, int n_heads,
                         mla_stream_t stream);

/*
 * mla_cache_append - write the cache rows of new tokens, the step before the
 * decode (explainer Step 5, the paper's equation 9: the hidden vector is
 * projected down to the latent c = W^DKV h, 512 numbers; Step 7: the token's
 * one position key shared by all heads is k^R = RoPE(W^KR h), 64 numbers;
 * Step 8: the row kept is [c | k^R]):
 *     row[n, 0:512]   = W^DKV h[n]                     (fp32 accumulate)
 *     row[n, 512:576] = RoPE_pos(W^KR h[n])            (fp32, then the row to bf16)
 *     kv_pool[block_table[b, pos / 64], pos % 64, :] = row[n]
 * for token t of sequence b (n = b * q_len + t), at position
 * pos = seq_lens[b] - q_len + t: the lengths already count the new tokens, as
 * in mla_decode's causal mode.  A decode step is q_len = 1; a prefill of a
 * prompt of L tokens is q_len = L with seq_lens = L.
 *
 * RoPE (the pages give no formula; the reading taken): coordinates (2i, 2i+1)
 * of k^R form pair i, turned counter-clockwise by pos * rope_base^(-2i/64):
 *     (x0, x1) -> (x0 cos a - x1 sin a, x0 sin a + x1 cos a).
 *
 * h            [batch * q_len, d_model] bf16, the new tokens' hidden vectors
 * w_dkv        [512, d_model] bf16, row r gives c[r] = W^DKV[r,:] . h
 * w_kr         [64, d_model] bf16, likewise for k^R before the rotation
 * block_table  [batch, max_pages] int32, device; seq_lens [batch] int32, device
 * rope_base    > 1 (10000 for DeepSeek-V2 shapes)
 * kv_pool      [num_pages, 64, 576] bf16, written in place; only the rows of
 *              the new tokens change.  The call needs no workspace.
 * A token whose position is negative or beyond the block table, or whose page
 * is outside [0, num_pages), is not written: the status word records
 * MLA_DEV_BAD_SEQ_LEN or MLA_DEV_BAD_BLOCK_TABLE.  Two new tokens mapped to the
 * same pool row race; the caller's block table must not do that.
 * Limits: 1 <= batch * q_len <= 2^20; d_model a multiple of 64, at most 65536.
 */
mla_status_t mla_cache_append(const void *h, const void *w_dkv, const void *w_kr, const int32_t *block_table,
                              const int32_t *seq_lens, int batch, int q_len, int d_model, int num_pages,
                              int max_pages, float rope_base, void *kv_pool, mla_stream_t stream);

/*
 * mla_cache_append_compressed - the cache write with token-level compression
 * (the DeepSeek page's "KV cache compression" section: consecutive tokens are
 * grouped in blocks of m, and each block keeps one key-value vector, the
 * component-wise weighted sum of its tokens' vectors, with weights from a
 * softmax over the block's tokens of each component of z = W^Z x).  Here the
 * vector is the 576-number cache row of each token as mla_cache_append writes
 * it (k^R turned at the token's own position), and z = W^Z h:
 *     row[g, k] = sum_i w[i, k] * row_tok[g*m + i, k],
 *     w[i, k]   = exp(z[g*m + i, k]) / sum_j exp(z[g*m + j, k])
 * The merged row of block j of sequence b goes to compressed position
 * P = seq_lens[b] - n_blocks + j (seq_lens counts compressed rows, the new ones
 * included) and merges the tokens at positions P*m .. P*m + m - 1, h rows
 * (b * n_blocks + j) * m + i.  mla_decode then runs on the compressed cache
 * unchanged (each compressed row is one "token").  Only whole blocks are written.
 *
 * h      [batch * n_blocks * m, d_model] bf16; w_dkv [512, d_model], w_kr [64, d_model],
 * w_z    [576, d_model] bf16 (row-major, z[k] = W^Z[k,:] . h)
 * m      tokens per block: a power of two, 1 to 128 (1: the plain cache write)
 * Other arguments, limits and device-side checks as mla_cache_append (positions and
 * pages are compressed ones); batch * n_blocks * m <= 2^20.
 */
mla_status_t mla_cache_append_compressed(const void *h, const void *w_dkv, const void *w_kr, const void *w_z,
                                         const int32_t *block_table, const int32_t *seq_lens, int batch,
                                         int n_blocks, int m, int d_model, int num_pages, int max_pages,
                                         float rope_base, void *kv_pool, mla_stream_t stream);

/*
 * The indexer path (the DeepSeek page, "KV cache data movement minimization"):
 * every cached token also keeps a small index vector k_idx, paged exactly like
 * the latent cache (same block table, same 64-token pages).  A decoding token
 * scores every cached token with one dot product against its index query q_idx,
 * keeps the k best, and attends over those tokens only, so the latent rows read
 * are k per sequence instead of L_b.  The pages leave the query side of the
 * index score open; the reading taken is a per-sequence index query of the
 * index vectors' width, supplied by the caller.
 *
 * mla_index_scores - the index scores of every cached token:
 *     scores[b, t] = q_idx[b, :] . idx_pool[block_table[b, t / 64], t % 64, :]
 * for t < L_b = seq_lens[b] (fp32 products and sums); entries t >= L_b are not
 * written.  A token on a page outside [0, num_pages) gets a NaN score and sets
 * MLA_DEV_BAD_BLOCK_TABLE.
 *
 * q_idx        [batch, d_idx] bf16
 * idx_pool     [num_pages, 64, d_idx] bf16
 * block_table  [batch, max_pages] int32, device; seq_lens [batch] int32, device
 * scores       [batch, max_pages * 64] float32 (output)
 * Limits: d_idx in {32, 64, 128, 256}; 1 <= batch <= 65536.
 */
mla_status_t mla_index_scores(const void *q_idx, const void *idx_pool, const int32_t *block_table,
                              const int32_t *seq_lens, int batch, int d_idx, int num_pages, int max_pages,
                              float *scores, mla_stream_t stream);

/*
 * mla_index_scores_e4m3 - the same scores over an index cache held in 8 bits: every index
 * vector is d_idx FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * subnormals at exponent 0, S.1111.111 NaN, no infinity) and one float32 scale per token:
 *     scores[b, t] = idx_scale[p, t % 64] * sum_d q_idx[b, d] * value(idx_codes[p, t % 64, d]),
 *     p = block_table[b, t / 64]
 * (each product and the sum in fp32, then the scale).  Half the index bytes of the bf16 form.
 * idx_codes [num_pages, 64, d_idx] uint8, 16-byte aligned; idx_scale [num_pages, 64] float32.
 * Other arguments, limits and device-side checks as mla_index_scores.
 */
mla_status_t mla_index_scores_e4m3(const void *q_idx, const void *idx_codes, const float *idx_scale,
                                   const int32_t *block_table, const int32_t *seq_lens, int batch, int d_idx,
                                   int num_pages, int max_pages, float *scores, mla_stream_t stream);

/*
 * mla_topk_gather - the k best tokens of each sequence and their cache rows.
 * Sequence b selects the min(k, L_b) positions with the largest scores[b, t],
 * t < L_b; equal scores go to the lower position first, and a NaN score ranks
 * below every number (-inf included).  Outputs:
 *     sel_index[b, 0:n]        the selected positions, ascending; -1 after them
 *     sel_pool[b*npk + j]      page j of sequence b's selected rows, npk = ceil(k / 64):
 *                              row i is kv_pool's row of position sel_index[b, i];
 *                              rows i >= n are zero
 *     sel_block_table[b, j]    b * npk + j
 *     sel_lens[b]              n = min(k, L_b)
 * so mla_decode(q_abs, sel_pool, sel_block_table, sel_lens, ..., num_pages = batch * npk,
 * max_pages = npk, causal = 0) attends over exactly the selected tokens.
 *
 * scores           [batch, max_pages * 64] float32 (from mla_index_scores)
 * kv_pool          [num_pages, 64, 576] bf16; block_table [batch, max_pages] int32
 * sel_index        [batch, k] int32; sel_pool [batch * npk, 64, 576] bf16;
 * sel_block_table  [batch, npk] int32; sel_lens [batch] int32 (all outputs, device)
 * A selected row on a page outside [0, num_pages) is written as zeros and sets
 * MLA_DEV_BAD_BLOCK_TABLE.
 * Limits: 1 <= k <= 2^18; 1 <= batch <= 65536.
 */
mla_status_t mla_topk_gather(const float *scores, const int32_t *seq_lens, const void *kv_pool,
                             const int32_t *block_table, int batch, int num_pages, int max_pages, int k,
                             int32_t *sel_index, void *sel_pool, int32_t *sel_block_table, int32_t *sel_lens,
                             mla_stream_t stream);

/*
 * mla_decode_sparse_workspace_size - bytes of workspace mla_decode_sparse needs
 * (the scores, the selection and its compact pool, and mla_decode's workspace).
 * Returns 0 for invalid sizes.
 */
size_t mla_decode_sparse_workspace_size(int batch, int max_pages, int k);

/*
 * mla_decode_sparse - the indexer decode of one new token per sequence:
 * mla_index_scores, mla_topk_gather, then mla_decode (non-causal) over the
 * selected rows: for every sequence b and head h,
 *     o_lat[b, 0, h] = sum_{t in S_b} softmax_t(scale * q_abs[b, 0, h] . row_t) row_t[0:512]
 *     lse[b, 0, h]   = log sum_{t in S_b} exp(scale * q_abs[b, 0, h] . row_t)
 * where S_b = the selected positions.  q_abs [batch, 1, 128, 576] bf16; sel_index
 * [batch, k] int32 receives the selection when not NULL.  idx_scale NULL: idx_pool is the bf16
 * index cache of mla_index_scores; otherwise idx_pool holds E4M3 codes and idx_scale their
 * per-token scales, as mla_index_scores_e4m3.  Other arguments as above
 * and as mla_decode; workspace of at least mla_decode_sparse_workspace_size() bytes,
 * 16-byte aligned, not shared by overlapping calls.  A selection of at most 16 pages per
 * sequence (k <= 1024) is decoded without splitting a sequence, and the top-k kernel writes that
 * decode plan itself: four kernels are enqueued (five for larger k).
 */
mla_status_t mla_decode_sparse(const void *q_abs, const void *q_idx, const void *kv_pool, const void *idx_pool,
                               const float *idx_scale, const int32_t *block_table, const int32_t *seq_lens,
                               int batch, int n_heads, int d_idx, int num_pages, int max_pages, int k, float scale,
                               void *o_lat, float *lse, int32_t *sel_index, void *workspace,
                               size_t workspace_bytes, mla_stream_t stream);

/*
 * mla_get_device_status - synchronise `stream`, then read and clear the
 * library's device status word on the current device (MLA_DEV_* bits).
 * Returns MLA_ERR_DEVICE_FAULT if any bit was set, MLA_ERR_CUDA if the stream
 * reported an error, MLA_OK otherwise.  err_word may be NULL.
 *
 * There is one word per device, shared by every call, stream and host thread
 * of the process on that device: kernels only ever set bits in it (atomic OR),
 * and this call reads and clears it after synchronising `stream` alone.  A bit
 * set by work on another stream may therefore be reported here, or missed if
 * that work has not finished; callers that need per-stream attribution keep
 * one stream per device, or synchronise the device before reading.
 */
mla_status_t mla_get_device_status(mla_stream_t stream, uint32_t *err_word);

/*
 * mla_cache_bytes - bytes of latent cache for `tokens` tokens over `layers`
 * layers: tokens * layers * (d_c + d_r) * bytes_per_elem (explainer Step 8:
 * 512 + 64 = 576 numbers per token per layer).  Host only.
 */
uint64_t mla_cache_bytes(int64_t tokens, int layers, int d_c, int d_r, int bytes_per_elem);

/* Human-readable name of a status code (static string). */
const char *mla_status_string(mla_status_t status);

/* Library ABI version (major * 100 + minor). */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
