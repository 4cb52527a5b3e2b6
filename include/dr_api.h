/*
 * dr_api.h -- C ABI of libdecoderattn.so, the decode step of a MusicGen-style
 * multi-codebook audio-token decoder (the Parler-TTS decoder) on NVIDIA GB300
 * (sm_103a).
 *
 * Four operations make up one decode step:
 *   dr_kv_append            write this step's key/value into the cache;
 *   dr_decode_self_attn     one-query causal self-attention over the valid
 *                           length of a static (contiguous) or paged cache,
 *                           bf16 or FP8 E4M3;
 *   dr_decode_cross_attn    one-query attention over the description
 *                           encoder's keys and values;
 *   dr_sample_topk_delayed  temperature, top-k, softmax and categorical draw
 *                           for every codebook in one kernel, under the
 *                           delay pattern.
 * dr_decode_layer does the first three for one layer in one launch; the
 * decoder's two ends around them are dr_lm_head (the merged codebook heads
 * on the newest position, writing the logits the sampler reads) and
 * dr_embed_tokens (the merged embedding lookup of the drawn tokens).
 *
 * Conventions shared by every call
 *   - Every pointer argument except `stream` is a DEVICE pointer owned by the
 *     caller.  The library allocates nothing, keeps no pointer after a call
 *     returns, and never synchronises with the host.
 *   - `stream` is a cudaStream_t passed as an opaque pointer (NULL = the
 *     legacy default stream).  Work is enqueued on it asynchronously; the
 *     calls are free of host-device synchronisation.
 *   - bf16 means IEEE bfloat16 (the upper 16 bits of a binary32), stored as
 *     2-byte values.  Tensors are dense and row-major in the order given.
 *   - Host-checkable mistakes (null pointers, bad sizes, misalignment) return
 *     an error status before anything is enqueued.  A failed launch returns
 *     DR_ERR_CUDA.
 *   - Mistakes only the device can see (a length above the capacity, a block
 *     id outside the pool, an append position past the end) never trap: the
 *     kernel clamps or skips the offending row or block and, when `err_flag`
 *     is non-NULL, ORs a DR_ERRF_* bit into *err_flag (a device int32 the
 *     caller zeroes and reads back when it chooses).
 *   - Head dimension D must be 64 (DR_ERR_UNSUPPORTED otherwise); keys and
 *     values have as many heads H as the query (plain multi-head attention).
 *   - Calls on the same stream are ordered; the library holds no state
 *     between calls, so calls on different streams may overlap as long as
 *     they do not write the same buffers.
 */
#ifndef DR_API_H
#define DR_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dr_status {
    DR_OK = 0,
    DR_ERR_INVALID_ARG = 1, /* null pointer, size out of range, misaligned pointer */
    DR_ERR_UNSUPPORTED = 2, /* a valid but unimplemented shape (D != 64, block_size != 16, C > 16, V > 2048,
                               more than 65535 sampler rows) */
    DR_ERR_CUDA = 3         /* the CUDA runtime refused the launch */
} dr_status;

typedef enum dr_kv_layout {
    DR_KV_CONTIGUOUS = 0, /* static cache: k, v are [B][H][max_len][D] */
    DR_KV_PAGED = 1       /* block pool: k, v are [num_blocks][H][block_size][D] */
} dr_kv_layout;

typedef enum dr_dtype { DR_BF16 = 0, DR_F32 = 1 } dr_dtype;

/* Storage format of a self-attention KV cache. */
typedef enum dr_kv_dtype {
    DR_KV_BF16 = 0,    /* bf16 keys and values */
    DR_KV_FP8_E4M3 = 1 /* OCP FP8 E4M3 codes: key = code * k_scale, value = code * v_scale */
} dr_kv_dtype;

/* Device-side error bits (see err_flag above). */
#define DR_ERRF_SEQ_LEN 1  /* a seq_len / enc_len entry outside [1, capacity]; it was clamped */
#define DR_ERRF_BLOCK_ID 2 /* a needed block-table entry outside [0, num_blocks); its keys were skipped */
#define DR_ERRF_POS 4      /* an append position outside [0, capacity) or on an unmapped block; row skipped */
#define DR_ERRF_TOKEN 8    /* a token outside [0, V) in dr_embed_tokens; that codebook's row was skipped */
#define DR_ERRF_TIMEOUT 16 /* a bounded on-chip wait gave up (never expected); that CTA's results were not written */

/* Sampler flags. */
#define DR_SAMPLE_ADVANCE 1 /* after drawing, step[b] += 1 for every row b */

/*
 * A self-attention KV cache (one decoder layer).
 *
 * Static cache (Optimized Parler TTS, "Analysis and improvements": the static
 * caches for causal and cross attention that CUDA-graph capture needs,
 * preallocated to a maximum length):
 *   layout = DR_KV_CONTIGUOUS; k, v = [B][H][max_len][D]; key j of row
 *   (b, h) at ((b*H + h)*max_len + j)*D.  Capacity = max_len keys per row.
 * Paged cache (same page, "Future work" item 1: a PagedAttention-style cache
 * so that no full static cache has to be kept or moved):
 *   layout = DR_KV_PAGED; k, v = [num_blocks][H][block_size][D];
 *   block_table = [B][max_blocks_per_seq] int32; key j of row b lives in block
 *   block_table[b][j / block_size], slot j % block_size; entries a row does
 *   not use may hold any value (conventionally -1).  block_size must be 16.
 *   Capacity = max_blocks_per_seq * block_size keys per row.
 * Element format (kv_dtype): bf16, or FP8 E4M3 codes (the same page's
 * "Future work" item 1 asks for less KV traffic; 8-bit codes halve it).  An
 * e4m3 cache stores code = e4m3(fl32(x / scale)) (IEEE division, round to
 * nearest even, saturating at +-448) and is read back as code * scale, with
 * k_scale for keys and v_scale for values (both > 0; ignored for bf16).
 * k and v must be 16-byte aligned.  The struct itself is read on the host
 * during the call only.
 */
typedef struct dr_kv_cache {
    int32_t layout;             /* dr_kv_layout */
    int32_t max_len;            /* contiguous: keys per (b, h) row; ignored when paged */
    int32_t block_size;         /* paged: keys per block (16); ignored when contiguous */
    int32_t num_blocks;         /* paged: blocks in the pool */
    int32_t max_blocks_per_seq; /* paged: row stride of block_table */
    int32_t kv_dtype;           /* dr_kv_dtype */
    void *k;                    /* keys (device) */
    void *v;                    /* values (device) */
    const int32_t *block_table; /* paged: [B][max_blocks_per_seq] int32 (device); NULL when contiguous */
    float k_scale;              /* e4m3 only: key = code * k_scale */
    float v_scale;              /* e4m3 only: value = code * v_scale */
} dr_kv_cache;

/*
 * dr_kv_append -- store this step's key and value of every row.
 * Source: Optimized Parler TTS, "Analysis and improvements" (static cache
 * for causal attention; each decode step adds one key/value per row).
 *
 *   k_new, v_new : [B][H][D] bf16 (device, 16-byte aligned); quantised to
 *                  e4m3 codes when the cache is DR_KV_FP8_E4M3
 *   pos          : [B] int32 (device); row b's key/value go to position pos[b]
 *                  (the row's valid length becomes pos[b] + 1 for the
 *                  self-attention that follows)
 *   err_flag     : nullable device int32; DR_ERRF_POS is ORed in when
 *                  pos[b] is outside [0, capacity) or, paged, its block-table
 *                  entry is outside the pool; that row is not written.
 * Writes exactly B*H*D elements into each of cache->k and cache->v.
 */
dr_status dr_kv_append(const dr_kv_cache *cache, const void *k_new, const void *v_new, const int32_t *pos, int B,
                       int H, int D, int32_t *err_flag, void *stream);

/*
 * dr_decode_self_attn -- single-query causal self-attention of one decode
 * step over the valid part of a KV cache.
 * Source: Optimized Parler TTS, "Analysis and improvements": the static-cache
 * attention kernel took ~95 us because it moved the whole preallocated cache,
 * against ~13 us for the eager kernel that reads the valid length only; and
 * "Future work" item 1 (paged cache).
 *
 * For every row b and head h:
 *   s_j = scale * (q[b,h,:] . K[b,h,j,:])  for j in [0, seq_len[b])
 *   out[b,h,:] = sum_j softmax(s)_j V[b,h,j,:]
 * Only the seq_len[b] valid keys of each row are read.  Causality for a
 * single query means it sees every valid key, including the one appended in
 * this step.  Accumulation is fp32; the result is written in out_dtype.
 *
 *   q        : [B][H][D] bf16 (device, 16-byte aligned)
 *   cache    : see dr_kv_cache
 *   seq_len  : [B] int32 (device), keys attended per row, 1 <= seq_len[b] <=
 *              capacity; entries outside are clamped to [0, capacity] and
 *              flagged DR_ERRF_SEQ_LEN (a row of length 0 outputs zeros)
 *   max_seq_len_hint : an upper bound the caller knows for max_b seq_len[b]
 *              (<= 0: the capacity).  It only tunes how each row's keys are
 *              split across CTAs (dr_plan_splits); any value gives a result
 *              within the stated accuracy, and the same hint on the same
 *              device gives the same bits (a different split changes only
 *              the order of the fp32 sums).
 *   scale    : softmax scale; <= 0 selects 1/sqrt(D)
 *   out      : [B][H][D] in out_dtype (DR_BF16: round to nearest even)
 *   err_flag : nullable device int32 (DR_ERRF_SEQ_LEN, DR_ERRF_BLOCK_ID)
 */
dr_status dr_decode_self_attn(const void *q, const dr_kv_cache *cache, const int32_t *seq_len, int B, int H, int D,
                              int max_seq_len_hint, float scale, void *out, dr_dtype out_dtype, int32_t *err_flag,
                              void *stream);

/*
 * dr_decode_cross_attn -- single-query attention over the description
 * encoder's keys and values (recomputed every decode step).
 * Source: Optimized Parler TTS, architecture overview (the description,
 * encoded by Flan-T5, is used through cross-attention in the decoder's
 * attention layers) and "Speeding up Parler TTS decoder" (throughput falls
 * as the description grows, because of this cross-attention).
 *
 *   q        : [B][H][D] bf16 (device, 16-byte aligned)
 *   k_enc, v_enc : [B][H][Lc_max][D] bf16 (device, 16-byte aligned)
 *   enc_len  : [B] int32 (device), description length per row, 1 <=
 *              enc_len[b] <= Lc_max (clamped and flagged otherwise)
 *   scale, out, out_dtype, err_flag : as for dr_decode_self_attn
 */
dr_status dr_decode_cross_attn(const void *q, const void *k_enc, const void *v_enc, const int32_t *enc_len, int B,
                               int H, int D, int Lc_max, float scale, void *out, dr_dtype out_dtype,
                               int32_t *err_flag, void *stream);

/*
 * dr_decode_layer -- one decoder layer's attention work of a decode step in
 * one launch: the KV append, the self-attention and the cross-attention.
 * Source: the same passages as the three calls above; fusing them is the
 * launch-count reduction the page's profile motivates (Optimized Parler TTS,
 * "Analysis and improvements": the decoder is overhead-bound, the GPU waits
 * between small kernels).
 *
 * Equivalent to, in this order,
 *   dr_kv_append(cache, k_new, v_new, pos = seq_len - 1, ...)
 *   dr_decode_self_attn(q, cache, seq_len, ..., out, ...)
 *   dr_decode_cross_attn(q_cross, k_enc, v_enc, enc_len, ..., Lc_max, ..., out_cross, ...)
 * with results within the same tolerances (the key at seq_len[b]-1 is taken
 * from k_new/v_new directly and also stored into the cache; rows whose
 * seq_len is outside [1, capacity] are not appended and flag DR_ERRF_POS and
 * DR_ERRF_SEQ_LEN).  Arguments are as for those calls; out and out_cross are
 * both [B][H][D] in out_dtype.  B <= 32767.
 */
dr_status dr_decode_layer(const void *q, const dr_kv_cache *cache, const void *k_new, const void *v_new,
                          const int32_t *seq_len, const void *q_cross, const void *k_enc, const void *v_enc,
                          const int32_t *enc_len, int Lc_max, int B, int H, int D, int max_seq_len_hint, float scale,
                          void *out, void *out_cross, dr_dtype out_dtype, int32_t *err_flag, void *stream);

/*
 * dr_sample_topk_delayed -- one kernel that turns the logits of every
 * codebook of every row into this step's tokens.
 * Source: Optimized Parler TTS, "Future work" item 2 (temperature scaling,
 * top-k and softmax, run as more than ten kernels, should be one fused
 * kernel), "Analysis and improvements" (sampling without a GPU-CPU
 * synchronisation) and the architecture overview (nine DAC codebooks, one
 * token each per step, in a delayed pattern).
 *
 * For every row b and codebook c (0-based):
 *   if step[b] <= c : tokens[b][c] = pad_id (delay pattern: codebook c starts
 *                     one step after codebook c-1); probs row = 0
 *   else:
 *     x_i  = fl32(logits[b][c][i] / temperature), IEEE round-to-nearest
 *     K    = the top_k indices by x descending, equal x -> lower index first
 *     u_i  = (2*(w >> 9) + 1) * 2^-24, w = word (i mod 4) of
 *            Philox4x32-10(counter = {i/4, c, step[b], b},
 *                          key = {seed[b] bits 0-31, bits 32-63})
 *     tokens[b][c] = argmax over i in K of x_i - log(-log(u_i))  (Gumbel-max:
 *                    a categorical draw from softmax over K); equal scores
 *                    -> lower index
 *     probs[b][c][i] = exp(x_i - max_K x) / sum_K exp(x_j - max_K x) for i in
 *                    K, 0 elsewhere (uniform 1/top_k over K if all of K is -inf)
 * Philox4x32-10: Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
 * SC'11.
 *
 *   logits   : [B][C][ldv] float32 (device); columns [V, ldv) are never read.
 *              NaN logits give an undefined (but in-range or pad) token.
 *              Where some x_i are +inf (an infinite logit, or a temperature
 *              so small that logit / temperature overflows), the token is the
 *              lowest such index and the probabilities are undefined.
 *   B        : batch rows, 1..65535 (DR_ERR_UNSUPPORTED above)
 *   C        : codebooks, 1..16          V : vocabulary, 1..2048, V <= ldv
 *   temperature : > 0 and finite          top_k : 1..V
 *   seeds    : [B] uint64 (device)
 *   step     : [B] int32 (device); read, and incremented when flags has
 *              DR_SAMPLE_ADVANCE (after every codebook of the row has read it)
 *   tokens   : [B][C] int32 (device, written)
 *   probs    : nullable [B][C][V] float32 (device, written when non-NULL)
 */
dr_status dr_sample_topk_delayed(const float *logits, int B, int C, int V, int ldv, float temperature, int top_k,
                                 const uint64_t *seeds, int32_t *step, int32_t pad_id, int32_t *tokens, float *probs,
                                 int flags, void *stream);

/*
 * dr_embed_tokens -- the next step's decoder input from this step's tokens:
 *   out[b][d] = sum_{c=0..C-1} table[c*V + tokens[b][c]][d]
 * Source: Optimized Parler TTS, "Analysis and improvements", other
 * optimizations item 3: the nine codebook embedding lookups merged into one
 * (one merged table, one gather of C rows per batch row).
 *
 *   C      : codebooks, 1..16 (DR_ERR_UNSUPPORTED above 16, as for the sampler)
 *   tokens : [B][C] int32 (device), e.g. the tokens dr_sample_topk_delayed wrote
 *   table  : [C*V][Dm] bf16 (device, 16-byte aligned); codebook c's rows start at c*V
 *   out    : [B][Dm] in out_dtype (device, 16-byte aligned); fp32 sum in c order
 *   Dm     : a multiple of 8
 *   err_flag : nullable; DR_ERRF_TOKEN when a token is outside [0, V) (that
 *            term is left out of the sum)
 */
dr_status dr_embed_tokens(const int32_t *tokens, const void *table, int B, int C, int V, int Dm, void *out,
                          dr_dtype out_dtype, int32_t *err_flag, void *stream);

/*
 * dr_lm_head -- logits of the newest position from the merged codebook heads:
 *   logits[b][c][v] = sum_k hidden[b][k] * W[c*V + v][k]
 * Source: Optimized Parler TTS, "Analysis and improvements", other
 * optimizations items 1-2: the LM head computed for the last position only,
 * and the nine codebook heads merged into one weight matrix.
 *
 *   hidden : [B][K] bf16 (device, 16-byte aligned), the newest position's hidden state
 *   W      : [C*V][K] bf16 (device, 16-byte aligned)
 *   logits : [B][C][ldv] float32 (device), ldv >= V; columns [V, ldv) untouched.
 *            The layout dr_sample_topk_delayed reads.
 *   K      : 256, 512, 768, 1024, 1536 or 2048 (DR_ERR_UNSUPPORTED otherwise)
 *   err_flag : nullable device int32; DR_ERRF_TIMEOUT if a tensor-core CTA's
 *            bounded pipeline wait gave up (its logits are then not written)
 * fp32 accumulation.  Below 4 batch rows each logit is one CUDA-core dot
 * product in a fixed order; from 4 rows on the head is a dense contraction
 * on the tensor cores (tcgen05.mma, bf16 in, fp32 accumulate in tensor
 * memory, K consumed 16 at a time; when the batch is one tile of up to 32
 * rows and the 128-row weight slabs are fewer than the SMs, the two halves of
 * K are accumulated apart and added, the first half's sum first).
 */
dr_status dr_lm_head(const void *hidden, const void *W, int B, int K, int C, int V, int ldv, float *logits,
                     int32_t *err_flag, void *stream);

/*
 * dr_lm_head_stall_test -- TEST HOOK, never needed in use.  The same call as
 * dr_lm_head, except that the CTAs of 128-row weight slab `stall_slab` (logit
 * rows c*V + v in [128*stall_slab, 128*stall_slab + 128)) never load their
 * first K chunk.  The CTA's bounded pipeline wait for it then runs out (after
 * about 2 s): DR_ERRF_TIMEOUT is ORed into *err_flag, that slab's logits are
 * left unwritten, the CTA frees its tensor memory and exits, and every other
 * logit is written as by dr_lm_head.  Nothing faults or hangs, and later calls
 * on the same context work normally.  The tests use it to check the failure
 * path of the waits; the paper has no counterpart.
 *   B >= 4 (the tensor-core head; DR_ERR_UNSUPPORTED below), 0 <= stall_slab
 *   < ceil(C*V / 128) (DR_ERR_INVALID_ARG otherwise); the rest as dr_lm_head.
 */
dr_status dr_lm_head_stall_test(const void *hidden, const void *W, int B, int K, int C, int V, int ldv, float *logits,
                                int32_t *err_flag, int stall_slab, void *stream);

/*
 * dr_decode_self_attn_stall_test -- TEST HOOK, never needed in use.  The
 * same call as dr_decode_self_attn, except that CTA 1 of row
 * stall_row = b*H + h never sends its softmax state to the row's CTA rank 0.
 * That CTA's bounded wait for the state then runs out (after about 2 s):
 * DR_ERRF_TIMEOUT is ORed into *err_flag, that row's output is left
 * unwritten, and every other row is written as by dr_decode_self_attn.
 * Nothing faults or hangs, and later calls on the same context work
 * normally.  The tests use it to check the failure path of the cluster
 * merge's wait; the paper has no counterpart.
 *   0 <= stall_row < B*H (DR_ERR_INVALID_ARG otherwise).  The call must run
 *   the kernel variant whose split rows merge through that wait: at least 2
 *   CTAs per row (dr_plan_splits) and more than 4 CTAs per SM in all
 *   (DR_ERR_UNSUPPORTED otherwise).  The rest as dr_decode_self_attn.
 */
dr_status dr_decode_self_attn_stall_test(const void *q, const dr_kv_cache *cache, const int32_t *seq_len, int B, int H,
                                        int D, int max_seq_len_hint, float scale, void *out, dr_dtype out_dtype,
                                        int32_t *err_flag, int stall_row, void *stream);

/*
 * dr_plan_splits -- host-only query: how many CTAs (one thread-block
 * cluster) share each (b, h) row of an attention call with this batch,
 * head count, length bound and KV storage type (DR_KV_BF16 or
 * DR_KV_FP8_E4M3; the description-encoder rows of dr_decode_cross_attn are
 * DR_KV_BF16) on a GPU with num_sms SMs.  Each CTA of the cluster takes an
 * equal run of whole 16-key blocks of the row.  The plan: at most 256 KiB
 * of K+V per CTA at the longest row, at least 6 CTAs per SM when the rows
 * alone are fewer, at least 64 keys per CTA, at most 8 CTAs -- or 16 (a
 * non-portable cluster) when 8 would each take at least 256 keys and 16 per
 * row come to at most 2 CTAs per SM (a few long rows: batch 1).  Pure
 * arithmetic; touches no device.  Returns 1 for non-positive sizes or an
 * unknown kv_dtype.
 */
int dr_plan_splits(int B, int H, int max_len, int kv_dtype, int num_sms);

/* Static, NUL-terminated description of a status code. */
const char *dr_status_string(dr_status s);

#ifdef __cplusplus
}
#endif

#endif /* DR_API_H */
