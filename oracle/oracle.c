/*
 * Plain, slow CPU oracle for one decode step of a MusicGen-style
 * multi-codebook audio-token decoder (the Parler-TTS decoder).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two sides meet only through seeded input tensors.
 *
 * Every quantity is computed from its plain definition, in double precision
 * unless the method fixes a precision (the temperature division is IEEE
 * float, because the top-k decision is taken on the scaled float values).
 * No blocking, no online softmax, no split of the key range: scores, one
 * softmax, one weighted sum.
 *
 * Sources ("Optimized Parler TTS" page):
 *   - "Analysis and improvements", item 1 of the CUDA-graph list: static
 *     caches for both cross and causal attention, preallocated to a maximum
 *     length; the attention kernel should touch only the valid length
 *     (eager ~13 us versus ~95 us for the whole static cache).
 *   - "Future work", item 1: a paged (block-table) cache instead of the
 *     static one.
 *   - "Future work", item 2: one fused sampler doing temperature scaling,
 *     top-k and softmax (the categorical draw that follows them).
 *   - The architecture overview: nine DAC codebooks decoded in parallel
 *     under a delayed pattern, one token per codebook per step; the
 *     description enters through cross-attention.
 * Philox4x32-10 follows Salmon, Moraes, Dror and Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3" (SC'11), section 3 (Philox S-box and key
 * schedule).
 *
 * Readings where the page is silent (each also listed in the design notes):
 *   - attention scale defaults to 1/sqrt(D); a one-token query attends to
 *     every valid key, including the one appended in the same step;
 *   - no positional term inside attention (q and k are taken as given);
 *   - top-k is taken on the temperature-scaled float values; equal values
 *     are ordered by lower index first;
 *   - the draw is Gumbel-max over the top-k set, u from Philox4x32-10 with
 *     key = seed, counter = (i / 4, codebook, step, batch row), word i % 4;
 *   - delay pattern: codebook c emits pad_id while step <= c (0-based).
 *
 * Parity pins: the closed forms, brute-force enumerations, published Philox
 * known-answer vectors and statistical checks live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 decoding: a bfloat16 is the upper half of an IEEE binary32.     */
/* ------------------------------------------------------------------ */
double oracle_bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------ */
/* Attention of one query over an explicit list of n keys and values.   */
/*   s_j = scale * sum_d q_d k_{j,d}                                    */
/*   p_j = exp(s_j - max_i s_i) / sum_i exp(s_i - max_i s_i)            */
/*   o_d = sum_j p_j v_{j,d}                                             */
/* keys/values: n rows of d bf16 values, row-major.  out: d doubles.    */
/* psum (nullable) receives sum_j p_j, which must be 1.                 */
/* n == 0 has no defined result: out is zero and psum is 0.             */
/* ------------------------------------------------------------------ */
void oracle_attend(const uint16_t *q, const uint16_t *keys, const uint16_t *values, int64_t n, int d,
                   double scale, double *out, double *psum) {
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (psum) *psum = 0.0;
    if (n <= 0) return;

    double *s = (double *)malloc((size_t)n * sizeof(double));
    double smax = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int e = 0; e < d; ++e)
            dot += oracle_bf16_to_double(q[e]) * oracle_bf16_to_double(keys[j * d + e]);
        s[j] = scale * dot;
        if (s[j] > smax) smax = s[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - smax);
        denom += s[j];
    }
    double total = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = s[j] / denom;
        total += p;
        for (int e = 0; e < d; ++e) out[e] += p * oracle_bf16_to_double(values[j * d + e]);
    }
    if (psum) *psum = total;
    free(s);
}

/* ------------------------------------------------------------------ */
/* Static (contiguous) cache, layout [B][H][max_len][D].                */
/* Row (b,h) attends keys 0 .. seq_len[b]-1.  out: [B][H][D] doubles.   */
/* Used for causal self-attention over the static cache and for         */
/* cross-attention over the description encoder's keys and values      */
/* (there seq_len is the description length of each row).              */
/* ------------------------------------------------------------------ */
void oracle_attn_contiguous(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int H, int D,
                            int max_len, const int32_t *seq_len, double scale, double *out) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t row = ((size_t)b * H + h);
            const uint16_t *kr = k + row * (size_t)max_len * D;
            const uint16_t *vr = v + row * (size_t)max_len * D;
            oracle_attend(q + row * D, kr, vr, seq_len[b], D, scale, out + row * D, NULL);
        }
}

/* Attention of one (b,h) row of a contiguous cache (for sampled checks). */
void oracle_attn_contiguous_row(const uint16_t *q_row, const uint16_t *k_row, const uint16_t *v_row, int D,
                                int n, double scale, double *out_row) {
    oracle_attend(q_row, k_row, v_row, n, D, scale, out_row, NULL);
}

/* ------------------------------------------------------------------ */
/* Paged cache: pool [num_blocks][H][block_size][D]; block_table        */
/* [B][max_blocks_per_seq].  Logical key j of row b lives in block      */
/* block_table[b][j / block_size], slot j % block_size.                 */
/* The oracle gathers the logical sequence, then attends it.            */
/* Returns 0, or -1 when a needed table entry is outside the pool.      */
/* ------------------------------------------------------------------ */
int oracle_attn_paged_row(const uint16_t *q_row, const uint16_t *k_pool, const uint16_t *v_pool,
                          const int32_t *table_row, int num_blocks, int block_size, int H, int h, int D, int n,
                          double scale, double *out_row) {
    uint16_t *kg = (uint16_t *)malloc((size_t)(n > 0 ? n : 1) * D * sizeof(uint16_t));
    uint16_t *vg = (uint16_t *)malloc((size_t)(n > 0 ? n : 1) * D * sizeof(uint16_t));
    for (int j = 0; j < n; ++j) {
        int32_t blk = table_row[j / block_size];
        if (blk < 0 || blk >= num_blocks) {
            free(kg);
            free(vg);
            return -1;
        }
        size_t src = (((size_t)blk * H + h) * block_size + (size_t)(j % block_size)) * D;
        memcpy(kg + (size_t)j * D, k_pool + src, (size_t)D * sizeof(uint16_t));
        memcpy(vg + (size_t)j * D, v_pool + src, (size_t)D * sizeof(uint16_t));
    }
    oracle_attend(q_row, kg, vg, n, D, scale, out_row, NULL);
    free(kg);
    free(vg);
    return 0;
}

int oracle_attn_paged(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool, const int32_t *block_table,
                      int max_blocks_per_seq, int num_blocks, int block_size, int B, int H, int D,
                      const int32_t *seq_len, double scale, double *out) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t row = ((size_t)b * H + h);
            int rc = oracle_attn_paged_row(q + row * D, k_pool, v_pool, block_table + (size_t)b * max_blocks_per_seq,
                                           num_blocks, block_size, H, h, D, seq_len[b], scale, out + row * D);
            if (rc) return rc;
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* KV append: the new key/value of row b is written at position pos[b]. */
/* ------------------------------------------------------------------ */
void oracle_kv_append_contiguous(uint16_t *k, uint16_t *v, const uint16_t *k_new, const uint16_t *v_new,
                                 const int32_t *pos, int B, int H, int D, int max_len) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t row = (size_t)b * H + h;
            size_t dst = (row * (size_t)max_len + (size_t)pos[b]) * D;
            memcpy(k + dst, k_new + row * D, (size_t)D * sizeof(uint16_t));
            memcpy(v + dst, v_new + row * D, (size_t)D * sizeof(uint16_t));
        }
}

void oracle_kv_append_paged(uint16_t *k_pool, uint16_t *v_pool, const int32_t *block_table, int max_blocks_per_seq,
                            int block_size, const uint16_t *k_new, const uint16_t *v_new, const int32_t *pos, int B,
                            int H, int D) {
    for (int b = 0; b < B; ++b) {
        int32_t blk = block_table[(size_t)b * max_blocks_per_seq + pos[b] / block_size];
        int slot = pos[b] % block_size;
        for (int h = 0; h < H; ++h) {
            size_t row = (size_t)b * H + h;
            size_t dst = (((size_t)blk * H + h) * block_size + (size_t)slot) * D;
            memcpy(k_pool + dst, k_new + row * D, (size_t)D * sizeof(uint16_t));
            memcpy(v_pool + dst, v_new + row * D, (size_t)D * sizeof(uint16_t));
        }
    }
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11).                                */
/* One round: two 32x32->64 products of the even counter words with     */
/* the Philox multipliers; the high halves are XORed with the odd       */
/* counter words and the round key, and the words are permuted.         */
/* The two key words are bumped by the Weyl constants (golden ratio and */
/* sqrt(3)-1, as 32-bit fractions) between rounds.                      */
/* ------------------------------------------------------------------ */
static const uint32_t PHILOX_M0 = 0xD2511F53u, PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W0 = 0x9E3779B9u, PHILOX_W1 = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t p0 = (uint64_t)PHILOX_M0 * x0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * x2;
        uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
        uint32_t y1 = (uint32_t)p1;
        uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
        uint32_t y3 = (uint32_t)p0;
        x0 = y0;
        x1 = y1;
        x2 = y2;
        x3 = y3;
    }
    out[0] = x0;
    out[1] = x1;
    out[2] = x2;
    out[3] = x3;
}

/* Uniform in (0,1) for vocabulary entry i of codebook c, row b, step:   */
/* w = word (i mod 4) of Philox4x32-10(counter = {i/4, c, step, b},      */
/* key = {low 32 bits of seed, high 32 bits of seed}); u = (2*(w>>9)+1)  */
/* / 2^24, an odd multiple of 2^-24 (exact in binary32 and binary64).    */
double oracle_uniform(uint64_t seed, int32_t b, int32_t c, int32_t step, int32_t i) {
    uint32_t ctr[4] = {(uint32_t)i >> 2, (uint32_t)c, (uint32_t)step, (uint32_t)b};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    uint32_t word = w[(uint32_t)i & 3u];
    return (double)(2u * (word >> 9) + 1u) / 16777216.0;
}

/* ------------------------------------------------------------------ */
/* Sampler for one (b, c) row.                                           */
/*  1. delay pattern: codebook c is not yet started while step <= c and */
/*     emits pad_id (probabilities row is all zero);                     */
/*  2. temperature: x_i = fl32(logit_i / T);                            */
/*  3. top-k: order entries by x descending, then index ascending; the   */
/*     first k form the candidate set;                                   */
/*  4. softmax over the candidate set (optional output);                 */
/*  5. categorical draw by Gumbel-max: argmax over the set of            */
/*     x_i - log(-log(u_i)); equal scores go to the lower index.        */
/* margin: best minus second-best perturbed score (+inf if there is no   */
/* second candidate, or if every candidate score is -inf).               */
/* topk_out (nullable): the k candidate indices in ascending order.      */
/* Returns 0, or -1 on invalid input (NaN logit, k out of range, T<=0).  */
/* ------------------------------------------------------------------ */
typedef struct {
    float x;
    int32_t i;
} oracle_entry;

static int oracle_entry_order(const void *pa, const void *pb) {
    const oracle_entry *a = (const oracle_entry *)pa, *b = (const oracle_entry *)pb;
    if (a->x > b->x) return -1;
    if (a->x < b->x) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

static int oracle_int_order(const void *pa, const void *pb) {
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

int oracle_sample_row(const float *logits, int V, float temperature, int top_k, uint64_t seed, int32_t b, int32_t c,
                      int32_t step, int32_t pad_id, int32_t *token, double *margin, double *probs,
                      int32_t *topk_out) {
    if (!(temperature > 0.0f) || top_k < 1 || top_k > V) return -1;
    if (probs)
        for (int i = 0; i < V; ++i) probs[i] = 0.0;
    if (step <= c) {
        *token = pad_id;
        if (margin) *margin = INFINITY;
        if (topk_out)
            for (int r = 0; r < top_k; ++r) topk_out[r] = -1;
        return 0;
    }

    oracle_entry *e = (oracle_entry *)malloc((size_t)V * sizeof(oracle_entry));
    for (int i = 0; i < V; ++i) {
        if (isnan(logits[i])) {
            free(e);
            return -1;
        }
        volatile float xi = logits[i] / temperature; /* binary32 division, round to nearest */
        e[i].x = xi;
        e[i].i = i;
    }
    qsort(e, (size_t)V, sizeof(oracle_entry), oracle_entry_order);

    /* Gumbel-max over the first top_k entries. */
    double best = -INFINITY, second = -INFINITY;
    int32_t best_i = -1;
    for (int r = 0; r < top_k; ++r) {
        double u = oracle_uniform(seed, b, c, step, e[r].i);
        double score = (double)e[r].x - log(-log(u));
        if (best_i < 0 || score > best || (score == best && e[r].i < best_i)) {
            if (best_i >= 0) second = best;
            best = score;
            best_i = e[r].i;
        } else if (score > second) {
            second = score;
        }
    }
    *token = best_i;
    if (margin) {
        if (top_k == 1 || best == -INFINITY)
            *margin = INFINITY;
        else
            *margin = best - second;
    }

    if (probs) {
        double xmax = (double)e[0].x;
        if (xmax == -INFINITY) {
            for (int r = 0; r < top_k; ++r) probs[e[r].i] = 1.0 / top_k;
        } else {
            double z = 0.0;
            for (int r = 0; r < top_k; ++r) z += exp((double)e[r].x - xmax);
            for (int r = 0; r < top_k; ++r) probs[e[r].i] = exp((double)e[r].x - xmax) / z;
        }
    }
    if (topk_out) {
        for (int r = 0; r < top_k; ++r) topk_out[r] = e[r].i;
        qsort(topk_out, (size_t)top_k, sizeof(int32_t), oracle_int_order);
    }
    free(e);
    return 0;
}

/* All rows of a [B][C][ldv] logits tensor.  tokens: [B][C]; margins,    */
/* probs ([B][C][V]) and topk ([B][C][k]) are nullable.                  */
int oracle_sample(const float *logits, int B, int C, int V, int ldv, float temperature, int top_k,
                  const uint64_t *seeds, const int32_t *steps, int32_t pad_id, int32_t *tokens, double *margins,
                  double *probs, int32_t *topk) {
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c) {
            size_t row = (size_t)b * C + c;
            int rc = oracle_sample_row(logits + row * (size_t)ldv, V, temperature, top_k, seeds[b], b, c, steps[b],
                                       pad_id, tokens + row, margins ? margins + row : NULL,
                                       probs ? probs + row * (size_t)V : NULL, topk ? topk + row * (size_t)top_k : NULL);
            if (rc) return rc;
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Merged codebook embedding lookup (Optimized Parler TTS, "Analysis    */
/* and improvements", other optimizations item 3: the nine embedding    */
/* lookups merged into one).  The decoder input of the next step is the */
/* sum over codebooks of each codebook's embedding of its token:        */
/*   x[b][d] = sum_c table[c*V + tokens[b][c]][d]                        */
/* table: [C*V][Dm] bf16 (codebook c's rows at c*V); tokens: [B][C].     */
/* Returns 0, or -1 when a token is outside [0, V).                     */
/* ------------------------------------------------------------------ */
int oracle_embed_tokens(const int32_t *tokens, const uint16_t *table, int B, int C, int V, int Dm, double *out) {
    for (int b = 0; b < B; ++b) {
        for (int d = 0; d < Dm; ++d) out[(size_t)b * Dm + d] = 0.0;
        for (int c = 0; c < C; ++c) {
            int32_t t = tokens[(size_t)b * C + c];
            if (t < 0 || t >= V) return -1;
            const uint16_t *row = table + ((size_t)c * V + (size_t)t) * Dm;
            for (int d = 0; d < Dm; ++d) out[(size_t)b * Dm + d] += oracle_bf16_to_double(row[d]);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Merged LM head on the last position (same page, other optimizations  */
/* items 1-2: the head evaluated only for the newest position, and the  */
/* nine codebook heads merged into one weight matrix):                  */
/*   logits[b][n] = sum_k hidden[b][k] * W[n][k],  n = c*V + v           */
/* hidden: [B][K] bf16; W: [N][K] bf16; out: [B][N] doubles.            */
/* ------------------------------------------------------------------ */
void oracle_lm_head(const uint16_t *hidden, const uint16_t *W, int B, int K, int N, double *out) {
    for (int b = 0; b < B; ++b)
        for (int n = 0; n < N; ++n) {
            double s = 0.0;
            for (int k = 0; k < K; ++k)
                s += oracle_bf16_to_double(hidden[(size_t)b * K + k]) * oracle_bf16_to_double(W[(size_t)n * K + k]);
            out[(size_t)b * N + n] = s;
        }
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 KV cache (the page's "Future work" item 1 asks for a cache  */
/* that loads memory bandwidth less; an 8-bit KV format halves the      */
/* bytes).  E4M3 follows the OCP 8-bit floating point specification:    */
/* 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0    */
/* holds subnormals m/8 * 2^-6; S.1111.111 is NaN; no infinities; the   */
/* largest finite magnitude is 1.75 * 2^8 = 448.                        */
/* ------------------------------------------------------------------ */
double oracle_e4m3_to_double(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = (m / 8.0) * ldexp(1.0, -6);
    else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -v : v;
}

/* Round to the nearest E4M3 value, ties to the even code (mantissa LSB 0), */
/* magnitudes at or above 448 saturating to 448 (the "satfinite" rule),     */
/* NaN to 0x7F.  Brute force over the 127 non-negative finite codes.        */
uint8_t oracle_double_to_e4m3(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    uint8_t best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Quantising append: code = E4M3(fl32(x / scale)) with x the bf16 value   */
/* (binary32 division, round to nearest).  k_new/v_new [B][H][D] bf16;    */
/* contiguous fp8 cache [B][H][max_len][D].                                */
static uint8_t quantize(uint16_t bf16, float scale) {
    volatile float q = (float)oracle_bf16_to_double(bf16) / scale;
    return oracle_double_to_e4m3((double)q);
}

void oracle_kv_append_fp8_contiguous(uint8_t *k, uint8_t *v, const uint16_t *k_new, const uint16_t *v_new,
                                     const int32_t *pos, int B, int H, int D, int max_len, float k_scale,
                                     float v_scale) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t row = (size_t)b * H + h;
            size_t dst = (row * (size_t)max_len + (size_t)pos[b]) * D;
            for (int e = 0; e < D; ++e) {
                k[dst + e] = quantize(k_new[row * D + e], k_scale);
                v[dst + e] = quantize(v_new[row * D + e], v_scale);
            }
        }
}

void oracle_kv_append_fp8_paged(uint8_t *k_pool, uint8_t *v_pool, const int32_t *block_table,
                                int max_blocks_per_seq, int block_size, const uint16_t *k_new,
                                const uint16_t *v_new, const int32_t *pos, int B, int H, int D, float k_scale,
                                float v_scale) {
    for (int b = 0; b < B; ++b) {
        int32_t blk = block_table[(size_t)b * max_blocks_per_seq + pos[b] / block_size];
        int slot = pos[b] % block_size;
        for (int h = 0; h < H; ++h) {
            size_t row = (size_t)b * H + h;
            size_t dst = (((size_t)blk * H + h) * block_size + (size_t)slot) * D;
            for (int e = 0; e < D; ++e) {
                k_pool[dst + e] = quantize(k_new[row * D + e], k_scale);
                v_pool[dst + e] = quantize(v_new[row * D + e], v_scale);
            }
        }
    }
}

/* Attention over n fp8 keys/values: k_j = decode(code) * k_scale,       */
/* v_j = decode(code) * v_scale; then the plain definition as above.     */
void oracle_attend_fp8(const uint16_t *q, const uint8_t *keys, const uint8_t *values, int64_t n, int d,
                       double scale, double k_scale, double v_scale, double *out) {
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (n <= 0) return;
    double *s = (double *)malloc((size_t)n * sizeof(double));
    double smax = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int e = 0; e < d; ++e)
            dot += oracle_bf16_to_double(q[e]) * (oracle_e4m3_to_double(keys[j * d + e]) * k_scale);
        s[j] = scale * dot;
        if (s[j] > smax) smax = s[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - smax);
        denom += s[j];
    }
    for (int64_t j = 0; j < n; ++j) {
        double p = s[j] / denom;
        for (int e = 0; e < d; ++e) out[e] += p * (oracle_e4m3_to_double(values[j * d + e]) * v_scale);
    }
    free(s);
}

void oracle_attn_fp8_contiguous(const uint16_t *q, const uint8_t *k, const uint8_t *v, int B, int H, int D,
                                int max_len, const int32_t *seq_len, double scale, double k_scale, double v_scale,
                                double *out) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t row = (size_t)b * H + h;
            oracle_attend_fp8(q + row * D, k + row * (size_t)max_len * D, v + row * (size_t)max_len * D, seq_len[b],
                              D, scale, k_scale, v_scale, out + row * D);
        }
}

int oracle_attn_fp8_paged(const uint16_t *q, const uint8_t *k_pool, const uint8_t *v_pool, const int32_t *block_table,
                          int max_blocks_per_seq, int num_blocks, int block_size, int B, int H, int D,
                          const int32_t *seq_len, double scale, double k_scale, double v_scale, double *out) {
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            size_t row = (size_t)b * H + h;
            int n = seq_len[b];
            uint8_t *kg = (uint8_t *)malloc((size_t)(n > 0 ? n : 1) * D);
            uint8_t *vg = (uint8_t *)malloc((size_t)(n > 0 ? n : 1) * D);
            for (int j = 0; j < n; ++j) {
                int32_t blk = block_table[(size_t)b * max_blocks_per_seq + j / block_size];
                if (blk < 0 || blk >= num_blocks) {
                    free(kg);
                    free(vg);
                    return -1;
                }
                size_t src = (((size_t)blk * H + h) * block_size + (size_t)(j % block_size)) * D;
                memcpy(kg + (size_t)j * D, k_pool + src, (size_t)D);
                memcpy(vg + (size_t)j * D, v_pool + src, (size_t)D);
            }
            oracle_attend_fp8(q + row * D, kg, vg, n, D, scale, k_scale, v_scale, out + row * D);
            free(kg);
            free(vg);
        }
    return 0;
}
