// extern "C" boundary of libdecoderattn.so: argument checks, split planning
// and launches.  Nothing here allocates device memory or synchronises with
// the host, so every entry point can be enqueued inside CUDA-graph capture
// (Optimized Parler TTS, "Analysis and improvements": static buffers and
// sampling without a GPU-CPU synchronisation are what make the decode step
// capturable as one graph).
#include <math.h>

#include <atomic>

#include "dr_internal.h"

namespace dr {

int max_cluster_size() { return 8; }

int current_device_sms() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

}  // namespace dr

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Validates a cache description; on success stores the keys a row can hold in *cap.
dr_status check_cache(const dr_kv_cache *c, int *cap) {
    if (!c || !c->k || !c->v) return DR_ERR_INVALID_ARG;
    if (!aligned16(c->k) || !aligned16(c->v)) return DR_ERR_INVALID_ARG;
    if (c->kv_dtype != DR_KV_BF16 && c->kv_dtype != DR_KV_FP8_E4M3) return DR_ERR_INVALID_ARG;
    if (c->kv_dtype == DR_KV_FP8_E4M3) {
        if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f) || isinf(c->k_scale) || isinf(c->v_scale))
            return DR_ERR_INVALID_ARG;
        if (!aligned16(c->k) || !aligned16(c->v)) return DR_ERR_INVALID_ARG;
    }
    if (c->layout == DR_KV_CONTIGUOUS) {
        if (c->max_len < 1) return DR_ERR_INVALID_ARG;
        *cap = c->max_len;
        return DR_OK;
    }
    if (c->layout == DR_KV_PAGED) {
        if (!c->block_table || c->num_blocks < 1 || c->max_blocks_per_seq < 1) return DR_ERR_INVALID_ARG;
        if (c->block_size != dr::kBlockKeys) return DR_ERR_UNSUPPORTED;
        if ((long long)c->max_blocks_per_seq * c->block_size > 0x7FFFFFFFLL) return DR_ERR_INVALID_ARG;
        *cap = c->max_blocks_per_seq * c->block_size;
        return DR_OK;
    }
    return DR_ERR_INVALID_ARG;
}

dr_status check_dims(int B, int H, int D) {
    if (B < 1 || H < 1 || B > 65535 || H > 65535) return DR_ERR_INVALID_ARG;
    if (D != dr::kHeadDim) return DR_ERR_UNSUPPORTED;
    return DR_OK;
}

dr_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DR_OK : DR_ERR_CUDA; }

float softmax_scale_log2(float scale, int D) {
    const float s = scale > 0.f ? scale : 1.0f / sqrtf((float)D);
    return s * 1.4426950408889634f;   // log2(e): the kernel works in base 2
}

void fill_self(dr::AttnParams &p, const void *q, const void *k, const void *v, const int32_t *lens,
               const int32_t *table, int B, int H, int cap, int max_blocks, int num_blocks, float scale, void *out,
               dr_dtype out_dtype, int32_t *err_flag, bool fp8 = false, float k_scale = 1.f, float v_scale = 1.f) {
    p = dr::AttnParams{};
    p.q = static_cast<const uint16_t *>(q);
    p.k = k;
    p.v = v;
    p.lens = lens;
    p.table = table;
    p.B = B;
    p.H = H;
    p.cap = cap;
    p.max_blocks = max_blocks;
    p.num_blocks = num_blocks;
    p.kv_fp8 = fp8 ? 1 : 0;
    p.k_scale = fp8 ? k_scale : 1.f;
    p.v_scale = fp8 ? v_scale : 1.f;
    // an e4m3 key is code * k_scale: fold k_scale into the query scale, v_scale into the output
    p.qscale = softmax_scale_log2(scale, dr::kHeadDim) * p.k_scale;
    p.out_scale = p.v_scale;
    p.xqscale = softmax_scale_log2(scale, dr::kHeadDim);
    p.out = out;
    p.out_f32 = out_dtype == DR_F32;
    p.err = err_flag;
}

void fill_cache(dr::AttnParams &p, const void *q, const dr_kv_cache *c, const int32_t *lens, int B, int H, int cap,
                float scale, void *out, dr_dtype out_dtype, int32_t *err_flag) {
    const bool paged = c->layout == DR_KV_PAGED;
    fill_self(p, q, c->k, c->v, lens, paged ? c->block_table : nullptr, B, H, cap, paged ? c->max_blocks_per_seq : 0,
              paged ? c->num_blocks : 0, scale, out, out_dtype, err_flag, c->kv_dtype == DR_KV_FP8_E4M3, c->k_scale,
              c->v_scale);
}

dr_status check_attn_args(const void *q, const int32_t *lens, void *out, dr_dtype out_dtype, float scale) {
    if (!q || !lens || !out || !aligned16(q)) return DR_ERR_INVALID_ARG;
    if (out_dtype != DR_BF16 && out_dtype != DR_F32) return DR_ERR_INVALID_ARG;
    if (!(scale == scale) || isinf(scale)) return DR_ERR_INVALID_ARG;
    return DR_OK;
}

int length_bound(const dr::AttnParams &p, int hint) { return (hint > 0 && hint < p.cap) ? hint : p.cap; }

int self_splits(const dr::AttnParams &p, int hint, int sms) {
    return dr_plan_splits(p.B, p.H, length_bound(p, hint), p.kv_fp8 ? DR_KV_FP8_E4M3 : DR_KV_BF16, sms);
}

dr_status launch(const dr::AttnParams &p, bool paged, int hint, void *stream) {
    const int sms = dr::current_device_sms();
    if (sms <= 0) return DR_ERR_CUDA;
    return from_cuda(dr::launch_decode_attn(p, paged, self_splits(p, hint, sms), static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int dr_plan_splits(int B, int H, int max_len, int kv_dtype, int num_sms) {
    if (B < 1 || H < 1 || max_len < 1 || num_sms < 1) return 1;
    if (kv_dtype != DR_KV_BF16 && kv_dtype != DR_KV_FP8_E4M3) return 1;
    constexpr long long kCtaBytes = 256 * 1024;   // K+V bytes per CTA at the longest row
    constexpr long long kFillCtasPerSm = 6;
    const long long rows = (long long)B * H;
    const long long key_bytes = 2LL * dr::kHeadDim * (kv_dtype == DR_KV_FP8_E4M3 ? 1 : 2);
    const long long tiles = (max_len + dr::kBlockKeys - 1) / dr::kBlockKeys;
    // At most kCtaBytes of K+V per CTA at the longest row: ragged rows spread
    // evenly, and each CTA streams enough to amortise its share of the merge...
    long long s = ((long long)max_len * key_bytes + kCtaBytes - 1) / kCtaBytes;
    // ...and at least kFillCtasPerSm CTAs per SM when the rows alone are fewer...
    const long long fill = (kFillCtasPerSm * num_sms + rows - 1) / rows;
    if (fill > s) s = fill;
    // ...but never fewer than 4 tiles (64 keys) per CTA, nor more than one portable cluster...
    const long long by_tiles = (tiles + 3) / 4;
    if (s > by_tiles) s = by_tiles;
    if (s > dr::max_cluster_size()) s = dr::max_cluster_size();
    // ...except for a few long rows (small batch): when 16 CTAs per row still leave room for the next launch's
    // grid (at most 2 CTAs per SM) and 8 CTAs would each stream 16 tiles or more, one non-portable cluster of
    // 16 halves every CTA's chain of dependent tiles (batch 1, 2048 + 64 keys: 4.87 -> 4.53 us per layer;
    // with 8 tiles per CTA, or more CTAs per SM, 16-CTA clusters were slower).
    if (s == dr::max_cluster_size() && rows * 16 <= 2LL * num_sms && tiles >= 16LL * 8) s = 16;
    return s < 1 ? 1 : (int)s;
}

dr_status dr_kv_append(const dr_kv_cache *cache, const void *k_new, const void *v_new, const int32_t *pos, int B,
                       int H, int D, int32_t *err_flag, void *stream) {
    dr_status st = check_dims(B, H, D);
    if (st != DR_OK) return st;
    int cap = 0;
    st = check_cache(cache, &cap);
    if (st != DR_OK) return st;
    if (!k_new || !v_new || !pos || !aligned16(k_new) || !aligned16(v_new)) return DR_ERR_INVALID_ARG;
    dr::AppendParams p;
    p.k = cache->k;
    p.v = cache->v;
    p.kv_fp8 = cache->kv_dtype == DR_KV_FP8_E4M3;
    p.k_scale = cache->k_scale;
    p.v_scale = cache->v_scale;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.pos = pos;
    p.table = cache->block_table;
    p.B = B;
    p.H = H;
    p.cap = cap;
    p.max_blocks = cache->max_blocks_per_seq;
    p.num_blocks = cache->num_blocks;
    p.err = err_flag;
    return from_cuda(dr::launch_kv_append(p, cache->layout == DR_KV_PAGED, static_cast<cudaStream_t>(stream)));
}

dr_status dr_decode_self_attn(const void *q, const dr_kv_cache *cache, const int32_t *seq_len, int B, int H, int D,
                              int max_seq_len_hint, float scale, void *out, dr_dtype out_dtype, int32_t *err_flag,
                              void *stream) {
    dr_status st = check_dims(B, H, D);
    if (st != DR_OK) return st;
    int cap = 0;
    st = check_cache(cache, &cap);
    if (st != DR_OK) return st;
    st = check_attn_args(q, seq_len, out, out_dtype, scale);
    if (st != DR_OK) return st;
    dr::AttnParams p;
    fill_cache(p, q, cache, seq_len, B, H, cap, scale, out, out_dtype, err_flag);
    return launch(p, cache->layout == DR_KV_PAGED, max_seq_len_hint, stream);
}

dr_status dr_decode_self_attn_stall_test(const void *q, const dr_kv_cache *cache, const int32_t *seq_len, int B, int H,
                                        int D, int max_seq_len_hint, float scale, void *out, dr_dtype out_dtype,
                                        int32_t *err_flag, int stall_row, void *stream) {
    if (B < 1 || H < 1 || stall_row < 0 || (long long)stall_row >= (long long)B * H) return DR_ERR_INVALID_ARG;
    dr_status st = check_dims(B, H, D);
    if (st != DR_OK) return st;
    int cap = 0;
    st = check_cache(cache, &cap);
    if (st != DR_OK) return st;
    st = check_attn_args(q, seq_len, out, out_dtype, scale);
    if (st != DR_OK) return st;
    dr::AttnParams p;
    fill_cache(p, q, cache, seq_len, B, H, cap, scale, out, out_dtype, err_flag);
    p.stall_row = stall_row;
    const int sms = dr::current_device_sms();
    if (sms <= 0) return DR_ERR_CUDA;
    // only the streaming variant (a grid larger than 4 CTAs per SM) with split rows waits on an mbarrier
    const int splits = self_splits(p, max_seq_len_hint, sms);
    if (splits < 2 || (long long)splits * H * B <= 4LL * sms) return DR_ERR_UNSUPPORTED;
    return from_cuda(dr::launch_decode_attn(p, cache->layout == DR_KV_PAGED, splits, static_cast<cudaStream_t>(stream)));
}

dr_status dr_decode_cross_attn(const void *q, const void *k_enc, const void *v_enc, const int32_t *enc_len, int B,
                               int H, int D, int Lc_max, float scale, void *out, dr_dtype out_dtype,
                               int32_t *err_flag, void *stream) {
    dr_status st = check_dims(B, H, D);
    if (st != DR_OK) return st;
    if (!k_enc || !v_enc || Lc_max < 1 || !aligned16(k_enc) || !aligned16(v_enc)) return DR_ERR_INVALID_ARG;
    st = check_attn_args(q, enc_len, out, out_dtype, scale);
    if (st != DR_OK) return st;
    dr::AttnParams p;
    fill_self(p, q, k_enc, v_enc, enc_len, nullptr, B, H, Lc_max, 0, 0, scale, out, out_dtype, err_flag);
    return launch(p, false, Lc_max, stream);
}

dr_status dr_decode_layer(const void *q, const dr_kv_cache *cache, const void *k_new, const void *v_new,
                          const int32_t *seq_len, const void *q_cross, const void *k_enc, const void *v_enc,
                          const int32_t *enc_len, int Lc_max, int B, int H, int D, int max_seq_len_hint, float scale,
                          void *out, void *out_cross, dr_dtype out_dtype, int32_t *err_flag, void *stream) {
    dr_status st = check_dims(B, H, D);
    if (st != DR_OK) return st;
    if (B > 32767) return DR_ERR_INVALID_ARG;   // self and cross rows share the grid's z dimension
    int cap = 0;
    st = check_cache(cache, &cap);
    if (st != DR_OK) return st;
    st = check_attn_args(q, seq_len, out, out_dtype, scale);
    if (st != DR_OK) return st;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return DR_ERR_INVALID_ARG;
    if (!q_cross || !k_enc || !v_enc || !enc_len || !out_cross || Lc_max < 1) return DR_ERR_INVALID_ARG;
    if (!aligned16(q_cross) || !aligned16(k_enc) || !aligned16(v_enc)) return DR_ERR_INVALID_ARG;
    const bool paged = cache->layout == DR_KV_PAGED;
    dr::AttnParams p;
    fill_cache(p, q, cache, seq_len, B, H, cap, scale, out, out_dtype, err_flag);
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.xq = static_cast<const uint16_t *>(q_cross);
    p.xk = static_cast<const uint16_t *>(k_enc);
    p.xv = static_cast<const uint16_t *>(v_enc);
    p.xlens = enc_len;
    p.xcap = Lc_max;
    p.xout = out_cross;
    // A description row takes one CTA of its own (packed, one row per CTA) when
    // the standalone plan gives it one, or when it is no longer than one self
    // CTA's share of the longest self row; otherwise it is split like the self rows.
    const int sms = dr::current_device_sms();
    if (sms <= 0) return DR_ERR_CUDA;
    const int s_self = self_splits(p, max_seq_len_hint, sms);
    const int self_tiles = (length_bound(p, max_seq_len_hint) + dr::kBlockKeys - 1) / dr::kBlockKeys;
    const int cross_tiles = (Lc_max + dr::kBlockKeys - 1) / dr::kBlockKeys;
    p.xpacked = dr_plan_splits(B, H, Lc_max, DR_KV_BF16, sms) == 1 ||
                cross_tiles <= (self_tiles + s_self - 1) / s_self;
    return from_cuda(dr::launch_decode_attn(p, paged, s_self, static_cast<cudaStream_t>(stream)));
}

dr_status dr_sample_topk_delayed(const float *logits, int B, int C, int V, int ldv, float temperature, int top_k,
                                 const uint64_t *seeds, int32_t *step, int32_t pad_id, int32_t *tokens, float *probs,
                                 int flags, void *stream) {
    if (!logits || !seeds || !step || !tokens) return DR_ERR_INVALID_ARG;
    if (B < 1 || C < 1 || V < 1 || ldv < V) return DR_ERR_INVALID_ARG;
    // one CTA row per batch row: the grid's y dimension holds at most 65535
    if (B > 65535 || C > dr::kMaxCodebooks || V > dr::kMaxVocab) return DR_ERR_UNSUPPORTED;
    if (top_k < 1 || top_k > V) return DR_ERR_INVALID_ARG;
    if (!(temperature > 0.f) || isinf(temperature)) return DR_ERR_INVALID_ARG;
    if (flags & ~DR_SAMPLE_ADVANCE) return DR_ERR_INVALID_ARG;
    dr::SampleParams p;
    p.logits = logits;
    p.seeds = seeds;
    p.step = step;
    p.tokens = tokens;
    p.probs = probs;
    p.B = B;
    p.C = C;
    p.V = V;
    p.ldv = ldv;
    p.top_k = top_k;
    p.pad_id = pad_id;
    p.flags = flags;
    p.temperature = temperature;
    return from_cuda(dr::launch_sample(p, static_cast<cudaStream_t>(stream)));
}

dr_status dr_embed_tokens(const int32_t *tokens, const void *table, int B, int C, int V, int Dm, void *out,
                          dr_dtype out_dtype, int32_t *err_flag, void *stream) {
    if (!tokens || !table || !out || !aligned16(table) || !aligned16(out)) return DR_ERR_INVALID_ARG;
    if (B < 1 || B > 0x7FFFFFFF || C < 1 || V < 1 || Dm < 8 || Dm % 8 != 0) return DR_ERR_INVALID_ARG;
    if (out_dtype != DR_BF16 && out_dtype != DR_F32) return DR_ERR_INVALID_ARG;
    // the kernel keeps one token per codebook in registers, up to kMaxCodebooks of them
    if (C > dr::kMaxCodebooks) return DR_ERR_UNSUPPORTED;
    dr::EmbedParams p;
    p.tokens = tokens;
    p.table = static_cast<const uint16_t *>(table);
    p.out = out;
    p.B = B;
    p.C = C;
    p.V = V;
    p.Dm = Dm;
    p.out_f32 = out_dtype == DR_F32;
    p.err = err_flag;
    return from_cuda(dr::launch_embed_tokens(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// dr_lm_head's checks and launch; stall_slab >= 0 only from the test hook below.
dr_status lm_head_call(const void *hidden, const void *W, int B, int K, int C, int V, int ldv, float *logits,
                       int32_t *err_flag, int stall_slab, void *stream) {
    if (!hidden || !W || !logits || !aligned16(hidden) || !aligned16(W)) return DR_ERR_INVALID_ARG;
    if (B < 1 || C < 1 || V < 1 || ldv < V || K < 1) return DR_ERR_INVALID_ARG;
    if ((long long)C * V > 0x7FFFFFFFLL) return DR_ERR_INVALID_ARG;
    const int kc = K / 256;
    if (K % 256 != 0 || !(kc == 1 || kc == 2 || kc == 3 || kc == 4 || kc == 6 || kc == 8)) return DR_ERR_UNSUPPORTED;
    dr::LmHeadParams p;
    p.hidden = static_cast<const uint16_t *>(hidden);
    p.W = static_cast<const uint16_t *>(W);
    p.logits = logits;
    p.B = B;
    p.K = K;
    p.C = C;
    p.V = V;
    p.ldv = ldv;
    p.err = err_flag;
    p.stall_slab = stall_slab;
    return from_cuda(dr::launch_lm_head(p, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

dr_status dr_lm_head(const void *hidden, const void *W, int B, int K, int C, int V, int ldv, float *logits,
                     int32_t *err_flag, void *stream) {
    return lm_head_call(hidden, W, B, K, C, V, ldv, logits, err_flag, -1, stream);
}

dr_status dr_lm_head_stall_test(const void *hidden, const void *W, int B, int K, int C, int V, int ldv, float *logits,
                                int32_t *err_flag, int stall_slab, void *stream) {
    // only the tensor-core head has pipeline waits; the slab must exist
    if (B < dr::kLmHeadTensorCoreMinBatch) return DR_ERR_UNSUPPORTED;
    if (C < 1 || V < 1 || stall_slab < 0 || (long long)stall_slab * 128 >= (long long)C * V) return DR_ERR_INVALID_ARG;
    return lm_head_call(hidden, W, B, K, C, V, ldv, logits, err_flag, stall_slab, stream);
}

const char *dr_status_string(dr_status s) {
    switch (s) {
        case DR_OK: return "ok";
        case DR_ERR_INVALID_ARG: return "invalid argument";
        case DR_ERR_UNSUPPORTED: return "unsupported shape";
        case DR_ERR_CUDA: return "CUDA launch failed";
    }
    return "unknown status";
}

}  // extern "C"
