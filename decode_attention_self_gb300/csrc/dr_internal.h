// Internal declarations shared by the translation units of libdecoderattn.so.
// Launch helpers take validated arguments; the extern "C" layer in dr_api.cu
// owns all argument checking.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dr_api.h"

namespace dr {

constexpr int kHeadDim = 64;     // D: the only head dimension built
constexpr int kBlockKeys = 16;   // keys per paged block, and per attention tile
constexpr int kMaxCodebooks = 16;
constexpr int kMaxVocab = 2048;

// Launch `kern` with programmatic dependent launch enabled and, when
// cluster_x > 1, as clusters of cluster_x CTAs along x.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
#ifndef DR_NO_PDL
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
#endif
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Largest thread-block cluster used for one (b, h) row of attention.
int max_cluster_size();

// SM count of the current device (cached per device).
int current_device_sms();

struct AttnParams {
    const uint16_t *q;       // [B][H][64] bf16 bits
    const void *k;           // contiguous [B][H][cap][64] or paged [NB][H][16][64], bf16 or e4m3
    const void *v;
    const int32_t *lens;     // [B]
    const int32_t *table;    // paged: [B][max_blocks]
    int32_t B, H;
    int32_t cap;             // keys a row can hold
    int32_t max_blocks;      // paged: block-table row stride
    int32_t num_blocks;      // paged: pool size
    int32_t kv_fp8;          // 1: the cache holds e4m3 codes (k = code * k_scale, v = code * v_scale)
    float qscale;            // softmax scale * log2(e) (* k_scale for an e4m3 cache)
    float k_scale, v_scale;  // e4m3 cache scales (used by the fused append)
    float out_scale;         // v_scale for an e4m3 cache, else 1
    void *out;               // [B][H][64]
    int32_t out_f32;
    int32_t *err;
    // Fused decode-layer launch only (see dr_decode_layer): this step's key and
    // value, stored at position lens[b]-1 of the cache and used from registers,
    // and a second set of B rows attending the description encoder's keys (bf16).
    const uint16_t *k_new;   // [B][H][64] or null
    const uint16_t *v_new;
    const uint16_t *xq;      // cross rows: [B][H][64] or null (no cross rows)
    const uint16_t *xk;      // [B][H][xcap][64]
    const uint16_t *xv;
    const int32_t *xlens;    // [B]
    int32_t xcap;
    float xqscale;           // softmax scale * log2(e) for the cross rows
    void *xout;              // [B][H][64]
    int32_t xpacked;         // 1: one CTA per cross row, gridDim.x rows per cluster; 0: rows split like self rows
    // Test hook (streaming variant only): CTA 1 of row b*H + h == stall_row never sends its state, so rank 0's
    // bounded wait for it runs out; -1 (every ordinary call): none.
    int32_t stall_row = -1;
};

cudaError_t launch_decode_attn(const AttnParams &p, bool paged, int splits, cudaStream_t stream);

struct AppendParams {
    void *k, *v;                     // bf16 or e4m3 cache
    const uint16_t *k_new, *v_new;   // [B][H][64]
    const int32_t *pos;              // [B]
    const int32_t *table;            // paged only
    int32_t B, H, cap, max_blocks, num_blocks;
    int32_t kv_fp8;                  // quantise to e4m3: code = e4m3(fl32(x / scale))
    float k_scale, v_scale;
    int32_t *err;
};

cudaError_t launch_kv_append(const AppendParams &p, bool paged, cudaStream_t stream);

struct SampleParams {
    const float *logits;     // [B][C][ldv]
    const uint64_t *seeds;   // [B]
    int32_t *step;           // [B]
    int32_t *tokens;         // [B][C]
    float *probs;            // nullable [B][C][V]
    int32_t B, C, V, ldv, top_k, pad_id, flags;
    float temperature;
};

cudaError_t launch_sample(const SampleParams &p, cudaStream_t stream);

struct EmbedParams {
    const int32_t *tokens;   // [B][C]
    const uint16_t *table;   // [C*V][Dm] bf16
    void *out;               // [B][Dm] bf16 or f32
    int32_t B, C, V, Dm, out_f32;
    int32_t *err;
};

cudaError_t launch_embed_tokens(const EmbedParams &p, cudaStream_t stream);

struct LmHeadParams {
    const uint16_t *hidden;  // [B][K] bf16
    const uint16_t *W;       // [C*V][K] bf16
    float *logits;           // [B][C][ldv]
    int32_t B, K, C, V, ldv;
    int32_t *err;
    // Test hook (tensor-core head only): the CTAs of this 128-row weight slab never load their first K chunk,
    // so their bounded pipeline wait runs out; -1 (every ordinary call): none.
    int32_t stall_slab = -1;
};

cudaError_t launch_lm_head(const LmHeadParams &p, cudaStream_t stream);

// Batches from this size on run the merged head on the tensor cores (tcgen05).
constexpr int kLmHeadTensorCoreMinBatch = 4;
cudaError_t launch_lm_head_tc(const LmHeadParams &p, int32_t *err, cudaStream_t stream);

}  // namespace dr
