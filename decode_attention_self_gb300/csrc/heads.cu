// The decoder's per-step input and output ends around the attention:
//
//   embed_tokens_kernel -- the next step's decoder input: for every row, the sum
//     over the codebooks of each codebook's embedding of the token it emitted
//     (Optimized Parler TTS, "Analysis and improvements", other optimizations
//     item 3: the nine embedding lookups merged into one gather from one
//     merged table [C*V][Dm]).
//   lm_head_kernel -- the merged LM head on the newest position only (same
//     list, items 1-2: the head evaluated for the last position, the nine
//     codebook heads merged into one weight matrix [C*V][K]), writing fp32
//     logits straight into the sampler's [B][C][ldv] layout.
//
// The embedding gathers C rows of Dm bf16 per batch row (HBM/launch bound).  At
// small batch the head is a matrix-vector product bound by streaming the
// C*V x K bf16 weights once: the CUDA-core kernel here applies every weight row
// to all B hidden vectors from shared memory (fp32 accumulation).  From
// kLmHeadTensorCoreMinBatch rows on it is a dense contraction and runs on the
// tensor cores (lm_head_tc.cu).
#include "dr_device.cuh"
#include "dr_internal.h"

namespace dr {
namespace {

// ---------------------------------------------------------------------------
// embedding: one CTA per batch row, each thread 8 consecutive dims (16 bytes)
// ---------------------------------------------------------------------------
constexpr int kEmbThreads = 128;

__global__ void __launch_bounds__(kEmbThreads) embed_tokens_kernel(const EmbedParams p) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    const int chunks = p.Dm / 8;
    // the row's tokens first (the same for every thread), so that all C row loads are in flight at once
    int tok[kMaxCodebooks];
    bool ok[kMaxCodebooks];
#pragma unroll
    for (int c = 0; c < kMaxCodebooks; ++c) {
        tok[c] = c < p.C ? __ldg(p.tokens + (size_t)b * p.C + c) : 0;
        ok[c] = c < p.C && (unsigned)tok[c] < (unsigned)p.V;
        if (c < p.C && !ok[c] && threadIdx.x == 0) flag_error(p.err, DR_ERRF_TOKEN);
    }
    for (int ch = threadIdx.x; ch < chunks; ch += kEmbThreads) {
        uint4 e[kMaxCodebooks];
#pragma unroll
        for (int c = 0; c < kMaxCodebooks; ++c)
            if (ok[c]) e[c] = ld_ro16(p.table + ((size_t)c * p.V + tok[c]) * p.Dm + ch * 8);
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
        for (int c = 0; c < kMaxCodebooks; ++c) {   // fp32 sum in codebook order
            if (!ok[c]) continue;
            float f[8];
            unpack8(e[c], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += f[j];
        }
        if (p.out_f32) {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + (size_t)b * p.Dm + ch * 8);
            o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        } else {
            uint4 w;
            w.x = (uint32_t)f32_to_bf16_rn(acc[0]) | ((uint32_t)f32_to_bf16_rn(acc[1]) << 16);
            w.y = (uint32_t)f32_to_bf16_rn(acc[2]) | ((uint32_t)f32_to_bf16_rn(acc[3]) << 16);
            w.z = (uint32_t)f32_to_bf16_rn(acc[4]) | ((uint32_t)f32_to_bf16_rn(acc[5]) << 16);
            w.w = (uint32_t)f32_to_bf16_rn(acc[6]) | ((uint32_t)f32_to_bf16_rn(acc[7]) << 16);
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + (size_t)b * p.Dm + ch * 8) = w;
        }
    }
}

// ---------------------------------------------------------------------------
// LM head below kLmHeadTensorCoreMinBatch rows: a persistent grid of one wave
// (KC <= 4: four CTAs per SM).  Warp w of the grid takes weight rows w, w + W,
// w + 2W, ... (W = warps in the grid); lane l holds the 16-byte chunks l,
// l+32, ... of its current row while the next row's loads are in flight, and
// dots it with every hidden vector (staged once in shared memory).  Each logit
// is the same fp32 sum in the same order as a per-row kernel would make it.
// ---------------------------------------------------------------------------
constexpr int kHeadWarps = 8;
constexpr int kHeadThreads = kHeadWarps * 32;
static_assert(kLmHeadTensorCoreMinBatch <= 4, "the hidden vectors of the CUDA-core head fit shared memory");

template <int KC>   // 16-byte chunks per lane per row: K = 256 * KC
constexpr int head_ctas_per_sm() { return KC <= 4 ? 4 : 2; }

template <int KC>
__global__ void __launch_bounds__(kHeadThreads, head_ctas_per_sm<KC>()) lm_head_kernel(const LmHeadParams p) {
    extern __shared__ uint4 s_hidden[];   // [B][K/8]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.C * p.V;
    const int kchunks = 32 * KC;
    const size_t row_elems = (size_t)kchunks * 8;
    const int gw = (int)gridDim.x * kHeadWarps;
    const int n0 = (int)blockIdx.x * kHeadWarps + warp;
    // The weights are parameters, not an output of the previous kernel: warm L2 with this warp's first two
    // rows while that kernel drains, then wait for it.
    if (lane == 0) {
        if (n0 < N) prefetch_l2(p.W + (size_t)n0 * row_elems, (uint32_t)kchunks * 16u);
        if (n0 + gw < N) prefetch_l2(p.W + (size_t)(n0 + gw) * row_elems, (uint32_t)kchunks * 16u);
    }
    pdl_wait();
    pdl_trigger();

    uint4 cur[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j)
        cur[j] = n0 < N ? ld_stream16(p.W + (size_t)n0 * row_elems + (size_t)(lane + 32 * j) * 8) : make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < p.B * kchunks; i += kHeadThreads) s_hidden[i] = ld_ro16(p.hidden + (size_t)i * 8);
    __syncthreads();

    for (int n = n0; n < N; n += gw) {
        const int nn = n + gw;
        uint4 nxt[KC];
#pragma unroll
        for (int j = 0; j < KC; ++j)
            nxt[j] = nn < N ? ld_stream16(p.W + (size_t)nn * row_elems + (size_t)(lane + 32 * j) * 8)
                            : make_uint4(0, 0, 0, 0);
        const int c = n / p.V, vi = n - c * p.V;
        for (int bb = 0; bb < p.B; ++bb) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                float h[8], w[8];
                unpack8(s_hidden[bb * kchunks + lane + 32 * j], h);
                unpack8(cur[j], w);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(h[e], w[e], acc);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
            if (lane == 0) p.logits[((size_t)bb * p.C + c) * p.ldv + vi] = acc;
        }
#pragma unroll
        for (int j = 0; j < KC; ++j) cur[j] = nxt[j];
    }
}

template <int KC>
cudaError_t launch_head(const LmHeadParams &p, cudaStream_t stream) {
    const int N = p.C * p.V;
    const int by_rows = (N + kHeadWarps - 1) / kHeadWarps;
    const int one_wave = head_ctas_per_sm<KC>() * current_device_sms();
    const unsigned grid = (unsigned)(by_rows < one_wave ? by_rows : one_wave);
    const size_t smem = (size_t)p.B * 32 * KC * sizeof(uint4);
    return launch_kernel(lm_head_kernel<KC>, dim3(grid), dim3(kHeadThreads), smem, stream, 1u, p);
}

}  // namespace

cudaError_t launch_embed_tokens(const EmbedParams &p, cudaStream_t stream) {
    return launch_kernel(embed_tokens_kernel, dim3((unsigned)p.B), dim3(kEmbThreads), 0, stream, 1u, p);
}

cudaError_t launch_lm_head(const LmHeadParams &p, cudaStream_t stream) {
    if (p.B >= kLmHeadTensorCoreMinBatch) return launch_lm_head_tc(p, p.err, stream);
    switch (p.K / 256) {
        case 1: return launch_head<1>(p, stream);
        case 2: return launch_head<2>(p, stream);
        case 3: return launch_head<3>(p, stream);
        case 4: return launch_head<4>(p, stream);
        case 6: return launch_head<6>(p, stream);
        case 8: return launch_head<8>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dr
