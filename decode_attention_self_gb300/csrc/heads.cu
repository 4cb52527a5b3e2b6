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
// LM head: warp w of CTA g owns weight rows n = (g*kWarps + w)*kRows + r.
// Lane l holds the 16-byte chunks l, l+32, ... of each of its rows (K/256 per
// row) for the whole launch; hidden vectors are staged kBatch at a time in
// shared memory and every row is dotted with each of them.
// ---------------------------------------------------------------------------
constexpr int kHeadWarps = 8;
constexpr int kHeadThreads = kHeadWarps * 32;
constexpr int kRows = 2;      // weight rows per warp
constexpr int kBatch = 16;    // hidden vectors per shared-memory stage

template <int KC>   // 16-byte chunks per lane per row: K = 256 * KC
__global__ void __launch_bounds__(kHeadThreads) lm_head_kernel(const LmHeadParams p) {
    extern __shared__ uint4 s_hidden[];   // [kBatch][K/8]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = (blockIdx.x * kHeadWarps + warp) * kRows;
    const int N = p.C * p.V;
    const int kchunks = 32 * KC;
    // The weights are parameters, not an output of the previous kernel: warm L2 with this warp's rows
    // (contiguous) while that kernel drains, then wait for it.
    if (lane == 0 && n0 < N)
        prefetch_l2(p.W + (size_t)n0 * (kchunks * 8), (uint32_t)(min(kRows, N - n0) * kchunks * 16));
    pdl_wait();
    pdl_trigger();

    uint4 wr[kRows][KC];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
        const int n = n0 + r;
#pragma unroll
        for (int j = 0; j < KC; ++j)
            wr[r][j] = n < N ? ld_stream16(p.W + (size_t)n * (kchunks * 8) + (size_t)(lane + 32 * j) * 8)
                             : make_uint4(0, 0, 0, 0);
    }

    for (int b0 = 0; b0 < p.B; b0 += kBatch) {
        const int nb = min(kBatch, p.B - b0);
        __syncthreads();   // the previous stage is no longer read
        for (int i = threadIdx.x; i < nb * kchunks; i += kHeadThreads) {
            const int bb = i / kchunks, ch = i - bb * kchunks;
            s_hidden[i] = ld_ro16(p.hidden + ((size_t)(b0 + bb) * kchunks + ch) * 8);
        }
        __syncthreads();
        for (int bb = 0; bb < nb; ++bb) {
            float acc[kRows];
#pragma unroll
            for (int r = 0; r < kRows; ++r) acc[r] = 0.f;
#pragma unroll
            for (int j = 0; j < KC; ++j) {
                float h[8];
                unpack8(s_hidden[bb * kchunks + lane + 32 * j], h);
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    float w[8];
                    unpack8(wr[r][j], w);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[r] = fmaf(h[e], w[e], acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[r] += __shfl_xor_sync(0xFFFFFFFFu, acc[r], o);
            }
            if (lane < kRows) {
                const int n = n0 + lane;
                float v = acc[0];
#pragma unroll
                for (int r = 1; r < kRows; ++r)
                    if (lane == r) v = acc[r];
                if (n < N) {
                    const int c = n / p.V, vi = n - c * p.V;
                    p.logits[((size_t)(b0 + bb) * p.C + c) * p.ldv + vi] = v;
                }
            }
        }
    }
}

template <int KC>
cudaError_t launch_head(const LmHeadParams &p, cudaStream_t stream) {
    const int N = p.C * p.V;
    const int rows_per_cta = kHeadWarps * kRows;
    const unsigned grid = (unsigned)((N + rows_per_cta - 1) / rows_per_cta);
    const size_t smem = (size_t)kBatch * 32 * KC * sizeof(uint4);
    auto kern = lm_head_kernel<KC>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(kern, dim3(grid), dim3(kHeadThreads), smem, stream, 1u, p);
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
