// KV append: store this step's key and value of every (b, h) row.
//
// Source: Optimized Parler TTS, "Analysis and improvements" -- a static cache
// for causal attention, preallocated so that the decode step can be captured
// as one CUDA graph; and "Future work" item 1, the paged alternative.
//
// One thread moves 8 elements of k and of v (16 bytes of bf16, or 8 e4m3 codes
// quantised from them): B*H*8 threads.  The write position comes from device
// memory, so the same launch (or captured graph) serves every step.
#include "dr_device.cuh"
#include "dr_internal.h"

namespace dr {
namespace {

constexpr int kThreads = 256;

template <bool kPaged, bool kFp8>
__global__ void __launch_bounds__(kThreads) kv_append_kernel(const AppendParams p) {
    pdl_wait();
    pdl_trigger();
    const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
    const long long total = (long long)p.B * p.H * 8;
    if (idx >= total) return;
    const int chunk = (int)(idx & 7);
    const long long row = idx >> 3;
    const int b = (int)(row / p.H);
    const int h = (int)(row - (long long)b * p.H);
    const int pos = __ldg(p.pos + b);
    if (pos < 0 || pos >= p.cap) {
        if (h == 0 && chunk == 0) flag_error(p.err, DR_ERRF_POS);
        return;
    }
    size_t dst;   // element offset of the row's slot
    if constexpr (kPaged) {
        const int blk = __ldg(p.table + (size_t)b * p.max_blocks + pos / kBlockKeys);
        if ((unsigned)blk >= (unsigned)p.num_blocks) {
            if (h == 0 && chunk == 0) flag_error(p.err, DR_ERRF_POS);
            return;
        }
        dst = (((size_t)blk * p.H + h) * kBlockKeys + (size_t)(pos % kBlockKeys)) * kHeadDim;
    } else {
        dst = ((size_t)row * p.cap + (size_t)pos) * kHeadDim;
    }
    const size_t src = (size_t)row * kHeadDim + chunk * 8;
    const uint4 kn = ld_ro16(p.k_new + src);
    const uint4 vn = ld_ro16(p.v_new + src);
    if constexpr (kFp8) {
        uint8_t *k = static_cast<uint8_t *>(p.k), *v = static_cast<uint8_t *>(p.v);
        *reinterpret_cast<uint2 *>(k + dst + chunk * 8) = quantize8_e4m3(kn, p.k_scale);
        *reinterpret_cast<uint2 *>(v + dst + chunk * 8) = quantize8_e4m3(vn, p.v_scale);
    } else {
        uint16_t *k = static_cast<uint16_t *>(p.k), *v = static_cast<uint16_t *>(p.v);
        *reinterpret_cast<uint4 *>(k + dst + chunk * 8) = kn;
        *reinterpret_cast<uint4 *>(v + dst + chunk * 8) = vn;
    }
}

}  // namespace

cudaError_t launch_kv_append(const AppendParams &p, bool paged, cudaStream_t stream) {
    const long long total = (long long)p.B * p.H * 8;
    const unsigned grid = (unsigned)((total + kThreads - 1) / kThreads);
    auto kern = p.kv_fp8 ? (paged ? kv_append_kernel<true, true> : kv_append_kernel<false, true>)
                         : (paged ? kv_append_kernel<true, false> : kv_append_kernel<false, false>);
    return launch_kernel(kern, dim3(grid), dim3(kThreads), 0, stream, 1u, p);
}

}  // namespace dr
