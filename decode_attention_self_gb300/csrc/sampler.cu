// Fused sampler: temperature, top-k, softmax and categorical draw for every
// codebook of every row, in one kernel, under the delay pattern.
//
// Source: Optimized Parler TTS, "Future work" item 2 -- temperature scaling,
// top-k and softmax ran as more than ten kernels with global-memory round
// trips and should be one fused kernel; "Analysis and improvements" --
// sampling without a GPU-CPU synchronisation; the architecture overview --
// nine DAC codebooks, one token each per step, in a delayed pattern.
//
// Grid (C, B): one CTA of NT threads per (codebook c, row b), NT = 256, or 128
// when the grid would not fit the GPU at once with 256.  A CTA
//   1. reads its V logits once (element i = t + NT j stays in thread t's
//      registers), divides by T with IEEE round-to-nearest and maps each float
//      to an order-preserving uint32 key;
//   2. finds the top_k-th largest key tau by an 8-bit radix select of up to 4
//      passes: double-buffered shared-memory histograms (shared atomics), one
//      warp scanning each in descending digit order, two barriers per pass.
//      When the digit bin that holds the top_k-th key holds exactly the keys
//      still needed, the whole bin is kept and the select stops there;
//   3. keeps every key above the threshold plus, when the select ran to a full
//      key, the lowest-index entries equal to tau (their rank in index order
//      comes from warp ballots), so ties go to the lower index exactly, and
//      compacts the kept indices into a shared list;
//   4. draws by Gumbel-max over the list, spread evenly over the threads:
//      u_i from Philox4x32-10 (Salmon et al., SC'11) keyed by the row's seed,
//      counter (i/4, c, step, b); argmax of x_i - log(-log u_i), equal scores
//      to the lower index;
//   5. optionally writes the softmax over the kept set.
// A codebook with step[b] <= c emits pad_id (delay pattern).  With
// DR_SAMPLE_ADVANCE the C CTAs of a row form one thread-block cluster; after a
// cluster barrier -- every CTA has read step[b] -- rank 0 increments it.
//
// Latency-bound: the 39 KB of logits of a row are nanoseconds of HBM time; the
// cost is the chain of dependent on-chip passes.
#include <cooperative_groups.h>
#include <math.h>

#include "dr_device.cuh"
#include "dr_internal.h"

namespace cg = cooperative_groups;

namespace dr {
namespace {

// Threads per CTA: 256 while the grid fits the GPU at once with four such CTAs per SM (the register bound);
// 128 for larger grids, so that twice the CTAs are resident and the grid still runs as one wave (batch 128:
// 1152 CTAs, in clusters of 9 with DR_SAMPLE_ADVANCE).
constexpr int kWideThreads = 256;
constexpr int kNarrowThreads = 128;
constexpr int kWideCtasPerSm = 4;

// Philox4x32-10, Salmon, Moraes, Dror and Shaw, SC'11, section 3.
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;   // golden-ratio Weyl increment
            k1 += 0xBB67AE85u;   // sqrt(3) - 1 Weyl increment
        }
        const uint32_t lo0 = 0xD2511F53u * x.x, hi0 = __umulhi(0xD2511F53u, x.x);
        const uint32_t lo1 = 0xCD9E8D57u * x.z, hi1 = __umulhi(0xCD9E8D57u, x.z);
        x = make_uint4(hi1 ^ x.y ^ k0, lo1, hi0 ^ x.w ^ k1, lo0);
    }
    return x;
}

__device__ __forceinline__ uint32_t order_key(float x) {
    uint32_t u = __float_as_uint(x);
    if (u == 0x80000000u) u = 0u;   // -0 sorts with +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ bool better(float s, int i, float bs, int bi) {
    return s > bs || (s == bs && i < bi);
}

// Block-wide exclusive prefix sum of one value per thread (all threads call).
template <int kWarps>
__device__ __forceinline__ int block_exclusive_scan(int v, int *s_warp, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const int s = s_warp[w];
        if (w < warp) before += s;
        total += s;
    }
    __syncthreads();   // s_warp may be reused right after
    return before + inc - v;
}

template <int EPT, int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads == kNarrowThreads ? 8 : kWideCtasPerSm) sample_kernel(const SampleParams p) {
    constexpr int kWarps = kThreads / 32;
    __shared__ uint32_t s_hist[2][256];
    __shared__ int s_sel[3];   // selected digit, keys still needed, keys in the digit's bin
    __shared__ uint32_t s_bal[EPT][kWarps];
    __shared__ int s_scan[kWarps];
    __shared__ int s_list[kMaxVocab];
    __shared__ float s_rf[kWarps];
    __shared__ int s_ri[kWarps];

    pdl_wait();
    const int c = blockIdx.x;
    const int b = blockIdx.y;
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    // The row's logits are loaded before the step is known, so that the two loads are in flight together (a
    // padded codebook does not use them; the row exists either way).
    const float *row = p.logits + ((size_t)b * p.C + c) * (size_t)p.ldv;
    float lg[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int i = t + kThreads * j;
        lg[j] = i < p.V ? __ldg(row + i) : 0.f;
    }
    const int step = p.step[b];
    const bool active = step > c;   // delay pattern: codebook c is padded while step <= c
    float *prow = p.probs ? p.probs + ((size_t)b * p.C + c) * (size_t)p.V : nullptr;

    if (!active) {
        if (t == 0) p.tokens[(size_t)b * p.C + c] = p.pad_id;
        if (prow)
            for (int i = t; i < p.V; i += kThreads) prow[i] = 0.f;
    } else {
        // Only the order keys stay in registers; key_value() inverts the map.
        uint32_t key[EPT];
        uint32_t valid = 0;
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int i = t + kThreads * j;
            key[j] = 0u;
            if (i < p.V) {
                key[j] = order_key(__fdiv_rn(lg[j], p.temperature));
                valid |= 1u << j;
            }
        }
        for (int i = t; i < 256; i += kThreads) {
            s_hist[0][i] = 0u;
            s_hist[1][i] = 0u;
        }
        __syncthreads();

        // ---- radix select of the top_k-th largest key ------------------------
        uint32_t prefix = 0u, pmask = 0u;
        int kk = p.top_k;
        bool whole_bin = false;   // the threshold bin is kept whole: no tie ranking needed
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            uint32_t *hist = s_hist[pass & 1];
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                if (((valid >> j) & 1u) && (key[j] & pmask) == prefix) atomicAdd(&hist[(key[j] >> shift) & 255u], 1u);
            }
            __syncthreads();
            for (int i = t; i < 256; i += kThreads) s_hist[(pass + 1) & 1][i] = 0u;   // free now: clear it for the next pass
            if (warp == 0) {
                // lane l scans digits 255 - 8l down to 248 - 8l; a warp scan orders the lanes
                uint32_t c8[8], sum = 0u;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    c8[e] = hist[255 - 8 * lane - e];
                    sum += c8[e];
                }
                uint32_t inc = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                    if (lane >= o) inc += n;
                }
                uint32_t before = inc - sum;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (before < (uint32_t)kk && (uint32_t)kk <= before + c8[e]) {
                        s_sel[0] = 255 - 8 * lane - e;
                        s_sel[1] = kk - (int)before;
                        s_sel[2] = (int)c8[e];
                    }
                    before += c8[e];
                }
            }
            __syncthreads();
            prefix |= (uint32_t)s_sel[0] << shift;
            pmask |= 0xFFu << shift;
            kk = s_sel[1];
            if (kk == s_sel[2]) {   // the same in every thread
                whole_bin = true;
                break;
            }
        }
        const uint32_t tau = prefix;   // without whole_bin: kk entries equal to tau are taken, lowest index first

        // ---- membership: keys above the threshold, and ties in index order ------
        uint32_t member = 0u;
        int nmine = 0;
        if (whole_bin) {
#pragma unroll
            for (int j = 0; j < EPT; ++j)
                if (((valid >> j) & 1u) && (key[j] & pmask) >= prefix) {
                    member |= 1u << j;
                    ++nmine;
                }
        } else {
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ((valid >> j) & 1u) && key[j] == tau);
                if (lane == 0) s_bal[j][warp] = bal;
            }
            __syncthreads();
            const uint32_t lt_mask = (1u << lane) - 1u;
            int ties_before = 0;
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                int row_before = 0, row_total = 0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const int n = __popc(s_bal[j][w]);
                    if (w < warp) row_before += n;
                    row_total += n;
                }
                if ((valid >> j) & 1u) {
                    bool take = key[j] > tau;
                    if (key[j] == tau)
                        take = ties_before + row_before + __popc(s_bal[j][warp] & lt_mask) < kk;
                    if (take) {
                        member |= 1u << j;
                        ++nmine;
                    }
                }
                ties_before += row_total;
            }
        }
        // compact the kept indices (top_k of them) into s_list
        int total = 0;
        int slot = block_exclusive_scan<kWarps>(nmine, s_scan, total);
#pragma unroll
        for (int j = 0; j < EPT; ++j)
            if ((member >> j) & 1u) s_list[slot++] = t + kThreads * j;
        __syncthreads();

        // ---- Gumbel-max draw over the list -------------------------------------
        const uint64_t seed = p.seeds[b];
        const uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFull), k1 = (uint32_t)(seed >> 32);
        float best = -INFINITY;
        int best_i = 0x7FFFFFFF;
        for (int r = t; r < total; r += kThreads) {
            const int i = s_list[r];
            const float x = __fdiv_rn(__ldg(row + i), p.temperature);   // same rounding as the key
            const uint4 w4 = philox4x32_10(make_uint4((uint32_t)i >> 2, (uint32_t)c, (uint32_t)step, (uint32_t)b),
                                           k0, k1);
            const uint32_t w = (i & 3) == 0 ? w4.x : (i & 3) == 1 ? w4.y : (i & 3) == 2 ? w4.z : w4.w;
            const float u = (float)(2u * (w >> 9) + 1u) * 0x1p-24f;   // exact odd multiple of 2^-24
            const float s = x - logf(-logf(u));
            if (better(s, i, best, best_i)) {
                best = s;
                best_i = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, best_i, o);
            if (better(os, oi, best, best_i)) {
                best = os;
                best_i = oi;
            }
        }
        if (lane == 0) {
            s_rf[warp] = best;
            s_ri[warp] = best_i;
        }
        __syncthreads();
        if (t == 0) {
            float bs = s_rf[0];
            int bi = s_ri[0];
            for (int w = 1; w < kWarps; ++w)
                if (better(s_rf[w], s_ri[w], bs, bi)) {
                    bs = s_rf[w];
                    bi = s_ri[w];
                }
            // NaN scores are never `better`: a set of NaN members alone leaves bi at its start value.  The
            // token is then undefined but stays a member of the kept set, so it is in range.
            p.tokens[(size_t)b * p.C + c] = bi == 0x7FFFFFFF ? s_list[0] : bi;
        }

        // ---- optional softmax over the kept set -------------------------------
        if (prow) {
            float xm = -INFINITY;
#pragma unroll
            for (int j = 0; j < EPT; ++j)
                if ((member >> j) & 1u) xm = fmaxf(xm, key_value(key[j]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) xm = fmaxf(xm, __shfl_xor_sync(0xFFFFFFFFu, xm, o));
            __syncthreads();   // s_rf is reused
            if (lane == 0) s_rf[warp] = xm;
            __syncthreads();
            xm = s_rf[0];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) xm = fmaxf(xm, s_rf[w]);
            float z = 0.f;
            if (xm != -INFINITY) {
#pragma unroll
                for (int j = 0; j < EPT; ++j)
                    if ((member >> j) & 1u) z += expf(key_value(key[j]) - xm);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
            }
            __syncthreads();
            if (lane == 0) s_rf[warp] = z;
            __syncthreads();
            z = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) z += s_rf[w];
            const float uniform = 1.0f / (float)p.top_k;
#pragma unroll
            for (int j = 0; j < EPT; ++j) {
                const int i = t + kThreads * j;
                if (i < p.V) {
                    float pr = 0.f;
                    if ((member >> j) & 1u)
                        pr = (xm == -INFINITY) ? uniform : __fdiv_rn(expf(key_value(key[j]) - xm), z);
                    prow[i] = pr;
                }
            }
        }
    }

    pdl_trigger();
    if (p.flags & DR_SAMPLE_ADVANCE) {
        // every thread of every codebook CTA of this row has read step[b] before it changes
        if (gridDim.x > 1) cg::this_cluster().sync();
        else __syncthreads();
        if (blockIdx.x == 0 && t == 0) p.step[b] = step + 1;
    }
}

template <int EPT, int kThreads>
cudaError_t launch_ept(const SampleParams &p, cudaStream_t stream) {
    const bool clustered = (p.flags & DR_SAMPLE_ADVANCE) && p.C > 1;
    auto kern = sample_kernel<EPT, kThreads>;
    if (clustered && p.C > 8) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(kern, dim3((unsigned)p.C, (unsigned)p.B, 1), dim3(kThreads), 0, stream,
                         clustered ? (unsigned)p.C : 1u, p);
}

}  // namespace

cudaError_t launch_sample(const SampleParams &p, cudaStream_t stream) {
    const long long ctas = (long long)p.B * p.C;
    if (ctas <= (long long)kWideCtasPerSm * current_device_sms()) {
        const int ept = (p.V + kWideThreads - 1) / kWideThreads;
        if (ept <= 1) return launch_ept<1, kWideThreads>(p, stream);
        if (ept <= 2) return launch_ept<2, kWideThreads>(p, stream);
        if (ept <= 4) return launch_ept<4, kWideThreads>(p, stream);
        if (ept <= 5) return launch_ept<5, kWideThreads>(p, stream);
        return launch_ept<8, kWideThreads>(p, stream);
    }
    const int ept = (p.V + kNarrowThreads - 1) / kNarrowThreads;
    if (ept <= 2) return launch_ept<2, kNarrowThreads>(p, stream);
    if (ept <= 4) return launch_ept<4, kNarrowThreads>(p, stream);
    if (ept <= 9) return launch_ept<9, kNarrowThreads>(p, stream);
    return launch_ept<16, kNarrowThreads>(p, stream);
}

}  // namespace dr
