// Fused sampler: temperature, top-k, softmax and categorical draw for every
// codebook of every row, in one kernel, under the delay pattern.
//
// Source: Optimized Parler TTS, "Future work" item 2 -- temperature scaling,
// top-k and softmax ran as more than ten kernels with global-memory round
// trips and should be one fused kernel; "Analysis and improvements" --
// sampling without a GPU-CPU synchronisation; the architecture overview --
// nine DAC codebooks, one token each per step, in a delayed pattern.
//
// One CTA per batch row b; inside it one group of 64 threads (two warps) per
// codebook c.  A group
//   1. reads its V logits once into registers, divides by T with IEEE
//      round-to-nearest and maps each float to an order-preserving uint32 key;
//   2. finds the k-th largest key tau by a 4-pass, 8-bit radix select over
//      shared-memory histograms (no sort, no second read of the logits);
//   3. takes every key > tau plus the lowest-index entries equal to tau
//      (their rank in index order comes from warp ballots), so ties go to the
//      lower index exactly;
//   4. draws by Gumbel-max over that set: u from Philox4x32-10 (Salmon et
//      al., SC'11) keyed by the row's seed, counter (i/4, c, step, b), then
//      argmax of x_i - log(-log u_i), equal scores to the lower index;
//   5. optionally writes softmax probabilities over the set.
// Codebooks c with step[b] <= c emit pad_id (delay pattern).  With DR_SAMPLE_ADVANCE, thread 0 increments
// step[b] after a CTA-wide barrier, when every group has read it.
//
// Latency-bound: 39 KB of logits per row at B = 1 is nanoseconds of HBM
// time; the cost is the dependent passes, kept on-chip.
#include <math.h>

#include "dr_device.cuh"
#include "dr_internal.h"

namespace dr {
namespace {

constexpr int kGroup = 64;   // threads per codebook

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

template <int EPT>
__global__ void __launch_bounds__(kMaxCodebooks *kGroup) sample_kernel(const SampleParams p) {
    __shared__ uint32_t s_hist[kMaxCodebooks][256];
    __shared__ uint32_t s_bal[kMaxCodebooks][EPT][2];
    __shared__ uint32_t s_scan[kMaxCodebooks][2];
    __shared__ int s_sel[kMaxCodebooks][2];
    __shared__ float s_rf[kMaxCodebooks][2];
    __shared__ int s_ri[kMaxCodebooks][2];

    const int b = blockIdx.x;
    const int c = threadIdx.x / kGroup;
    const int t = threadIdx.x % kGroup;
    const int wg = t >> 5;
    const int lane = threadIdx.x & 31;
    const int step = p.step[b];
    const uint64_t seed = p.seeds[b];
    const bool active = step > c;   // delay pattern: codebook c is padded while step <= c
    const float *row = p.logits + ((size_t)b * p.C + c) * (size_t)p.ldv;

    // Only the order keys stay in registers; key_value() inverts the map.
    uint32_t key[EPT];
    uint32_t valid = 0;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int i = t + kGroup * j;
        key[j] = 0u;
        if (active && i < p.V) {
            key[j] = order_key(__fdiv_rn(__ldg(row + i), p.temperature));
            valid |= 1u << j;
        }
    }

    // ---- radix select of the top_k-th largest key -------------------------
    uint32_t prefix = 0u, pmask = 0u;
    int kk = p.top_k;
    uint32_t inc = 0u, tot = 0u;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int q = t; q < 256; q += kGroup) s_hist[c][q] = 0u;
        __syncthreads();
        if (active) {
#pragma unroll
            for (int j = 0; j < EPT; ++j)
                if (((valid >> j) & 1u) && (key[j] & pmask) == prefix)
                    atomicAdd(&s_hist[c][(key[j] >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (active) {
            // thread t owns bins 255-4t .. 252-4t, i.e. descending digit order
            const int top = 255 - 4 * t;
            tot = s_hist[c][top] + s_hist[c][top - 1] + s_hist[c][top - 2] + s_hist[c][top - 3];
            inc = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t n = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += n;
            }
            if (lane == 31) s_scan[c][wg] = inc;
        }
        __syncthreads();
        if (active) {
            const uint32_t before = inc - tot + (wg ? s_scan[c][0] : 0u);
            if (before < (uint32_t)kk && (uint32_t)kk <= before + tot) {
                uint32_t acc = before;
                int digit = 255 - 4 * t - 3;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int bin = 255 - 4 * t - q;
                    const uint32_t hq = s_hist[c][bin];
                    if (acc + hq >= (uint32_t)kk) {
                        digit = bin;
                        break;
                    }
                    acc += hq;
                }
                s_sel[c][0] = digit;
                s_sel[c][1] = kk - (int)acc;
            }
        }
        __syncthreads();
        if (active) {
            prefix |= (uint32_t)s_sel[c][0] << shift;
            pmask |= 0xFFu << shift;
            kk = s_sel[c][1];
        }
    }
    const uint32_t tau = prefix;   // the top_k-th largest key; kk entries equal to tau are taken

    // ---- membership: keys above tau, and the first kk ties in index order ----
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ((valid >> j) & 1u) && key[j] == tau);
        if (lane == 0) s_bal[c][j][wg] = bal;
    }
    __syncthreads();
    uint32_t member = 0u;
    if (active) {
        const uint32_t lt_mask = (1u << lane) - 1u;
        int ties_before = 0;
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const uint32_t b0 = s_bal[c][j][0], b1 = s_bal[c][j][1];
            if ((valid >> j) & 1u) {
                if (key[j] > tau) {
                    member |= 1u << j;
                } else if (key[j] == tau) {
                    const int rank = ties_before + (wg ? __popc(b0) : 0) + __popc((wg ? b1 : b0) & lt_mask);
                    if (rank < kk) member |= 1u << j;
                }
            }
            ties_before += __popc(b0) + __popc(b1);
        }
    }

    // ---- Gumbel-max draw over the members ---------------------------------
    float best = -INFINITY;
    int best_i = 0x7FFFFFFF;
    if (active) {
        const uint32_t k0 = (uint32_t)(seed & 0xFFFFFFFFull), k1 = (uint32_t)(seed >> 32);
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            if ((member >> j) & 1u) {
                const int i = t + kGroup * j;
                const uint4 r = philox4x32_10(make_uint4((uint32_t)i >> 2, (uint32_t)c, (uint32_t)step, (uint32_t)b),
                                              k0, k1);
                const uint32_t w = (i & 3) == 0 ? r.x : (i & 3) == 1 ? r.y : (i & 3) == 2 ? r.z : r.w;
                const float u = (float)(2u * (w >> 9) + 1u) * 0x1p-24f;   // exact odd multiple of 2^-24
                const float g = -logf(-logf(u));
                const float s = key_value(key[j]) + g;
                if (better(s, i, best, best_i)) {
                    best = s;
                    best_i = i;
                }
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
            s_rf[c][wg] = best;
            s_ri[c][wg] = best_i;
        }
    }
    __syncthreads();
    if (t == 0) {
        int tok = p.pad_id;
        if (active) {
            tok = better(s_rf[c][1], s_ri[c][1], s_rf[c][0], s_ri[c][0]) ? s_ri[c][1] : s_ri[c][0];
        }
        p.tokens[(size_t)b * p.C + c] = tok;
    }

    // ---- optional softmax over the members --------------------------------
    if (p.probs) {
        float xm = -INFINITY;
#pragma unroll
        for (int j = 0; j < EPT; ++j)
            if ((member >> j) & 1u) xm = fmaxf(xm, key_value(key[j]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) xm = fmaxf(xm, __shfl_xor_sync(0xFFFFFFFFu, xm, o));
        __syncthreads();   // s_rf is reused below
        if (lane == 0) s_rf[c][wg] = xm;
        __syncthreads();
        xm = fmaxf(s_rf[c][0], s_rf[c][1]);
        float z = 0.f;
        if (xm != -INFINITY) {
#pragma unroll
            for (int j = 0; j < EPT; ++j)
                if ((member >> j) & 1u) z += expf(key_value(key[j]) - xm);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
        }
        __syncthreads();
        if (lane == 0) s_rf[c][wg] = z;
        __syncthreads();
        z = s_rf[c][0] + s_rf[c][1];
        float *prow = p.probs + ((size_t)b * p.C + c) * (size_t)p.V;
        const float uniform = 1.0f / (float)p.top_k;
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int i = t + kGroup * j;
            if (i < p.V) {
                float pr = 0.f;
                if ((member >> j) & 1u) pr = (xm == -INFINITY) ? uniform : __fdiv_rn(expf(key_value(key[j]) - xm), z);
                prow[i] = pr;
            }
        }
    }

    if (p.flags & DR_SAMPLE_ADVANCE) {
        __syncthreads();   // every group has read step[b]
        if (threadIdx.x == 0) p.step[b] = step + 1;
    }
}

template <int EPT>
cudaError_t launch_ept(const SampleParams &p, cudaStream_t stream) {
    sample_kernel<EPT><<<(unsigned)p.B, (unsigned)(p.C * kGroup), 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sample(const SampleParams &p, cudaStream_t stream) {
    const int ept = (p.V + kGroup - 1) / kGroup;
    if (ept <= 4) return launch_ept<4>(p, stream);
    if (ept <= 8) return launch_ept<8>(p, stream);
    if (ept <= 17) return launch_ept<17>(p, stream);
    return launch_ept<32>(p, stream);
}

}  // namespace dr
