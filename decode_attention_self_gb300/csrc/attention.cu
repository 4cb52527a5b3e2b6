// Single-query decode attention over the valid part of a KV cache.
//
// Source: Optimized Parler TTS, "Analysis and improvements" -- the attention
// kernel of a static-cache decoder must not move the whole preallocated cache
// (~95 us) when only the valid length is needed (~13 us eager); "Future work"
// item 1 -- a paged cache.  Cross-attention over the description encoder's
// keys and values is the same computation on a contiguous [B][H][Lc_max][D]
// tensor.
//
// Work decomposition (one launch, no workspace, no second kernel):
//   grid = (S, H, B), one thread-block cluster of S CTAs per (b, h) row.
//   The row's valid keys are cut into 16-key tiles (a tile is one paged
//   block, or 2 KiB of K plus 2 KiB of V of a contiguous row); CTA s of the
//   cluster takes an equal run of tiles, so a long row is spread over S SMs
//   and every CTA of a cluster finishes at about the same time.
//   Inside a CTA, warp w takes tiles w, w+4, ...; inside a warp, lane
//   (g, e) = (lane / 8, lane % 8) owns dims 8e..8e+7 of keys g, g+4, g+8,
//   g+12 of the tile, so each 16-byte load instruction of the warp reads
//   512 contiguous bytes.  Each lane group keeps an fp32 online-softmax state
//   (running max m, running sum l, acc[8]); states are merged with warp
//   shuffles, then across warps in shared memory, then across the cluster's
//   CTAs through distributed shared memory by CTA rank 0.
//
// Roofline: a key costs 256 bytes (64 bf16 of K and of V) and ~260 flops, so
// the kernel is bound by HBM bandwidth; there is no dense contraction for the
// tensor cores (one query row).
#include <cooperative_groups.h>

#include "dr_device.cuh"
#include "dr_internal.h"

namespace cg = cooperative_groups;

namespace dr {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kD = kHeadDim;
constexpr int kTile = kBlockKeys;

struct SoftmaxPartial {
    float m;         // max of scaled log2-domain scores
    float l;         // sum of 2^(s - m)
    float acc[kD];   // sum of 2^(s - m) * v
};

// Merge (m2, l2, a2) into (m, l, a); an empty state has m = -inf, l = 0, a = 0.
template <int N>
__device__ __forceinline__ void merge_state(float &m, float &l, float (&a)[N], float m2, float l2,
                                            const float (&a2)[N]) {
    const float mm = fmaxf(m, m2);
    if (mm == -INFINITY) return;
    const float w1 = exp2f(m - mm);
    const float w2 = exp2f(m2 - mm);
    l = l * w1 + l2 * w2;
#pragma unroll
    for (int j = 0; j < N; ++j) a[j] = a[j] * w1 + a2[j] * w2;
    m = mm;
}

// One lane group's online-softmax update with a 16-key tile: this lane holds
// dims 8*sub..8*sub+7 of keys t+grp, t+grp+4, t+grp+8, t+grp+12.
__device__ __forceinline__ void consume_tile(const uint4 (&kw)[4], const uint4 (&vw)[4], const float (&qf)[8], int t,
                                             int grp, int key1, float &m, float &l, float (&acc)[8]) {
    float sc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float kf[8];
        unpack8(kw[u], kf);
        float d = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) d = fmaf(qf[j], kf[j], d);
        d += __shfl_xor_sync(0xFFFFFFFFu, d, 1);
        d += __shfl_xor_sync(0xFFFFFFFFu, d, 2);
        d += __shfl_xor_sync(0xFFFFFFFFu, d, 4);
        sc[u] = (t + grp + 4 * u < key1) ? d : -INFINITY;
    }
    const float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    const float mn = fmaxf(m, mt);
    if (mn == -INFINITY) return;   // this lane group had no valid key yet
    const float corr = exp2f(m - mn);
    l *= corr;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] *= corr;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float pu = exp2f(sc[u] - mn);
        l += pu;
        float vf[8];
        unpack8(vw[u], vf);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = fmaf(pu, vf[j], acc[j]);
    }
    m = mn;
}

// kPipelined: each warp keeps the next tile's loads in flight while it
// computes the current one (twice the bytes in flight per warp, at ~100
// registers instead of 64).  Chosen when the whole grid is resident at once,
// i.e. when occupancy is not what limits the bytes in flight.  Both variants
// perform the same arithmetic in the same order.
template <bool kPaged, bool kPipelined, bool kFused>
__global__ void __launch_bounds__(kThreads, kPipelined ? 4 : 8) decode_attn_kernel(const AttnParams p) {
    __shared__ float s_wm[kWarps], s_wl[kWarps];
    __shared__ float s_wacc[kWarps][kD];
    __shared__ SoftmaxPartial s_part;

    const int h = blockIdx.y;
    // Fused launches carry the B self rows along z, then the cross rows: split
    // like the self rows (z = B + b), or packed one row per CTA (row b =
    // (z - B) * gridDim.x + x) when a cross row is short enough for one CTA.
    const bool cross = kFused && p.xq != nullptr && (int)blockIdx.z >= p.B;
    const bool packed = cross && p.xpacked;
    const int split = packed ? 0 : (int)blockIdx.x;
    const int nsplit = packed ? 1 : (int)gridDim.x;
    const int b = !cross ? (int)blockIdx.z
                         : packed ? ((int)blockIdx.z - p.B) * (int)gridDim.x + (int)blockIdx.x : (int)blockIdx.z - p.B;
    if (b >= p.B) return;   // tail of the packed region (no cluster barrier is reached there)
    const bool paged = kPaged && !cross;
    const uint16_t *qsrc = cross ? p.xq : p.q;
    const uint16_t *kcache = cross ? p.xk : p.k;
    const uint16_t *vcache = cross ? p.xv : p.v;
    const int cap = cross ? p.xcap : p.cap;
    void *outp = cross ? p.xout : p.out;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int grp = lane >> 3;   // which key of each group of 4
    const int sub = lane & 7;    // which 8 dims

    int L = __ldg((cross ? p.xlens : p.lens) + b);
    // Fused append: this step's key goes to slot L-1 (only for a valid length).
    int newpos = -1;
    if (kFused && !cross && p.k_new != nullptr && L >= 1 && L <= cap) newpos = L - 1;
    if (L < 1 || L > cap) {
        if (split == 0 && h == 0 && threadIdx.x == 0) {
            flag_error(p.err, DR_ERRF_SEQ_LEN);
            if (kFused && !cross && p.k_new != nullptr) flag_error(p.err, DR_ERRF_POS);
        }
        L = L < 0 ? 0 : (L > cap ? cap : L);
    }
    const int ntiles = (L + kTile - 1) / kTile;
    const int per = (ntiles + nsplit - 1) / nsplit;
    const int key0 = min(split * per, ntiles) * kTile;
    const int key1 = min(key0 + per * kTile, L);

    const size_t row = (size_t)b * p.H + h;
    float qf[8];
    unpack8(ld_ro16(qsrc + row * kD + sub * 8), qf);
#pragma unroll
    for (int j = 0; j < 8; ++j) qf[j] *= p.qscale;

    float m = -INFINITY, l = 0.f;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;

    // Issue the 16-byte loads of tile t (zeros past key1 or for an unmapped block).
    // Fused: the key at newpos is this step's k_new/v_new, taken from the inputs
    // and stored into its cache slot by the same lanes.
    auto load_tile = [&](int t, uint4 (&kw)[4], uint4 (&vw)[4]) -> bool {
        const uint16_t *kt;
        const uint16_t *vt;
        bool ok = true;
        if (paged) {
            const int blk = __ldg(p.table + (size_t)b * p.max_blocks + t / kTile);
            ok = (unsigned)blk < (unsigned)p.num_blocks;
            const size_t off = ok ? ((size_t)blk * p.H + h) * (size_t)(kTile * kD) : 0;
            kt = kcache + off;
            vt = vcache + off;
        } else {
            const size_t off = (row * (size_t)cap + (size_t)t) * kD;
            kt = kcache + off;
            vt = vcache + off;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = grp + 4 * u;
            if (ok && t + r < key1) {
                if (kFused && t + r == newpos) {
                    kw[u] = ld_ro16(p.k_new + row * kD + sub * 8);
                    vw[u] = ld_ro16(p.v_new + row * kD + sub * 8);
                    *reinterpret_cast<uint4 *>(const_cast<uint16_t *>(kt) + r * kD + sub * 8) = kw[u];
                    *reinterpret_cast<uint4 *>(const_cast<uint16_t *>(vt) + r * kD + sub * 8) = vw[u];
                } else {
                    kw[u] = ld_stream16(kt + r * kD + sub * 8);
                    vw[u] = ld_stream16(vt + r * kD + sub * 8);
                }
            } else {
                kw[u] = make_uint4(0, 0, 0, 0);
                vw[u] = make_uint4(0, 0, 0, 0);
            }
        }
        if (kFused && !ok && t <= newpos && newpos < t + kTile && lane == 0) flag_error(p.err, DR_ERRF_POS);
        return ok;
    };

    if constexpr (kPipelined) {
        uint4 kw[4], vw[4];
        int t = key0 + warp * kTile;
        bool ok = t < key1 ? load_tile(t, kw, vw) : true;
        for (; t < key1; t += kWarps * kTile) {
            uint4 nk[4] = {}, nv[4] = {};
            const int tn = t + kWarps * kTile;
            const bool nok = tn < key1 ? load_tile(tn, nk, nv) : true;
            if (ok) consume_tile(kw, vw, qf, t, grp, key1, m, l, acc);
            else if (lane == 0) flag_error(p.err, DR_ERRF_BLOCK_ID);   // warp-uniform: the tile is skipped
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                kw[u] = nk[u];
                vw[u] = nv[u];
            }
            ok = nok;
        }
    } else {
        for (int t = key0 + warp * kTile; t < key1; t += kWarps * kTile) {
            uint4 kw[4], vw[4];
            if (load_tile(t, kw, vw)) consume_tile(kw, vw, qf, t, grp, key1, m, l, acc);
            else if (lane == 0) flag_error(p.err, DR_ERRF_BLOCK_ID);   // warp-uniform: the tile is skipped
        }
    }

    // Lanes sub, sub+8, sub+16, sub+24 hold the same dims for different keys.
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
        const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, off);
        float a2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a2[j] = __shfl_xor_sync(0xFFFFFFFFu, acc[j], off);
        merge_state(m, l, acc, m2, l2, a2);
    }
    if (grp == 0) {
        if (sub == 0) {
            s_wm[warp] = m;
            s_wl[warp] = l;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) s_wacc[warp][sub * 8 + j] = acc[j];
    }
    __syncthreads();
    if (threadIdx.x < kD) {
        const int d = threadIdx.x;
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, s_wm[w]);
        float ls = 0.f, o = 0.f;
        if (mm != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float wt = exp2f(s_wm[w] - mm);
                ls += wt * s_wl[w];
                o += wt * s_wacc[w][d];
            }
        }
        s_part.acc[d] = o;
        if (d == 0) {
            s_part.m = mm;
            s_part.l = ls;
        }
    }

    float *out_f = reinterpret_cast<float *>(outp) + row * kD;
    uint16_t *out_h = reinterpret_cast<uint16_t *>(outp) + row * kD;

    if (nsplit == 1) {
        __syncthreads();
        if (threadIdx.x < kD) {
            const int d = threadIdx.x;
            const float o = s_part.l > 0.f ? s_part.acc[d] / s_part.l : 0.f;
            if (p.out_f32) out_f[d] = o;
            else out_h[d] = f32_to_bf16_rn(o);
        }
        return;
    }

    // Cluster-wide merge of the S partial states (CTA rank == split).
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();   // every CTA's s_part is complete and visible
    if (split == 0 && threadIdx.x < kD) {
        const int d = threadIdx.x;
        float mm = -INFINITY;
        for (int r = 0; r < nsplit; ++r) {
            const SoftmaxPartial *pr = cluster.map_shared_rank(&s_part, r);
            mm = fmaxf(mm, pr->m);
        }
        float ls = 0.f, o = 0.f;
        if (mm != -INFINITY) {
            for (int r = 0; r < nsplit; ++r) {
                const SoftmaxPartial *pr = cluster.map_shared_rank(&s_part, r);
                const float wt = exp2f(pr->m - mm);
                ls += wt * pr->l;
                o += wt * pr->acc[d];
            }
        }
        o = ls > 0.f ? o / ls : 0.f;
        if (p.out_f32) out_f[d] = o;
        else out_h[d] = f32_to_bf16_rn(o);
    }
    cluster.sync();   // keep every CTA's shared memory alive until rank 0 has read it
}

template <bool kPaged, bool kPipelined, bool kFused>
cudaError_t launch_variant(const AttnParams &p, int splits, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    unsigned zrows = (unsigned)p.B;
    if (kFused && p.xq) zrows += p.xpacked ? (unsigned)((p.B + splits - 1) / splits) : (unsigned)p.B;
    cfg.gridDim = dim3((unsigned)splits, (unsigned)p.H, zrows);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 1 : 0;
    auto kern = decode_attn_kernel<kPaged, kPipelined, kFused>;
    if (splits > 8) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// CTAs of the pipelined kernel that fit on one SM at once (up to 112 registers x 128 threads).
constexpr int kPipelinedCtasPerSm = 4;

template <bool kFused>
cudaError_t launch_layout(const AttnParams &p, bool paged, int splits, cudaStream_t stream) {
    long long ctas = (long long)splits * p.H * p.B;
    if (kFused && p.xq) ctas += (long long)p.H * (p.xpacked ? p.B : (long long)splits * p.B);
    const bool pipelined = ctas <= (long long)kPipelinedCtasPerSm * current_device_sms();
    if (paged)
        return pipelined ? launch_variant<true, true, kFused>(p, splits, stream)
                         : launch_variant<true, false, kFused>(p, splits, stream);
    return pipelined ? launch_variant<false, true, kFused>(p, splits, stream)
                     : launch_variant<false, false, kFused>(p, splits, stream);
}

}  // namespace

cudaError_t launch_decode_attn(const AttnParams &p, bool paged, int splits, cudaStream_t stream) {
    const bool fused = p.k_new != nullptr || p.xq != nullptr;
    return fused ? launch_layout<true>(p, paged, splits, stream) : launch_layout<false>(p, paged, splits, stream);
}

}  // namespace dr
