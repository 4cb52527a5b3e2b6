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
//   CTAs in CTA rank 0's shared memory (distributed shared memory): a grid
//   resident as a whole (small batch) pushes the states and meets at one
//   cluster barrier; a larger grid sends them with remote stores that complete
//   on an mbarrier of rank 0, so that the other CTAs exit at once.
//
// Overlap with the previous kernel on the stream (programmatic dependent
// launch): before waiting for it, each warp prefetches its tiles' K and V rows,
// and the query row, into L2; a grid that is resident as a whole then lets the
// next kernel launch at once, a larger one after its streaming.
//
// Self caches are bf16 or e4m3 (one byte per element with per-tensor k/v
// scales, the KV-format trait below); the description encoder's K/V are bf16.
//
// Roofline: a key costs 256 bytes (64 bf16 of K and of V; 128 for e4m3) and
// ~260 flops, so the kernel is bound by HBM bandwidth; there is no dense
// contraction for the tensor cores (one query row).
#include <cooperative_groups.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "dr_device.cuh"
#include "dr_internal.h"

namespace cg = cooperative_groups;

namespace dr {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kD = kHeadDim;
constexpr int kTile = kBlockKeys;
constexpr int kMaxSplits = 8;       // CTAs per row of the streaming variant: one portable cluster
constexpr int kMaxSplitsWide = 16;  // of the pipelined variant: one non-portable cluster (small batch)

struct SoftmaxPartial {
    float m;         // max of scaled log2-domain scores
    float l;         // sum of 2^(s - m)
    float acc[kD];   // sum of 2^(s - m) * v
};

// Storage formats of a KV cache and the lane layout that streams them.  A key's
// 64 dims are spread over kLanesPerKey lanes, each moving kDims consecutive
// dims: 8 bf16 (16 bytes) or 8 e4m3 codes (8 bytes), so one load instruction
// of a warp reads 4 consecutive key rows (512 or 256 contiguous bytes).
// (Four lanes per key with 16 e4m3 codes each was measured slower: the extra
// merge level and register pressure outweighed the shorter reductions.)
struct Bf16Kv {
    using Chunk = uint4;
    static constexpr int kElemBytes = 2;
    static constexpr int kLanesPerKey = 8;
    static constexpr int kDims = 8;   // dims per lane: [sub*8, sub*8 + 8)
    __device__ static Chunk zero() { return make_uint4(0, 0, 0, 0); }
    __device__ static Chunk load(const uint8_t *p) { return ld_stream16(p); }
    __device__ static void store(uint8_t *p, const Chunk &c) { *reinterpret_cast<uint4 *>(p) = c; }
    __device__ static void unpack(const Chunk &c, float (&f)[kDims]) { unpack8(c, f); }
    // This lane's chunk (dims sub*8 .. sub*8 + 7) of this step's key or value row src_row [D] bf16, in the
    // cache's format.  kWarpNewRow: the whole warp must call new_row; else only the lanes that need it.
    static constexpr bool kWarpNewRow = false;
    __device__ static Chunk new_row(const uint16_t *src_row, float, int, int sub) { return ld_ro16(src_row + sub * 8); }
};
struct Fp8Kv {
    using Chunk = uint2;
    static constexpr int kElemBytes = 1;
    static constexpr int kLanesPerKey = 8;
    static constexpr int kDims = 8;
    __device__ static Chunk zero() { return make_uint2(0, 0); }
    __device__ static Chunk load(const uint8_t *p) { return ld_stream8(p); }
    __device__ static void store(uint8_t *p, const Chunk &c) { *reinterpret_cast<uint2 *>(p) = c; }
    __device__ static void unpack(const Chunk &c, float (&f)[kDims]) { unpack8_e4m3(c, f); }
    // The same for an e4m3 cache: code = e4m3(fl32(x / scale)), round to nearest even, saturating.  The IEEE
    // divisions are spread over the warp -- lane L quantises dims 2L and 2L + 1 -- and each lane gathers its
    // eight codes from lanes 4 sub .. 4 sub + 3 (a lane group alone would do 16 dependent divisions).
    static constexpr bool kWarpNewRow = true;
    __device__ static Chunk new_row(const uint16_t *src_row, float scale, int lane, int sub) {
        const uint32_t two = __ldg(reinterpret_cast<const uint32_t *>(src_row) + lane);
        const uint32_t codes = (uint32_t)__nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(bf16_lo(two), scale), __fdiv_rn(bf16_hi(two), scale)), __NV_SATFINITE, __NV_E4M3);
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = __shfl_sync(0xFFFFFFFFu, codes, 4 * sub + i);
        return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(const_cast<void *>(p));
}

// The address of the same shared-memory variable in CTA rank 0 of the cluster.
__device__ __forceinline__ uint32_t map_rank0(uint32_t local) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(local));
    return r;
}

// Remote stores of one and of two floats into another CTA's shared memory that complete their bytes as
// transactions on an mbarrier of that CTA (st.async: no reply, the sender may exit at once).
__device__ __forceinline__ void st_async_f32(uint32_t remote, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote),
                 "r"(__float_as_uint(v)), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_f32x2(uint32_t remote, float a, float b, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(remote),
                 "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(remote_bar)
                 : "memory");
}

// Wait for phase `parity` of a shared-memory mbarrier whose transactions other CTAs of the cluster complete
// (acquire at cluster scope).  Bounded: false after about 2 s of clock cycles (never expected; the caller
// flags DR_ERRF_TIMEOUT instead of hanging).
__device__ __forceinline__ bool cluster_mbar_wait(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > (4LL << 30)) return false;
    }
}

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

// Lazy rescaling: the running reference m only moves when a score exceeds it
// by more than this (log2 units), so weights stay below 2^8 and the
// accumulator is rescaled rarely instead of on every tile.  Any reference
// gives the same softmax: states carry (m, l, acc) relative to their own m.
constexpr float kRescaleSlack = 8.0f;

// One lane group's online-softmax update with a 16-key tile.  With G = 32 /
// kLanesPerKey lane groups, group grp holds keys t + grp + G*u (u < 16 / G) and
// this lane the kDims dims [sub*kDims, (sub+1)*kDims) of each.  kFull: every key
// of the tile is valid (no masking).
template <typename KV, bool kFull>
__device__ __forceinline__ void consume_tile(const typename KV::Chunk (&kw)[16 * KV::kLanesPerKey / 32],
                                             const typename KV::Chunk (&vw)[16 * KV::kLanesPerKey / 32],
                                             const float (&qf)[KV::kDims], int t, int grp, int key1, float &m,
                                             float &l, float (&acc)[KV::kDims]) {
    constexpr int kLpk = KV::kLanesPerKey, kGroups = 32 / kLpk, kKeys = kTile / kGroups, kDims = KV::kDims;
    float sc[kKeys];
#pragma unroll
    for (int u = 0; u < kKeys; ++u) {
        float kf[kDims];
        KV::unpack(kw[u], kf);
        // even and odd dims in two partial sums: one packed f32x2 FMA per pair of dims
        float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kDims; j += 2)
            d2 = __ffma2_rn(make_float2(qf[j], qf[j + 1]), make_float2(kf[j], kf[j + 1]), d2);
        float d = d2.x + d2.y;
#pragma unroll
        for (int off = 1; off < kLpk; off <<= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, off);
        sc[u] = (kFull || t + grp + kGroups * u < key1) ? d : -INFINITY;
    }
    float mt = sc[0];
#pragma unroll
    for (int u = 1; u < kKeys; ++u) mt = fmaxf(mt, sc[u]);
    if (mt > m + kRescaleSlack) {   // also taken for the first valid key (m = -inf)
        const float corr = fast_exp2(m - mt);
        l *= corr;
#pragma unroll
        for (int j = 0; j < kDims; ++j) acc[j] *= corr;
        m = mt;
    }
    if (m == -INFINITY) return;   // this lane group had no valid key yet
#pragma unroll
    for (int u = 0; u < kKeys; ++u) {
        const float pu = fast_exp2(sc[u] - m);
        l += pu;
        float vf[kDims];
        KV::unpack(vw[u], vf);
#pragma unroll
        for (int j = 0; j < kDims; j += 2) {   // packed f32x2 FMA: two IEEE fmas per instruction
            const float2 a = __ffma2_rn(make_float2(pu, pu), make_float2(vf[j], vf[j + 1]),
                                        make_float2(acc[j], acc[j + 1]));
            acc[j] = a.x;
            acc[j + 1] = a.y;
        }
    }
}

// Which rows an attend_range body serves.
enum RowKind { kSelfRows, kCrossRows, kEitherRows };

// Stream this CTA's tiles [key0, key1) of row (b, h) through the online softmax
// (warp w takes tiles w, w+4, ...).  kKind selects the self rows, the
// description-encoder rows of a fused launch (contiguous bf16), or either at
// run time (one loop body for both when the self cache is bf16 too, which
// keeps the fused kernel's registers down).  kPipelined keeps the next
// tile's loads in flight while the current one is consumed.  Launch
// parameters are read from the parameter space, not copied into registers.
template <typename KV, bool kPaged, bool kPipelined, bool kAppend, RowKind kKind>
__device__ __forceinline__ void attend_range(const AttnParams &p, bool cross_row, int b, int h, int key0, int key1,
                                             int newpos, int warp, int lane, float *s_wm, float *s_wl,
                                             float (*s_wacc)[kD]) {
    using Chunk = typename KV::Chunk;
    constexpr int kLpk = KV::kLanesPerKey, kGroups = 32 / kLpk, kKeys = kTile / kGroups, kDims = KV::kDims;
    constexpr size_t kRowBytes = (size_t)kD * KV::kElemBytes;
    const int grp = lane / kLpk, sub = lane % kLpk;
    const size_t row = (size_t)b * p.H + h;
    const bool cross = kKind == kCrossRows || (kKind == kEitherRows && cross_row);
    const bool paged = kPaged && !cross;
    const uint8_t *kc = reinterpret_cast<const uint8_t *>(cross ? p.xk : p.k);
    const uint8_t *vc = reinterpret_cast<const uint8_t *>(cross ? p.xv : p.v);
    const size_t lane_off = (size_t)sub * kDims * KV::kElemBytes;   // this lane's chunk of a key row

    // this lane's query dims, pre-scaled (the softmax scale in log2 units; times k_scale for e4m3)
    float qf[kDims];
    auto load_query = [&]() {
        const uint16_t *qrow = (cross ? p.xq : p.q) + row * kD + sub * kDims;
        const float qscale = cross ? p.xqscale : p.qscale;
#pragma unroll
        for (int c8 = 0; c8 < kDims / 8; ++c8) {
            float f[8];
            unpack8(ld_ro16(qrow + 8 * c8), f);
#pragma unroll
            for (int j = 0; j < 8; ++j) qf[8 * c8 + j] = f[j] * qscale;
        }
    };
    float m = -INFINITY, l = 0.f;
    float acc[kDims];
#pragma unroll
    for (int j = 0; j < kDims; ++j) acc[j] = 0.f;

    // Issue the loads of tile t (zeros past key1 or for an unmapped block).  With
    // kAppend, the key at newpos is this step's k_new/v_new, converted to the
    // cache format, stored into its cache slot and used from registers.
    auto tile_base = [&](int t, bool &ok) -> size_t {
        ok = true;
        if (paged) {
            const int blk = __ldg(p.table + (size_t)b * p.max_blocks + t / kTile);
            ok = (unsigned)blk < (unsigned)p.num_blocks;
            return ok ? ((size_t)blk * p.H + h) * (size_t)kTile * kRowBytes : 0;
        }
        return (row * (size_t)(cross ? p.xcap : p.cap) + (size_t)t) * kRowBytes;
    };
    auto load_tile = [&](int t, Chunk (&kw)[kKeys], Chunk (&vw)[kKeys]) -> bool {
        bool ok;
        const size_t base = tile_base(t, ok);
        Chunk knew = KV::zero(), vnew = KV::zero();
        if (KV::kWarpNewRow && kAppend && t <= newpos && newpos < t + kTile) {   // the same in the whole warp
            knew = KV::new_row(p.k_new + row * kD, p.k_scale, lane, sub);
            vnew = KV::new_row(p.v_new + row * kD, p.v_scale, lane, sub);
        }
#pragma unroll
        for (int u = 0; u < kKeys; ++u) {
            const int rr = grp + kGroups * u;
            const size_t off = base + (size_t)rr * kRowBytes + lane_off;
            if (ok && t + rr < key1) {
                if (kAppend && t + rr == newpos) {
                    kw[u] = KV::kWarpNewRow ? knew : KV::new_row(p.k_new + row * kD, p.k_scale, lane, sub);
                    vw[u] = KV::kWarpNewRow ? vnew : KV::new_row(p.v_new + row * kD, p.v_scale, lane, sub);
                    KV::store(const_cast<uint8_t *>(kc) + off, kw[u]);
                    KV::store(const_cast<uint8_t *>(vc) + off, vw[u]);
                } else {
                    kw[u] = KV::load(kc + off);
                    vw[u] = KV::load(vc + off);
                }
            } else {
                kw[u] = KV::zero();
                vw[u] = KV::zero();
            }
        }
        if (kAppend && !ok && t <= newpos && newpos < t + kTile && lane == 0) flag_error(p.err, DR_ERRF_POS);
        return ok;
    };
    // Whole tiles away from the appended key need no per-key checks.
    auto full_tile = [&](int t) -> bool {
        return t + kTile <= key1 && !(kAppend && newpos >= t && newpos < t + kTile);
    };
    auto load_full = [&](int t, Chunk (&kw)[kKeys], Chunk (&vw)[kKeys]) -> bool {
        bool ok;
        const size_t base = tile_base(t, ok);
        if (ok) {
            const uint8_t *kp = kc + base + (size_t)grp * kRowBytes + lane_off;
            const uint8_t *vp = vc + base + (size_t)grp * kRowBytes + lane_off;
#pragma unroll
            for (int u = 0; u < kKeys; ++u) {
                kw[u] = KV::load(kp + (size_t)kGroups * u * kRowBytes);
                vw[u] = KV::load(vp + (size_t)kGroups * u * kRowBytes);
            }
        }
        return ok;
    };

    if constexpr (kPipelined) {
        Chunk kw[kKeys], vw[kKeys];
        int t = key0 + warp * kTile;
        bool full = t < key1 && full_tile(t);
        bool ok = t < key1 ? (full ? load_full(t, kw, vw) : load_tile(t, kw, vw)) : true;
        // The first tile's loads go out before the query is waited for (measured: batch 1, 24 layers of
        // 1024 + 1024 keys, 4.02 -> 3.90 us per layer).
        load_query();
        for (; t < key1; t += kWarps * kTile) {
            Chunk nk[kKeys] = {}, nv[kKeys] = {};
            const int tn = t + kWarps * kTile;
            const bool nfull = tn < key1 && full_tile(tn);
            const bool nok = tn < key1 ? (nfull ? load_full(tn, nk, nv) : load_tile(tn, nk, nv)) : true;
            if (!ok) {
                if (lane == 0) flag_error(p.err, DR_ERRF_BLOCK_ID);   // warp-uniform: the tile is skipped
            } else if (full) {
                consume_tile<KV, true>(kw, vw, qf, t, grp, key1, m, l, acc);
            } else {
                consume_tile<KV, false>(kw, vw, qf, t, grp, key1, m, l, acc);
            }
#pragma unroll
            for (int u = 0; u < kKeys; ++u) {
                kw[u] = nk[u];
                vw[u] = nv[u];
            }
            ok = nok;
            full = nfull;
        }
    } else {
        load_query();
        for (int t = key0 + warp * kTile; t < key1; t += kWarps * kTile) {
            Chunk kw[kKeys], vw[kKeys];
            if (full_tile(t)) {
                if (load_full(t, kw, vw)) consume_tile<KV, true>(kw, vw, qf, t, grp, key1, m, l, acc);
                else if (lane == 0) flag_error(p.err, DR_ERRF_BLOCK_ID);
            } else {
                if (load_tile(t, kw, vw)) consume_tile<KV, false>(kw, vw, qf, t, grp, key1, m, l, acc);
                else if (lane == 0) flag_error(p.err, DR_ERRF_BLOCK_ID);
            }
        }
    }

    // Lanes sub, sub + kLpk, ... hold the same dims for different keys: merge them,
    // then lane group 0 publishes the warp's partial state.
#pragma unroll
    for (int off = kLpk; off < 32; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
        const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, off);
        float a2[kDims];
#pragma unroll
        for (int j = 0; j < kDims; ++j) a2[j] = __shfl_xor_sync(0xFFFFFFFFu, acc[j], off);
        merge_state(m, l, acc, m2, l2, a2);
    }
    if (grp == 0) {
        if (sub == 0) {
            s_wm[warp] = m;
            s_wl[warp] = l;
        }
#pragma unroll
        for (int j = 0; j < kDims; ++j) s_wacc[warp][sub * kDims + j] = acc[j];
    }
}

// L2 prefetch of the K and V rows of warp `warp`'s first kPrefetchTiles tiles
// (the pipelined variant, whose whole grid is resident at once, takes up to 64,
// its whole range for rows of up to 4096 keys per CTA; the streaming variant
// its first two), issued before the kernel waits for its predecessor on the
// stream.  Only a hint: the
// length and the block table may still be changing (the predecessor may write
// them), so they are read with relaxed loads, every address is checked against
// the row's capacity or the block pool, and the real loads after the wait use
// the final values.  L2 is coherent with the predecessor's writes.
template <typename KV, bool kPaged, int kPrefetchTiles>
__device__ __forceinline__ void prefetch_tiles(const AttnParams &p, bool cross, int b, int h, int split,
                                                     int nsplit, int warp) {
    constexpr uint32_t kRowBytes = (uint32_t)kD * KV::kElemBytes;
    const int cap = cross ? p.xcap : p.cap;
    int L = ld_relaxed((cross ? p.xlens : p.lens) + b);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int ntiles = (L + kTile - 1) / kTile;
    const int per = (ntiles + nsplit - 1) / nsplit;
    const int key0 = min(split * per, ntiles) * kTile;
    const int key1 = min(key0 + per * kTile, L);
    const uint8_t *kc = reinterpret_cast<const uint8_t *>(cross ? p.xk : p.k);
    const uint8_t *vc = reinterpret_cast<const uint8_t *>(cross ? p.xv : p.v);
    for (int i = 0; i < kPrefetchTiles; ++i) {
        const int t = key0 + (warp + i * kWarps) * kTile;
        if (t >= key1) break;
        size_t base;
        uint32_t bytes;
        if (kPaged) {
            const int blk = ld_relaxed(p.table + (size_t)b * p.max_blocks + t / kTile);
            if ((unsigned)blk >= (unsigned)p.num_blocks) break;
            base = ((size_t)blk * p.H + h) * kTile * kRowBytes;
            bytes = kTile * kRowBytes;
        } else {
            base = (((size_t)b * p.H + h) * (size_t)cap + (size_t)t) * kRowBytes;
            bytes = (uint32_t)min(kTile, cap - t) * kRowBytes;
        }
        prefetch_l2(kc + base, bytes);
        prefetch_l2(vc + base, bytes);
    }
}

// kPipelined: each warp keeps the next tile's loads in flight while it
// computes the current one (twice the bytes in flight per warp, at ~110
// registers instead of 64-72).  Chosen when the whole grid is resident at
// once, i.e. when occupancy is not what limits the bytes in flight.  Both
// variants perform the same arithmetic in the same order.
//
// Occupancy of the streaming variant: 8 CTAs per SM (64 registers), except
// for the fused bf16 layer kernel, which at 64 registers spilled 40-48 bytes
// per thread; bounded at 6 CTAs per SM it takes 72 registers, so 7 CTAs fit
// per SM, and runs faster (batch 32 ragged, paged: 34.8 -> 33.4 us per layer;
// batch 128: 186.0 -> 185.4 us).
template <typename KV, bool kFused>
constexpr int streaming_min_ctas() { return kFused && std::is_same<KV, Bf16Kv>::value ? 6 : 8; }

template <typename KV, bool kPaged, bool kPipelined, bool kFused>
__global__ void __launch_bounds__(kThreads, kPipelined ? 4 : streaming_min_ctas<KV, kFused>())
    decode_attn_kernel(const AttnParams p) {
    __shared__ float s_wm[kWarps], s_wl[kWarps];
    __shared__ float s_wacc[kWarps][kD];
    // rank 0 of a cluster collects the CTAs' states here
    __shared__ alignas(16) SoftmaxPartial s_parts[kPipelined ? kMaxSplitsWide : kMaxSplits];
    __shared__ alignas(8) uint64_t s_parts_bar;   // streaming variant, rank 0: the other CTAs' states have landed

    const int h = blockIdx.y;
    // Fused launches carry the B self rows along z, then the cross rows: split
    // like the self rows (z = B + b), or packed one row per CTA (row b =
    // (z - B) * gridDim.x + x) when a cross row is short enough for one CTA.
    const bool cross = kFused && p.xq != nullptr && (int)blockIdx.z >= p.B;
    const bool packed = cross && p.xpacked;
    const int split = packed ? 0 : (int)blockIdx.x;
    const int nsplit = packed ? 1 : (int)gridDim.x;
    int b = !cross ? (int)blockIdx.z
                   : packed ? ((int)blockIdx.z - p.B) * (int)gridDim.x + (int)blockIdx.x : (int)blockIdx.z - p.B;
    if (b >= p.B) return;   // tail of the packed region (no cluster barrier is reached there)
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // A split row's CTAs later write into CTA rank 0's shared memory; that needs every CTA of the cluster
    // to have started.  Announce it now, and wait for the others just before the write.  In the streaming
    // variant rank 0 first sets up the mbarrier on which the other CTAs' states will land (expecting their
    // bytes), and its arrive releases that set-up to them; otherwise the arrive orders nothing.
    if (nsplit > 1) {
        if (!kPipelined && split == 0) {
            if (threadIdx.x == 0) {
                asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&s_parts_bar)) : "memory");
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&s_parts_bar)),
                             "r"((uint32_t)((nsplit - 1) * (kD + 2) * sizeof(float)))
                             : "memory");
                asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            }
            asm volatile("barrier.cluster.arrive.aligned;" ::: "memory");
        } else {
            asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
        }
    }

    // While the previous kernel on the stream drains, warm L2 with this warp's tiles; then wait for it.
    if (lane == 0) {
        if (cross) prefetch_tiles<Bf16Kv, false, kPipelined ? 64 : 2>(p, true, b, h, split, nsplit, warp);
        else prefetch_tiles<KV, kPaged, kPipelined ? 64 : 2>(p, false, b, h, split, nsplit, warp);
        // The query row, and this step's key and value rows, 128 bytes each: the first dependent loads after
        // the wait (batch 1, 24 layers of 1024 + 1024 keys in turn: 4.34 -> 4.02 us per layer).
        if (warp == 0) {
            const size_t qrow = ((size_t)b * p.H + h) * kD;
            prefetch_l2((cross ? p.xq : p.q) + qrow, kD * 2);
            if (kFused && !cross && p.k_new != nullptr) {
                prefetch_l2(p.k_new + qrow, kD * 2);
                prefetch_l2(p.v_new + qrow, kD * 2);
            }
        }
    }
    pdl_wait();
    // The row index taken through a warp shuffle (the same value): measured, the compiler then schedules the
    // row's address arithmetic so that the standalone bf16 kernel on a paged cache streams 4-13% faster
    // (batch 32: 32.8 -> 28.3 us); the other variants time the same either way.
    b = __shfl_sync(0xFFFFFFFFu, b, 0);
    // The next kernel on the stream may start launching: at once when this grid is resident as a whole
    // (its CTAs take free slots and prefetch), else once the streaming is done (below), so that they do
    // not take the slots of this grid's later waves.
    if (kPipelined) pdl_trigger();

    const size_t row = (size_t)b * p.H + h;
    const int cap = cross ? p.xcap : p.cap;
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

    if constexpr (kFused && std::is_same<KV, Bf16Kv>::value) {
        attend_range<KV, kPaged, kPipelined, true, kEitherRows>(p, cross, b, h, key0, key1, newpos, warp, lane, s_wm,
                                                                 s_wl, s_wacc);
    } else if constexpr (kFused) {
        if (cross)
            attend_range<Bf16Kv, false, kPipelined, false, kCrossRows>(p, true, b, h, key0, key1, -1, warp, lane, s_wm,
                                                                      s_wl, s_wacc);
        else
            attend_range<KV, kPaged, kPipelined, true, kSelfRows>(p, false, b, h, key0, key1, newpos, warp, lane, s_wm,
                                                                 s_wl, s_wacc);
    } else {
        attend_range<KV, kPaged, kPipelined, false, kSelfRows>(p, false, b, h, key0, key1, -1, warp, lane, s_wm, s_wl,
                                                              s_wacc);
    }
    if (!kPipelined) pdl_trigger();
    // an e4m3 value is code * v_scale: the kernel accumulates codes and scales the result
    const float out_scale = cross ? 1.0f : p.out_scale;

    __syncthreads();
    void *outp = cross ? p.xout : p.out;
    const int d = threadIdx.x;   // threads d < kD each own output dim d
    const size_t oidx = row * kD + d;
    auto store = [&](float o) {
        if (p.out_f32) reinterpret_cast<float *>(outp)[oidx] = o;
        else reinterpret_cast<uint16_t *>(outp)[oidx] = f32_to_bf16_rn(o);
    };
    // CTA merge of the warps' states (m and l come out the same in every thread)
    float mm = -INFINITY, ls = 0.f, o = 0.f;
    if (d < kD) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, s_wm[w]);
        if (mm != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float wt = exp2f(s_wm[w] - mm);
                ls += wt * s_wl[w];
                o += wt * s_wacc[w][d];
            }
        }
    }
    if (nsplit == 1) {   // the same for every CTA of a cluster
        if (d < kD) store(ls > 0.f ? o / ls * out_scale : 0.f);
        return;
    }

    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every CTA of the cluster has started
    if constexpr (!kPipelined) {
        // Cluster merge of the streaming variant: every other CTA sends its state to slot `split` of rank
        // 0's shared memory with remote stores that complete bytes on rank 0's mbarrier, and exits; rank 0
        // waits for those bytes and merges, its own state first.  The CTAs that finish early free their SM
        // at once (batch 32: fused layer 35.7 -> 34.8 us; batch 128: 187.3 -> 186.0 us).
        if (split != 0) {
            if (split == 1 && (long long)row == p.stall_row) return;   // test hook: this state never arrives
            if (d < kD) {
                const uint32_t bar = map_rank0(smem_addr(&s_parts_bar));
                SoftmaxPartial *slot = &s_parts[split];
                st_async_f32(map_rank0(smem_addr(&slot->acc[d])), o, bar);
                if (d == 0) st_async_f32x2(map_rank0(smem_addr(&slot->m)), mm, ls, bar);
            }
            return;
        }
        if (d >= kD) return;
        if (!cluster_mbar_wait(&s_parts_bar, 0)) {
            if (d == 0) flag_error(p.err, DR_ERRF_TIMEOUT);
            return;
        }
        float m0 = mm;
        for (int r = 1; r < nsplit; ++r) m0 = fmaxf(m0, s_parts[r].m);
        float l0 = 0.f, o0 = 0.f;
        if (m0 != -INFINITY) {
            const float w0 = exp2f(mm - m0);
            l0 = w0 * ls;
            o0 = w0 * o;
            for (int r = 1; r < nsplit; ++r) {
                const float wt = exp2f(s_parts[r].m - m0);
                l0 += wt * s_parts[r].l;
                o0 += wt * s_parts[r].acc[d];
            }
        }
        store(l0 > 0.f ? o0 / l0 * out_scale : 0.f);
        return;
    }

    // Cluster merge of the pipelined variant (a grid resident as a whole): every CTA pushes its state into
    // slot `split` of rank 0's shared memory, then one cluster barrier, which every thread of the cluster
    // reaches (release / acquire), makes all of them visible to rank 0.  Nothing reads another CTA's shared
    // memory after the barrier, so the other CTAs may exit at once.  (The remote-store merge above is slower
    // here: batch 1, 24 layers of 1024 + 1024 keys, 3.86 -> 4.01 us per layer.)
    cg::cluster_group cluster = cg::this_cluster();
    if (d < kD) {
        SoftmaxPartial *slot = cluster.map_shared_rank(&s_parts[split], 0);
        slot->acc[d] = o;
        if (d == 0) {
            slot->m = mm;
            slot->l = ls;
        }
    }
    cluster.sync();
    if (split != 0 || d >= kD) return;
    mm = -INFINITY;
    for (int r = 0; r < nsplit; ++r) mm = fmaxf(mm, s_parts[r].m);
    ls = 0.f;
    o = 0.f;
    if (mm != -INFINITY) {
        for (int r = 0; r < nsplit; ++r) {
            const float wt = exp2f(s_parts[r].m - mm);
            ls += wt * s_parts[r].l;
            o += wt * s_parts[r].acc[d];
        }
    }
    store(ls > 0.f ? o / ls * out_scale : 0.f);
}

template <typename KV, bool kPaged, bool kPipelined, bool kFused>
cudaError_t launch_variant(const AttnParams &p, int splits, cudaStream_t stream) {
    unsigned zrows = (unsigned)p.B;
    if (kFused && p.xq) zrows += p.xpacked ? (unsigned)((p.B + splits - 1) / splits) : (unsigned)p.B;
    auto kern = decode_attn_kernel<KV, kPaged, kPipelined, kFused>;
    // rank 0 has one state slot per CTA of its cluster
    if (splits < 1 || splits > (kPipelined ? kMaxSplitsWide : kMaxSplits)) return cudaErrorInvalidValue;
    if (splits > 8) {   // clusters of more than 8 CTAs are non-portable: allowed per kernel
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(kern, dim3((unsigned)splits, (unsigned)p.H, zrows), dim3(kThreads), 0, stream,
                         (unsigned)splits, p);
}

// CTAs of the pipelined kernel that fit on one SM at once (up to 112 registers x 128 threads).
constexpr int kPipelinedCtasPerSm = 4;

template <typename KV, bool kFused>
cudaError_t launch_layout(const AttnParams &p, bool paged, int splits, cudaStream_t stream) {
    long long ctas = (long long)splits * p.H * p.B;
    if (kFused && p.xq) ctas += (long long)p.H * (p.xpacked ? p.B : (long long)splits * p.B);
    const bool pipelined = ctas <= (long long)kPipelinedCtasPerSm * current_device_sms();
    if (!pipelined && splits > kMaxSplits) return cudaErrorInvalidValue;   // the plan keeps wide clusters resident
    if (paged)
        return pipelined ? launch_variant<KV, true, true, kFused>(p, splits, stream)
                         : launch_variant<KV, true, false, kFused>(p, splits, stream);
    return pipelined ? launch_variant<KV, false, true, kFused>(p, splits, stream)
                     : launch_variant<KV, false, false, kFused>(p, splits, stream);
}

}  // namespace

cudaError_t launch_decode_attn(const AttnParams &p, bool paged, int splits, cudaStream_t stream) {
    const bool fused = p.k_new != nullptr || p.xq != nullptr;
    if (p.kv_fp8)
        return fused ? launch_layout<Fp8Kv, true>(p, paged, splits, stream)
                     : launch_layout<Fp8Kv, false>(p, paged, splits, stream);
    return fused ? launch_layout<Bf16Kv, true>(p, paged, splits, stream)
                 : launch_layout<Bf16Kv, false>(p, paged, splits, stream);
}

}  // namespace dr
