// Merged LM head on the 5th-generation tensor cores, for decode batches large
// enough to make the head a dense contraction (Optimized Parler TTS, "Analysis
// and improvements", other optimizations items 1-2: the head on the last
// position only, the nine codebook heads merged into one weight matrix).
//
//   logits^T[n, b] = sum_k W[n, k] * hidden[b, k]       (n = c*V + v)
//
// One CTA computes a 128-row slab of W against a tile of up to 128 batch rows
// over its share of K: the weight slab is the MMA's M = 128 operand A, the batch
// tile its N operand B, both K-major bf16 in shared memory with the 128-byte
// swizzle, and the fp32 accumulator lives in tensor memory (128 lanes x N
// columns).
//   warp 0, lane 0 : TMA producer -- cp.async.bulk.tensor.2d loads of 64-wide K
//                    chunks of A and B into a ring of up to 4 stages, completion counted
//                    on the stage's "full" mbarrier;
//   warp 1, lane 0 : MMA issuer -- four tcgen05.mma (K = 16 each) per chunk,
//                    tcgen05.commit to the stage's "empty" mbarrier, and a last
//                    commit to "done";
//   all 4 warps    : epilogue -- warp w reads TMEM lanes 32w..32w+31 with
//                    tcgen05.ld and writes fp32 logits into the sampler layout.
// Split K (batch tiles of up to 32 rows): when the weight slabs alone are fewer
// than the SMs, K is cut in two and the two CTAs of a cluster each accumulate
// one half.  Each stages the half of its partial accumulator that the other
// owns in its (then idle) stage ring; after a cluster barrier each CTA adds the
// two partials for its own batch columns, rank 0's first, reading the other's
// through distributed shared memory.  Whenever the grid has more CTAs than the
// GPU has SMs, the ring is cut to at most 112 KB so that two CTAs share an SM
// and the grid runs as one wave.
// Every mbarrier wait is bounded: a wait that runs out sets DR_ERRF_TIMEOUT
// and the CTA skips the rest of its work (a correct launch never gets there);
// both cluster barriers are reached on every path.
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "dr_device.cuh"
#include "dr_internal.h"

namespace dr {
namespace {

constexpr int kThreads = 128;
constexpr int kTileN = 128;          // W rows per CTA (MMA M)
constexpr int kChunkK = 64;          // K elements per stage: one 128-byte swizzled row
constexpr int kMaxStages = 4;
constexpr int kTwoPerSmBytes = 110 * 1024;   // stage ring small enough for two CTAs per SM (with alignment)
constexpr int kMaxBatchTile = 128;   // MMA N (a multiple of 16); larger batches take more tiles
constexpr int kMaxSplitK = 2;
constexpr long long kWaitLimit = 4LL << 30;   // clock cycles (about 2 s)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitLimit) return false;
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row
// groups 1024 bytes apart (start address, leading / stride byte offsets >> 4,
// descriptor version 1, swizzle mode 2 = 128B).
__device__ __forceinline__ uint64_t smem_desc(const void *p) {
    const uint64_t addr = smem_u32(p);
    return ((addr & 0x3FFFFull) >> 4) | (1ull << 16) | ((1024ull >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// tcgen05.ld of 32 (or 8) consecutive fp32 accumulator columns starting at
// column c0, TMEM lanes 32w .. 32w+31 (one row per thread of warp w).
__device__ __forceinline__ void tmem_ld32(uint32_t tmem, int warp, int c0, uint32_t (&r)[32]) {
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t tmem, int warp, int c0, uint32_t (&r)[8]) {
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct TcParams {
    float *logits;     // [B][C][ldv]
    int32_t B, K, C, V, ldv, btile, tmem_cols;
    int32_t ksplit;    // CTAs (one cluster along x) that share a weight slab's K range
    int32_t stages;    // depth of the stage ring, <= kMaxStages
    int32_t *err;
    int32_t stall_slab;   // test hook: this slab's CTAs never load their first chunk (-1: none)
};

__global__ void __launch_bounds__(kThreads, 2)
    lm_head_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                      const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[kMaxStages], empty[kMaxStages], done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag, cta_ok;

    if (threadIdx.x == 0) {   // fetch the two tensor-map descriptors early
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_h)) : "memory");
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ks = p.ksplit;
    const int kpart = (int)blockIdx.x % ks;   // rank in the cluster
    const int n0 = ((int)blockIdx.x / ks) * kTileN;
    const int b0 = blockIdx.y * p.btile;
    const int N = p.C * p.V;
    const int chunks = p.K / kChunkK / ks;
    const int kc0 = kpart * chunks;
    const uint32_t bytes_a = kTileN * kChunkK * 2;
    const uint32_t bytes_b = (uint32_t)p.btile * kChunkK * 2;

    // 1024-byte aligned stage ring: A stages, then B stages
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sa = base;
    uint8_t *sb = base + p.stages * bytes_a;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        abort_flag = 0;
        cta_ok = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                     "r"(p.tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    // The weight boxes of the first ring round go into L2 now, a hint issued before the wait (the weights may
    // in principle be an earlier kernel's output, so the loads themselves come after it): batch 4-32 about
    // 0.3 us faster; prefetching the whole slab this way was slower at most batches.
    if (warp == 0 && lane == 0) {
        const int npf = chunks < p.stages ? chunks : p.stages;
        for (int kc = 0; kc < npf; ++kc)
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                             reinterpret_cast<uint64_t>(&map_w)),
                         "r"((kc0 + kc) * kChunkK), "r"(n0)
                         : "memory");
    }
    // Everything above is set-up that reads nothing an earlier kernel writes, so it overlaps the previous
    // kernel's tail; the hidden states and the logits' buffer are used only after this wait.
    pdl_wait();

    if (warp == 0 && lane == 0) {
        // producer: stage s of round `round` (parity round & 1) waits for the MMAs of round - 1.
        // (Test hook: the stalled slab's producer starts at chunk 1, so stage 0 of round 0 is never armed nor
        // loaded and the MMA issuer's wait for it runs out.)
        int kc = 0, s = 0, round = 0;
        if (n0 == p.stall_slab * kTileN) kc = s = 1;
        for (; kc < chunks; ++kc) {
            if (round > 0 && !mbar_wait(&empty[s], (round - 1) & 1)) {
                abort_flag = 1;
                flag_error(p.err, DR_ERRF_TIMEOUT);
                break;
            }
            mbar_expect_tx(&full[s], bytes_a + bytes_b);
            tma_load_2d(sa + s * bytes_a, &map_w, (kc0 + kc) * kChunkK, n0, &full[s]);
            tma_load_2d(sb + s * bytes_b, &map_h, (kc0 + kc) * kChunkK, b0, &full[s]);
            if (++s == p.stages) {
                s = 0;
                ++round;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        const uint32_t idesc = instr_desc(kTileN, p.btile);
        bool ok = true;
        for (int kc = 0, s = 0, round = 0; kc < chunks; ++kc) {
            if (!mbar_wait(&full[s], round & 1)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
            for (int k = 0; k < kChunkK / 16; ++k) {
                const uint64_t a = smem_desc(sa + s * bytes_a + k * 32);
                const uint64_t b = smem_desc(sb + s * bytes_b + k * 32);
                mma_bf16(tmem, a, b, idesc, (kc | k) != 0);
            }
            mma_commit(&empty[s]);   // the stage is free once these MMAs have read it
            if (++s == p.stages) {
                s = 0;
                ++round;
            }
        }
        if (!ok) {
            abort_flag = 1;
            flag_error(p.err, DR_ERRF_TIMEOUT);
        }
        mma_commit(&done);
    }
    __syncwarp();
    // The producer and the MMA issuer set abort_flag with plain shared stores; this barrier orders them before
    // the epilogue reads it, so that every warp of the CTA takes the same decision to write or not.
    __syncthreads();

    pdl_trigger();
    // epilogue: warp w owns TMEM lanes (W rows) 32w .. 32w+31
    const bool finished = __all_sync(0xFFFFFFFFu, mbar_wait(&done, 0));   // warp-uniform for tcgen05.ld
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!finished) {
        if (lane == 0) flag_error(p.err, DR_ERRF_TIMEOUT);
        cta_ok = 0;
    }
    const int row = warp * 32 + lane;
    const int n = n0 + row;
    const int c = n / p.V, v = n - c * p.V;
    const bool have = finished && !abort_flag;
    if (ks == 1) {
        if (have)
            for (int c0 = 0; c0 < p.btile; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem, warp, c0, r);
                // valid columns of this group: inside the tile (btile need not be a multiple of 32; the
                // columns past it belong to the next tile) and inside the batch.  The addresses are one
                // base plus a stride per column: computing each column's full index took 82-92 registers
                // instead of 64, and the head ran up to 20% slower.
                const int lim = min(p.btile, p.B - b0) - c0;
                if (n < N) {
                    float *dst = p.logits + ((size_t)(b0 + c0) * p.C + c) * p.ldv + v;
                    const size_t stride = (size_t)p.C * p.ldv;
                    if (lim >= 32) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) dst[j * stride] = __uint_as_float(r[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < lim) dst[j * stride] = __uint_as_float(r[j]);
                    }
                }
            }
    } else {
        // Two CTAs: this one owns batch columns [kpart * half, (kpart + 1) * half).  It stages the
        // other half of its partial, [column][128 rows] fp32, in its idle stage ring for the peer.
        const int half = p.btile / 2;   // a multiple of 8
        const int own0 = kpart * half, other0 = (kpart ^ 1) * half;
        float *staged = reinterpret_cast<float *>(base);
        if (have)
            for (int c0 = 0; c0 < half; c0 += 8) {
                uint32_t r[8];
                tmem_ld8(tmem, warp, other0 + c0, r);
#pragma unroll
                for (int j = 0; j < 8; ++j) staged[(c0 + j) * kTileN + row] = __uint_as_float(r[j]);
            }
        cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
        cluster.sync();   // both partials (and both CTAs' status) are staged and visible
        const unsigned peer = (unsigned)(kpart ^ 1);
        const bool peer_ok = *cluster.map_shared_rank(&cta_ok, peer) != 0 &&
                             *cluster.map_shared_rank(&abort_flag, peer) == 0;
        const float *theirs = cluster.map_shared_rank(staged, peer);
        if (have && peer_ok)
            for (int c0 = 0; c0 < half; c0 += 8) {
                uint32_t r[8];
                tmem_ld8(tmem, warp, own0 + c0, r);
                float t[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) t[j] = theirs[(c0 + j) * kTileN + row];   // 8 loads in flight
                if (n < N) {
                    const int lim = p.B - (b0 + own0 + c0);   // columns of this group inside the batch
                    float *dst = p.logits + ((size_t)(b0 + own0 + c0) * p.C + c) * p.ldv + v;
                    const size_t stride = (size_t)p.C * p.ldv;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        // rank 0's partial first
                        const float sum = kpart == 0 ? __uint_as_float(r[j]) + t[j] : t[j] + __uint_as_float(r[j]);
                        if (j < lim) dst[j * stride] = sum;
                    }
                }
            }
        cluster.sync();   // keep the staged halves alive until both CTAs have read them
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(p.tmem_cols));
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2D bf16 tensor [rows][K] (row stride K*2 bytes), box [box_rows][64], 128-byte swizzle.
bool encode_2d(CUtensorMap *map, const void *ptr, int rows, int K, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kChunkK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Batch rows per CTA tile: a multiple of 16 (the MMA's N granularity), at most 128.  Above 32 rows, while the
// weight slabs alone leave SMs idle, the batch is cut into at least two tiles, so that every slab has two CTAs
// (measured on the 77 slabs of the 9 x 1088-row head: batch 128 10.6 -> 9.4 us, batch 64 9.0 -> 8.5 us); up
// to 32 rows, one tile and the K split over a CTA pair do that instead.
int lm_head_tc_batch_tile(int B, int mtiles, int sms) {
    int tiles = (B + kMaxBatchTile - 1) / kMaxBatchTile;
    if (B > 32 && tiles < 2 && mtiles < sms) tiles = 2;
    const int t = (((B + tiles - 1) / tiles + 15) / 16) * 16;
    return t > kMaxBatchTile ? kMaxBatchTile : t;
}

cudaError_t launch_lm_head_tc(const LmHeadParams &p, int32_t *err, cudaStream_t stream) {
    const int N = p.C * p.V;
    TcParams tp;
    tp.logits = p.logits;
    tp.B = p.B;
    tp.K = p.K;
    tp.C = p.C;
    tp.V = p.V;
    tp.ldv = p.ldv;
    const int mtiles = (N + kTileN - 1) / kTileN;
    const int sms = current_device_sms();
    tp.btile = lm_head_tc_batch_tile(p.B, mtiles, sms);
    int cols = 32;
    while (cols < tp.btile) cols <<= 1;
    tp.tmem_cols = cols;
    tp.err = err;
    tp.stall_slab = p.stall_slab;
    const int ntiles = (p.B + tp.btile - 1) / tp.btile;
    // Split K in two for small batch tiles when the weight slabs alone leave SMs idle; with more CTAs
    // than SMs the ring shrinks so that two CTAs share an SM (one wave).
    tp.ksplit = (tp.btile <= 32 && mtiles * ntiles <= sms && (p.K / kChunkK) % kMaxSplitK == 0) ? kMaxSplitK : 1;
    const int stage_bytes = (kTileN + tp.btile) * kChunkK * 2;
    tp.stages = mtiles * ntiles * tp.ksplit > sms ? kTwoPerSmBytes / stage_bytes : kMaxStages;
    if (tp.stages > kMaxStages) tp.stages = kMaxStages;
    CUtensorMap map_w, map_h;
    if (!encode_2d(&map_w, p.W, N, p.K, kTileN) || !encode_2d(&map_h, p.hidden, p.B, p.K, tp.btile))
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)tp.stages * stage_bytes;
    const cudaError_t e = cudaFuncSetAttribute(lm_head_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(mtiles * tp.ksplit), (unsigned)ntiles);
    return launch_kernel(lm_head_tc_kernel, grid, dim3(kThreads), smem, stream, (unsigned)tp.ksplit, map_w, map_h,
                         tp);
}

}  // namespace dr
