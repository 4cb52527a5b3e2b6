// Small device helpers: bf16 unpacking, streaming loads, error bits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dr {

// A bf16 is the upper half of a binary32: widening is a shift or a mask.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 &w, float (&f)[8]) {
    f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
    f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
    f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

// 16-byte read-only load of data read once per call: bypass L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 8-byte read-only streaming load (8 e4m3 codes).
__device__ __forceinline__ uint2 ld_stream8(const void *p) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// 8 e4m3 codes (byte i of the pair = element i) -> 8 floats, through CUDA's fp8 conversions.
__device__ __forceinline__ void unpack8_e4m3(const uint2 &c, float (&f)[8]) {
    const uint32_t w[2] = {c.x, c.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const __half2 lo(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFFu), __NV_E4M3));
        const __half2 hi(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3));
        const float2 a = __half22float2(lo), b = __half22float2(hi);
        f[4 * i + 0] = a.x;
        f[4 * i + 1] = a.y;
        f[4 * i + 2] = b.x;
        f[4 * i + 3] = b.y;
    }
}

// 16-byte read-only load through the normal cached path (small, reused data).
__device__ __forceinline__ uint4 ld_ro16(const void *p) {
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// 2^x with the SFU's approximate base-2 exponential (PTX ex2.approx.ftz.f32:
// about 2 ulp; 2^-inf = +0).  Used for softmax weights, where the attention
// tolerance is orders of magnitude looser.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation: it may start while the previous kernel on
// the stream is finishing, so it waits for that kernel (and the visibility of
// its writes) before its first global memory access, and lets the next kernel
// start launching once its own main work is done.  Without the launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() {
#ifndef DR_NO_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_trigger() {
#ifndef DR_NO_PDL
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Relaxed (gpu scope) load: a value that another grid may still be writing,
// read without a data race (used only for prefetch hints).
__device__ __forceinline__ int ld_relaxed(const int32_t *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple
// of 16).  A hint: it changes no data and L2 stays coherent with every writer.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void flag_error(int32_t *err, int bits) {
    if (err) atomicOr(err, bits);
}

// 8 bf16 values -> 8 e4m3 codes: code = e4m3(fl32(x / scale)) with IEEE
// division and CUDA's round-to-nearest-even, saturating conversion.
__device__ __forceinline__ uint2 quantize8_e4m3(const uint4 &w, float scale) {
    float f[8];
    unpack8(w, f);
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        pk[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(f[2 * i], scale), __fdiv_rn(f[2 * i + 1], scale)), __NV_SATFINITE, __NV_E4M3);
    return make_uint2(pk[0] | (pk[1] << 16), pk[2] | (pk[3] << 16));
}

// fp32 -> bf16 bits, IEEE round to nearest even (CUDA's conversion intrinsic).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

}  // namespace dr
