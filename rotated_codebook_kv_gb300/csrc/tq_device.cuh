// tq_device.cuh -- small device helpers shared by the kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#define TQ_DEVERR_SLOT_RANGE 0x1u
#define TQ_DEVERR_BLOCK_RANGE 0x2u
#define TQ_DEVERR_SEQ_RANGE 0x4u
#define TQ_DEVERR_TIMEOUT 0x8u

namespace tq {

__device__ __forceinline__ float bf16_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint16_t double_to_bf16_bits(double x)
{
    return __bfloat16_as_ushort(__double2bfloat16(x));
}

// Error-free sum: s + e == a + b exactly (Knuth's TwoSum).  The _rn
// intrinsics are never contracted into FMAs by the compiler.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Compensated dot-product step (Ogita, Rump & Oishi, "Accurate sum and dot
// product", 2005): (s, c) accumulates a * b with the product split exactly.
__device__ __forceinline__ void dot2_step(float &s, float &c, float a, float b)
{
    const float p = __fmul_rn(a, b);
    const float ep = __fmaf_rn(a, b, -p);
    float t, et;
    two_sum(s, p, t, et);
    s = t;
    c = __fadd_rn(c, __fadd_rn(et, ep));
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Asynchronous prefetch of [p, p + bytes) into L2 by the bulk-copy engine; no
// registers or shared memory are held.  p and bytes must be multiples of 16
// and the range must lie inside one allocation.
__device__ __forceinline__ void l2_prefetch_bulk(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 16-byte global load issued exactly where written: a volatile asm statement
// is neither sunk past a barrier to its first use nor re-issued later, which
// the compiler may do with read-only loads.  p must be 16-byte aligned.
__device__ __forceinline__ uint4 ld_pinned(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int64_t ld_pinned_s64(const int64_t *p)
{
    int64_t v;
    asm volatile("ld.global.nc.s64 %0, [%1];" : "=l"(v) : "l"(p));
    return v;
}

}  // namespace tq
