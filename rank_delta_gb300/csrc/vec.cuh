// 16-byte bf16 vector loads, bf16 -> f32 widening and warp reductions.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace rd {

__device__ __forceinline__ uint4 ld_16(const uint16_t *p)
{
    return *reinterpret_cast<const uint4 *>(p);
}

// Read-only path (data not written during the kernel).
__device__ __forceinline__ uint4 ld_nc_16(const uint16_t *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// bf16 bits -> f32: the bf16 value is the upper half of the f32 pattern.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// acc + sum_{j<8} a[j] * b[j] over two 8 x bf16 vectors, in index order.
__device__ __forceinline__ float dot8_acc(float acc, uint4 a, uint4 b)
{
    acc = fmaf(bf_lo(a.x), bf_lo(b.x), acc);
    acc = fmaf(bf_hi(a.x), bf_hi(b.x), acc);
    acc = fmaf(bf_lo(a.y), bf_lo(b.y), acc);
    acc = fmaf(bf_hi(a.y), bf_hi(b.y), acc);
    acc = fmaf(bf_lo(a.z), bf_lo(b.z), acc);
    acc = fmaf(bf_hi(a.z), bf_hi(b.z), acc);
    acc = fmaf(bf_lo(a.w), bf_lo(b.w), acc);
    acc = fmaf(bf_hi(a.w), bf_hi(b.w), acc);
    return acc;
}

// acc + sum_{j<8} b[j] * h[j], b bf16, h f32 (two float4).
__device__ __forceinline__ float dot8_bf_f32(float acc, uint4 b, float4 h0, float4 h1)
{
    acc = fmaf(bf_lo(b.x), h0.x, acc);
    acc = fmaf(bf_hi(b.x), h0.y, acc);
    acc = fmaf(bf_lo(b.y), h0.z, acc);
    acc = fmaf(bf_hi(b.y), h0.w, acc);
    acc = fmaf(bf_lo(b.z), h1.x, acc);
    acc = fmaf(bf_hi(b.z), h1.y, acc);
    acc = fmaf(bf_lo(b.w), h1.z, acc);
    acc = fmaf(bf_hi(b.w), h1.w, acc);
    return acc;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float v)
{
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t *>(&b);
}

} // namespace rd
