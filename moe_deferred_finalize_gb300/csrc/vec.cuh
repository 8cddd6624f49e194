// Device helpers shared by the finalize kernels: bf16 <-> fp32 conversion,
// 16-byte and scalar vector access with the cache behaviour each operand
// wants, warp reduction, routing-weight decoding.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_finalize.h"

namespace moef {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);   // .x -> low half
    return *reinterpret_cast<uint32_t *>(&b);
}

template <int VEC>
struct VecOps;

// 16-byte vectors of 8 bf16 values.
template <>
struct VecOps<8> {
    using V = uint4;
    // Gathered expert rows: read-only for the kernel's lifetime and read once.
    static __device__ __forceinline__ V load_row(const uint16_t *p) {
        V r;
        asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
            : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
            : "l"(p));
        return r;
    }
    // Dense per-token operands (may alias an output when run in place).
    static __device__ __forceinline__ V load(const uint16_t *p) {
        return __ldcs(reinterpret_cast<const uint4 *>(p));
    }
    // Small operands reused by every token (gamma).
    static __device__ __forceinline__ V load_reused(const uint16_t *p) {
        return __ldg(reinterpret_cast<const uint4 *>(p));
    }
    static __device__ __forceinline__ void store(uint16_t *p, V v) {
        __stcs(reinterpret_cast<uint4 *>(p), v);
    }
    static __device__ __forceinline__ void to_f32(const V &v, float f[8]) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
    static __device__ __forceinline__ V from_f32(const float f[8]) {
        V v;
        v.x = pack_bf16x2(f[0], f[1]);
        v.y = pack_bf16x2(f[2], f[3]);
        v.z = pack_bf16x2(f[4], f[5]);
        v.w = pack_bf16x2(f[6], f[7]);
        return v;
    }
};

// Single bf16 values: any H, any 2-byte alignment.
template <>
struct VecOps<1> {
    using V = unsigned short;
    static __device__ __forceinline__ V load_row(const uint16_t *p) {
        return __ldg(reinterpret_cast<const unsigned short *>(p));
    }
    static __device__ __forceinline__ V load(const uint16_t *p) {
        return __ldcs(reinterpret_cast<const unsigned short *>(p));
    }
    static __device__ __forceinline__ V load_reused(const uint16_t *p) {
        return __ldg(reinterpret_cast<const unsigned short *>(p));
    }
    static __device__ __forceinline__ void store(uint16_t *p, V v) {
        __stcs(reinterpret_cast<unsigned short *>(p), v);
    }
    static __device__ __forceinline__ void to_f32(const V &v, float f[1]) {
        f[0] = __uint_as_float(static_cast<uint32_t>(v) << 16);
    }
    static __device__ __forceinline__ V from_f32(const float f[1]) {
        return __bfloat16_as_ushort(__float2bfloat16_rn(f[0]));
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Routing weight of slot i, decoded exactly to fp32.
__device__ __forceinline__ float decode_weight(const void *weights, int wkind, int64_t i) {
    if (wkind == MOEF_W_FP32) return __ldg(static_cast<const float *>(weights) + i);
    if (wkind == MOEF_W_BF16)
        return __uint_as_float(
            static_cast<uint32_t>(__ldg(static_cast<const unsigned short *>(weights) + i)) << 16);
    // packed (expert_id << 16) | bf16(weight): the low half, moved up
    return __uint_as_float(
        static_cast<uint32_t>(__ldg(static_cast<const int *>(weights) + i)) << 16);
}

}  // namespace
}  // namespace moef
