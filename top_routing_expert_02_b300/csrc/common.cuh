// Shared device helpers of the MoE-layer forward library (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_b300.h"

// Bits of the sticky device status word (read and cleared by moe_check).
#define MOE_DEV_TIMEOUT 1u      // a pipeline wait ran past its limit
#define MOE_DEV_BAD_EXPERT 2u   // an expert id outside [0, E) reached dispatch

// One status word per device that loads the library; zero at module load.
__device__ unsigned int g_moe_status;

__device__ __forceinline__ void moe_flag(unsigned bits) { atomicOr(&g_moe_status, bits); }

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t u16) { return __uint_as_float(u16 << 16); }

// Eight bf16 (one 16-byte vector) -> eight floats.
__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float* f)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Two floats -> packed bf16x2, round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Exact-erf GELU and SiLU in fp32 (CUDA's erff / expf).
__device__ __forceinline__ float gelu_f32(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }
__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

static inline int ceil_div_i(long long a, long long b) { return (int)((a + b - 1) / b); }
