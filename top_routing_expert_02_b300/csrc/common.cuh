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

// Programmatic dependent launch: the next kernel in the stream may start
// (launch_dependents); wait until the kernel before this one has finished and
// its memory is visible (wait).  Both are no-ops for a kernel launched
// without the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// Routing variants of the top-k step.  Group-limited routing (the ms-swift
// Megatron acceleration page, §3.2 EP bullet: pick the token's expert group,
// then Top-k inside it): experts form n_group contiguous groups of gsz; a
// group scores its largest logit; the topk_group best groups (ties: lower
// group) are kept and the k experts are chosen among theirs.  n_group = 1 is
// plain top-k.  lse, when set, receives log sum_e exp(l[t,e]) per token for
// the router z-loss; logits, when set, receives the logits themselves.
struct RouteSel {
    int n_group;      // 1..32
    int gsz;          // E / n_group
    int topk_group;   // 1..n_group
    float* lse;       // [T] or nullptr
    float* logits;    // [T, E] (bias included) or nullptr: kept for the backward
};

// Group mask of one token (bit g set: group g kept), lane l holding the
// logits of experts l, l+32, ...: topk_group rounds of warp argmax over the
// experts of groups not yet kept; the winner's group is kept next.  The
// argmax orders by (logit desc, index asc), so equal group scores go to the
// lower group.  All ones when n_group = 1.
template <int EPL>
__device__ __forceinline__ unsigned keep_groups(const float* l, const int* grp, int E, const RouteSel& sel,
                                                int lane)
{
    if (sel.n_group <= 1) return 0xffffffffu;
    unsigned keep = 0;
    for (int r = 0; r < sel.topk_group; ++r) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((keep >> grp[i]) & 1u) && (l[i] > bv || (l[i] == bv && e < bi))) {
                bv = l[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (bi < E) keep |= 1u << (bi / sel.gsz);
    }
    return keep;
}

static inline int ceil_div_i(long long a, long long b) { return (int)((a + b - 1) / b); }
