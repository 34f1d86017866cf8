// Router on the tensor cores for bf16 x: logits, softmax, top-k and the
// per-block probability sums of 128 tokens per block.
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §1.1 / §2.1
// step 1 (a light linear layer scores the experts, each token keeps its
// Top-K); the deployment guide "细粒度专家并行部署实践与优化指南" §七 takes the top-k
// of the softmaxed gate probabilities.  Ties go to the lower expert index.
//
// The fp32 router weight is split exactly into three bf16 parts,
// W = W0 + W1 + W2 (each part holds the next 8 significant bits), stacked as
// one [3*E_pad, d] bf16 matrix.  x is bf16, so each product x*Wi is exact in
// fp32 and the tensor core accumulates in fp32: the logits carry fp32
// accuracy at tensor-core speed, and the router stays bound by the HBM read
// of x at every E (on CUDA cores it is FP32-bound from E of about 16 up).
//
// One block per 128 tokens, 6 warps: TMA producer (x tile 128x64 + the
// stacked weight), one MMA-issuing thread (M=128, N = 3*E_pad in one or two
// MMAs), 4 epilogue warps with one token per thread: the thread reads its
// token's accumulator row from TMEM, forms l = (a0 + a1) + a2 + b, and keeps
// the running max and a sorted top-k list in registers; a second pass sums
// exp(l - max); a third forms p = exp(l - max) / sum, reduces it over the 128
// tokens (warp shuffles, then the 4 warps in a fixed order) into this block's
// row of partial sums.  route_finalize then adds the rows in block order.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"

namespace rtc {

constexpr int BM = 128, BK = 64, THREADS = 192, MAX_STAGES = 8;
constexpr int A_BYTES = BM * BK * 2;
constexpr int MAX_EPAD = 160;   // 3 * E_pad <= 480 TMEM columns

struct Args {
    const float* bias;
    int T, E, E_pad, k, renorm;
    int nk;          // K blocks of 64
    int nb_chunks;   // MMAs per K step (1 or 2)
    int nb_rows;     // N of each MMA (rows of one weight box)
    int stages;
    int stage_bytes;
    uint32_t tmem_cols;
    int32_t* idx;
    float* gate;
    float* partial;  // [gridDim.x, E]
    unsigned long long wait_limit;
};

// W (fp32 [E, d]) -> stacked bf16 [3*E_pad, d]: rows [0,E_pad) W0, [E_pad,2E_pad) W1,
// [2E_pad,3E_pad) W2; rows of experts >= E are zero.  W0 = rn(W), W1 = rn(W - W0),
// W2 = rn(W - W0 - W1); both differences are exact in fp32.
__global__ void split_weight_kernel(const float* __restrict__ W, int E, int E_pad, int d,
                                    uint16_t* __restrict__ Ws)
{
    const long long n = (long long)E_pad * d;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(i / d);
        float w = e < E ? __ldg(W + i) : 0.f;
        __nv_bfloat16 b0 = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(b0);
        __nv_bfloat16 b1 = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(b1);
        __nv_bfloat16 b2 = __float2bfloat16_rn(r2);
        Ws[i] = *reinterpret_cast<uint16_t*>(&b0);
        Ws[n + i] = *reinterpret_cast<uint16_t*>(&b1);
        Ws[2 * n + i] = *reinterpret_cast<uint16_t*>(&b2);
    }
}

// Insert (v, e) into the descending list tv/ti of KMAX entries; an equal
// value already present stays ahead (it has the lower expert index).
template <int KMAX>
__device__ __forceinline__ void topk_insert(float (&tv)[KMAX], int (&ti)[KMAX], float v, int e)
{
    if (!(v > tv[KMAX - 1])) return;
#pragma unroll
    for (int j = KMAX - 1; j > 0; --j) {
        if (v > tv[j - 1]) {
            tv[j] = tv[j - 1];
            ti[j] = ti[j - 1];
        } else if (v > tv[j]) {
            tv[j] = v;
            ti[j] = e;
        }
    }
    if (v > tv[0]) {
        tv[0] = v;
        ti[0] = e;
    }
}

template <int KMAX>
__global__ void __launch_bounds__(THREADS, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const Args g)
{
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES], acc_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ float red[4][MAX_EPAD];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem0 = (ptx::smem_u32(dsmem) + 1023u) & ~1023u;
    const int t0 = blockIdx.x * BM;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < g.stages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&acc_bar), 1);
        ptx::fence_mbar_init();
        ptx::tma_prefetch_desc(&tmX);
        ptx::tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), g.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;
    const uint64_t limit = g.wait_limit;
    const int b_box_bytes = g.nb_rows * 128;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int fills = 0;
            bool ok = true;
            for (int kb = 0; kb < g.nk; ++kb) {
                if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), phase ^ 1u, limit)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
                const uint32_t sa = smem0 + stage * g.stage_bytes;
                ptx::mbar_arrive_expect_tx(fb, g.stage_bytes);
                ptx::tma_load_2d(sa, &tmX, fb, kb * BK, t0);
                for (int c = 0; c < g.nb_chunks; ++c)
                    ptx::tma_load_2d(sa + A_BYTES + c * b_box_bytes, &tmW, fb, kb * BK, c * g.nb_rows);
                ++fills;
                if (++stage == g.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            for (int f = fills - 1; f >= 0 && f >= fills - g.stages; --f)
                if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[f % g.stages]), (uint32_t)((f / g.stages) & 1), limit)) {
                    moe_flag(MOE_DEV_TIMEOUT);
                    break;
                }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(128, g.nb_rows);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = 0; kb < g.nk; ++kb) {
                if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), phase, limit)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sa = smem0 + stage * g.stage_bytes, sb = sa + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    for (int c = 0; c < g.nb_chunks; ++c)
                        ptx::mma_bf16(tmem_base + (uint32_t)(c * g.nb_rows), ptx::sdesc_kmajor_sw128(sa + kk * 32),
                                      ptx::sdesc_kmajor_sw128(sb + c * b_box_bytes + kk * 32), idesc,
                                      (kb | kk) != 0);
                ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
                if (++stage == g.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            // arrives once every MMA issued above has completed (also on the error path)
            ptx::mma_commit(ptx::smem_u32(&acc_bar));
        }
    } else {
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int t = t0 + r;
        const bool valid = t < g.T;
        const bool waited = ptx::mbar_wait(ptx::smem_u32(&acc_bar), 0, limit);
        const bool all_ok = __all_sync(0xffffffffu, waited);
        if (!all_ok) moe_flag(MOE_DEV_TIMEOUT);
        ptx::tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
        const int E = g.E, Ep = g.E_pad;

        float tv[KMAX];
        int ti[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            tv[j] = -INFINITY;
            ti[j] = 0x7fffffff;
        }
        float mx = -INFINITY;
        // pass 1: running max and top-k
        for (int e0 = 0; e0 < Ep; e0 += 16) {
            uint32_t a0[16], a1[16], a2[16];
            ptx::tmem_ld16(tb + e0, a0);
            ptx::tmem_ld16(tb + Ep + e0, a1);
            ptx::tmem_ld16(tb + 2 * Ep + e0, a2);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = e0 + i;
                if (e < E) {
                    const float l = (__uint_as_float(a0[i]) + __uint_as_float(a1[i])) + __uint_as_float(a2[i]) +
                                    (g.bias ? __ldg(g.bias + e) : 0.f);
                    mx = fmaxf(mx, l);
                    topk_insert<KMAX>(tv, ti, l, e);
                }
            }
        }
        // pass 2: softmax denominator
        float s = 0.f;
        for (int e0 = 0; e0 < Ep; e0 += 16) {
            uint32_t a0[16], a1[16], a2[16];
            ptx::tmem_ld16(tb + e0, a0);
            ptx::tmem_ld16(tb + Ep + e0, a1);
            ptx::tmem_ld16(tb + 2 * Ep + e0, a2);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = e0 + i;
                if (e < E) {
                    const float l = (__uint_as_float(a0[i]) + __uint_as_float(a1[i])) + __uint_as_float(a2[i]) +
                                    (g.bias ? __ldg(g.bias + e) : 0.f);
                    s += expf(l - mx);
                }
            }
        }
        // pass 3: probabilities, summed over this block's tokens per expert
        for (int e0 = 0; e0 < Ep; e0 += 16) {
            uint32_t a0[16], a1[16], a2[16];
            ptx::tmem_ld16(tb + e0, a0);
            ptx::tmem_ld16(tb + Ep + e0, a1);
            ptx::tmem_ld16(tb + 2 * Ep + e0, a2);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = e0 + i;
                float p = 0.f;
                if (e < E && valid) {
                    const float l = (__uint_as_float(a0[i]) + __uint_as_float(a1[i])) + __uint_as_float(a2[i]) +
                                    (g.bias ? __ldg(g.bias + e) : 0.f);
                    p = expf(l - mx) / s;
                }
#pragma unroll
                for (int o = 16; o; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
                if (lane == 0) red[q][e] = p;
            }
        }
        if (valid) {
            float chosen = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < g.k) chosen += expf(tv[j] - mx) / s;
#pragma unroll
            for (int j = 0; j < KMAX; ++j)
                if (j < g.k) {
                    const float pj = expf(tv[j] - mx) / s;
                    g.idx[(size_t)t * g.k + j] = ti[j];
                    g.gate[(size_t)t * g.k + j] = g.renorm ? pj / chosen : pj;
                }
        }
        ptx::tc_fence_before();
        ptx::named_bar_sync(1, 128);
        for (int e = r; e < E; e += 128)
            g.partial[(size_t)blockIdx.x * E + e] = ((red[0][e] + red[1][e]) + red[2][e]) + red[3][e];
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, g.tmem_cols);
    }
}

}  // namespace rtc
