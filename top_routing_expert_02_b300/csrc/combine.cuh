// Combine (the return All-to-All of expert parallelism, here an
// un-permutation in HBM) and the auxiliary load-balance loss.
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §2.1 step 5:
// expert outputs go back to their tokens' original positions; the
// deployment guide "细粒度专家并行部署实践与优化指南" §七 gathers them back the same
// way.  The gate product already sits inside y_perm (expert down-projection
// epilogue), so the combine is a plain sum over the k slots of a token.
// Aux loss: §5.1 of the tutorial, L = alpha * num_experts * sum_i f_i P_i.
#pragma once
#include "common.cuh"

namespace combine {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;

// One warp: f_e = counts[e] / T, P_e = prob_sum[e] / T, fixed-order fp64 sum
// (lane-strided partial sums, then a butterfly).
__device__ __forceinline__ void aux_loss_warp(const int32_t* __restrict__ counts, const float* __restrict__ prob_sum,
                                              long long T, int E, float alpha, float* __restrict__ loss, int lane)
{
    double s = 0.0;
    for (int e = lane; e < E; e += 32)
        s += ((double)counts[e] / (double)T) * ((double)prob_sum[e] / (double)T);
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) *loss = (float)((double)alpha * (double)E * s);
}

// Optional auxiliary loss computed by the first warp of a combine launch
// (saves the aux-loss launch; loss == nullptr: none).  Its inputs (counts,
// prob_sum) come from routing and dispatch, which have finished before the
// expert GEMMs, so it runs before the wait for y_perm.
struct AuxArgs {
    const int32_t* counts;
    const float* prob_sum;
    long long T;
    int E;
    float alpha;
    float* loss;
};

// One warp per (token, chunk of 128 16-byte vectors of its row): each lane
// sums four vectors of the token's k rows in j order (fp32) and rounds once.
// The rows go in pairs whose eight loads are all issued before their sums,
// unconditionally: a dropped slot (-1) reads row 0 and adds -0.0, which is
// an exact identity for every fp32 value (x + -0 = x, also for x = +0 and
// -0), so the result has the bits of skipping it.  A token with no kept slot
// gets zeros.  The slot rows of the token are loaded once per task, one per
// lane, and handed out by shuffles.
constexpr int CHUNK_VEC = 128;   // 16-byte vectors per chunk (4 per lane)
constexpr int ROWS_PER_BATCH = 2;

template <bool BF16>
__global__ void __launch_bounds__(THREADS)
combine_kernel(const uint4* __restrict__ y_perm, const int32_t* __restrict__ slot_row, int T, int k,
               int vec16, uint4* __restrict__ y, AuxArgs aux)
{
    constexpr int V = CHUNK_VEC / 32, KB = ROWS_PER_BATCH;
    const int lane = threadIdx.x & 31;
    if (aux.loss && blockIdx.x == 0 && threadIdx.x < 32)
        aux_loss_warp(aux.counts, aux.prob_sum, aux.T, aux.E, aux.alpha, aux.loss, lane);
    pdl_wait();   // launched as a programmatic dependent of the kernel writing y_perm
    const int nchunk = (vec16 + CHUNK_VEC - 1) / CHUNK_VEC;
    const long long tasks = (long long)T * nchunk;
    const long long warps_total = (long long)gridDim.x * WARPS;
    for (long long task = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5); task < tasks; task += warps_total) {
        const int t = (int)(task / nchunk);
        const int v0 = (int)(task - (long long)t * nchunk) * CHUNK_VEC + lane;
        const int my_row = lane < k ? __ldg(slot_row + (size_t)t * k + lane) : -1;   // k <= 16
        float acc[V][8];
#pragma unroll
        for (int u = 0; u < V; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] = 0.f;
        for (int j0 = 0; j0 < k; j0 += KB) {
            uint4 q[KB][V];
            bool ok[KB];
#pragma unroll
            for (int jj = 0; jj < KB; ++jj) {
                const int r = __shfl_sync(0xffffffffu, my_row, (j0 + jj) & 31);
                ok[jj] = j0 + jj < k && r >= 0;
                const uint4* src = y_perm + (size_t)(ok[jj] ? r : 0) * vec16;
#pragma unroll
                for (int u = 0; u < V; ++u)
                    q[jj][u] = v0 + 32 * u < vec16 ? ldg_nc_v4(src + v0 + 32 * u) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int jj = 0; jj < KB; ++jj)
#pragma unroll
                for (int u = 0; u < V; ++u) {
                    if (BF16) {
                        float f[8];
                        unpack_bf16x8(q[jj][u], f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[u][i] += ok[jj] ? f[i] : -0.0f;
                    } else {
                        acc[u][0] += ok[jj] ? __uint_as_float(q[jj][u].x) : -0.0f;
                        acc[u][1] += ok[jj] ? __uint_as_float(q[jj][u].y) : -0.0f;
                        acc[u][2] += ok[jj] ? __uint_as_float(q[jj][u].z) : -0.0f;
                        acc[u][3] += ok[jj] ? __uint_as_float(q[jj][u].w) : -0.0f;
                    }
                }
        }
#pragma unroll
        for (int u = 0; u < V; ++u) {
            const int v = v0 + 32 * u;
            if (v >= vec16) break;
            uint4 o;
            if (BF16) {
                o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                o.w = pack_bf16x2(acc[u][6], acc[u][7]);
            } else {
                o = make_uint4(__float_as_uint(acc[u][0]), __float_as_uint(acc[u][1]), __float_as_uint(acc[u][2]),
                               __float_as_uint(acc[u][3]));
            }
            y[(size_t)t * vec16 + v] = o;
        }
    }
}

// The aux loss alone (one warp).
__global__ void aux_loss_kernel(const int32_t* __restrict__ counts, const float* __restrict__ prob_sum,
                                long long T, int E, float alpha, float* __restrict__ loss)
{
    aux_loss_warp(counts, prob_sum, T, E, alpha, loss, threadIdx.x);
}

// Router z-loss (the ms-swift ETP page names a routing z-loss that spreads
// the router's choices; its formula is the one of ST-MoE, Zoph et al. 2022,
// eq. 5): loss = beta * (1/T) * sum_t lse[t]^2.  One block: each thread sums
// the squares of its elements (16-byte loads, eight in flight, when lse is
// 16-byte aligned) in fp32 with Kahan compensation -- a single block has few
// fp64 units, and compensated fp32 keeps the sum within a few fp32 ulps for
// any T -- then the per-thread sums go through a fixed shared-memory tree in
// fp64; the result does not depend on timing.
constexpr int ZL_THREADS = 1024;

struct Kahan {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float v)
    {
        const float y = v - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
};

__global__ void __launch_bounds__(ZL_THREADS)
z_loss_kernel(const float* __restrict__ lse, long long T, float beta, float* __restrict__ loss)
{
    __shared__ double sh[ZL_THREADS];
    Kahan k;
    long long done = 0;
    if ((reinterpret_cast<uintptr_t>(lse) & 15u) == 0) {
        const float4* v = reinterpret_cast<const float4*>(lse);
        const long long n4 = T / 4;
        for (long long i0 = threadIdx.x; i0 < n4; i0 += 8 * ZL_THREADS) {
            float4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const long long i = i0 + (long long)u * ZL_THREADS;
                q[u] = i < n4 ? __ldg(v + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                k.add(q[u].x * q[u].x);
                k.add(q[u].y * q[u].y);
                k.add(q[u].z * q[u].z);
                k.add(q[u].w * q[u].w);
            }
        }
        done = n4 * 4;
    }
    for (long long t = done + threadIdx.x; t < T; t += ZL_THREADS) {
        const float x = __ldg(lse + t);
        k.add(x * x);
    }
    sh[threadIdx.x] = (double)k.s - (double)k.c;
    __syncthreads();
    for (int w = ZL_THREADS / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) *loss = (float)((double)beta * sh[0] / (double)T);
}

}  // namespace combine
