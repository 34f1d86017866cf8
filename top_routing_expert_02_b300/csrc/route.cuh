// Router: logits = x W^T + b (fp32), softmax over E, top-k by warp argmax,
// and per-block partial sums of the probabilities.
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §1.1 (the
// router is a light linear layer choosing Top-K experts per token) and §2.1
// step 1; the deployment guide "细粒度专家并行部署实践与优化指南" §七 takes top-k of
// the softmaxed gate probabilities.  Ties go to the lower expert index.
//
// Layout: one block = 8 warps; each warp owns TW tokens; lane l owns experts
// l, l+32, ... (EPL of them).  d is walked in 32-wide chunks staged in shared
// memory (x tile as fp32, W chunk transposed so a warp reads 32 consecutive
// experts).  Each logit is one fp32 FMA chain over c = 0..d-1 in order, so
// results do not depend on the launch shape.
#pragma once
#include "common.cuh"

namespace route {

constexpr int WARPS = 8;
constexpr int THREADS = WARPS * 32;
constexpr int DK = 32;

template <int EPL, int TW, bool BF16>
__global__ void __launch_bounds__(THREADS)
route_kernel(const void* __restrict__ x, const float* __restrict__ W, const float* __restrict__ bias,
             int T, int d, int E, int k, int renorm, int32_t* __restrict__ idx_out,
             float* __restrict__ gate_out, float* __restrict__ partial, RouteSel sel)
{
    constexpr int EP = 32 * EPL;
    constexpr int TM = WARPS * TW;
    __shared__ float xs[TM][DK];
    __shared__ float wsm[DK][EP + 1];
    __shared__ float red[WARPS][EP];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * TM;

    // experts E..EP-1 do not exist: keep their staged weights at zero
    for (int v = tid; v < DK * (EP - E); v += THREADS) wsm[v / (EP - E)][E + v % (EP - E)] = 0.f;

    float acc[TW][EPL];
#pragma unroll
    for (int a = 0; a < TW; ++a)
#pragma unroll
        for (int i = 0; i < EPL; ++i) acc[a][i] = 0.f;

    for (int c0 = 0; c0 < d; c0 += DK) {
        if (BF16) {
            for (int v = tid; v < TM * (DK / 8); v += THREADS) {
                const int r = v / (DK / 8), q = v % (DK / 8), t = t0 + r;
                float f[8];
                if (t < T) {
                    unpack_bf16x8(ldg_nc_v4((const uint16_t*)x + (size_t)t * d + c0 + q * 8), f);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) f[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) xs[r][q * 8 + i] = f[i];
            }
        } else {
            for (int v = tid; v < TM * (DK / 4); v += THREADS) {
                const int r = v / (DK / 4), q = v % (DK / 4), t = t0 + r;
                uint4 u = make_uint4(0, 0, 0, 0);
                if (t < T) u = ldg_nc_v4((const float*)x + (size_t)t * d + c0 + q * 4);
                xs[r][q * 4 + 0] = __uint_as_float(u.x);
                xs[r][q * 4 + 1] = __uint_as_float(u.y);
                xs[r][q * 4 + 2] = __uint_as_float(u.z);
                xs[r][q * 4 + 3] = __uint_as_float(u.w);
            }
        }
        for (int v = tid; v < E * (DK / 4); v += THREADS) {
            const int e = v / (DK / 4), q = v % (DK / 4);
            const uint4 u = ldg_nc_v4(W + (size_t)e * d + c0 + q * 4);
            wsm[q * 4 + 0][e] = __uint_as_float(u.x);
            wsm[q * 4 + 1][e] = __uint_as_float(u.y);
            wsm[q * 4 + 2][e] = __uint_as_float(u.z);
            wsm[q * 4 + 3][e] = __uint_as_float(u.w);
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < DK; ++c) {
            float xv[TW], wv[EPL];
#pragma unroll
            for (int a = 0; a < TW; ++a) xv[a] = xs[warp * TW + a][c];
#pragma unroll
            for (int i = 0; i < EPL; ++i) wv[i] = wsm[c][lane + 32 * i];
#pragma unroll
            for (int a = 0; a < TW; ++a)
#pragma unroll
                for (int i = 0; i < EPL; ++i) acc[a][i] = fmaf(xv[a], wv[i], acc[a][i]);
        }
        __syncthreads();
    }

    float psum[EPL];
    int grp[EPL];   // group of each of this lane's experts
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        psum[i] = 0.f;
        grp[i] = (lane + 32 * i) / sel.gsz;
    }

#pragma unroll
    for (int a = 0; a < TW; ++a) {
        const int t = t0 + warp * TW + a;   // uniform across the warp
        if (t >= T) break;
        float l[EPL], p[EPL];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            l[i] = (e < E) ? acc[a][i] + (bias ? __ldg(bias + e) : 0.f) : -INFINITY;
            mx = fmaxf(mx, l[i]);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            p[i] = (lane + 32 * i < E) ? expf(l[i] - mx) : 0.f;
            s += p[i];
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (sel.lse && lane == 0) sel.lse[t] = mx + logf(s);
        if (sel.logits) {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i < E) sel.logits[(size_t)t * E + lane + 32 * i] = l[i];
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            p[i] = p[i] / s;
            psum[i] += p[i];
        }
        const unsigned gkeep = keep_groups<EPL>(l, grp, E, sel, lane);

        // k rounds of warp argmax on (logit desc, index asc) over the kept groups
        unsigned taken = 0;
        int my_e = 0;
        float my_p = 0.f, chosen = 0.f;
        for (int j = 0; j < k; ++j) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && ((gkeep >> grp[i]) & 1u) &&
                    (l[i] > bv || (l[i] == bv && e < bi))) {
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
            float pv = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == bi) {
                    pv = p[i];
                    taken |= 1u << i;
                }
            const float pw = __shfl_sync(0xffffffffu, pv, bi & 31);
            chosen += pw;
            if (lane == j) {
                my_e = bi;
                my_p = pw;
            }
        }
        if (lane < k) {
            idx_out[(size_t)t * k + lane] = my_e;
            gate_out[(size_t)t * k + lane] = renorm ? my_p / chosen : my_p;
        }
    }

#pragma unroll
    for (int i = 0; i < EPL; ++i) red[warp][lane + 32 * i] = psum[i];
    __syncthreads();
    for (int e = tid; e < E; e += THREADS) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) s += red[w][e];
        partial[(size_t)blockIdx.x * E + e] = s;
    }
}

// prob_sum[e] = sum over blocks of partial[b][e], in a fixed order (fp64).
constexpr int FIN_THREADS = 1024;
__global__ void __launch_bounds__(FIN_THREADS)
route_finalize(const float* __restrict__ partial, int nblk, int E, float* __restrict__ prob_sum)
{
    __shared__ double part[FIN_THREADS];
    const int parts = FIN_THREADS / E;   // >= 4 since E <= 256
    const int e = threadIdx.x % E, g = threadIdx.x / E;
    double s = 0.0;
    if (g < parts)
        for (int b = g; b < nblk; b += parts) s += (double)partial[(size_t)b * E + e];
    part[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x < E) {
        double tot = 0.0;
        for (int q = 0; q < parts; ++q) tot += part[q * E + threadIdx.x];
        prob_sum[threadIdx.x] = (float)tot;
    }
}

}  // namespace route
