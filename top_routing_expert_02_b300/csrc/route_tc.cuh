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
// route_logits_kernel: S blocks per 128-token tile (S > 1 splits d when there
// are too few tiles to fill the GPU), 6 warps each: TMA producer (x tile
// 128x64 + the stacked weight), one MMA-issuing thread (M=128, N = 3*E_pad in
// one or two MMAs), 4 epilogue warps that turn the accumulator row of each
// token into its partial logits (a0 + a1) + a2 and store them.
// route_finish_*_kernel: adds each token's S partial rows in split order plus
// the bias, takes the softmax and the top-k on (logit desc, index asc), and
// sums the probabilities per block; prob_sum_kernel then adds the block rows
// with one fixed-shape tree per expert.  E <= 32: one lane per token (all E logits in
// registers, sorted top-k insertion); larger E: one warp per token (lane l
// owns experts l, l+32, ... sorted in registers; k rounds of two redux.sync
// over order-preserving keys).
// Every sum runs in a fixed order, so the result is the same bits on every run.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"

namespace rtc {

constexpr int BM = 128, BK = 64, THREADS = 192, MAX_STAGES = 8;
constexpr int A_BYTES = BM * BK * 2;
constexpr int MAX_EPAD = 160;   // 3 * E_pad <= 480 TMEM columns
constexpr int MAX_SPLITS = 16;  // blocks per 128-token tile

struct Args {
    int T, E_pad;
    int nk;          // K blocks of 64 in d
    int S;           // K splits: blocks per 128-token tile
    int nb_chunks;   // MMAs per K step (1 or 2)
    int nb_rows;     // N of each MMA (rows of one weight box)
    int stages;
    int stage_bytes;
    uint32_t tmem_cols;
    float* part;     // [S, T, E_pad] partial logits
    unsigned long long wait_limit;
};

// W (fp32 [E, d]) -> stacked bf16 [3*E_pad, d]: rows [0,E_pad) W0, [E_pad,2E_pad) W1,
// [2E_pad,3E_pad) W2; rows of experts >= E are zero.  W0 = rn(W), W1 = rn(W - W0),
// W2 = rn(W - W0 - W1); both differences are exact in fp32.
__global__ void split_weight_kernel(const float* __restrict__ W, int E, int E_pad, int d,
                                    uint16_t* __restrict__ Ws)
{
    const long long n = (long long)E_pad * d;
    const long long i0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = i0; i < n; i += stride) {
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

// Block (tile, s): tile = blockIdx.x / S covers tokens [128*tile, 128*tile + 128),
// split s covers K blocks [s*nk/S, (s+1)*nk/S).  Each block walks its K range
// starting at a block-dependent offset (wrapping around), so that the blocks
// running at the same time read different columns of the stacked weight
// instead of all hitting the same lines of L2.
__global__ void __launch_bounds__(THREADS, 1)
route_logits_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const Args g)
{
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES], acc_bar;
    __shared__ uint32_t tmem_base_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem0 = (ptx::smem_u32(dsmem) + 1023u) & ~1023u;
    const int tile = blockIdx.x / g.S, split = blockIdx.x - tile * g.S;
    const int t0 = tile * BM;
    const int kb0 = (int)((long long)split * g.nk / g.S), kb1 = (int)((long long)(split + 1) * g.nk / g.S);
    const int nkb = kb1 - kb0;
    const int rot = nkb > 0 ? (int)(((long long)tile * 5) % nkb) : 0;   // first K block of this block's walk

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
            for (int i = 0; i < nkb; ++i) {
                const int kb = kb0 + (i + rot) % nkb;
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
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(128, g.nb_rows);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
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
                                      (i > 0 || kk > 0) ? 1u : 0u);
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
        __syncwarp();
    } else {
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int t = t0 + r;
        const int Ep = g.E_pad;
        const bool waited = ptx::mbar_wait(ptx::smem_u32(&acc_bar), 0, limit);
        if (!__all_sync(0xffffffffu, waited)) moe_flag(MOE_DEV_TIMEOUT);
        ptx::tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
        float* row = g.part + ((size_t)split * g.T + t) * Ep;
        for (int e0 = 0; e0 < Ep; e0 += 16) {
            uint32_t a0[16], a1[16], a2[16];
            ptx::tmem_ld16(tb + e0, a0);
            ptx::tmem_ld16(tb + Ep + e0, a1);
            ptx::tmem_ld16(tb + 2 * Ep + e0, a2);
            ptx::tmem_ld_wait();
            if (t < g.T) {
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    float4 v;
                    v.x = (__uint_as_float(a0[i]) + __uint_as_float(a1[i])) + __uint_as_float(a2[i]);
                    v.y = (__uint_as_float(a0[i + 1]) + __uint_as_float(a1[i + 1])) + __uint_as_float(a2[i + 1]);
                    v.z = (__uint_as_float(a0[i + 2]) + __uint_as_float(a1[i + 2])) + __uint_as_float(a2[i + 2]);
                    v.w = (__uint_as_float(a0[i + 3]) + __uint_as_float(a1[i + 3])) + __uint_as_float(a2[i + 3]);
                    *reinterpret_cast<float4*>(row + e0 + i) = v;
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, g.tmem_cols);
    }
}

constexpr int FIN_THREADS = 256;   // warp-per-token finisher
constexpr int FIN_WARPS = FIN_THREADS / 32;
constexpr int LANE_THREADS = 64;   // lane-per-token finisher: small blocks spread few tokens over many SMs
constexpr int LANE_WARPS = LANE_THREADS / 32;

// Sum of the S partial logits of token t, expert e, in split order (four
// loads in flight at a time).
__device__ __forceinline__ float sum_splits(const float* __restrict__ part, int S, int T, int E_pad, int t, int e)
{
    const size_t plane = (size_t)T * E_pad;
    const float* p = part + (size_t)t * E_pad + e;
    float acc = __ldcg(p);
    for (int s0 = 1; s0 < S; s0 += 4) {
        float v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = s0 + u < S ? __ldcg(p + (size_t)(s0 + u) * plane) : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (s0 + u < S) acc += v[u];
    }
    return acc;
}

// Per-block probability sums (rows in warp order) -> psum[block].
template <int NW>
__device__ __forceinline__ void block_prob_sums(float (*red)[256], int E, float* __restrict__ psum)
{
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += NW * 32) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += red[w][e];
        psum[(size_t)blockIdx.x * E + e] = v;
    }
}

// prob_sum[e] = sum over the R block rows of psum[:, e]: one block per expert,
// a fixed-shape tree (strided fp64 partial sums, then a shared-memory tree).
__global__ void __launch_bounds__(256) prob_sum_kernel(const float* __restrict__ psum, int R, int E,
                                                       float* __restrict__ prob_sum)
{
    __shared__ double sh[256];
    const int e = blockIdx.x;
    double acc = 0.0;
    for (int b = threadIdx.x; b < R; b += 256) acc += (double)__ldg(psum + (size_t)b * E + e);
    sh[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) prob_sum[e] = (float)sh[0];
}

// E <= 32: one lane per token, its E logits in registers.
template <int EMAX, int KMAX>
__global__ void __launch_bounds__(LANE_THREADS)
route_finish_lane_kernel(const float* __restrict__ part, int S, int T, int E, int E_pad, int k, int renorm,
                         const float* __restrict__ bias, int32_t* __restrict__ idx_out,
                         float* __restrict__ gate_out, float* __restrict__ psum, RouteSel sel)
{
    __shared__ float red[LANE_WARPS][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float bia[EMAX], acc_p[EMAX];
    int grp[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        bia[e] = (bias && e < E) ? __ldg(bias + e) : 0.f;
        acc_p[e] = 0.f;
        grp[e] = e / sel.gsz;
    }
    for (int t = (blockIdx.x * LANE_WARPS + warp) * 32 + lane; t < T; t += gridDim.x * LANE_THREADS) {
        float l[EMAX];
        // this token's E_pad partial logits of split 0, then the other splits in order
#pragma unroll
        for (int e4 = 0; e4 < EMAX; e4 += 4) {
            const float4 a = e4 < E_pad ? __ldcg(reinterpret_cast<const float4*>(part + (size_t)t * E_pad + e4))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            l[e4] = a.x;
            l[e4 + 1] = a.y;
            l[e4 + 2] = a.z;
            l[e4 + 3] = a.w;
        }
        for (int sp = 1; sp < S; sp += 2) {   // two splits' loads in flight, added in split order
            const float* row = part + ((size_t)sp * T + t) * E_pad;
            const bool two = sp + 1 < S;
            float4 q[EMAX / 4], r[EMAX / 4];
#pragma unroll
            for (int e4 = 0; e4 < EMAX; e4 += 4) {
                const bool in = e4 < E_pad;
                q[e4 / 4] = in ? __ldcg(reinterpret_cast<const float4*>(row + e4)) : make_float4(0.f, 0.f, 0.f, 0.f);
                r[e4 / 4] = (in && two) ? __ldcg(reinterpret_cast<const float4*>(row + (size_t)T * E_pad + e4))
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int e4 = 0; e4 < EMAX; e4 += 4) {
                l[e4] += q[e4 / 4].x;
                l[e4 + 1] += q[e4 / 4].y;
                l[e4 + 2] += q[e4 / 4].z;
                l[e4 + 3] += q[e4 / 4].w;
                if (two) {
                    l[e4] += r[e4 / 4].x;
                    l[e4 + 1] += r[e4 / 4].y;
                    l[e4 + 2] += r[e4 / 4].z;
                    l[e4 + 3] += r[e4 / 4].w;
                }
            }
        }
        float tv[KMAX];
        int ti[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            tv[j] = -INFINITY;
            ti[j] = 0x7fffffff;
        }
#pragma unroll
        for (int e = 0; e < EMAX; ++e) l[e] = (e < E) ? l[e] + bia[e] : -INFINITY;
        // group-limited routing: keep the topk_group groups of largest max logit
        // (strict > scanning up the index keeps the lower group on ties)
        unsigned gkeep = 0xffffffffu;
        if (sel.n_group > 1) {
            gkeep = 0;
            for (int r = 0; r < sel.topk_group; ++r) {
                float bv = -INFINITY;
                int bg = -1;
#pragma unroll
                for (int e = 0; e < EMAX; ++e)
                    if (e < E && !((gkeep >> grp[e]) & 1u) && (bg < 0 || l[e] > bv)) {
                        bv = l[e];
                        bg = grp[e];
                    }
                if (bg >= 0) gkeep |= 1u << bg;
            }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            mx = fmaxf(mx, l[e]);
            if (e < E && ((gkeep >> grp[e]) & 1u)) {
                // insert into the descending top list; equal values keep the lower index ahead
                const float v = l[e];
                if (v > tv[KMAX - 1]) {
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
            }
        }
        float p[EMAX], s = 0.f;
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            p[e] = (e < E) ? expf(l[e] - mx) : 0.f;
            s += p[e];
        }
        if (sel.lse) sel.lse[t] = mx + logf(s);
        if (sel.logits) {
#pragma unroll
            for (int e = 0; e < EMAX; ++e)
                if (e < E) sel.logits[(size_t)t * E + e] = l[e];
        }
#pragma unroll
        for (int e = 0; e < EMAX; ++e) acc_p[e] += p[e] / s;
        float chosen = 0.f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            if (j < k) chosen += expf(tv[j] - mx) / s;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            if (j < k) {
                const float pj = expf(tv[j] - mx) / s;
                idx_out[(size_t)t * k + j] = ti[j];
                gate_out[(size_t)t * k + j] = renorm ? pj / chosen : pj;
            }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        float v = acc_p[e];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[warp][e] = v;
    }
    block_prob_sums<LANE_WARPS>(red, E, psum);
}

// Order-preserving map of a float onto uint32 (a < b  <=>  key(a) < key(b) for
// non-NaN values), so that one redux.sync finds a warp's maximum; key 0 lies
// below every float and marks "not selectable".
__device__ __forceinline__ unsigned fkey(float v)
{
    const unsigned u = __float_as_uint(v);
    return u ^ ((u & 0x80000000u) ? 0xffffffffu : 0x80000000u);
}
__device__ __forceinline__ float fkey_value(unsigned k)
{
    return __uint_as_float(k ^ ((k & 0x80000000u) ? 0x80000000u : 0xffffffffu));
}

// Sorts a lane's EPL (key, expert) pairs by key descending, expert ascending.
template <int EPL>
__device__ __forceinline__ void sort_lane(unsigned (&ck)[EPL], int (&ce)[EPL])
{
    auto cx = [&](int a, int b) {
        if (ck[b] > ck[a] || (ck[b] == ck[a] && ce[b] < ce[a])) {
            const unsigned tk = ck[a];
            ck[a] = ck[b];
            ck[b] = tk;
            const int te = ce[a];
            ce[a] = ce[b];
            ce[b] = te;
        }
    };
    if (EPL == 2) {
        cx(0, 1);
    } else if (EPL == 4) {
        cx(0, 1); cx(2, 3); cx(0, 2); cx(1, 3); cx(1, 2);
    } else if (EPL == 8) {   // Batcher's odd-even merge sort, 19 comparators
        cx(0, 1); cx(2, 3); cx(4, 5); cx(6, 7);
        cx(0, 2); cx(1, 3); cx(4, 6); cx(5, 7);
        cx(1, 2); cx(5, 6);
        cx(0, 4); cx(1, 5); cx(2, 6); cx(3, 7);
        cx(2, 4); cx(3, 5);
        cx(1, 2); cx(3, 4); cx(5, 6);
    }
}

// E > 32: one warp per token, lane l owns experts l, l+32, ...  The softmax
// maximum is one redux.sync over order-preserving keys.  For the top-k every
// lane sorts its EPL candidates (key descending, expert ascending); each of
// the k rounds takes the largest head key over the warp (redux max), then the
// lowest expert id among the lanes holding it (redux min: ties go to the
// lower index), and the winning lane drops its head.
template <int EPL>
__global__ void __launch_bounds__(FIN_THREADS, 4)
route_finish_warp_kernel(const float* __restrict__ part, int S, int T, int E, int E_pad, int k, int renorm,
                         const float* __restrict__ bias, int32_t* __restrict__ idx_out,
                         float* __restrict__ gate_out, float* __restrict__ psum, RouteSel sel)
{
    __shared__ float red[FIN_WARPS][256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float bia[EPL], acc_p[EPL];
    int grp[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        bia[i] = (bias && e < E) ? __ldg(bias + e) : 0.f;
        acc_p[i] = 0.f;
        grp[i] = e / sel.gsz;
    }
    for (int t = blockIdx.x * FIN_WARPS + warp; t < T; t += gridDim.x * FIN_WARPS) {
        float l[EPL];
        unsigned km = 0u;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            l[i] = (e < E) ? sum_splits(part, S, T, E_pad, t, e) + bia[i] : -INFINITY;
            km = max(km, fkey(l[i]));
        }
        const float mx = fkey_value(__reduce_max_sync(0xffffffffu, km));
        float p[EPL], s = 0.f;
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
        for (int i = 0; i < EPL; ++i) acc_p[i] += p[i] / s;
        const unsigned gkeep = keep_groups<EPL>(l, grp, E, sel, lane);
        unsigned ck[EPL];
        int ce[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            ce[i] = e;
            ck[i] = (e < E && ((gkeep >> grp[i]) & 1u)) ? fkey(l[i]) : 0u;
        }
        sort_lane<EPL>(ck, ce);
        int my_e = 0;
        float my_p = 0.f, chosen = 0.f;
        for (int j = 0; j < k; ++j) {
            const unsigned m = __reduce_max_sync(0xffffffffu, ck[0]);
            const unsigned w = __reduce_min_sync(0xffffffffu, ck[0] == m ? (unsigned)ce[0] : 0xffffffffu);
            const float pw = expf(fkey_value(m) - mx) / s;   // the winner's probability, as p[] above
            chosen += pw;
            if (lane == j) {
                my_e = (int)w;
                my_p = pw;
            }
            if ((unsigned)ce[0] == w) {   // the winning lane drops its head
#pragma unroll
                for (int i = 0; i + 1 < EPL; ++i) {
                    ck[i] = ck[i + 1];
                    ce[i] = ce[i + 1];
                }
                ck[EPL - 1] = 0u;
            }
        }
        if (lane < k) {
            idx_out[(size_t)t * k + lane] = my_e;
            gate_out[(size_t)t * k + lane] = renorm ? my_p / chosen : my_p;
        }
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) red[warp][lane + 32 * i] = acc_p[i];
    block_prob_sums<FIN_WARPS>(red, E, psum);
}

}  // namespace rtc
