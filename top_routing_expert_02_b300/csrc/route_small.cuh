// Router of bf16 x for few experts (E <= 8) on the CUDA cores, fused: logits,
// softmax, top-k and the per-block probability sums in one kernel.
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §1.1 / §2.1
// step 1 (a light linear layer scores the experts, each token keeps its
// Top-K); the deployment guide "细粒度专家并行部署实践与优化指南" §七 takes the top-k
// of the softmaxed gate probabilities.  Ties go to the lower expert index.
//
// Why CUDA cores.  With E <= 8 the router is 2·E flops per byte of x: far
// below what the tensor cores would need to matter, and the step is a read
// of x.  Plain per-thread copies (cp.async, 16 bytes per lane, a warp reading
// 512 contiguous bytes of one row) stream x without the weight split, the
// tensor-memory set-up and the column boxes of the tensor-core router.
//
// Work split.  A block has d / 8 threads; thread c owns the eight columns
// [8c, 8c + 8) of x and holds W[e][8c .. 8c + 7] for every expert in
// registers (fp32, loaded once).  The block owns tokens [b·tpc, (b+1)·tpc):
// each thread copies its 16 bytes of each token's row into a ring of RING
// token slots in shared memory (one cp.async group per token; a thread reads
// back only what it copied, so no barrier guards the ring) and, per token,
// forms E partial dot products over its eight columns (the even and the odd
// columns as two fp32 FMA chains in column order, issued as paired FMAs,
// then added).  Per pair of tokens the 16 partials are summed over the
// warp's 32 lanes by a transposing butterfly (each step halves the values
// per lane), and lane 2q holds the warp's sum for (token q / 8, expert q % 8).
// After the loop the warps' sums meet in shared memory: the logit of
// (token, e) is the sum over warps in warp order, plus the bias.  Four lanes
// per token then take the softmax and the top-k (rfu::finish_token), and the
// block writes its per-expert sums of p, which prob_sum_kernel adds in a
// fixed order.  A call gives the same bits every run.
//
// Numerics: x (bf16) is exact in fp32; each logit is a fixed tree of fp32
// sums of four-term FMA chains (d / 4 leaves), so its error is a few fp32
// units of the largest partial sums.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"
#include "route_fused.cuh"

namespace rsm {

constexpr int EMAX = 8;            // experts per token (W rows held per thread, zero-padded)
constexpr int CW = 8;              // columns per thread: one 16-byte vector of bf16
constexpr int RING = 16;           // token rows of x in flight per block
constexpr int NT = 2;              // tokens per butterfly
constexpr int MAX_THREADS = 512;   // d <= 4096
constexpr int TPC_MAX = 64;        // tokens per block

struct Args {
    const uint16_t* x;   // [T, d] bf16
    const float* W;      // [E, d]
    const float* bias;   // [E] or nullptr
    int T, d, E, k, renorm;
    int tpc;             // tokens per block
    int32_t* idx;        // [T, k]
    float* gate;         // [T, k]
    float* psum;         // [gridDim.x, E] per-block probability sums
    RouteSel sel;        // group-limited routing, lse and logits out
};

// Shared memory: the x ring [RING][d] bf16, then the warps' logit sums
// [warps][tpc][EMAX] fp32.
inline size_t smem_bytes(int d, int tpc)
{
    return (size_t)RING * d * 2 + (size_t)(d / 256) * tpc * EMAX * sizeof(float);
}

// Two fp32 values in one 64-bit register (low: first) and the paired FMA of
// sm_100-class SMs: each half is an ordinary fp32 fma (round to nearest).
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float sum2(uint64_t p)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
    return lo + hi;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// One butterfly step over lanes l and l ^ OFF: a lane keeps its first H
// values and adds the partner's second H.  The two lanes hold the halves in
// opposite order (see the lane layout below), so each ends with the sums of
// a different half.
template <int H, int OFF>
__device__ __forceinline__ void fold(float* v)
{
#pragma unroll
    for (int i = 0; i < H; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[H + i], OFF);
}

template <int KMAX>
__global__ void __launch_bounds__(MAX_THREADS, 1) route_small_kernel(const Args g)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = blockDim.x >> 5;
    const int d = g.d, E = g.E;
    const int t0 = blockIdx.x * g.tpc;
    const int n = min(g.tpc, g.T - t0);          // tokens of this block (>= 1)
    const uint32_t ring = ptx::smem_u32(smem);
    float* const red = reinterpret_cast<float*>(smem + (size_t)RING * d * 2);   // [nw][tpc][EMAX]
    // Lane layout of the 16 partials of a token pair, so that the butterfly
    // needs no selects: value slot jj * 8 + e of lane l belongs to token
    // jj ^ b4 of the pair and to expert e ^ em, em = 4 b3 + 2 b2 + b1 (b the
    // bits of l).  Lanes l and l ^ 16 hold the two tokens in opposite order,
    // lanes l and l ^ 8 / 4 / 2 the expert halves / quarters / pairs; after
    // the four halving steps lane l holds (token b4, expert em) -- slot q = l / 2.
    const int b4 = (lane >> 4) & 1, em = (lane >> 1) & 7;

    pdl_launch_dependents();   // prob_sum_kernel may launch; it waits for this grid
    pdl_wait();                // a programmatic dependent of the work before it (which may write x or W)

    // the first RING rows of the block's tokens into the ring, one group per token
    const uint16_t* xs = g.x + (size_t)t0 * d + tid * CW;
#pragma unroll 1
    for (int j = 0; j < RING; ++j) {
        if (j < n) ptx::cp_async_16(ring + (uint32_t)(j * d * 2 + tid * 16), xs + (size_t)j * d);
        ptx::cp_async_commit();
    }
    // this thread's eight columns of W as four (even, odd) column pairs, for
    // the experts in this lane's order (zero past E)
    uint64_t w[EMAX][CW / 2];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int ge = e ^ em;
        if (ge < E) {
            const float4* src = reinterpret_cast<const float4*>(g.W + (size_t)ge * d + tid * CW);
            const float4 a = __ldg(src), b = __ldg(src + 1);
            w[e][0] = pack2(a.x, a.y);
            w[e][1] = pack2(a.z, a.w);
            w[e][2] = pack2(b.x, b.y);
            w[e][3] = pack2(b.z, b.w);
        } else {
#pragma unroll
            for (int p = 0; p < CW / 2; ++p) w[e][p] = 0ull;
        }
    }

#pragma unroll 1
    for (int j0 = 0; j0 < n; j0 += NT) {
        // both tokens of the pair are the two oldest copy groups in flight
        ptx::cp_async_wait<RING - NT>();
        float v[NT * EMAX];
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) {
            const int j = j0 + (jj ^ b4);        // this lane's token for value slots jj * 8 ..
            uint64_t xp[CW / 2];                 // (even, odd) column pairs of x, exact in fp32
            if (j < n) {
                const uint4 q = ptx::ld_shared_v4(ring + (uint32_t)((j % RING) * d * 2 + tid * 16));
                const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) xp[m] = pack2(__uint_as_float(wd[m] << 16), __uint_as_float(wd[m] & 0xffff0000u));
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m) xp[m] = 0ull;
            }
            // per expert: the even and the odd columns as two FMA chains, then their sum
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                uint64_t a = fma2(xp[0], w[e][0], 0ull);
#pragma unroll
                for (int m = 1; m < CW / 2; ++m) a = fma2(xp[m], w[e][m], a);
                v[jj * EMAX + e] = sum2(a);
            }
        }
        // refill the pair's slots RING tokens ahead; the warp barrier orders
        // this thread's reads of the slots before the copies that overwrite them
        __syncwarp();
#pragma unroll
        for (int jj = 0; jj < NT; ++jj) {
            const int j = j0 + jj;
            if (j + RING < n)
                ptx::cp_async_16(ring + (uint32_t)((j % RING) * d * 2 + tid * 16), xs + (size_t)(j + RING) * d);
            ptx::cp_async_commit();
        }
        // the warp's sums: four halving steps, then the pair (l, l ^ 1); lane
        // 2q holds (token q / 8, expert q % 8) of the pair
        fold<8, 16>(v);
        fold<4, 8>(v);
        fold<2, 4>(v);
        fold<1, 2>(v);
        const float other = __shfl_xor_sync(0xffffffffu, v[0], 1);
        if ((lane & 1) == 0) {
            const int q = lane >> 1;
            const int jj = q / EMAX, e = q % EMAX;
            if (j0 + jj < n) red[((size_t)warp * g.tpc + j0 + jj) * EMAX + e] = v[0] + other;
        }
    }
    ptx::cp_async_wait<0>();
    __syncthreads();

    // softmax / top-k of the block's tokens, four lanes per token (eight per warp)
    constexpr int G = 4, EPL = EMAX / G;
    const int sub = lane & (G - 1);
    for (int base = warp * (32 / G); base < n; base += nw * (32 / G)) {
        const int tau = base + lane / G;
        const bool valid = tau < n;
        const int t = t0 + (valid ? tau : 0);
        float l[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = sub + G * i;
            float s = 0.f;
            if (valid && e < E) {
                for (int ww = 0; ww < nw; ++ww) s += red[((size_t)ww * g.tpc + tau) * EMAX + e];
                s += g.bias ? __ldg(g.bias + e) : 0.f;
                if (g.sel.logits) g.sel.logits[(size_t)t * E + e] = s;
            }
            l[i] = s;
        }
        rfu::finish_token<G, EPL, KMAX>(l, sub, E, g.k, g.renorm, valid, t, g.sel, g.idx, g.gate);
        // p back into warp 0's row of the token (read above only by these lanes)
        if (valid) {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (sub + G * i < E) red[(size_t)tau * EMAX + sub + G * i] = l[i];
        }
    }
    __syncthreads();
    // this block's per-expert sums of p, in token order
    if (tid < E) g.psum[(size_t)blockIdx.x * E + tid] = rfu::column_sum(red, n, EMAX, tid);
}

}  // namespace rsm
