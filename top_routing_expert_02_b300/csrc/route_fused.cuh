// Router of bf16 x on the tensor cores, fused: logits, softmax, top-k and the
// per-CTA probability sums in one kernel.
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §1.1 / §2.1
// step 1 (a light linear layer scores the experts, each token keeps its
// Top-K); the deployment guide "细粒度专家并行部署实践与优化指南" §七 takes the top-k
// of the softmaxed gate probabilities.  Ties go to the lower expert index.
//
// Arithmetic.  The fp32 router weight is split exactly into three bf16 parts,
// W = W0 + W1 + W2 (each part holds the next 8 significant bits; both
// differences are exact in fp32).  x is bf16, so every product x*Wi is exact
// and the logits keep fp32 accuracy at tensor-core speed.  The tensor core's
// fp32 accumulator loses up to about one unit in the last place of the
// running sum per MMA, always in the same direction, so over all of d the
// error of the W0 sum would grow linearly with d.  The W0 accumulator is
// therefore cut into chunks of KC K blocks (KC*64 columns): two TMEM buffers
// alternate, and while the MMAs fill one, the other is added (fp32, round to
// nearest) into a running W0 sum kept in TMEM.  W1 and W2 (about 2^-8 and
// 2^-16 of the size) share one accumulator over the whole range: its error
// is relative to its own small size.
//
// The split runs once per call (split_weight_kernel, into the workspace);
// the router kernel is launched as its programmatic dependent, so its set-up
// and the first x tiles overlap the split, and only the weight loads wait
// for it.
//
// Work split.  A CTA owns TPB 128-token tiles (TPB = 2 while the TMEM columns
// allow, so each weight block serves 256 tokens); a cluster of S CTAs shares
// them (S > 1 splits d when there are too few tiles to fill the GPU): CTA s
// covers K blocks [s*nk/S, (s+1)*nk/S).  Each CTA has 7 warps:
//   warp 0      TMA producer of the x ring: per K block the TPB x tiles (128
//               tokens x 64 columns each), as many blocks ahead as the ring
//               holds (x comes from HBM: the ring is deep)
//   warp 6      TMA producer of the weight ring: the three stacked parts (3
//               E_pad rows x 64) per K block (they stay in L2: a short ring)
//   warp 1      TMEM allocation and the single thread issuing tcgen05.mma
//               (M = 128 tokens, K = 16 per instruction)
//   warps 2-5   add each finished chunk into an fp32 sum (in TMEM, or in
//               registers); at the end, the partial logits of the tiles'
//               rows (thread = TMEM lane = token row)
// Two accumulator layouts.  E_pad <= 32 (FUSED_PARTS): one MMA per tile and
// K step covers all three parts (N = 3 E_pad), so each x tile is read once
// per step; TMEM per tile [chunk buffer 0 (3 E_pad) | chunk buffer 1 (3 E_pad)
// | sum (E_pad)], and a chunk adds W0 + (W1 + W2) into the sum.  Larger
// E_pad: W0 (N = E_pad) into a chunk buffer and W1, W2 together (N = 2 E_pad)
// into their own columns, TMEM per tile [W0 chunk buffer 0 | W0 chunk buffer
// 1 | W1 | W2], E_pad each, the W0 sum in the accumulator warps' registers;
// two tiles fit up to E_pad = 64 (they share each weight block, halving its
// traffic).
// The partial logits of the S CTAs meet in shared memory: CTA s takes tokens
// [s*TPC, (s+1)*TPC), TPC = 128*TPB/S; every CTA pushes the rows of those
// tokens to CTA s with one bulk copy into its shared memory (distributed
// shared memory, completion counted on CTA s's mbarrier), and CTA s adds the
// S partial logits in split order plus the bias.  For E <= 64 it then takes
// the softmax, the top-k and its per-expert sums of p itself (finish_token:
// four lanes per token); for larger E it writes the fp32 logits and
// route_finish_kernel (a programmatic dependent, many blocks per SM to hide
// the latency of the longer per-token chains) does that.  For E <= 64 each
// CTA adds its probability sums into 64-bit fixed-point accumulators and the
// CTA that finishes last writes prob_sum (integer adds: the bits do not
// depend on the order); for larger E prob_sum_kernel adds the per-block rows
// in a fixed order.  A call gives the same bits every run.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"

namespace rfu {

constexpr int BM = 128, BK = 64;
constexpr int THREADS = 224;
constexpr int WARPS = THREADS / 32;
constexpr int MAX_XSTAGES = 12;             // x ring
constexpr int MAX_WSTAGES = 12;             // weight-part ring
constexpr int KC = 4;                       // K blocks per W0 accumulator chunk
constexpr int X_BYTES = BM * BK * 2;        // one x tile, 16 KB
constexpr int MAX_EPAD = 128;               // 4 * E_pad TMEM columns <= 512
constexpr int MAX_SPLITS = 4;               // cluster size (larger clusters of one-SM CTAs may not all fit at once)
constexpr int ACC_THREADS = 128;            // warps 2-5

struct Args {
    int T, d, E, E_pad, k, renorm;
    int nk;             // K blocks of 64 over d
    int S;              // CTAs per token group (cluster size)
    int TPB;            // 128-token tiles per CTA (1 or 2)
    int xstages;        // x ring: TPB tiles of 16 KB per stage
    int wstages;        // weight ring: 3 E_pad x 64 bf16 per stage
    uint32_t tmem_cols;
    const float* bias;  // [E] or nullptr
    int32_t* idx;       // [T, k]              (E <= 64: finished in this kernel)
    float* gate;        // [T, k]
    float* psum;        // [gridDim.x, E]      per-CTA probability sums
    RouteSel sel;       // group-limited routing, lse and logits out
    float* logits;      // [T, E] fp32 out (E > 64): the logits for route_finish_kernel
    // E <= 64: the per-CTA probability sums go into E 64-bit fixed-point
    // accumulators (zeroed by the split kernel, like the count of CTAs done);
    // the CTA that counts itself in last writes prob_sum
    unsigned long long* psum_fx;
    unsigned* done;
    float* prob_sum;
    unsigned long long wait_limit;
};
// Fixed-point scale of the probability-sum accumulators: integer adds are
// exact and associative, so the result does not depend on which CTA adds
// first; per CTA the rounding error is at most 2^-33, and T * 2^32 < 2^63.
constexpr double PSUM_FX_SCALE = 4294967296.0;

// Arguments of the finishing kernel.
struct FinArgs {
    int T, E, k, renorm;
    const float* logits;  // [T, E]
    int32_t* idx;         // [T, k]
    float* gate;          // [T, k]
    float* psum;          // [gridDim.x, E]: per-block probability sums
    RouteSel sel;         // group-limited routing, lse out (its logits pointer is unused here)
};

// Shared memory after the main loop (reusing the stage ring): the partial
// logits of the CTA's rows, [TPB * 128][E_pad + 4]; the rows the other CTAs
// of the cluster push for the tokens this CTA finishes, [S][TPC][E_pad + 4]
// (the same size).  Rows are RPITCH = E_pad + 4 floats long (4 times an odd
// number, since E_pad is a multiple of 16): the accumulator threads write
// their rows with 16-byte stores (eight lanes per 128 bytes hit eight
// different 16-byte bank groups), the finishing lanes read with a stride of
// four floats (the four lanes of eight tokens hit 32 different banks), and a
// thread per expert summing a column hits its own bank.
__host__ __device__ constexpr int rpitch(int E_pad) { return E_pad + 4; }
__host__ __device__ constexpr int red_bytes(int TPB, int E_pad) { return TPB * BM * rpitch(E_pad) * 4; }
__host__ __device__ constexpr int finish_smem_bytes(int TPB, int E_pad) { return 2 * red_bytes(TPB, E_pad); }
// TMEM columns of one 128-token tile in the two accumulator layouts.
__host__ __device__ constexpr int tile_tmem_cols(bool fused_parts, int E_pad) { return fused_parts ? 7 * E_pad : 4 * E_pad; }

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to the
// shared memory of a CTA of the cluster (dst and bar: shared::cluster
// addresses); completion is counted in bytes on that CTA's mbarrier.
__device__ __forceinline__ void bulk_push(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// W (fp32 [E, d]) -> stacked bf16 [3*E_pad, d]: rows [0,E_pad) W0, [E_pad,2E_pad) W1,
// [2E_pad,3E_pad) W2; rows of experts >= E are zero.  W0 = rn(W), W1 = rn(W - W0),
// W2 = rn(W - W0 - W1); both differences are exact in fp32.  Eight columns per thread.
// It also zeroes the fixed-point probability-sum accumulators of the call.
__global__ void __launch_bounds__(256) split_weight_kernel(const float* __restrict__ W, int E, int E_pad, int d,
                                                           uint4* __restrict__ Ws, unsigned long long* __restrict__ psum_fx,
                                                           unsigned* __restrict__ done)
{
    pdl_launch_dependents();
    // the router's probability-sum accumulators and its count of finished CTAs
    // (every later kernel of the call starts its use of them after this grid)
    if (psum_fx && blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) psum_fx[e] = 0ull;
        if (threadIdx.x == 0) *done = 0u;
    }
    const int d8 = d / 8;
    const long long n8 = (long long)E_pad * d8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const int e = (int)(i / d8);
        float w[8];
        if (e < E) {
            const float4* src = reinterpret_cast<const float4*>(W) + 2 * i;   // row e, columns 8 (i - e d8) ..
            const float4 a = __ldg(src), b = __ldg(src + 1);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) w[u] = 0.f;
        }
        uint32_t h0[4], h1[4], h2[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float q0[2], q1[2], q2[2];
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const float x = w[2 * u + v];
                q0[v] = __bfloat162float(__float2bfloat16_rn(x));
                const float r1 = x - q0[v];
                q1[v] = __bfloat162float(__float2bfloat16_rn(r1));
                q2[v] = r1 - q1[v];
            }
            h0[u] = pack_bf16x2(q0[0], q0[1]);   // exact: q0 and q1 are bf16 values
            h1[u] = pack_bf16x2(q1[0], q1[1]);
            h2[u] = pack_bf16x2(q2[0], q2[1]);   // the rounding of the last residual
        }
        Ws[i] = make_uint4(h0[0], h0[1], h0[2], h0[3]);
        Ws[n8 + i] = make_uint4(h1[0], h1[1], h1[2], h1[3]);
        Ws[2 * n8 + i] = make_uint4(h2[0], h2[1], h2[2], h2[3]);
    }
}

// FUSED_PARTS: chunk `buf` (W0 + (W1 + W2) from its three part blocks) of the
// tile whose TMEM columns start at tb added into that tile's sum at column
// 6 E_pad (or copied, for the first chunk), by one accumulator warp (its 32
// TMEM lanes).
__device__ __forceinline__ void drain_chunk_fp(uint32_t tb, int Ep, int buf, bool first)
{
    const uint32_t sum_col = (uint32_t)(6 * Ep), buf_col = (uint32_t)(buf * 3 * Ep);
    for (int e0 = 0; e0 < Ep; e0 += 16) {
        uint32_t v[16], v1[16], v2[16], a[16];
        ptx::tmem_ld16(tb + buf_col + (uint32_t)e0, v);
        ptx::tmem_ld16(tb + buf_col + (uint32_t)(Ep + e0), v1);
        ptx::tmem_ld16(tb + buf_col + (uint32_t)(2 * Ep + e0), v2);
        if (!first) ptx::tmem_ld16(tb + sum_col + (uint32_t)e0, a);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const float c = __uint_as_float(v[u]) + (__uint_as_float(v1[u]) + __uint_as_float(v2[u]));
            v[u] = __float_as_uint(first ? c : __uint_as_float(a[u]) + c);
        }
        ptx::tmem_st16(tb + sum_col + (uint32_t)e0, v);
    }
    ptx::tmem_st_wait();
}

// Softmax and top-k of one token held by a group of four lanes (xor-1 and
// xor-2 shuffles stay inside the group): lane sub holds the logits of experts
// sub, sub + 4, ... in l[] (entries past E unused).  The maximum and the
// softmax sum combine over the four lanes in a fixed order; each lane sorts
// its candidates (logit desc, index asc) and k rounds of a four-lane argmax
// of the list heads give the winners, in order.  On return l[] holds p
// (softmax probabilities); lane 0 of a valid token has written idx, gate and
// lse.  Every lane of the warp must call it (shuffles).  The exponentials use
// the hardware approximation (__expf): its relative error on arguments in
// [-30, 0] is a few units in the last place, far inside the 1e-5 bar of the
// gates and probability sums, and the top-k decision uses the logits alone.
template <int G, int EPL, int KMAX>
__device__ __forceinline__ void finish_token(float (&l)[EPL], int sub, int E, int k, int renorm, bool valid, int t,
                                             const RouteSel& sel, int32_t* __restrict__ idx_out,
                                             float* __restrict__ gate_out)
{
    static_assert(G == 4 || G == 8 || G == 16, "G consecutive lanes share a token");
    const bool grouped = sel.n_group > 1;
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        if (sub + G * i < E) mx = fmaxf(mx, l[i]);
#pragma unroll
    for (int o = 1; o < G; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // group-limited routing: keep the topk_group groups holding the best
    // remaining logit, ordered by (logit desc, expert asc)
    unsigned gkeep = 0xffffffffu;
    if (grouped) {
        gkeep = 0;
        for (int rr = 0; rr < sel.topk_group; ++rr) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = sub + G * i;
                if (e < E && !((gkeep >> (e / sel.gsz)) & 1u) && (l[i] > bv || (l[i] == bv && e < bi))) {
                    bv = l[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 1; o < G; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (bi < E) gkeep |= 1u << (bi / sel.gsz);
        }
    }
    // this lane's candidates, sorted: descending, an equal value keeps the
    // lower expert ahead (experts ascend with i)
    float tv[KMAX];
    int ti[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        tv[j] = -INFINITY;
        ti[j] = 0x7fffffff;
    }
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = sub + G * i;
        const float v = l[i];
        if (e < E && v > tv[KMAX - 1] && (!grouped || ((gkeep >> (e / sel.gsz)) & 1u))) {
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
    // softmax over all E: this lane's terms in expert order, then the G
    // lanes' sums in a fixed butterfly
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        if (sub + G * i < E) {
            l[i] = __expf(l[i] - mx);
            s += l[i];
        }
#pragma unroll
    for (int o = 1; o < G; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.f / s;
    if (valid && sel.lse && sub == 0) sel.lse[t] = mx + logf(s);
#pragma unroll
    for (int i = 0; i < EPL; ++i) l[i] *= inv;
    // the k winners: each round the best list head of the G lanes (logit
    // desc, expert asc); the lane holding it drops it
    int widx[KMAX];
    float wp[KMAX];
    float chosen = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
            float bv = tv[0];
            int bi = ti[0];
#pragma unroll
            for (int o = 1; o < G; o <<= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (ti[0] == bi) {
#pragma unroll
                for (int u = 0; u + 1 < KMAX; ++u) {
                    tv[u] = tv[u + 1];
                    ti[u] = ti[u + 1];
                }
                tv[KMAX - 1] = -INFINITY;
                ti[KMAX - 1] = 0x7fffffff;
            }
            wp[j] = __expf(bv - mx) * inv;   // the winner's probability, as in l[]
            widx[j] = bi;
            chosen += wp[j];
        }
    }
    if (valid && sub == 0) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            if (j < k) {
                idx_out[(size_t)t * k + j] = widx[j];
                gate_out[(size_t)t * k + j] = renorm ? wp[j] / chosen : wp[j];
            }
    }
}

// Per-expert sums of p over `n` rows (pitch P floats) of shared memory: eight
// interleaved partial sums in row order, combined in a fixed order.
__device__ __forceinline__ float column_sum(const float* rows, int n, int P, int e)
{
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    int r = 0;
    for (; r + 8 <= n; r += 8) {
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] += rows[(size_t)(r + u) * P + e];
    }
    for (; r < n; ++r) acc[0] += rows[(size_t)r * P + e];
    return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

template <int EMAX, int KMAX>
__global__ void __launch_bounds__(THREADS, 1)
route_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const Args g)
{
    constexpr bool FP = EMAX <= 32;
    constexpr bool FINISH_HERE = EMAX <= 64;   // larger E: route_finish_kernel, at higher occupancy
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t xfull[MAX_XSTAGES], xempty[MAX_XSTAGES], wfull[MAX_WSTAGES], wempty[MAX_WSTAGES];
    __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2], fin_bar, recv_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ float bias_sh[MAX_EPAD];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem0 = (ptx::smem_u32(dsmem) + 1023u) & ~1023u;
    uint8_t* const gsmem = dsmem + (smem0 - ptx::smem_u32(dsmem));
    const int S = g.S, TPB = g.TPB;
    const int group = blockIdx.x / S, split = blockIdx.x - group * S;
    const int row0 = group * TPB * BM;          // first token of this CTA's tiles
    const int kb0 = (int)((long long)split * g.nk / S), kb1 = (int)((long long)(split + 1) * g.nk / S);
    const int nkb = kb1 - kb0;
    const int rot = nkb > 0 ? group % nkb : 0;   // staggered walk: concurrent groups read different W columns
    const int nch = (nkb + KC - 1) / KC;
    const int Ep = g.E_pad, P = rpitch(Ep);
    const uint32_t tile_cols = (uint32_t)tile_tmem_cols(FP, Ep);
    const uint64_t limit = g.wait_limit;
    const int TPC = TPB * BM / S;                 // tokens this CTA finishes
    const uint32_t slice_bytes = (uint32_t)(TPC * P * 4);   // one CTA's partial rows of them
    const uint32_t xstage_bytes = (uint32_t)(TPB * X_BYTES), wstage_bytes = (uint32_t)(3 * Ep * 128);
    const uint32_t wring = smem0 + (uint32_t)g.xstages * xstage_bytes;   // weight ring after the x ring
    // x fills issued by the x producer before the block-wide barrier below
    const int xpre = nkb < g.xstages ? nkb : g.xstages;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < g.xstages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&xfull[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&xempty[s]), 1);
        }
        for (int s = 0; s < g.wstages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&wfull[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&wempty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&accf_bar[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&acce_bar[b]), ACC_THREADS);
        }
        ptx::mbar_init(ptx::smem_u32(&fin_bar), 1);
        ptx::mbar_init(ptx::smem_u32(&recv_bar), 1);
        ptx::fence_mbar_init();
        // the other S-1 CTAs push their partial rows of this CTA's tokens
        if (S > 1) ptx::mbar_arrive_expect_tx(ptx::smem_u32(&recv_bar), (uint32_t)(S - 1) * slice_bytes);
        ptx::tma_prefetch_desc(&tmX);
        ptx::tma_prefetch_desc(&tmW);
        // the first pass of the x ring needs no free slot: it starts here, while
        // the other warps allocate TMEM and load the bias
        int kb = kb0 + rot;
        for (int i = 0; i < xpre; ++i) {
            const uint32_t fb = ptx::smem_u32(&xfull[i]);
            const uint32_t dst = smem0 + (uint32_t)i * xstage_bytes;
            ptx::mbar_arrive_expect_tx(fb, xstage_bytes);
            ptx::tma_load_2d(dst, &tmX, fb, kb * BK, row0);
            if (TPB > 1) ptx::tma_load_2d(dst + X_BYTES, &tmX, fb, kb * BK, row0 + BM);
            if (++kb == kb1) kb = kb0;
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), g.tmem_cols);
        ptx::tmem_relinquish();
    }
    for (int e = threadIdx.x; e < Ep; e += THREADS) bias_sh[e] = (g.bias && e < g.E) ? __ldg(g.bias + e) : 0.f;
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;
    // the stacked parts [W0; W1; W2] of a K block: one box of 3 E_pad rows when
    // that is at most 256 rows, else one box per part
    const bool w_one_box = 3 * Ep <= 256;

    if (warp == 0 || warp == 6) {
        // ------------------------------------------------ TMA producers: x ring (warp 0), weight ring (warp 6)
        if (lane == 0) {
            const bool xring = warp == 0;
            const int nst = xring ? g.xstages : g.wstages;
            uint64_t* full = xring ? xfull : wfull;
            uint64_t* empty = xring ? xempty : wempty;
            const uint32_t sbytes = xring ? xstage_bytes : wstage_bytes;
            const uint32_t base = xring ? smem0 : wring;
            // the x ring fills before the weight split has finished; the
            // weight producer waits for it (programmatic dependent launch)
            if (!xring) pdl_wait();
            const int i0 = xring ? xpre : 0;       // the x ring's first fills went out before the barrier
            int stage = i0 % nst;
            uint32_t phase = (uint32_t)((i0 / nst) & 1);
            int fills = i0;
            bool ok = true;
            int kb = kb0 + (rot + i0) % (nkb > 0 ? nkb : 1);   // K blocks walked from kb0 + rot, wrapping at kb1
            for (int i = i0; i < nkb; ++i) {
                if (!ptx::mbar_wait(ptx::smem_u32(&empty[stage]), phase ^ 1u, limit)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = ptx::smem_u32(&full[stage]);
                const uint32_t dst = base + (uint32_t)stage * sbytes;
                ptx::mbar_arrive_expect_tx(fb, sbytes);
                if (xring) {
                    ptx::tma_load_2d(dst, &tmX, fb, kb * BK, row0);
                    if (TPB > 1) ptx::tma_load_2d(dst + X_BYTES, &tmX, fb, kb * BK, row0 + BM);
                } else if (w_one_box) {
                    ptx::tma_load_2d(dst, &tmW, fb, kb * BK, 0);
                } else {
                    for (int p = 0; p < 3; ++p) ptx::tma_load_2d(dst + p * Ep * 128, &tmW, fb, kb * BK, p * Ep);
                }
                ++fills;
                if (++kb == kb1) kb = kb0;
                if (++stage == nst) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            // the last stages' copies must have landed before shared memory is reused or freed
            for (int f = fills - 1; f >= 0 && f >= fills - nst; --f) {
                if (!ptx::mbar_wait(ptx::smem_u32(&full[f % nst]), (uint32_t)((f / nst) & 1), limit)) {
                    moe_flag(MOE_DEV_TIMEOUT);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            // FUSED_PARTS: one MMA (N = 3 E_pad) per tile and K step into the
            // chunk buffer; otherwise W0 (N = E_pad) into its chunk buffer and
            // W1, W2 together (N = 2 E_pad, rows E_pad .. 3 E_pad of the weight
            // block) into their own columns.  Descriptors advance by adding
            // byte offsets / 16 to the start-address field.
            const uint32_t idesc_a = ptx::idesc_bf16_f32(BM, FP ? 3 * Ep : Ep);
            const uint32_t idesc_b = ptx::idesc_bf16_f32(BM, 2 * Ep);
            const uint64_t xd0 = ptx::sdesc_kmajor_sw128(smem0), wd0 = ptx::sdesc_kmajor_sw128(wring);
            const uint64_t w12_off = (uint64_t)(Ep * 128) >> 4;
            int xs = 0, ws = 0;
            uint32_t xph = 0, wph = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
                const int c = i / KC, buf = c & 1;
                const bool first = (i % KC) == 0;
                // chunk c reuses the buffer of chunk c-2: wait until that one was added in
                if (first && c >= 2 &&
                    !ptx::mbar_wait(ptx::smem_u32(&acce_bar[buf]), (uint32_t)((c / 2 - 1) & 1), limit)) {
                    ok = false;
                    break;
                }
                if (!ptx::mbar_wait(ptx::smem_u32(&xfull[xs]), xph, limit) ||
                    !ptx::mbar_wait(ptx::smem_u32(&wfull[ws]), wph, limit)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t ad = xd0 + (((uint64_t)xs * xstage_bytes) >> 4);
                const uint64_t bd = wd0 + (((uint64_t)ws * wstage_bytes) >> 4);
                const uint32_t c0 = tmem_base + (uint32_t)(buf * (FP ? 3 : 1) * Ep);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
                    for (int tt = 0; tt < 2; ++tt) {
                        if (tt < TPB) {
                            const uint64_t a = ad + (uint64_t)((tt * X_BYTES + kk * 32) >> 4);
                            const uint64_t b = bd + (uint64_t)((kk * 32) >> 4);
                            const uint32_t toff = (uint32_t)tt * tile_cols;
                            ptx::mma_bf16(c0 + toff, a, b, idesc_a, (!first || kk > 0) ? 1u : 0u);
                            if (!FP)
                                ptx::mma_bf16(tmem_base + toff + (uint32_t)(2 * Ep), a, b + w12_off, idesc_b,
                                              (i > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                }
                ptx::mma_commit(ptx::smem_u32(&xempty[xs]));
                ptx::mma_commit(ptx::smem_u32(&wempty[ws]));
                const bool last = (i % KC) == KC - 1 || i == nkb - 1;
                if (last && c < nch - 1) ptx::mma_commit(ptx::smem_u32(&accf_bar[buf]));
                if (++xs == g.xstages) {
                    xs = 0;
                    xph ^= 1u;
                }
                if (++ws == g.wstages) {
                    ws = 0;
                    wph ^= 1u;
                }
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            // arrives once every MMA issued above has completed (also on the error path)
            ptx::mma_commit(ptx::smem_u32(&fin_bar));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ warps 2-5: chunk sums, partial logits
        const int q = warp & 3;                    // TMEM lanes 32q .. 32q+31
        const int r = q * 32 + lane;               // token row of each tile
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
        // one CTA owns at most two tiles, and only when E_pad <= 64
        constexpr int TMAX = EMAX <= 64 ? 2 : 1;
        constexpr int SR = FP ? 1 : EMAX;          // the W0 sum lives in registers when not FUSED_PARTS
        float sumr[TMAX][SR];
#pragma unroll
        for (int tt = 0; tt < TMAX; ++tt)
#pragma unroll
            for (int e = 0; e < SR; ++e) sumr[tt][e] = 0.f;
        bool ok = true;
        for (int c = 0; c + 1 < nch; ++c) {        // every chunk but the last into the sum
            const int buf = c & 1;
            const bool w = ptx::mbar_wait(ptx::smem_u32(&accf_bar[buf]), (uint32_t)((c >> 1) & 1), limit);
            if (!__all_sync(0xffffffffu, w)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int tt = 0; tt < TMAX; ++tt) {
                if (tt < TPB) {
                    const uint32_t tt_b = tb + (uint32_t)tt * tile_cols;
                    if (FP) {
                        drain_chunk_fp(tt_b, Ep, buf, c == 0);
                    } else {
#pragma unroll
                        for (int e0 = 0; e0 < SR; e0 += 16) {
                            if (e0 < Ep) {
                                uint32_t v[16];
                                ptx::tmem_ld16(tt_b + (uint32_t)(buf * Ep + e0), v);
                                ptx::tmem_ld_wait();
#pragma unroll
                                for (int u = 0; u < 16; ++u) sumr[tt][e0 + u] += __uint_as_float(v[u]);
                            }
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&acce_bar[buf]));
        }
        if (!ok) moe_flag(MOE_DEV_TIMEOUT);
        const bool fin = ptx::mbar_wait(ptx::smem_u32(&fin_bar), 0, limit);
        if (!__all_sync(0xffffffffu, fin)) moe_flag(MOE_DEV_TIMEOUT);
        ptx::tc_fence_after();
        // partial logits: (sum of the earlier chunks + the last chunk), and in
        // the per-part layout + (W1 + W2) accumulated over the whole range
        const int lb = (nch - 1) & 1;
#pragma unroll
        for (int tt = 0; tt < TMAX; ++tt) {
            if (tt < TPB) {
                const uint32_t tt_b = tb + (uint32_t)tt * tile_cols;
                float* red = reinterpret_cast<float*>(gsmem) + (size_t)(tt * BM + r) * P;
                if (FP) {
                    for (int e0 = 0; e0 < Ep; e0 += 16) {
                        uint32_t a0[16], a1[16], a2[16], as[16];
                        ptx::tmem_ld16(tt_b + (uint32_t)(lb * 3 * Ep + e0), a0);
                        ptx::tmem_ld16(tt_b + (uint32_t)(lb * 3 * Ep + Ep + e0), a1);
                        ptx::tmem_ld16(tt_b + (uint32_t)(lb * 3 * Ep + 2 * Ep + e0), a2);
                        if (nch >= 2) ptx::tmem_ld16(tt_b + (uint32_t)(6 * Ep + e0), as);
                        ptx::tmem_ld_wait();
                        float o[16];
#pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const float chunk = __uint_as_float(a0[u]) + (__uint_as_float(a1[u]) + __uint_as_float(a2[u]));
                            o[u] = nch >= 2 ? __uint_as_float(as[u]) + chunk : chunk;
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            reinterpret_cast<float4*>(red + e0)[u] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
                    }
                } else {
#pragma unroll
                    for (int e0 = 0; e0 < SR; e0 += 16) {
                        if (e0 < Ep) {
                            uint32_t a0[16], a1[16], a2[16];
                            ptx::tmem_ld16(tt_b + (uint32_t)(lb * Ep + e0), a0);
                            ptx::tmem_ld16(tt_b + (uint32_t)(2 * Ep + e0), a1);
                            ptx::tmem_ld16(tt_b + (uint32_t)(3 * Ep + e0), a2);
                            ptx::tmem_ld_wait();
                            float o[16];
#pragma unroll
                            for (int u = 0; u < 16; ++u) {
                                const float w0 = nch >= 2 ? sumr[tt][e0 + u] + __uint_as_float(a0[u]) : __uint_as_float(a0[u]);
                                o[u] = w0 + (__uint_as_float(a1[u]) + __uint_as_float(a2[u]));
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u)
                                reinterpret_cast<float4*>(red + e0)[u] =
                                    make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
                        }
                    }
                }
            }
        }
    }

    pdl_launch_dependents();   // the finishing kernel may launch; it waits for this grid's results
    // every CTA of the cluster has its partial rows in shared memory (the
    // proxy fence makes them visible to the bulk copies)
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    if (S > 1) ptx2::cluster_sync();
    else __syncthreads();

    // ---------------------------------------------------- exchange the partial rows, write the logits
    const int E = g.E;
    const int tbase = split * TPC;                // first token this CTA finishes, counted from row0
    const uint32_t recv0 = smem0 + (uint32_t)red_bytes(TPB, Ep);   // [S][TPC][P]
    if (S > 1 && threadIdx.x == 0) {
        for (int j = 0; j < S; ++j)
            if (j != split)
                bulk_push(ptx2::mapa(recv0 + (uint32_t)split * slice_bytes, (uint32_t)j),
                          smem0 + (uint32_t)j * slice_bytes, slice_bytes,
                          ptx2::mapa(ptx::smem_u32(&recv_bar), (uint32_t)j));
    }
    if (S > 1) {
        const bool w = ptx::mbar_wait(ptx::smem_u32(&recv_bar), 0, limit);
        if (!__all_sync(0xffffffffu, w)) moe_flag(MOE_DEV_TIMEOUT);
    }
    float* const red = reinterpret_cast<float*>(gsmem);
    const float* const recv = reinterpret_cast<const float*>(gsmem + red_bytes(TPB, Ep));
    if constexpr (FINISH_HERE) {
        // softmax / top-k of this CTA's tokens right here, four lanes per token
        // (eight tokens per warp); p goes back into the token's own row
        constexpr int G = 4, EPL = EMAX / G;
        const int sub = lane & (G - 1);
        for (int base = warp * (32 / G); base < TPC; base += WARPS * (32 / G)) {
            const int tau = base + lane / G;
            const int t = row0 + tbase + tau;
            const bool in_cta = tau < TPC;
            const bool valid = in_cta && t < g.T;
            float* row = red + (size_t)(tbase + (in_cta ? tau : 0)) * P;   // this CTA's own partial row
            // logits: the S partial rows added in split order, then the bias
            float l[EPL];
#pragma unroll
            for (int i = 0; i < EPL; ++i) l[i] = 0.f;
            if (valid) {
                for (int sp = 0; sp < S; ++sp) {
                    const float* src = sp == split ? row : recv + (size_t)(sp * TPC + tau) * P;
#pragma unroll
                    for (int i = 0; i < EPL; ++i)
                        if (sub + G * i < E) l[i] += src[sub + G * i];
                }
            }
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = sub + G * i;
                if (e < E) {
                    l[i] += bias_sh[e];
                    if (valid && g.sel.logits) g.sel.logits[(size_t)t * E + e] = l[i];
                }
            }
            finish_token<4, EPL, KMAX>(l, sub, E, g.k, g.renorm, valid, t, g.sel, g.idx, g.gate);
            if (in_cta) {
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (sub + G * i < E) row[sub + G * i] = valid ? l[i] : 0.f;
            }
        }
        __syncthreads();
        // this CTA's probability sums into the fixed-point accumulators; the
        // CTA that finishes last converts them into prob_sum
        __shared__ int is_last;
        for (int e = threadIdx.x; e < E; e += THREADS) {
            const float v = column_sum(red + (size_t)tbase * P, TPC, P, e);
            atomicAdd(g.psum_fx + e, (unsigned long long)__double2ll_rn((double)v * PSUM_FX_SCALE));
            __threadfence();
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            pdl_wait();   // the split kernel (which zeroed the accumulators) has finished
            is_last = atomicAdd(g.done, 1u) == gridDim.x - 1;
        }
        __syncthreads();
        if (is_last) {
            __threadfence();
            for (int e = threadIdx.x; e < E; e += THREADS)
                g.prob_sum[e] = (float)((double)(long long)__ldcg(g.psum_fx + e) * (1.0 / PSUM_FX_SCALE));
        }
    } else {
        // the logits of this CTA's tokens for the finishing kernel: the S
        // partial rows added in split order, then the bias; one warp per token
        for (int tau = warp; tau < TPC; tau += WARPS) {
            const int t = row0 + tbase + tau;
            if (t >= g.T) break;                  // tokens ascend with tau
            for (int e = lane; e < E; e += 32) {
                float acc = 0.f;
                for (int sp = 0; sp < S; ++sp)
                    acc += sp == split ? red[(size_t)(tbase + tau) * P + e] : recv[(size_t)(sp * TPC + tau) * P + e];
                g.logits[(size_t)t * E + e] = acc + bias_sh[e];
            }
        }
    }
    // every push into this CTA has landed (waited above); the ones it sent
    // have been read once every CTA is past this point
    if (S > 1) ptx2::cluster_sync();

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, g.tmem_cols);
    }
}

// Softmax, top-k and per-block probability sums from the logits [T, E] (for
// E > 64, where the fused kernel leaves them to this one): FIN_G lanes per
// token (16 logits per lane at E = 128: short per-lane candidate lists and a
// three-step butterfly per winner), FIN_TOKENS tokens per block.  Launched as
// a programmatic dependent of the logits kernel; many blocks per SM hide the
// latency of the dependent chains of finish_token.
constexpr int FIN_THREADS = 256;
constexpr int FIN_G = 8;
constexpr int FIN_TOKENS = FIN_THREADS / FIN_G;

template <int EMAX, int KMAX>
__global__ void __launch_bounds__(FIN_THREADS, KMAX <= 8 ? 4 : 2)
route_finish_kernel(const FinArgs g)
{
    constexpr int G = FIN_G, EPL = EMAX / G;
    __shared__ float pbuf[FIN_TOKENS][EMAX + 1];     // p of the block's tokens, for the per-expert sums
    pdl_launch_dependents();
    pdl_wait();                                      // the logits kernel has finished
    const int lane = threadIdx.x & 31, sub = lane & (G - 1);
    const int slot = threadIdx.x / G;                // token of the block handled by this group of G lanes
    const int t = blockIdx.x * FIN_TOKENS + slot;
    const bool valid = t < g.T;
    const int E = g.E;
    float l[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = sub + G * i;
        l[i] = (valid && e < E) ? __ldcg(g.logits + (size_t)t * E + e) : 0.f;
    }
    finish_token<G, EPL, KMAX>(l, sub, E, g.k, g.renorm, valid, t, g.sel, g.idx, g.gate);
#pragma unroll
    for (int i = 0; i < EPL; ++i)
        if (sub + G * i < E) pbuf[slot][sub + G * i] = valid ? l[i] : 0.f;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += FIN_THREADS)
        g.psum[(size_t)blockIdx.x * E + e] = column_sum(&pbuf[0][0], FIN_TOKENS, EMAX + 1, e);
}

// prob_sum[e] = sum over the R rows of psum[:, e]: one block per expert, a
// fixed-shape tree (strided fp64 partial sums, then a shared-memory tree), so
// the result does not depend on timing.
__global__ void __launch_bounds__(256) prob_sum_kernel(const float* __restrict__ psum, int R, int E,
                                                       float* __restrict__ prob_sum)
{
    __shared__ double sh[256];
    pdl_launch_dependents();   // the next step's first kernel may launch; it waits for this grid
    pdl_wait();   // launched as a programmatic dependent of the kernel writing psum
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

}  // namespace rfu
