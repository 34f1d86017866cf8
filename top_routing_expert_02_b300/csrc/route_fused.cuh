// Router of bf16 x on the tensor cores, fused: logits, softmax, top-k and the
// per-block probability sums of one 128-token tile in one kernel.
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
// Work split.  A cluster of S CTAs shares one 128-token tile (S > 1 splits d
// when there are too few tiles to fill the GPU); CTA s of the cluster covers
// K blocks [s*nk/S, (s+1)*nk/S).  Each CTA has 6 warps:
//   warp 0      TMA producer: per stage the x tile (128 tokens x 64 columns)
//               and the three weight parts (E_pad rows x 64 columns each)
//   warp 1      TMEM allocation and the single thread issuing tcgen05.mma
//               (M = 128 tokens, N = E_pad experts, one MMA per part per K=16)
//   warps 2-5   add each finished W0 chunk into the fp32 sum kept in TMEM;
//               at the end, the partial logits of the tile's rows (thread =
//               TMEM lane = token row)
// TMEM columns: [W0 chunk, buffer 0 | W0 chunk, buffer 1 | W1 + W2 | W0 sum],
// E_pad each.
// The partial logits of the S CTAs meet in distributed shared memory: CTA s
// finishes tokens [s*128/S, (s+1)*128/S) of the tile, adding the S partial rows
// in split order plus the bias, then takes the softmax, the top-k (sorted
// insertion per token on (logit desc, index asc)) and its per-expert sums of
// p.  Every sum has a fixed order, so a call gives the same bits every run.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"

namespace rfu {

constexpr int BM = 128, BK = 64;
constexpr int THREADS = 192;
constexpr int MAX_STAGES = 8;
constexpr int KC = 4;                       // K blocks per W0 accumulator chunk
constexpr int X_BYTES = BM * BK * 2;        // one x tile, 16 KB
constexpr int MAX_EPAD = 128;               // 4 * E_pad TMEM columns <= 512
constexpr int MAX_SPLITS = 8;               // portable cluster size
constexpr int ACC_THREADS = 128;            // warps 2-5

struct Args {
    int T, d, E, E_pad, k, renorm;
    int nk;             // K blocks of 64 over d
    int S;              // CTAs per tile (cluster size)
    int stages;
    int stage_bytes;    // x tile + three weight parts
    uint32_t tmem_cols;
    const float* bias;  // [E] or nullptr
    int32_t* idx;       // [T, k]
    float* gate;        // [T, k]
    float* psum;        // [gridDim.x, E]: per-CTA probability sums
    RouteSel sel;
    unsigned long long wait_limit;
};

__host__ __device__ constexpr int red_bytes(int E_pad) { return BM * E_pad * 4; }
__host__ __device__ constexpr int fin_bytes(int E_pad) { return BM * (E_pad + 1) * 4; }

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Programmatic dependent launch: the next kernel in the stream may start
// (launch_dependents); wait until the kernel before this one has finished and
// its memory is visible (wait).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// W (fp32 [E, d]) -> stacked bf16 [3*E_pad, d]: rows [0,E_pad) W0, [E_pad,2E_pad) W1,
// [2E_pad,3E_pad) W2; rows of experts >= E are zero.  W0 = rn(W), W1 = rn(W - W0),
// W2 = rn(W - W0 - W1); both differences are exact in fp32.  Eight columns per thread.
__global__ void __launch_bounds__(256) split_weight_kernel(const float* __restrict__ W, int E, int E_pad, int d,
                                                           uint4* __restrict__ Ws)
{
    pdl_launch_dependents();
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

// W0 chunk `buf` added into the W0 sum (or copied, for the first chunk), by
// one accumulator warp (its 32 TMEM lanes).
__device__ __forceinline__ void drain_chunk(uint32_t tb, int Ep, int buf, bool first)
{
    for (int e0 = 0; e0 < Ep; e0 += 16) {
        uint32_t v[16], a[16];
        ptx::tmem_ld16(tb + (uint32_t)(buf * Ep + e0), v);
        if (!first) ptx::tmem_ld16(tb + (uint32_t)(3 * Ep + e0), a);
        ptx::tmem_ld_wait();
        if (!first) {
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = __float_as_uint(__uint_as_float(a[u]) + __uint_as_float(v[u]));
        }
        ptx::tmem_st16(tb + (uint32_t)(3 * Ep + e0), v);
    }
    ptx::tmem_st_wait();
}

template <int KMAX>
__global__ void __launch_bounds__(THREADS, 2)
route_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const Args g)
{
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t accf_bar[2], acce_bar[2], fin_bar;
    __shared__ uint32_t tmem_base_sh;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem0 = (ptx::smem_u32(dsmem) + 1023u) & ~1023u;
    uint8_t* const gsmem = dsmem + (smem0 - ptx::smem_u32(dsmem));
    const int S = g.S;
    const int tile = blockIdx.x / S, split = blockIdx.x - tile * S;
    const int kb0 = (int)((long long)split * g.nk / S), kb1 = (int)((long long)(split + 1) * g.nk / S);
    const int nkb = kb1 - kb0;
    const int rot = nkb > 0 ? tile % nkb : 0;   // staggered walk: concurrent tiles read different W columns
    const int nch = (nkb + KC - 1) / KC;
    const int Ep = g.E_pad;
    const uint64_t limit = g.wait_limit;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < g.stages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&accf_bar[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&acce_bar[b]), ACC_THREADS);
        }
        ptx::mbar_init(ptx::smem_u32(&fin_bar), 1);
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

    if (warp == 0) {
        // ------------------------------------------------ TMA producer: x and weight parts
        if (lane == 0) {
            const int part_bytes = Ep * 128;
            const uint32_t tx_bytes = (uint32_t)(X_BYTES + 3 * part_bytes);
            auto kblock = [&](int i) { return kb0 + (i + rot) % nkb; };
            auto load_parts = [&](int i, int stage) {
                const uint32_t sb = smem0 + stage * g.stage_bytes + X_BYTES;
                const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
                for (int p = 0; p < 3; ++p) ptx::tma_load_2d(sb + p * part_bytes, &tmW, fb, kblock(i) * BK, p * Ep);
            };
            // the first stages' x tiles go out before the weight split has finished
            const int pre = nkb < g.stages ? nkb : g.stages;
            for (int i = 0; i < pre; ++i) {
                const uint32_t fb = ptx::smem_u32(&full_bar[i]);
                ptx::mbar_arrive_expect_tx(fb, tx_bytes);
                ptx::tma_load_2d(smem0 + i * g.stage_bytes, &tmX, fb, kblock(i) * BK, tile * BM);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) load_parts(i, i);
            int stage = pre % g.stages;
            uint32_t phase = pre == g.stages ? 1u : 0u;
            int fills = pre;
            bool ok = true;
            for (int i = pre; i < nkb; ++i) {
                if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), phase ^ 1u, limit)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
                ptx::mbar_arrive_expect_tx(fb, tx_bytes);
                ptx::tma_load_2d(smem0 + stage * g.stage_bytes, &tmX, fb, kblock(i) * BK, tile * BM);
                load_parts(i, stage);
                ++fills;
                if (++stage == g.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            // the last stages' copies must have landed before shared memory is reused or freed
            for (int f = fills - 1; f >= 0 && f >= fills - g.stages; --f) {
                const uint32_t bar = ptx::smem_u32(&full_bar[f % g.stages]);
                if (!ptx::mbar_wait(bar, (uint32_t)((f / g.stages) & 1), limit)) {
                    moe_flag(MOE_DEV_TIMEOUT);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_bf16_f32(BM, Ep);
            const uint32_t t_w12 = tmem_base + (uint32_t)(2 * Ep);
            const int part_bytes = Ep * 128;
            int stage = 0;
            uint32_t phase = 0;
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
                if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[stage]), phase, limit)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sa = smem0 + stage * g.stage_bytes, sb = sa + X_BYTES;
                const uint32_t t_w0 = tmem_base + (uint32_t)(buf * Ep);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t ad = ptx::sdesc_kmajor_sw128(sa + kk * 32);
                    ptx::mma_bf16(t_w0, ad, ptx::sdesc_kmajor_sw128(sb + kk * 32), idesc, (!first || kk > 0) ? 1u : 0u);
                    ptx::mma_bf16(t_w12, ad, ptx::sdesc_kmajor_sw128(sb + part_bytes + kk * 32), idesc,
                                  (i > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_bf16(t_w12, ad, ptx::sdesc_kmajor_sw128(sb + 2 * part_bytes + kk * 32), idesc, 1u);
                }
                ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
                const bool last = (i % KC) == KC - 1 || i == nkb - 1;
                if (last && c < nch - 1) ptx::mma_commit(ptx::smem_u32(&accf_bar[buf]));
                if (++stage == g.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            // arrives once every MMA issued above has completed (also on the error path)
            ptx::mma_commit(ptx::smem_u32(&fin_bar));
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ warps 2-5: W0 sums, partial logits
        const int q = warp & 3;                    // TMEM lanes 32q .. 32q+31
        const int r = q * 32 + lane;               // token row of the tile
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
        bool ok = true;
        for (int c = 0; c + 1 < nch; ++c) {        // every W0 chunk but the last into the sum
            const int buf = c & 1;
            const bool w = ptx::mbar_wait(ptx::smem_u32(&accf_bar[buf]), (uint32_t)((c >> 1) & 1), limit);
            if (!__all_sync(0xffffffffu, w)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            drain_chunk(tb, Ep, buf, c == 0);
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&acce_bar[buf]));
        }
        if (!ok) moe_flag(MOE_DEV_TIMEOUT);
        const bool fin = ptx::mbar_wait(ptx::smem_u32(&fin_bar), 0, limit);
        if (!__all_sync(0xffffffffu, fin)) moe_flag(MOE_DEV_TIMEOUT);
        ptx::tc_fence_after();
        // partial logits: (W0 sum + last W0 chunk) + (W1 + W2)
        const int lb = (nch - 1) & 1;
        float* red = reinterpret_cast<float*>(gsmem) + (size_t)r * Ep;
        for (int e0 = 0; e0 < Ep; e0 += 16) {
            uint32_t a0[16], a1[16], as[16];
            ptx::tmem_ld16(tb + (uint32_t)(lb * Ep + e0), a0);
            ptx::tmem_ld16(tb + (uint32_t)(2 * Ep + e0), a1);
            if (nch >= 2) ptx::tmem_ld16(tb + (uint32_t)(3 * Ep + e0), as);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; u += 4) {
                float v[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float s0 = nch >= 2 ? __uint_as_float(as[u + w]) + __uint_as_float(a0[u + w])
                                              : __uint_as_float(a0[u + w]);
                    v[w] = s0 + __uint_as_float(a1[u + w]);
                }
                *reinterpret_cast<float4*>(red + e0 + u) = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
    }

    pdl_launch_dependents();   // the probability-sum kernel may launch; it waits for this grid's results
    // every CTA of the cluster has its partial rows in shared memory
    ptx::tc_fence_before();
    if (S > 1) ptx2::cluster_sync();
    else __syncthreads();

    // ---------------------------------------------------- gather the S partial rows
    const int TPC = BM / S;                       // tokens this CTA finishes
    const int tbase = split * TPC;
    float* const L = reinterpret_cast<float*>(gsmem + red_bytes(Ep));   // [TPC][Ep + 1]
    const int LP = Ep + 1;
    {
        const int g4n = Ep / 4;
        const uint32_t red0 = smem0;
        for (int it = threadIdx.x; it < TPC * g4n; it += THREADS) {
            const int tau = it / g4n, e = (it - tau * g4n) * 4;
            const uint32_t off = (uint32_t)(((tbase + tau) * Ep + e) * 4);
            float4 s4;
            if (S == 1) {
                s4 = *reinterpret_cast<const float4*>(gsmem + off);
            } else {
                s4 = ld_cluster_f4(ptx2::mapa(red0 + off, 0));
                for (int sp = 1; sp < S; ++sp) {
                    const float4 v = ld_cluster_f4(ptx2::mapa(red0 + off, (uint32_t)sp));
                    s4.x += v.x;
                    s4.y += v.y;
                    s4.z += v.z;
                    s4.w += v.w;
                }
            }
            const float vals[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float bb = (g.bias && e + u < g.E) ? __ldg(g.bias + e + u) : 0.f;
                L[tau * LP + e + u] = vals[u] + bb;
            }
        }
    }
    // no CTA reads another's partial rows after this point
    if (S > 1) ptx2::cluster_sync();
    else __syncthreads();

    // ---------------------------------------------------- finish: one thread per token
    // (the row of logits is read from shared memory in each pass; rows are
    // E_pad + 1 floats apart, so the threads of a warp hit different banks)
    if (threadIdx.x < TPC) {
        const int tau = threadIdx.x;
        const int t = tile * BM + tbase + tau;
        float* row = L + tau * LP;
        const int E = g.E;
        if (t < g.T) {
            const RouteSel& sel = g.sel;
            // group-limited routing: keep the topk_group groups of largest max
            // logit (strict > scanning up the index keeps the lower group on ties)
            const bool grouped = sel.n_group > 1;
            unsigned gkeep = 0xffffffffu;
            if (grouped) {
                gkeep = 0;
                for (int rr = 0; rr < sel.topk_group; ++rr) {
                    float bv = -INFINITY;
                    int bg = -1;
                    for (int e = 0; e < E; ++e) {
                        const int ge = e / sel.gsz;
                        const float v = row[e];
                        if (!((gkeep >> ge) & 1u) && (bg < 0 || v > bv)) {
                            bv = v;
                            bg = ge;
                        }
                    }
                    if (bg >= 0) gkeep |= 1u << bg;
                }
            }
            // maximum and top-k (descending list; an equal value keeps the lower index ahead)
            float tv[KMAX];
            int ti[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                tv[j] = -INFINITY;
                ti[j] = 0x7fffffff;
            }
            float mx = -INFINITY;
            for (int e = 0; e < E; ++e) {
                const float v = row[e];
                mx = fmaxf(mx, v);
                if (v > tv[KMAX - 1] && (!grouped || ((gkeep >> (e / sel.gsz)) & 1u))) {
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
            float s = 0.f;
            for (int e = 0; e < E; ++e) s += expf(row[e] - mx);
            if (sel.lse) sel.lse[t] = mx + logf(s);
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
            for (int e = 0; e < E; ++e) {
                const float v = row[e];
                if (sel.logits) sel.logits[(size_t)t * E + e] = v;
                row[e] = expf(v - mx) / s;
            }
        } else {
            for (int e = 0; e < E; ++e) row[e] = 0.f;
        }
    }
    __syncthreads();
    // per-expert sums of p over this CTA's tokens, in token order
    for (int e = threadIdx.x; e < g.E; e += THREADS) {
        float v = 0.f;
        for (int tau = 0; tau < TPC; ++tau) v += L[tau * LP + e];
        g.psum[(size_t)blockIdx.x * g.E + e] = v;
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, g.tmem_cols);
    }
}

// prob_sum[e] = sum over the R rows of psum[:, e]: one block per expert, a
// fixed-shape tree (strided fp64 partial sums, then a shared-memory tree), so
// the result does not depend on timing.
__global__ void __launch_bounds__(256) prob_sum_kernel(const float* __restrict__ psum, int R, int E,
                                                       float* __restrict__ prob_sum)
{
    __shared__ double sh[256];
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
