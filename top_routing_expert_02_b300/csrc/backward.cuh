// Backward of the MoE layer: the kernels that are not grouped GEMMs.
//
// The pages train the layer through the same steps in reverse (the
// expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §2.1 and §5.1,
// whose auxiliary loss steers the router through its gradient; the deployment
// guide "细粒度专家并行部署实践与优化指南" 步骤三 item 3, the reverse exchange of the
// gradients); they give no formula, so these kernels compute the derivative of
// the forward.  With L = <dy, y> + aux_weight L_aux + z_weight L_z:
//   combine backward   do_r = g_r dy[t],  dgate[t,j] = <dy[t], o_r>
//                      (o_r = y_perm_r / g_r: the down projection before the gate)
//   activation backward dz = act'(z) da   (SwiGLU: da up silu'(gate) | da silu(gate))
//   router backward    dp from the gates (renormalised: (dgate_j - sum_i dgate_i g_i) / S)
//                      and from L_aux (aux_weight alpha E f_e / T); dl = p (dp - <p, dp>)
//                      + z_weight (2 beta / T) lse p
//   input gradient     dx[t] = sum over kept j of dx_perm[slot] + W^T dl[t]
//   router weights     dW = dl^T x, db = sum_t dl  (fixed-order sums)
// plus the transposes that feed the tensor-core GEMMs K-major operands.
#pragma once
#include "common.cuh"
#include "tiles.cuh"

namespace bwd {

// ----------------------------------------------------------- transposes ---

// dst[e][c][r] = src[e][r][c] for 2-byte elements, R and C multiples of 64.
// One 64x64 tile per block: 16-byte loads along c, 16-byte stores along r.
__global__ void __launch_bounds__(256)
transpose_experts_kernel(const uint16_t* __restrict__ src, int R, int C, uint16_t* __restrict__ dst)
{
    __shared__ uint16_t tile[64][64 + 2];
    const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
    const size_t slab = (size_t)blockIdx.z * R * C;
    for (int v = threadIdx.x; v < 64 * 8; v += 256) {
        const int r = v >> 3, q = v & 7;
        const uint4 u = ldg_nc_v4(src + slab + (size_t)(r0 + r) * C + c0 + q * 8);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            tile[r][q * 8 + 2 * i] = (uint16_t)(w[i] & 0xffffu);
            tile[r][q * 8 + 2 * i + 1] = (uint16_t)(w[i] >> 16);
        }
    }
    __syncthreads();
    for (int v = threadIdx.x; v < 64 * 8; v += 256) {
        const int c = v >> 3, q = v & 7;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (uint32_t)tile[q * 8 + 2 * i][c] | ((uint32_t)tile[q * 8 + 2 * i + 1][c] << 16);
        *reinterpret_cast<uint4*>(dst + slab + (size_t)(c0 + c) * R + r0 + q * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Segment-packed transpose for the weight-gradient GEMMs: expert e's rows
// src[offsets[e] + i][0..C) become columns 64 kstart[e] + i of dst [C, ld],
// zero for kept[e] <= i < 64 (kstart[e+1] - kstart[e]) (kstart = running sum
// of ceil(kept / 64)).  Block (x, y): columns 64x.., K block y of all experts.
__global__ void __launch_bounds__(256)
pack_segments_t_kernel(const uint16_t* __restrict__ src, const int32_t* __restrict__ offsets,
                       const int32_t* __restrict__ kept, int E, int C, long long ld, uint16_t* __restrict__ dst)
{
    __shared__ int kstart[257];
    __shared__ uint16_t tile[64][64 + 2];
    if (threadIdx.x < 32) build_mtile_prefix<64>(kept, E, kstart, threadIdx.x);
    __syncthreads();
    const int kb = blockIdx.y;
    if (kb >= kstart[E]) return;
    const int e = find_expert(kstart, E, kb);
    const int i0 = (kb - kstart[e]) * 64;        // first row of this block inside the segment
    const int n = __ldg(kept + e) - i0;         // rows of this block that exist (<= 64 valid)
    const int base = __ldg(offsets + e) + i0;
    const int c0 = blockIdx.x * 64;
    for (int v = threadIdx.x; v < 64 * 8; v += 256) {
        const int r = v >> 3, q = v & 7;
        uint4 u = make_uint4(0, 0, 0, 0);
        if (r < n) u = ldg_nc_v4(src + (size_t)(base + r) * C + c0 + q * 8);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            tile[r][q * 8 + 2 * i] = (uint16_t)(w[i] & 0xffffu);
            tile[r][q * 8 + 2 * i + 1] = (uint16_t)(w[i] >> 16);
        }
    }
    __syncthreads();
    for (int v = threadIdx.x; v < 64 * 8; v += 256) {
        const int c = v >> 3, q = v & 7;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (uint32_t)tile[q * 8 + 2 * i][c] | ((uint32_t)tile[q * 8 + 2 * i + 1][c] << 16);
        *reinterpret_cast<uint4*>(dst + (size_t)(c0 + c) * ld + (size_t)kb * 64 + q * 8) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// ------------------------------------------------------ combine backward ---

// One warp per token.  For each kept slot r = slot_row[t, j]:
//   do_perm[r] = g_r * dy[t]   (bf16),   dgate[t, j] = <dy[t], y_perm[r]> / g_r
// (y_perm holds g_r o_r); a dropped slot gets dgate 0 and no row.  Each lane
// works on four 16-byte vectors at a time (4 (k + 1) loads in flight).
constexpr int CB_THREADS = 256;
__global__ void __launch_bounds__(CB_THREADS)
combine_bwd_kernel(const uint4* __restrict__ dy, const int32_t* __restrict__ slot_row,
                   const float* __restrict__ row_gate, const uint4* __restrict__ y_perm, int T, int k, int vec16,
                   uint4* __restrict__ do_perm, float* __restrict__ dgate)
{
    const int lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * (CB_THREADS / 32);
    for (int t = blockIdx.x * (CB_THREADS / 32) + (threadIdx.x >> 5); t < T; t += warps_total) {
        int rows[16];
        float g[16], dot[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            rows[j] = (j < k) ? __ldg(slot_row + (size_t)t * k + j) : -1;
            g[j] = rows[j] >= 0 ? __ldg(row_gate + rows[j]) : 0.f;
            dot[j] = 0.f;
        }
        for (int v0 = lane; v0 < vec16; v0 += 128) {
            float f[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + 32 * u;
                unpack_bf16x8(v < vec16 ? ldg_nc_v4(dy + (size_t)t * vec16 + v) : make_uint4(0, 0, 0, 0), f[u]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (rows[j] < 0) continue;
                uint4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int v = v0 + 32 * u;
                    q[u] = v < vec16 ? ldg_nc_v4(y_perm + (size_t)rows[j] * vec16 + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int v = v0 + 32 * u;
                    if (v >= vec16) break;
                    float o[8];
                    unpack_bf16x8(q[u], o);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dot[j] = fmaf(f[u][i], o[i], dot[j]);
                    uint4 w;
                    w.x = pack_bf16x2(g[j] * f[u][0], g[j] * f[u][1]);
                    w.y = pack_bf16x2(g[j] * f[u][2], g[j] * f[u][3]);
                    w.z = pack_bf16x2(g[j] * f[u][4], g[j] * f[u][5]);
                    w.w = pack_bf16x2(g[j] * f[u][6], g[j] * f[u][7]);
                    do_perm[(size_t)rows[j] * vec16 + v] = w;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= k) break;
            float s = dot[j];
#pragma unroll
            for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == j) dgate[(size_t)t * k + j] = rows[j] >= 0 ? s / g[j] : 0.f;
        }
    }
}

// --------------------------------------------------- activation backward ---

// dz from z (pre-activation, bf16 [A, N1]) and da (bf16 [A, F]) over the kept
// rows A = offsets[E]; eight columns per thread step.
template <int ACT>
__global__ void __launch_bounds__(256)
act_bwd_kernel(const uint16_t* __restrict__ z, const uint16_t* __restrict__ da, const int32_t* __restrict__ offsets,
               int E, int F, uint16_t* __restrict__ dz)
{
    const long long A = __ldg(offsets + E);
    const int fv = F / 8;
    const int N1 = ACT == MOE_ACT_SWIGLU ? 2 * F : F;
    const long long total = A * fv;
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < total; i += (long long)gridDim.x * 256) {
        const long long r = i / fv;
        const int c = (int)(i - r * fv) * 8;
        float a[8], zg[8];
        unpack_bf16x8(ldg_nc_v4(da + r * F + c), a);
        unpack_bf16x8(ldg_nc_v4(z + r * N1 + c), zg);
        float o[8];
        if (ACT == MOE_ACT_SWIGLU) {
            float zu[8], ou[8];
            unpack_bf16x8(ldg_nc_v4(z + r * N1 + F + c), zu);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float s = 1.0f / (1.0f + expf(-zg[q]));
                const float silu = zg[q] * s;
                o[q] = a[q] * zu[q] * (s * (1.0f + zg[q] * (1.0f - s)));
                ou[q] = a[q] * silu;
            }
            *reinterpret_cast<uint4*>(dz + r * N1 + F + c) =
                make_uint4(pack_bf16x2(ou[0], ou[1]), pack_bf16x2(ou[2], ou[3]), pack_bf16x2(ou[4], ou[5]),
                           pack_bf16x2(ou[6], ou[7]));
        } else if (ACT == MOE_ACT_GELU) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float cdf = 0.5f * (1.0f + erff(zg[q] * 0.70710678118654752f));
                const float pdf = 0.39894228040143268f * expf(-0.5f * zg[q] * zg[q]);
                o[q] = a[q] * (cdf + zg[q] * pdf);
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = a[q];
        }
        *reinterpret_cast<uint4*>(dz + r * N1 + c) =
            make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                       pack_bf16x2(o[6], o[7]));
    }
}

// ------------------------------------------------------- router backward ---

// One warp per token, lane l owns experts l, l+32, ...  logits [T, E] are the
// forward's (bias included); counts are the f_e numerators (counts or kept).
//   aux_coef = aux_weight * alpha * E  (the kernel divides by T twice: f_e and P_e)
//   z_coef   = z_weight * beta         (the kernel applies 2 / T)
template <int EPL>
__global__ void __launch_bounds__(256)
route_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx, const float* __restrict__ dgate,
                 const int32_t* __restrict__ counts, int T, int E, int k, int renorm, float aux_coef, float z_coef,
                 float* __restrict__ dl)
{
    const int lane = threadIdx.x & 31;
    const float invT = 1.0f / (float)T;
    float daux[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        daux[i] = e < E ? aux_coef * ((float)__ldg(counts + e) * invT) * invT : 0.f;
    }
    for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += gridDim.x * 8) {
        float l[EPL], p[EPL], dp[EPL];
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            l[i] = e < E ? __ldg(logits + (size_t)t * E + e) : -INFINITY;
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
        const float lse = mx + logf(s);
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            p[i] = p[i] / s;
            dp[i] = daux[i];
        }
        // the k gates: probabilities of the chosen experts, their sum, sum_j dgate_j g_j
        float S = 0.f, dsum = 0.f;
        int ej[16];
        float pj[16], dgj[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= k) break;
            ej[j] = __ldg(idx + (size_t)t * k + j);
            dgj[j] = __ldg(dgate + (size_t)t * k + j);
            float v = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == ej[j]) v = p[i];
            pj[j] = __shfl_sync(0xffffffffu, v, ej[j] & 31);
            S += pj[j];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= k) break;
            dsum += dgj[j] * (pj[j] / S);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j >= k) break;
            const float add = renorm ? (dgj[j] - dsum) / S : dgj[j];
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i == ej[j]) dp[i] += add;
        }
        float pdp = 0.f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) pdp += p[i] * dp[i];
#pragma unroll
        for (int o = 16; o; o >>= 1) pdp += __shfl_xor_sync(0xffffffffu, pdp, o);
        const float zc = z_coef * 2.0f * invT * lse;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) dl[(size_t)t * E + e] = p[i] * (dp[i] - pdp) + zc * p[i];
        }
    }
}

// ------------------------------------------------------- input gradient ---

// dx[t][c] = sum_e dl[t,e] W[e,c] + sum over kept j of dx_perm[slot_row[t,j]][c].
// Block: GX_TOK tokens x 1024 columns, 4 adjacent columns per thread; dl is
// staged transposed in shared memory (dlT[e][token], read as 16-byte
// vectors), each W element is read once per block; fp32 sums in a fixed
// order (router part over e, then the kept slots in j order), one rounding.
constexpr int GX_TOK = 16;
constexpr int GX_COLS = 1024;
template <bool BF16>
__global__ void __launch_bounds__(256)
grad_x_kernel(const void* __restrict__ dx_perm, const int32_t* __restrict__ slot_row, const float* __restrict__ dl,
              const float* __restrict__ W, int T, int k, int E, int d, void* __restrict__ dx)
{
    __shared__ __align__(16) float dlT[256][GX_TOK];
    __shared__ int rows[GX_TOK][16];
    const int t0 = blockIdx.y * GX_TOK;
    const int c = blockIdx.x * GX_COLS + threadIdx.x * 4;
    for (int v = threadIdx.x; v < GX_TOK * E; v += 256) {
        const int tk = v / E, e = v - tk * E;
        dlT[e][tk] = (t0 + tk < T) ? __ldg(dl + (size_t)(t0 + tk) * E + e) : 0.f;
    }
    for (int v = threadIdx.x; v < GX_TOK * k; v += 256) {
        const int tk = v / k, j = v - tk * k;
        rows[tk][j] = (t0 + tk < T) ? __ldg(slot_row + (size_t)(t0 + tk) * k + j) : -1;
    }
    __syncthreads();
    if (c >= d) return;
    float acc[GX_TOK][4];
#pragma unroll
    for (int tk = 0; tk < GX_TOK; ++tk)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[tk][q] = 0.f;
    // W rows two experts ahead of the FMAs that use them
    float4 wn = __ldg(reinterpret_cast<const float4*>(W + c));
    float4 wnn = E > 1 ? __ldg(reinterpret_cast<const float4*>(W + (size_t)d + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int e = 0; e < E; ++e) {
        const float4 w = wn;
        wn = wnn;
        if (e + 2 < E) wnn = __ldg(reinterpret_cast<const float4*>(W + (size_t)(e + 2) * d + c));
#pragma unroll
        for (int t4 = 0; t4 < GX_TOK; t4 += 4) {
            const float4 l = *reinterpret_cast<const float4*>(&dlT[e][t4]);
            const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc[t4 + u][0] = fmaf(lv[u], w.x, acc[t4 + u][0]);
                acc[t4 + u][1] = fmaf(lv[u], w.y, acc[t4 + u][1]);
                acc[t4 + u][2] = fmaf(lv[u], w.z, acc[t4 + u][2]);
                acc[t4 + u][3] = fmaf(lv[u], w.w, acc[t4 + u][3]);
            }
        }
    }
#pragma unroll
    for (int tk = 0; tk < GX_TOK; ++tk) {
        if (t0 + tk >= T) continue;
        float a[4] = {acc[tk][0], acc[tk][1], acc[tk][2], acc[tk][3]};
        for (int j = 0; j < k; ++j) {
            const int r = rows[tk][j];
            if (r < 0) continue;
            if (BF16) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>((const uint16_t*)dx_perm + (size_t)r * d + c));
                a[0] += __uint_as_float(u.x << 16);
                a[1] += __uint_as_float(u.x & 0xffff0000u);
                a[2] += __uint_as_float(u.y << 16);
                a[3] += __uint_as_float(u.y & 0xffff0000u);
            } else {
                const float4 u = __ldg(reinterpret_cast<const float4*>((const float*)dx_perm + (size_t)r * d + c));
                a[0] += u.x;
                a[1] += u.y;
                a[2] += u.z;
                a[3] += u.w;
            }
        }
        if (BF16) {
            *reinterpret_cast<uint2*>((uint16_t*)dx + (size_t)(t0 + tk) * d + c) =
                make_uint2(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]));
        } else {
            *reinterpret_cast<float4*>((float*)dx + (size_t)(t0 + tk) * d + c) = make_float4(a[0], a[1], a[2], a[3]);
        }
    }
}

// ------------------------------------------------------ router weights ---

// partial[s][e][c] = sum over tokens t of split s of dl[t,e] x[t,c].
// Block (x, y, s): 1024 columns (4 adjacent per thread), 16 experts, token
// split s; dl staged 32 tokens at a time (read back as 16-byte vectors).
// The splits are summed in order by router_wgrad_sum_kernel.
constexpr int RW_EXP = 16;
constexpr int RW_COLS = 1024;

// Columns c..c+3 of x rows t..t+7 (as fp32; rows at or past tb read as 0).
template <bool BF16>
__device__ __forceinline__ void load_x_rows(const void* __restrict__ x, int t, int tb, int d, int c, float (&xv)[8][4])
{
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        if (t + u < tb) {
            if (BF16) {
                const uint2 w = __ldg(reinterpret_cast<const uint2*>((const uint16_t*)x + (size_t)(t + u) * d + c));
                xv[u][0] = __uint_as_float(w.x << 16);
                xv[u][1] = __uint_as_float(w.x & 0xffff0000u);
                xv[u][2] = __uint_as_float(w.y << 16);
                xv[u][3] = __uint_as_float(w.y & 0xffff0000u);
            } else {
                const float4 w = __ldg(reinterpret_cast<const float4*>((const float*)x + (size_t)(t + u) * d + c));
                xv[u][0] = w.x;
                xv[u][1] = w.y;
                xv[u][2] = w.z;
                xv[u][3] = w.w;
            }
        } else {
            xv[u][0] = xv[u][1] = xv[u][2] = xv[u][3] = 0.f;
        }
    }
}
template <bool BF16>
__global__ void __launch_bounds__(256)
router_wgrad_kernel(const float* __restrict__ dl, const void* __restrict__ x, int T, int E, int d, int tok_per_split,
                    float* __restrict__ partial)
{
    __shared__ __align__(16) float dls[32][RW_EXP];
    const int c = blockIdx.x * RW_COLS + threadIdx.x * 4;
    const int e0 = blockIdx.y * RW_EXP;
    const int s = blockIdx.z;
    const int ta = s * tok_per_split;
    const int tb = min(T, ta + tok_per_split);
    float acc[RW_EXP][4];
#pragma unroll
    for (int i = 0; i < RW_EXP; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = 0.f;
    for (int t0 = ta; t0 < tb; t0 += 32) {
        __syncthreads();
        for (int v = threadIdx.x; v < 32 * RW_EXP; v += 256) {
            const int tk = v / RW_EXP, i = v - tk * RW_EXP;
            dls[tk][i] = (t0 + tk < tb && e0 + i < E) ? __ldg(dl + (size_t)(t0 + tk) * E + e0 + i) : 0.f;
        }
        __syncthreads();
        if (c < d) {
            // eight token rows of x in flight at a time (rows past the split read as 0)
            for (int tk0 = 0; tk0 < 32; tk0 += 8) {
                float xv[8][4];
                load_x_rows<BF16>(x, t0 + tk0, tb, d, c, xv);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
#pragma unroll
                    for (int i4 = 0; i4 < RW_EXP; i4 += 4) {
                        const float4 l = *reinterpret_cast<const float4*>(&dls[tk0 + u][i4]);
                        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                        for (int v = 0; v < 4; ++v)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[i4 + v][q] = fmaf(lv[v], xv[u][q], acc[i4 + v][q]);
                    }
                }
            }
        }
    }
    if (c < d) {
#pragma unroll
        for (int i = 0; i < RW_EXP; ++i)
            if (e0 + i < E)
                *reinterpret_cast<float4*>(partial + ((size_t)s * E + e0 + i) * d + c) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
}

__global__ void __launch_bounds__(256)
router_wgrad_sum_kernel(const float* __restrict__ partial, int S, long long n, float* __restrict__ dW)
{
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
        float a = 0.f;
        for (int s = 0; s < S; ++s) a += __ldg(partial + (size_t)s * n + i);
        dW[i] = a;
    }
}

// ---------------------------------------------------------------------------
// Router gradients on the tensor cores.  dx_router = dl . W and dW = dl^T x
// are dense contractions over E and over T; their fp32 operands (dl, W) are
// split into bf16 parts, v = hi + lo with hi = rn(v), lo = rn(v - hi), so that
// bf16 MMAs with fp32 accumulation keep ~16 significant bits:
//   dl . W  ~ hi(dl).hi(W) + lo(dl).hi(W) + hi(dl).lo(W)     (one GEMM, K = 3 Ep)
//   dl^T x  = hi(dl)^T x + lo(dl)^T x                        (x is bf16: exact)
// Ep = E rounded up to 64; the padding experts are zero.
//
// router_grads_prep_kernel writes
//   dl3 [T, 3 Ep] bf16, row t = [hi(dl[t]) | lo(dl[t]) | hi(dl[t])]
//   W3  [3 Ep, d] bf16, rows   = [hi(W); hi(W); lo(W)]
// and the row segments of the two GEMMs: one segment [0, T) (seg1) and S
// equal token splits (segS) for the weight gradient.
__global__ void __launch_bounds__(256)
router_grads_prep_kernel(const float* __restrict__ dl, const float* __restrict__ W, int T, int E, int Ep, int d,
                         int S, uint16_t* __restrict__ dl3, uint16_t* __restrict__ W3, int32_t* __restrict__ seg1,
                         int32_t* __restrict__ segS)
{
    const long long n_dl = (long long)T * Ep, n_w = (long long)Ep * d;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_dl + n_w; i += stride) {
        if (i < n_dl) {
            const long long t = i / Ep;
            const int c = (int)(i - t * Ep);
            const float v = c < E ? __ldg(dl + t * E + c) : 0.f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
            uint16_t* row = dl3 + t * (3LL * Ep);
            row[c] = *reinterpret_cast<const uint16_t*>(&hi);
            row[Ep + c] = *reinterpret_cast<const uint16_t*>(&lo);
            row[2 * Ep + c] = *reinterpret_cast<const uint16_t*>(&hi);
        } else {
            const long long j = i - n_dl;
            const int e = (int)(j / d);
            const float v = e < E ? __ldg(W + j) : 0.f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(v);
            const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
            W3[j] = *reinterpret_cast<const uint16_t*>(&hi);
            W3[n_w + j] = *reinterpret_cast<const uint16_t*>(&hi);
            W3[2 * n_w + j] = *reinterpret_cast<const uint16_t*>(&lo);
        }
    }
    if (blockIdx.x == 0) {
        // seg1: offsets {0, T}, kept {T};  segS: offsets [S + 1], kept [S]
        if (threadIdx.x == 0) {
            seg1[0] = 0;
            seg1[1] = T;
            seg1[2] = T;
        }
        for (int s = threadIdx.x; s <= S; s += blockDim.x) {
            const int o = (int)((long long)s * T / S);
            segS[s] = o;
            if (s < S) segS[S + 1 + s] = (int)((long long)(s + 1) * T / S) - o;
        }
    }
}

// dx[t] = rn_bf16(zr[t] + sum_j dx_perm[slot_row[t, j]]): zr [T, d] fp32 is the
// router part dl . W, the slots are added in j order (dropped ones skipped).
// One warp per token, four 16-byte vectors (8 columns each) per lane in flight.
__global__ void __launch_bounds__(256)
grad_x_gather_kernel(const uint4* __restrict__ dx_perm, const int32_t* __restrict__ slot_row,
                     const float4* __restrict__ zr, int T, int k, int vec16, uint4* __restrict__ dx)
{
    const int lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * 8;
    for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += warps_total) {
        int rows[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) rows[j] = j < k ? __ldg(slot_row + (size_t)t * k + j) : -1;
        for (int v0 = lane; v0 < vec16; v0 += 128) {
            float acc[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + 32 * u;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                if (v < vec16) {
                    a = __ldcs(zr + ((size_t)t * vec16 + v) * 2);
                    b = __ldcs(zr + ((size_t)t * vec16 + v) * 2 + 1);
                }
                acc[u][0] = a.x; acc[u][1] = a.y; acc[u][2] = a.z; acc[u][3] = a.w;
                acc[u][4] = b.x; acc[u][5] = b.y; acc[u][6] = b.z; acc[u][7] = b.w;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (rows[j] < 0) continue;
                const uint4* src = dx_perm + (size_t)rows[j] * vec16;
                uint4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    q[u] = (v0 + 32 * u < vec16) ? ldg_nc_v4(src + v0 + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float f[8];
                    unpack_bf16x8(q[u], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[u][i] += f[i];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + 32 * u;
                if (v >= vec16) break;
                uint4 o;
                o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                o.w = pack_bf16x2(acc[u][6], acc[u][7]);
                dx[(size_t)t * vec16 + v] = o;
            }
        }
    }
}

// dW[e, c] = sum_s P[s, e, c] + sum_s P[s, Ep + e, c]  (hi part, then lo part,
// splits in order); P [S, 2 Ep, d] fp32 from the split weight-gradient GEMM.
__global__ void __launch_bounds__(256)
router_grads_reduce_kernel(const float4* __restrict__ P, int S, int E, int Ep, int d4, float4* __restrict__ dW)
{
    const long long n = (long long)E * d4, plane = 2LL * Ep * d4, lo_off = (long long)Ep * d4;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float4 h = __ldcs(P + i), l = __ldcs(P + lo_off + i);
        for (int s = 1; s < S; ++s) {
            const float4 a = __ldcs(P + s * plane + i), b = __ldcs(P + s * plane + lo_off + i);
            h.x += a.x; h.y += a.y; h.z += a.z; h.w += a.w;
            l.x += b.x; l.y += b.y; l.z += b.z; l.w += b.w;
        }
        dW[i] = make_float4(h.x + l.x, h.y + l.y, h.z + l.z, h.w + l.w);
    }
}

}  // namespace bwd
