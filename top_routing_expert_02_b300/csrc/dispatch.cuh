// Dispatch: capacity-limited slot assignment and the row permutation that
// replaces the All-to-All token exchange on one GPU.
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §2.1 steps
// 2-3 (mark each token with its target expert, exchange the tokens) and §2.2
// (expert capacity; tokens beyond it are dropped and take the residual path);
// §5.3 of the same page packs and sorts tokens so each expert's rows are
// contiguous.
//
// Assignments are numbered a = j*T + t (k-rank major, token minor): that is
// the order in which slots are granted.  Three kernels:
//   hist    per chunk of 1024 assignments, a histogram over experts
//   rank    per chunk: base of every expert from the earlier chunks, then the
//           stable rank of each assignment inside the chunk (warp match +
//           per-warp counts), giving its place in the expert's queue; kept
//           slots get a row of the permuted buffer
//   gather  x_perm[row] = x[row_token[row]] with 16-byte vector moves
#pragma once
#include "common.cuh"

namespace dispatch {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int CHUNK = 1024;
constexpr int MAX_E = 256;

__global__ void __launch_bounds__(THREADS)
hist_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int* __restrict__ hist)
{
    __shared__ int h[MAX_E];
    for (int e = threadIdx.x; e < E; e += THREADS) h[e] = 0;
    __syncthreads();
    const long long n = (long long)T * k;
    const long long a0 = (long long)blockIdx.x * CHUNK;
    bool bad = false;
    for (int i = threadIdx.x; i < CHUNK; i += THREADS) {
        const long long a = a0 + i;
        if (a >= n) break;
        const int j = (int)(a / T), t = (int)(a - (long long)j * T);
        const int e = __ldg(idx + (size_t)t * k + j);
        if (e >= 0 && e < E) atomicAdd(&h[e], 1);
        else bad = true;
    }
    if (bad) moe_flag(MOE_DEV_BAD_EXPERT);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += THREADS) hist[(size_t)blockIdx.x * E + e] = h[e];
}

__global__ void __launch_bounds__(THREADS)
rank_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate, int T, int k, int E, int cap,
            const int* __restrict__ hist, int nchunk, int32_t* __restrict__ counts, int32_t* __restrict__ kept,
            int32_t* __restrict__ offsets, int32_t* __restrict__ slot_row, int32_t* __restrict__ row_token,
            float* __restrict__ row_gate, int32_t* __restrict__ n_dropped)
{
    __shared__ int base[MAX_E], off[MAX_E + 1], running[MAX_E], scan[MAX_E];
    __shared__ int wcnt[WARPS][MAX_E];
    __shared__ int drop_part[THREADS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = blockIdx.x;

    // 1. place of this chunk in every expert's queue, and the totals
    int my_drop = 0;
    for (int e = tid; e < E; e += THREADS) {
        int before = 0, total = 0;
#pragma unroll 8
        for (int c = 0; c < nchunk; ++c) {
            const int v = __ldg(hist + (size_t)c * E + e);
            if (c < chunk) before += v;
            total += v;
        }
        base[e] = before;
        running[e] = 0;
        const int kp = total < cap ? total : cap;
        scan[e] = kp;
        if (chunk == 0) {
            counts[e] = total;
            kept[e] = kp;
        }
        my_drop += total - kp;
    }
    drop_part[tid] = my_drop;
    __syncthreads();
    // 2. exclusive scan of kept over experts (E <= 256, one pass per thread)
    if (tid == 0) {
        int s = 0;
        for (int e = 0; e < E; ++e) {
            off[e] = s;
            s += scan[e];
        }
        off[E] = s;
        if (chunk == 0) {
            int dsum = 0;
            for (int i = 0; i < THREADS; ++i) dsum += drop_part[i];
            *n_dropped = dsum;
        }
    }
    __syncthreads();
    if (chunk == 0)
        for (int e = tid; e <= E; e += THREADS) offsets[e] = off[e];

    // 3. stable rank inside the chunk, THREADS assignments per round; every
    //    round's expert id and gate are loaded up front (one memory latency)
    const long long n = (long long)T * k;
    const unsigned lt_mask = (1u << lane) - 1u;
    constexpr int ROUNDS = CHUNK / THREADS;
    int ev[ROUNDS];
    float gv[ROUNDS];
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        const long long a = (long long)chunk * CHUNK + (long long)r * THREADS + tid;
        ev[r] = -1;
        gv[r] = 0.f;
        if (a < n) {
            const int j = (int)(a / T), t = (int)(a - (long long)j * T);
            ev[r] = __ldg(idx + (size_t)t * k + j);
            gv[r] = __ldg(gate + (size_t)t * k + j);
        }
    }
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        for (int v = tid; v < WARPS * E; v += THREADS) wcnt[v / E][v % E] = 0;
        __syncthreads();
        const long long a = (long long)chunk * CHUNK + (long long)r * THREADS + tid;
        int e = -1, t = 0, j = 0;
        if (a < n) {
            j = (int)(a / T);
            t = (int)(a - (long long)j * T);
            e = ev[r];
            if (e < 0 || e >= E) e = -2;   // flagged by hist_kernel; the slot is dropped
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int intra = __popc(peers & lt_mask);
        if (e >= 0 && intra == 0) wcnt[warp][e] = __popc(peers);
        __syncthreads();
        if (a < n) {
            int32_t row = -1;
            if (e >= 0) {
                int pos = base[e] + running[e] + intra;
                for (int w = 0; w < warp; ++w) pos += wcnt[w][e];
                if (pos < cap) {
                    row = off[e] + pos;
                    row_token[row] = t;
                    row_gate[row] = gv[r];
                }
            }
            slot_row[(size_t)t * k + j] = row;
        }
        __syncthreads();
        for (int v = tid; v < E; v += THREADS) {
            int s = 0;
            for (int w = 0; w < WARPS; ++w) s += wcnt[w][v];
            running[v] += s;
        }
        __syncthreads();
    }
}

// hist + rank in one block for small T*k (<= SMALL_MAX assignments): 32 warps,
// warp w owns the contiguous assignments [w*per, (w+1)*per), at most
// SMALL_PER_LANE per lane, whose expert ids and gates are loaded once, all at
// the start (one memory latency instead of one per round).
//   1. per-warp expert histograms in shared memory
//   2. per expert: exclusive scan over the warps (the base of each warp's
//      run in the expert's queue), counts, kept, n_dropped; exclusive scan of
//      kept over experts gives offsets
//   3. each warp walks its range in order, 32 assignments at a time: the rank
//      inside the 32 (match_any) plus the warp's running count gives the
//      place in the expert's queue
// Same results as hist_kernel + rank_kernel, in one launch without the
// global histogram round trip.
constexpr int SMALL_THREADS = 1024;
constexpr int SMALL_WARPS = SMALL_THREADS / 32;
constexpr int SMALL_PER_LANE = 16;
constexpr int SMALL_MAX = SMALL_THREADS * SMALL_PER_LANE;

__global__ void __launch_bounds__(SMALL_THREADS)
dispatch_small_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate, int T, int k, int E, int cap,
                      int32_t* __restrict__ counts, int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
                      int32_t* __restrict__ slot_row, int32_t* __restrict__ row_token, float* __restrict__ row_gate,
                      int32_t* __restrict__ n_dropped)
{
    __shared__ int wh[SMALL_WARPS][MAX_E];
    __shared__ int off[MAX_E + 1];
    __shared__ int drop_w[SMALL_WARPS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = T * k;
    const int per = (n + SMALL_WARPS - 1) / SMALL_WARPS;
    const int a0 = warp * per, a1 = min(n, a0 + per);
    const unsigned lt_mask = (1u << lane) - 1u;

    // this lane's assignments a0 + 32 i + lane: expert (-1 none, -2 invalid) and gate
    int ev[SMALL_PER_LANE];
    float gv[SMALL_PER_LANE];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < SMALL_PER_LANE; ++i) {
        const int a = a0 + 32 * i + lane;
        ev[i] = -1;
        gv[i] = 0.f;
        if (a < a1) {
            const int j = a / T, t = a - j * T;
            ev[i] = __ldg(idx + (size_t)t * k + j);
            gv[i] = __ldg(gate + (size_t)t * k + j);
        }
    }
    for (int e = lane; e < E; e += 32) wh[warp][e] = 0;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < SMALL_PER_LANE; ++i) {
        if (a0 + 32 * i + lane >= a1) continue;
        if (ev[i] >= 0 && ev[i] < E) {
            atomicAdd(&wh[warp][ev[i]], 1);
        } else {
            ev[i] = -2;
            bad = true;
        }
    }
    if (bad) moe_flag(MOE_DEV_BAD_EXPERT);
    __syncthreads();

    // 2. warp bases, totals, kept; offsets by a scan over experts (warp 0)
    int kp = 0, dr = 0;
    if (tid < E) {
        int tot = 0;
        for (int w = 0; w < SMALL_WARPS; ++w) {
            const int c = wh[w][tid];
            wh[w][tid] = tot;
            tot += c;
        }
        kp = tot < cap ? tot : cap;
        dr = tot - kp;
        counts[tid] = tot;
        kept[tid] = kp;
        off[tid] = kp;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) dr += __shfl_xor_sync(0xffffffffu, dr, o);
    if (lane == 0) drop_w[warp] = dr;
    __syncthreads();
    if (warp == 0) {
        int d = drop_w[lane];
#pragma unroll
        for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        if (lane == 0) *n_dropped = d;
        // exclusive scan of kept over E <= 256 experts: lane l owns experts 8l .. 8l+7
        int v[8], sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            v[i] = e < E ? off[e] : 0;
            sum += v[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        int run = incl - sum;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane * 8 + i;
            if (e < E) off[e] = run;
            run += v[i];
        }
        if (lane == 31) off[E] = incl;
    }
    __syncthreads();
    for (int e = tid; e <= E; e += SMALL_THREADS) offsets[e] = off[e];

    // 3. ranks, in assignment order inside each warp's range
#pragma unroll
    for (int i = 0; i < SMALL_PER_LANE; ++i) {
        if (a0 + 32 * i >= a1) break;   // warp-uniform
        const int a = a0 + 32 * i + lane;
        const int e = ev[i];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int intra = __popc(peers & lt_mask);
        const int pos = e >= 0 ? wh[warp][e] + intra : 0;
        __syncwarp();
        if (e >= 0 && intra == 0) wh[warp][e] += __popc(peers);
        __syncwarp();
        if (a < a1) {
            const int j = a / T, t = a - j * T;
            int32_t row = -1;
            if (e >= 0 && pos < cap) {
                row = off[e] + pos;
                row_token[row] = t;
                row_gate[row] = gv[i];
            }
            slot_row[(size_t)t * k + j] = row;
        }
    }
}

// Row permutation, token-major: one warp per token reads x[t] once and writes
// it to every kept slot row of the token (slot_row[t, j] >= 0), so a token
// routed to k experts costs one read and k writes instead of k of each.
// Tokens strided over the grid; vec16 = 16-byte vectors per row; four loads in
// flight per lane.
__global__ void __launch_bounds__(THREADS)
scatter_tokens_kernel(const int32_t* __restrict__ slot_row, int T, int k, const uint4* __restrict__ x,
                      uint4* __restrict__ x_perm, int vec16)
{
    const int lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * WARPS;
    for (int t = blockIdx.x * WARPS + (threadIdx.x >> 5); t < T; t += warps_total) {
        int rows[16];
        bool any = false;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            rows[j] = j < k ? __ldg(slot_row + (size_t)t * k + j) : -1;
            any |= rows[j] >= 0;
        }
        if (!any) continue;   // every slot dropped: the row is never read
        const uint4* src = x + (size_t)t * vec16;
        int v = lane;
        for (; v + 96 < vec16; v += 128) {
            const uint4 a0 = ldg_nc_v4(src + v), a1 = ldg_nc_v4(src + v + 32);
            const uint4 a2 = ldg_nc_v4(src + v + 64), a3 = ldg_nc_v4(src + v + 96);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (rows[j] < 0) continue;
                uint4* dst = x_perm + (size_t)rows[j] * vec16;
                dst[v] = a0;
                dst[v + 32] = a1;
                dst[v + 64] = a2;
                dst[v + 96] = a3;
            }
        }
        for (; v < vec16; v += 32) {
            const uint4 a0 = ldg_nc_v4(src + v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (rows[j] >= 0) x_perm[(size_t)rows[j] * vec16 + v] = a0;
        }
    }
}

// dst[i] = src[index[i]] for i < n: one warp per row, 16-byte vectors (the
// regrouping of received rows in the expert-parallel exchange).
__global__ void __launch_bounds__(THREADS)
permute_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ index, long long n, int vec16,
                    uint4* __restrict__ dst)
{
    const int lane = threadIdx.x & 31;
    const long long warps_total = (long long)gridDim.x * WARPS;
    for (long long i = blockIdx.x * WARPS + (threadIdx.x >> 5); i < n; i += warps_total) {
        const uint4* s = src + (size_t)__ldg(index + i) * vec16;
        uint4* o = dst + (size_t)i * vec16;
        for (int v = lane; v < vec16; v += 32) o[v] = ldg_nc_v4(s + v);
    }
}

}  // namespace dispatch
