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
// the order in which slots are granted.  Three or four kernels, each a
// programmatic dependent of the one before (it launches while that one runs,
// and waits for it only where it reads its results):
//   hist    per chunk of CH assignments, a histogram over experts
//   scan    (large chunks) per expert, the exclusive prefix of the
//           histograms over chunks, in place, and the totals
//   rank    per chunk: base of every expert from the earlier chunks and the
//           totals (without the scan: threads split the chunks of an
//           expert), then the stable rank of each assignment inside the
//           chunk (warp match + per-warp counts), giving its place in the
//           expert's queue; kept slots get a row of the permuted buffer;
//           chunk 0 also writes counts, kept, offsets and n_dropped
//   scatter x_perm[row] = x[token] with 16-byte vector moves, x staged in
//           shared memory while the ranks are computed
// CH = 256 while T*k <= SMALL_CHUNK_MAX (many short chunks: enough blocks to
// spread the latency-bound ranking over the GPU), else 1024.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"

namespace dispatch {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int MAX_E = 256;
constexpr int SMALL_CHUNK = 256, LARGE_CHUNK = 1024;
constexpr long long SMALL_CHUNK_MAX = 65536;   // T*k up to this: chunks of SMALL_CHUNK

__host__ __device__ constexpr int chunk_size(long long n) { return n <= SMALL_CHUNK_MAX ? SMALL_CHUNK : LARGE_CHUNK; }

template <int CH>
__global__ void __launch_bounds__(THREADS)
hist_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int* __restrict__ hist)
{
    // idx is final once the router has finished; only then may the rank
    // kernel launch (it preloads idx and gate before its own wait)
    pdl_wait();
    pdl_launch_dependents();
    constexpr int R = CH / THREADS;
    __shared__ int h[MAX_E];
    for (int e = threadIdx.x; e < E; e += THREADS) h[e] = 0;
    const long long n = (long long)T * k;
    const long long a0 = (long long)blockIdx.x * CH;
    int ev[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long long a = a0 + r * THREADS + threadIdx.x;
        ev[r] = -1;
        if (a < n) {
            const int j = (int)(a / T), t = (int)(a - (long long)j * T);
            ev[r] = __ldg(idx + (size_t)t * k + j);
        }
    }
    __syncthreads();
    bool bad = false;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (a0 + r * THREADS + threadIdx.x >= n) continue;
        if (ev[r] >= 0 && ev[r] < E) atomicAdd(&h[ev[r]], 1);
        else bad = true;
    }
    if (bad) moe_flag(MOE_DEV_BAD_EXPERT);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += THREADS) hist[(size_t)blockIdx.x * E + e] = h[e];
}

// Lanes that share an expert's chunk sums in rank_kernel (no scan): the
// largest power of two P <= 32 with P * E <= THREADS.
__host__ __device__ constexpr int rank_lanes_per_expert(int E)
{
    return E <= 8 ? 32 : E <= 16 ? 16 : E <= 32 ? 8 : E <= 64 ? 4 : E <= 128 ? 2 : 1;
}
// The per-expert scan runs for large chunks (up to 2M chunks, where the rank
// blocks' own sums would grow with the chunk count).  With chunks of 256 (at
// most 256 chunks) the rank kernel sums them itself: a scan launch measured
// no faster even at 128 chunks of 64 experts.
__host__ __device__ constexpr bool use_chunk_scan(int, int, bool large) { return large; }

// Per expert, the exclusive prefix of the chunk histograms
// over chunks, in place (hist[c][e] becomes the assignments to e in chunks
// before c), and the total into counts[e].  One warp per expert, windows of
// 256 chunks: lane l loads its run of 8 at once, a warp scan orders the runs.
constexpr int SCAN_PER = 8;   // chunks per lane in one window of 256

__global__ void __launch_bounds__(THREADS)
scan_kernel(int* __restrict__ hist, int nchunk, int E, int32_t* __restrict__ counts)
{
    pdl_launch_dependents();   // the rank kernel preloads its chunk meanwhile
    pdl_wait();                // every histogram is written
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * WARPS + (threadIdx.x >> 5);
    if (e >= E) return;
    int carry = 0;   // assignments to e in the windows before
    for (int w0 = 0; w0 < nchunk; w0 += 32 * SCAN_PER) {
        const int c0 = w0 + lane * SCAN_PER;
        int v[SCAN_PER], run = 0;
#pragma unroll
        for (int i = 0; i < SCAN_PER; ++i) v[i] = c0 + i < nchunk ? __ldcg(hist + (size_t)(c0 + i) * E + e) : 0;
#pragma unroll
        for (int i = 0; i < SCAN_PER; ++i) run += v[i];
        int incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        int acc = carry + incl - run;   // before this lane's run of chunks
#pragma unroll
        for (int i = 0; i < SCAN_PER; ++i)
            if (c0 + i < nchunk) {
                hist[(size_t)(c0 + i) * E + e] = acc;
                acc += v[i];
            }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) counts[e] = carry;
}

template <int CH>
__global__ void __launch_bounds__(THREADS)
rank_kernel(const int32_t* __restrict__ idx, const float* __restrict__ gate, int T, int k, int E, int cap,
            const int* __restrict__ hist, int nchunk, int scanned, int32_t* __restrict__ counts,
            int32_t* __restrict__ kept, int32_t* __restrict__ offsets, int32_t* __restrict__ slot_row,
            int32_t* __restrict__ row_token, float* __restrict__ row_gate, int32_t* __restrict__ n_dropped)
{
    constexpr int R = CH / THREADS;
    __shared__ int base[MAX_E], off[MAX_E + 1], running[MAX_E];
    __shared__ int wcnt[WARPS][MAX_E];
    __shared__ int drop_w[WARPS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = blockIdx.x;
    pdl_launch_dependents();   // the row scatter preloads x meanwhile

    // this chunk's expert ids and gates (router outputs, final before the
    // histogram kernel started), loaded before the wait
    const long long n = (long long)T * k;
    int ev[R];
    float gv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const long long a = (long long)chunk * CH + (long long)r * THREADS + tid;
        ev[r] = -1;
        gv[r] = 0.f;
        if (a < n) {
            const int j = (int)(a / T), t = (int)(a - (long long)j * T);
            ev[r] = __ldg(idx + (size_t)t * k + j);
            gv[r] = __ldg(gate + (size_t)t * k + j);
        }
    }
    pdl_wait();   // every histogram is written

    // 1. per expert: the assignments of earlier chunks (base) and in all
    //    chunks (total).  scanned: scan_kernel has turned hist into that
    //    exclusive prefix over chunks and written the totals to counts (many
    //    chunks per expert).  Otherwise P threads (consecutive lanes, P a power
    //    of two) share an expert, each summing every P-th chunk; a butterfly
    //    over the P lanes adds their sums.
    const bool SCANNED = scanned != 0;
    int P = rank_lanes_per_expert(E);
    if (SCANNED) P = 1;
    const int e1 = tid / P, s1 = tid & (P - 1);
    int before = 0, total = 0;
    if (SCANNED) {
        if (e1 < E) {
            before = __ldcg(hist + (size_t)chunk * E + e1);
            total = __ldcg(counts + e1);
        }
    } else if (e1 < E) {
        const int* col = hist + e1;
        int c = s1;
        for (; c + 3 * P < nchunk; c += 4 * P) {
            const int v0 = __ldcg(col + (size_t)c * E), v1 = __ldcg(col + (size_t)(c + P) * E);
            const int v2 = __ldcg(col + (size_t)(c + 2 * P) * E), v3 = __ldcg(col + (size_t)(c + 3 * P) * E);
            total += v0 + v1 + v2 + v3;
            before += (c < chunk ? v0 : 0) + (c + P < chunk ? v1 : 0) + (c + 2 * P < chunk ? v2 : 0) +
                      (c + 3 * P < chunk ? v3 : 0);
        }
        for (; c < nchunk; c += P) {
            const int v = __ldcg(col + (size_t)c * E);
            total += v;
            before += c < chunk ? v : 0;
        }
    }
    for (int o = 1; o < P; o <<= 1) {   // P is uniform over the block
        total += __shfl_xor_sync(0xffffffffu, total, o);
        before += __shfl_xor_sync(0xffffffffu, before, o);
    }
    int dr = 0;
    if (e1 < E && s1 == 0) {
        const int kp = total < cap ? total : cap;
        base[e1] = before;
        running[e1] = 0;
        off[e1] = kp;
        dr = total - kp;
        if (chunk == 0) {
            if (!SCANNED) counts[e1] = total;
            kept[e1] = kp;
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) dr += __shfl_xor_sync(0xffffffffu, dr, o);
    if (lane == 0) drop_w[warp] = dr;
    __syncthreads();
    // 2. exclusive scan of kept over E <= 256 experts (warp 0: lane l owns
    //    experts 8l .. 8l+7); chunk 0 also writes n_dropped and offsets
    if (warp == 0) {
        if (chunk == 0) {
            int d = lane < WARPS ? drop_w[lane] : 0;
#pragma unroll
            for (int o = 16; o; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) *n_dropped = d;
        }
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
    if (chunk == 0)
        for (int e = tid; e <= E; e += THREADS) offsets[e] = off[e];

    // 3. stable rank inside the chunk, THREADS assignments per round
    const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        for (int v = tid; v < WARPS * E; v += THREADS) wcnt[v / E][v % E] = 0;
        __syncthreads();
        const long long a = (long long)chunk * CH + (long long)r * THREADS + tid;
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
        if (R > 1) {
            __syncthreads();
            for (int v = tid; v < E; v += THREADS) {
                int s = 0;
                for (int w = 0; w < WARPS; ++w) s += wcnt[w][v];
                running[v] += s;
            }
            __syncthreads();
        }
    }
}

// Row permutation, token-major: one warp per (token, 2 KB chunk of its row)
// reads that chunk of x[t] once and writes it to every kept slot row of the
// token (slot_row[t, j] >= 0), so a token routed to k experts costs one read
// and k writes instead of k of each, and a whole row's chunks run in separate
// warps at once.  One wave of resident blocks grid-strides over the tasks.
// Launched as a programmatic dependent of the ranking kernel: x does not
// depend on it, so before waiting for the ranks every warp starts bulk copies
// of the x chunks of its first SLOTS tasks into its own shared-memory slots
// (one mbarrier per warp counts their bytes); those chunks are written from
// shared memory once the ranks are final, later ones are loaded directly
// (four 16-byte vectors per lane, all in flight together), and skipped when
// every slot of the token was dropped.
constexpr int CHUNK_VEC = 128;                   // 16-byte vectors per chunk
constexpr int CHUNK_BYTES = CHUNK_VEC * 16;      // 2 KB
constexpr int SLOTS = 4;                         // staged chunks per warp
constexpr int SCATTER_SMEM = WARPS * SLOTS * CHUNK_BYTES;   // 64 KB of dynamic shared memory

__global__ void __launch_bounds__(THREADS)
scatter_tokens_kernel(const int32_t* __restrict__ slot_row, int T, int k, const uint4* __restrict__ x,
                      uint4* __restrict__ x_perm, int vec16, unsigned long long wait_limit)
{
    extern __shared__ __align__(128) uint8_t sbuf[];
    __shared__ __align__(8) uint64_t bar[WARPS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nchunk = (vec16 + CHUNK_VEC - 1) / CHUNK_VEC;
    const long long tasks = (long long)T * nchunk;
    const long long warps_total = (long long)gridDim.x * WARPS;
    const long long first = (long long)blockIdx.x * WARPS + warp;
    const uint32_t wbar = ptx::smem_u32(&bar[warp]);
    const uint32_t wbuf = ptx::smem_u32(sbuf) + (uint32_t)(warp * SLOTS * CHUNK_BYTES);
    auto chunk_vecs = [&](long long task) {
        const int c = (int)(task % nchunk);
        return min(CHUNK_VEC, vec16 - c * CHUNK_VEC);
    };
    int nst = 0;   // staged tasks of this warp
#pragma unroll
    for (int p = 0; p < SLOTS; ++p)
        if (first + p * warps_total < tasks) ++nst;
    if (lane == 0) {
        ptx::mbar_init(wbar, 1);
        ptx::fence_mbar_init();
        if (nst > 0) {
            uint32_t bytes = 0;
            for (int p = 0; p < nst; ++p) bytes += (uint32_t)chunk_vecs(first + p * warps_total) * 16u;
            ptx::mbar_arrive_expect_tx(wbar, bytes);
            for (int p = 0; p < nst; ++p) {
                const long long task = first + p * warps_total;
                const int t = (int)(task / nchunk), c = (int)(task - (long long)t * nchunk);
                ptx::bulk_load(wbuf + (uint32_t)(p * CHUNK_BYTES), x + (size_t)t * vec16 + (size_t)c * CHUNK_VEC,
                               (uint32_t)chunk_vecs(task) * 16u, wbar);
            }
        }
    }
    __syncwarp();
    pdl_wait();   // slot_row is final
    if (nst > 0 && !ptx::mbar_wait(wbar, 0, wait_limit)) {
        moe_flag(MOE_DEV_TIMEOUT);
        // the copies into this warp's slots must land before the block exits
        ptx::mbar_wait(wbar, 0, wait_limit);
        return;
    }
    int p = 0;
    for (long long task = first; task < tasks; task += warps_total, ++p) {
        const int t = (int)(task / nchunk);
        const int v0 = (int)(task - (long long)t * nchunk) * CHUNK_VEC + lane;
        const int32_t* sr = slot_row + (size_t)t * k;
        bool any = false;
        for (int j = 0; j < k; ++j) any |= __ldg(sr + j) >= 0;
        if (!any) continue;
        uint4 a[4];
        if (p < nst) {
            const uint32_t slot = wbuf + (uint32_t)(p * CHUNK_BYTES) + (uint32_t)lane * 16u;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v0 + 32 * u < vec16) a[u] = ptx::ld_shared_v4(slot + (uint32_t)(u * 512));
        } else {
            const uint4* src = x + (size_t)t * vec16;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v0 + 32 * u < vec16) a[u] = ldg_nc_v4(src + v0 + 32 * u);
        }
        for (int j = 0; j < k; ++j) {
            const int row = __ldg(sr + j);
            if (row < 0) continue;
            uint4* dst = x_perm + (size_t)row * vec16;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (v0 + 32 * u < vec16) dst[v0 + 32 * u] = a[u];
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
