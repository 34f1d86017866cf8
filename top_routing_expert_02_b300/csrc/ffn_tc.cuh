// bf16 grouped expert GEMMs on the 5th-generation tensor cores (tcgen05).
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §2.1 step 4
// (every expert runs its FFN on the rows it received) with the two-matrix
// expert d -> d_ff -> d of the ETP page "ETP专家并行加速MoE模型：ms-swift中稀疏架构的
// 极致优化".  Up:   h[r] = act(w1[e] . x_perm[r]);  down: y_perm[r] = row_gate[r]
// * (w2[e] . h[r]).  The activation lives in the up epilogue and the gate
// product in the down epilogue, so neither needs a pass of its own.
//
// One persistent block per SM, 6 warps (BN = 128, 192 or 256 output-tile
// columns, chosen per call for the best wave balance over the SMs):
//   warp 0     TMA producer: A tile 128x64 and B tile BNx64 (two BN/2-row
//              boxes) per stage, 128-byte swizzle, a ring as deep as shared
//              memory allows (6 / 5 / 4 stages)
//   warp 1     MMA issuer: tcgen05.mma M=128 N=BN K=16, fp32 accumulator in
//              TMEM, two accumulators so the epilogue of one tile overlaps
//              the main loop of the next
//   warps 2-5  epilogue: tcgen05.ld 32 columns at a time, activation or
//              gate scale in fp32, one rounding to bf16, masked stores
// Tiles never straddle experts: M-tile m of expert e starts at row
// offsets[e] + 128 m; rows past kept[e] are computed (they belong to the next
// expert or to the zero fill past the buffer) but never stored.  Tiles run
// M-fastest inside (expert, N-tile), so the blocks working at the same time
// share one weight tile through L2.  For SwiGLU the B tile pairs gate rows
// n..n+BN/2-1 with up rows F+n..F+n+BN/2-1, so accumulator columns [0,BN/2)
// are the gate and [BN/2,BN) the up projection of the same BN/2 outputs.
//
// Every wait is bounded by a cycle limit; a wait that runs out records
// MOE_DEV_TIMEOUT and its role stops, the other roles then run out too, and
// the block still drains its copies and frees TMEM before it exits.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"
#include "tiles.cuh"

namespace tcg {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;              // 16 KB
constexpr int THREADS = 192;

template <int BN>
struct Shape {
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int BH_BYTES = B_BYTES / 2;                       // one BN/2-row box
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (200 * 1024) / STAGE_BYTES > 6 ? 6 : (200 * 1024) / STAGE_BYTES;
    static constexpr int SMEM_DYN = STAGES * STAGE_BYTES + 1024;       // + slack for 1024-B alignment
    // weight-gradient mode: the same ring plus a 32x32 fp32 staging tile per
    // epilogue warp for the TMA stores of the output (fits next to 4 stages of 48 KB)
    static constexpr int WG_STAGES = STAGES;
    static constexpr int WG_STAGE_OUT = 32 * 32 * 4;
    static constexpr int WG_SMEM_DYN = WG_STAGES * STAGE_BYTES + 4 * WG_STAGE_OUT + 1024;
    static_assert(WG_SMEM_DYN <= 227 * 1024, "weight-gradient mode exceeds shared memory");
    static constexpr int ACC_COLS = BN;
    static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, BN);
};
constexpr int MAX_STAGES = 6;

// EPI_DGELU / EPI_DSWIGLU: activation backward fused into the da = do . w2[e]
// epilogue: the accumulator column c is da[:, c]; the epilogue reads the kept
// pre-activation z (in_z, row stride z_cols = N1) and writes dz (out, row
// stride z_cols): GELU dz = da (Phi(z) + z phi(z)); SwiGLU dz[:, c] = da
// z_up silu'(z_gate), dz[:, F + c] = da silu(z_gate).
enum { EPI_GELU = 0, EPI_SWIGLU = 1, EPI_IDENT = 2, EPI_GATE = 3, EPI_DGELU = 4, EPI_DSWIGLU = 5 };

struct Args {
    const int32_t* offsets;
    const int32_t* kept;
    int E;
    int K;             // reduction length (d for up, F for down)
    int n_tiles;       // N-tiles per expert
    int b_rows;        // rows of one expert's weight in the 2-D view [E*b_rows, K]
    int half_off;      // row offset of the second BN/2-row box of a B tile
    int n_step;        // output columns per tile: BN/2 (SwiGLU) or BN
    int out_cols;      // columns of the output (F for up, d for down)
    uint16_t* out;     // bf16 [rows_max, out_cols]
    const float* row_gate;
    const int32_t* row_token;   // gathered A: row r of the tile is x[row_token[r]]
    const uint8_t* a_base;      // gathered A: x
    uint32_t a_row_bytes;       // gathered A: bytes of one x row (x is below 4 GB)
    uint16_t* out_z;            // up projection, optional: the pre-activation, bf16 [rows_max, N1]
    const uint16_t* in_z;       // activation backward: the pre-activation, bf16 [rows_max, N1]
    int z_cols;                 // columns of out_z / in_z (N1)
    float* out_f32;             // weight gradient: fp32 [E, m_rows, out_cols]; identity epilogue: fp32
                                // [rows_max, out_cols]; nullptr: bf16 into out
    int m_tiles;                // weight gradient: M-tiles per expert, ceil(m_rows / BM)
    int m_rows;                 // weight gradient: rows M of each expert's gradient
    int lda;                    // MODE_WGRAD_ROWS: row stride of A in elements (>= m_rows)
    int n_fastest;              // tile order N-fastest inside an expert (default: M-fastest)
    int tail_halves;            // let a short last wave run as 128-column units (see unit_tile)
    int tma_store;              // gate epilogue: output tiles through shared memory and TMA stores
    unsigned long long wait_limit;
};

// Where the A operand and the K range come from:
//   MODE_ROWS    A = x_perm rows of the expert's segment (TMA box), K = 0..K-1
//   MODE_GATHER  A = x rows at row_token[] (cp.async), K = 0..K-1
//   MODE_BMN     A as MODE_ROWS; B stored MN-major, [E * K rows, N cols] (N
//                contiguous: w2[e] as [d, F] or w1[e] as [N1, d]), loaded as
//                four 64x64 boxes per stage -- the data-gradient GEMMs of the
//                backward run on the weights as they are, without transposes
//   MODE_WGRAD   weight gradients: A [M, ld] and B [N, ld] are transposed,
//                segment-packed activations; expert e contracts over its own
//                K columns [64 kstart[e], 64 kstart[e+1]) (kept[e] rounded up
//                to 64, zero padded); every expert has m_tiles M-tiles; the
//                output is fp32 or bf16 [E, M, N] (zeros for an expert with
//                no rows)
//   MODE_WGRAD_ROWS  weight gradients straight from the row-major activations:
//                A [rows, M] and B [rows, N] are both read MN-major (two and
//                four 64x64 boxes per stage, rows = K); expert e contracts over
//                rows [offsets[e], offsets[e] + kept[e]) in blocks of 64 rows.
//                The rows of a last, partial block that lie past the segment
//                are zeroed in shared memory by the MMA warp before its MMAs
//                read the stage, so neighbouring segments or unwritten rows
//                never leak in; output as MODE_WGRAD
enum { MODE_ROWS = 0, MODE_GATHER = 1, MODE_WGRAD = 2, MODE_BMN = 3, MODE_WGRAD_ROWS = 4 };

// Tile -> (expert, M-tile, N-tile): M-fastest inside an expert, so the blocks
// running together share the B tile (the weights); n_fastest: N-fastest, so
// they share the A tile instead.
__device__ __forceinline__ void decode_tile(const int* mstart, int E, int n_tiles, int tile, int& e, int& m,
                                            int& n, bool n_fastest = false)
{
    e = find_expert(mstart, E, tile / n_tiles);
    const int local = tile - mstart[e] * n_tiles;
    if (n_fastest) {
        m = local / n_tiles;
        n = local - m * n_tiles;
        return;
    }
    const int mt = mstart[e + 1] - mstart[e];
    n = local / mt;
    m = local - n * mt;
}

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// Units of work of a launch.  The tiles are dealt to the blocks round-robin,
// so a launch of W whole waves plus R < grid tiles ends with a wave in which
// grid - R blocks idle for a whole tile time.  When R <= grid / 2, those R
// tiles run instead as 2R units of half the columns (BN/2), one per block:
// the last wave takes about half as long.  Units [0, full) are whole tiles
// (hv = -1); unit full + 2i + h is half h of tile full + i.  A half computes
// the same dot products over the same K order as the whole tile, so the
// output bits do not change.
__device__ __forceinline__ int unit_tile(int u, int full, int& hv)
{
    if (u < full) {
        hv = -1;
        return u;
    }
    hv = (u - full) & 1;
    return full + ((u - full) >> 1);
}

// Byte offsets in x of the 32 rows lane `lane` copies for `tile` (rows
// 4i + lane/8, plus its 16-byte chunk lane%8); rows past the expert's segment
// repeat a valid token (they are computed, never stored).
template <int N>
__device__ __forceinline__ void gather_offsets(const Args& g, const int* mstart, int tile, int lane, uint32_t (&off)[N])
{
    int e, m, n;
    decode_tile(mstart, g.E, g.n_tiles, tile, e, m, n, g.n_fastest != 0);
    const int rowA = __ldg(g.offsets + e) + m * BM;
    const int rows_valid = __ldg(g.kept + e) - m * BM;
    const int first = __ldg(g.row_token + rowA);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const int r = 4 * i + (lane >> 3);
        const int tok = r < rows_valid ? __ldg(g.row_token + rowA + r) : first;
        off[i] = (uint32_t)tok * g.a_row_bytes + (uint32_t)(lane & 7) * 16u;
    }
}

// MODE_GATHER: the A rows are read straight from x at row_token[] (the dispatch
// permutation), so no permuted copy of x is materialised.  The 32 lanes of
// the producer warp copy them with 16-byte cp.async (lane l: chunk l % 8 of
// rows 4i + l / 8, written to the 128-byte-swizzled place a TMA box load would
// use), and each lane's copies of a stage arrive on its full barrier when they
// land (33 arrivals: 32 lanes + lane 0's TMA transaction arrival for the B
// tile).  Those are generic-proxy writes: the MMA thread fences them into the
// async proxy after its wait and before its tcgen05.mma reads them.
template <int EPI, int BN, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const Args g)
{
    constexpr bool GATHER = MODE == MODE_GATHER, BMN = MODE == MODE_BMN, WGR = MODE == MODE_WGRAD_ROWS;
    constexpr bool WGRAD = MODE == MODE_WGRAD || WGR;   // weight-gradient tiles and epilogue
    static_assert(!(BMN || WGR) || BN == 256, "MN-major B is staged as four 64-column boxes");
    using SH = Shape<BN>;
    constexpr int STAGES = WGRAD ? SH::WG_STAGES : SH::STAGES;
    constexpr int STAGE_BYTES = SH::STAGE_BYTES, BH_BYTES = SH::BH_BYTES;
    constexpr int ACC_COLS = SH::ACC_COLS, TMEM_COLS = SH::TMEM_COLS;
    constexpr int BOX_BYTES = BK * 128;   // one 64x64 bf16 box
    // fp32 output tiles of the MN-major identity GEMM go out through the same
    // shared-memory staging and TMA stores as the weight gradients
    // the forward projections (bf16 rows of y_perm or h): whole 32-row blocks go out by TMA
    // stores as well -- per-thread stores of 32 different rows per warp instruction measured
    // 12-14% of the down GEMM at the many-expert shapes, where each tile has only 24 K blocks.
    // FWD_TMA: the column-wise epilogues (gate, GELU, identity) through the path below;
    // FWD_TMA_SW: SwiGLU, whose 64-column output blocks pair 64 gate and 64 up columns
    constexpr bool FWD_TMA = MODE == MODE_ROWS && (EPI == EPI_GATE || EPI == EPI_GELU || EPI == EPI_IDENT);
    constexpr bool FWD_TMA_SW = MODE == MODE_ROWS && EPI == EPI_SWIGLU && BN % 128 == 0;
    // the data-gradient GEMM dx_perm = dz . w1[e] (MN-major weights, bf16 output) likewise
    constexpr bool BMN_TMA = BMN && EPI == EPI_IDENT;
    constexpr bool TMA_OUT_OK = WGRAD || (BMN && EPI == EPI_IDENT) || FWD_TMA;
    constexpr uint32_t IDESC = WGR ? ptx::idesc_bf16_f32(128, BN, true, true)
                               : BMN ? ptx::idesc_bf16_f32(128, BN, true) : SH::IDESC;
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES], tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int mstart[257];
    __shared__ int kstart[WGRAD ? 257 : 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t smem0 = (ptx::smem_u32(dsmem) + 1023u) & ~1023u;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full_bar[s]), GATHER ? 33 : 1);
            ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_u32(&tfull_bar[a]), 1);
            ptx::mbar_init(ptx::smem_u32(&tempty_bar[a]), 128);
        }
        ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
        ptx::fence_mbar_init();
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
        if (WGRAD) ptx::tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_base_sh), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // launched as a programmatic dependent: the kernel before it (which wrote
    // kept[], the A rows, row_gate) has finished once this returns
    pdl_wait();
    if (warp == 2) {
        if (WGRAD) {
            for (int e = lane; e <= g.E; e += 32) mstart[e] = e * g.m_tiles;
        } else {
            build_mtile_prefix<BM>(g.kept, g.E, mstart, lane);
        }
    }
    if (WGRAD && warp == 3) build_mtile_prefix<BK>(g.kept, g.E, kstart, lane);   // K blocks per expert
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const uint32_t tmem_base = tmem_base_sh;
    const int total_tiles = mstart[g.E] * g.n_tiles;
    // half-width units for a short last wave: plain x_perm rows, 256-column
    // tiles whose columns are independent outputs (not the SwiGLU pairing)
    constexpr bool HALVES = MODE == MODE_ROWS && BN == 256 && (EPI == EPI_GATE || EPI == EPI_GELU || EPI == EPI_IDENT);
    const int tail = total_tiles % (int)gridDim.x;
    const bool halves = HALVES && g.tail_halves != 0 && tail > 0 && 2 * tail <= (int)gridDim.x;
    const int full_units = total_tiles - (halves ? tail : 0);
    const int total_units = full_units + (halves ? 2 * tail : 0);
    constexpr uint32_t IDESC_HALF = ptx::idesc_bf16_f32(128, BN / 2);
    // TMA stores of the forward output only where the GEMM is not bound by streaming its weights:
    // with fewer than 3 M-tiles per expert on average each weight tile serves at most ~2 row
    // tiles, the loads keep the TMA unit busy, and the stores measured slower there (e64_zipf up
    // GEMM 127 -> 148 us); per-thread stores then
    const bool tma_rows = g.tma_store != 0 && mstart[g.E] >= 3 * g.E;
    const int nk = (g.K + BK - 1) / BK;
    const uint64_t limit = g.wait_limit;

    if (warp == 0) {
        if (GATHER || lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            uint32_t roff[GATHER ? 32 : 1];   // gathered rows: this lane's 32 offsets in x
            for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
                int hv;
                const int tile = unit_tile(u, full_units, hv);
                int e, m, n;
                decode_tile(mstart, g.E, g.n_tiles, tile, e, m, n, g.n_fastest != 0);
                const int rowA = WGRAD ? m * BM : __ldg(g.offsets + e) + m * BM;
                const int rowB0 = (WGRAD ? 0 : e * g.b_rows) + n * g.n_step;
                const int rowB1 = rowB0 + g.half_off;
                const int kb0 = WGRAD ? kstart[e] : 0;
                const int nkt = WGRAD ? kstart[e + 1] - kb0 : nk;
                const int rowK0 = WGR ? __ldg(g.offsets + e) : 0;   // first row of the expert's segment
                if (GATHER) gather_offsets(g, mstart, tile, lane, roff);
                for (int kb = 0; kb < nkt; ++kb) {
                    bool got = true;
                    if (lane == 0) got = ptx::mbar_wait(ptx::smem_u32(&empty_bar[stage]), phase ^ 1u, limit);
                    if (GATHER) got = __shfl_sync(0xffffffffu, got, 0);
                    if (!got) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::smem_u32(&full_bar[stage]);
                    const uint32_t sa = smem0 + stage * STAGE_BYTES;
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(fb, GATHER ? 2 * BH_BYTES : hv < 0 ? STAGE_BYTES : A_BYTES + BH_BYTES);
                        const int kx = (kb0 + kb) * BK;
                        if (WGR) {
                            // rows rowK0 + 64 kb.. (K); A columns m*128.. (M), B columns n*256.. (N)
                            const int ky = rowK0 + kb * BK;
#pragma unroll
                            for (int j = 0; j < 2; ++j) ptx::tma_load_2d(sa + j * BOX_BYTES, &tmA, fb, m * BM + 64 * j, ky);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                ptx::tma_load_2d(sa + A_BYTES + j * BOX_BYTES, &tmB, fb, n * BN + 64 * j, ky);
                        } else {
                            if (!GATHER) ptx::tma_load_2d(sa, &tmA, fb, kx, rowA);
                            if (BMN) {
                                // B rows e*K + kx.. (K), columns n*BN + 64j.. (N): four 64x64 boxes
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    ptx::tma_load_2d(sa + A_BYTES + j * BOX_BYTES, &tmB, fb, n * BN + 64 * j,
                                                     e * g.K + kx);
                            } else if (hv < 0) {
                                ptx::tma_load_2d(sa + A_BYTES, &tmB, fb, kx, rowB0);
                                ptx::tma_load_2d(sa + A_BYTES + BH_BYTES, &tmB, fb, kx, rowB1);
                            } else {
                                // half unit: the BN/2 weight rows of its columns, first in the stage
                                ptx::tma_load_2d(sa + A_BYTES, &tmB, fb, kx, hv ? rowB1 : rowB0);
                            }
                        }
                    }
                    if (GATHER) {
                        const uint8_t* src = g.a_base + (size_t)kb * (BK * 2);
                        const int c = lane & 7;
#pragma unroll
                        for (int i = 0; i < (GATHER ? 32 : 1); ++i) {
                            const int r = 4 * i + (lane >> 3);
                            ptx::cp_async_16(sa + r * 128 + ((c ^ (r & 7)) << 4), src + roff[i]);
                        }
                        ptx::cp_async_mbar_arrive_noinc(fb);
                    }
                    ++fills;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (GATHER) ptx::cp_async_wait<0>();
            if (lane == 0) {
                if (!ok) moe_flag(MOE_DEV_TIMEOUT);
                // drain: the last fill of every stage must have landed before exit
                for (long long f = fills - 1; f >= 0 && f >= fills - STAGES; --f) {
                    const int s = (int)(f % STAGES);
                    const uint32_t par = (uint32_t)((f / STAGES) & 1);
                    if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), par, limit)) {
                        moe_flag(MOE_DEV_TIMEOUT);
                        break;
                    }
                }
            }
        }
        __syncwarp();   // reconverge before the block-wide barrier below
    } else if (warp == 1) {
        // lane 0 issues the MMAs; in MODE_WGRAD_ROWS the whole warp runs the
        // loop (every lane waits and votes) to zero the tails of partial blocks
        if (lane == 0 || WGR) {
            auto wait = [&](uint64_t* bar, uint32_t par) {
                const bool w = ptx::mbar_wait(ptx::smem_u32(bar), par, limit);
                return WGR ? __all_sync(0xffffffffu, w) : w;
            };
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
                int hv;
                const int tile = unit_tile(u, full_units, hv);
                const uint32_t idesc = hv < 0 ? IDESC : IDESC_HALF;
                if (!wait(&tempty_bar[acc], aphase ^ 1u)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                int nkt = nk, kept_e = 0;
                if (WGRAD) {
                    int e, m, n;
                    decode_tile(mstart, g.E, g.n_tiles, tile, e, m, n, g.n_fastest != 0);
                    nkt = kstart[e + 1] - kstart[e];   // 0: nothing accumulates, the epilogue writes zeros
                    if (WGR) kept_e = __ldg(g.kept + e);
                }
                for (int kb = 0; kb < nkt; ++kb) {
                    if (!wait(&full_bar[stage], phase)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = smem0 + stage * STAGE_BYTES, sb = sa + A_BYTES;
                    if (WGR) {
                        const int valid = kept_e - kb * BK;   // rows of this block inside the segment (>= 1)
                        if (valid < BK) {
                            // rows [valid, 64) of the six boxes are whole 128-byte lines: zero them
                            for (int b6 = 0; b6 < 6; ++b6)
                                for (int c = valid * 8 + lane; c < BK * 8; c += 32)
                                    ptx::st_shared_v4(sa + b6 * BOX_BYTES + c * 16, 0u, 0u, 0u, 0u);
                            ptx::fence_proxy_async_smem();   // generic writes before the MMAs read them
                        }
                        __syncwarp();
                    }
                    if (lane == 0) {
                        if (GATHER) ptx::fence_proxy_async_smem();   // the A tile came through the generic proxy
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            // K-major: 16 K columns = 32 bytes on; MN-major: 16 K rows = 2048 bytes on
                            const uint64_t adesc = WGR ? ptx::sdesc_mnmajor_sw128(sa + kk * 2048, BOX_BYTES)
                                                       : ptx::sdesc_kmajor_sw128(sa + kk * 32);
                            const uint64_t bdesc = (BMN || WGR) ? ptx::sdesc_mnmajor_sw128(sb + kk * 2048, BOX_BYTES)
                                                                : ptx::sdesc_kmajor_sw128(sb + kk * 32);
                            ptx::mma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0);
                        }
                        ptx::mma_commit(ptx::smem_u32(&empty_bar[stage]));
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (lane == 0) ptx::mma_commit(ptx::smem_u32(&tfull_bar[acc]));
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            if (lane == 0) {
                if (!ok) moe_flag(MOE_DEV_TIMEOUT);
                // no MMA may still write TMEM when the block frees it
                ptx::mma_commit(ptx::smem_u32(&drain_bar));
                if (!ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, limit)) moe_flag(MOE_DEV_TIMEOUT);
            }
        }
        __syncwarp();   // reconverge before the block-wide barrier below
    } else {
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        const int r_in = q * 32 + lane;    // row of the tile owned by this thread
        int acc = 0;
        uint32_t aphase = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
            int hv;
            const int tile = unit_tile(u, full_units, hv);
            int e, m, n;
            decode_tile(mstart, g.E, g.n_tiles, tile, e, m, n, g.n_fastest != 0);
            const int rows_valid = WGRAD ? g.m_rows - m * BM : __ldg(g.kept + e) - m * BM;
            const int row = WGRAD ? e * g.m_rows + m * BM + r_in : __ldg(g.offsets + e) + m * BM + r_in;
            const bool rv = r_in < rows_valid;
            // the row's gate does not depend on the MMAs: its load is in flight during the wait
            const float gate_pre = (EPI == EPI_GATE && rv) ? __ldg(g.row_gate + row) : 0.f;
            const bool waited = ptx::mbar_wait(ptx::smem_u32(&tfull_bar[acc]), aphase, limit);
            if (!__all_sync(0xffffffffu, waited)) {
                moe_flag(MOE_DEV_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            if (TMA_OUT_OK && (WGRAD || g.out_f32 != nullptr || ((FWD_TMA || BMN_TMA) && tma_rows))) {
                const bool empty = WGRAD && kstart[e + 1] == kstart[e];
                const float gsc = gate_pre;   // gate epilogue: the row's gate
                // this warp's 32 rows all inside the expert's M rows: stage each block of
                // 32 rows x 128 bytes in shared memory (128-byte swizzle) and store it with
                // TMA; otherwise (a ragged last M-tile) masked per-thread stores
                const bool whole = rows_valid >= q * 32 + 32;
                const bool f32_out = g.out_f32 != nullptr;
                const uint32_t stg = smem0 + STAGES * STAGE_BYTES + q * SH::WG_STAGE_OUT;
                const int step = f32_out ? 32 : 64;   // output columns per 128-byte row block
                // a half-width unit: BN/2 columns from accumulator column 0
                const int ncols = hv < 0 ? BN : BN / 2;
                const int col0 = n * BN + (hv > 0 ? BN / 2 : 0);
#pragma unroll 1
                for (int c = 0; c < ncols; c += step) {
                    uint32_t av[32], bv[32];
                    if (!empty) {
                        ptx::tmem_ld32(tb + c, av);
                        if (!f32_out) ptx::tmem_ld32(tb + c + 32, bv);
                        ptx::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) av[i] = bv[i] = 0u;
                    }
                    if (EPI == EPI_GATE) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            av[i] = __float_as_uint(f32(av[i]) * gsc);
                            bv[i] = __float_as_uint(f32(bv[i]) * gsc);
                        }
                    } else if (EPI == EPI_GELU) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            av[i] = __float_as_uint(gelu_f32(f32(av[i])));
                            bv[i] = __float_as_uint(gelu_f32(f32(bv[i])));
                        }
                    }
                    const int col = col0 + c;
                    if (col >= g.out_cols) continue;
                    uint32_t w[32];   // this thread's 128 output bytes
                    if (f32_out) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) w[i] = av[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            w[i] = pack_bf16x2(f32(av[2 * i]), f32(av[2 * i + 1]));
                            w[16 + i] = pack_bf16x2(f32(bv[2 * i]), f32(bv[2 * i + 1]));
                        }
                    }
                    if (whole) {
                        if (lane == 0) ptx::bulk_wait_group_read<0>();   // the previous block has left smem
                        __syncwarp();
                        const uint32_t rb = stg + lane * 128;
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            ptx::st_shared_v4(rb + ((v ^ (lane & 7)) << 4), w[4 * v], w[4 * v + 1], w[4 * v + 2],
                                              w[4 * v + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&tmC, stg, col, row - lane);
                            ptx::bulk_commit_group();
                        }
                    } else if (rv) {
                        uint4* dst = f32_out ? reinterpret_cast<uint4*>(g.out_f32 + (size_t)row * g.out_cols + col)
                                             : reinterpret_cast<uint4*>(g.out + (size_t)row * g.out_cols + col);
#pragma unroll
                        for (int v = 0; v < 8; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                    }
                }
            } else if (FWD_TMA_SW && tma_rows) {
                // SwiGLU outputs in blocks of 64 columns (gate columns c.., up columns BN/2 + c..),
                // whole 32-row blocks staged in shared memory and stored by TMA
                const bool whole = rows_valid >= q * 32 + 32;
                const uint32_t stg = smem0 + STAGES * STAGE_BYTES + q * SH::WG_STAGE_OUT;
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 64) {
                    uint32_t w[32];   // this thread's 64 outputs
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        uint32_t gv[32], uv[32];
                        ptx::tmem_ld32(tb + c + 32 * h2, gv);
                        ptx::tmem_ld32(tb + BN / 2 + c + 32 * h2, uv);
                        ptx::tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[16 * h2 + i] = pack_bf16x2(silu_f32(f32(gv[2 * i])) * f32(uv[2 * i]),
                                                         silu_f32(f32(gv[2 * i + 1])) * f32(uv[2 * i + 1]));
                    }
                    const int col = n * (BN / 2) + c;
                    if (col >= g.out_cols) continue;
                    if (whole) {
                        if (lane == 0) ptx::bulk_wait_group_read<0>();   // the previous block has left smem
                        __syncwarp();
                        const uint32_t rb = stg + lane * 128;
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            ptx::st_shared_v4(rb + ((v ^ (lane & 7)) << 4), w[4 * v], w[4 * v + 1], w[4 * v + 2],
                                              w[4 * v + 3]);
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            ptx::tma_store_2d(&tmC, stg, col, row - lane);
                            ptx::bulk_commit_group();
                        }
                    } else if (rv) {
                        uint4* dst = reinterpret_cast<uint4*>(g.out + (size_t)row * g.out_cols + col);
#pragma unroll
                        for (int v = 0; v < 8; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                    }
                }
            } else if (EPI == EPI_SWIGLU) {
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    uint32_t gv[32], uv[32];
                    ptx::tmem_ld32(tb + c, gv);
                    ptx::tmem_ld32(tb + BN / 2 + c, uv);
                    ptx::tmem_ld_wait();
                    const int col = n * (BN / 2) + c;
                    if (rv && col < g.out_cols && g.out_z) {
                        // keep the pre-activation (gate | up) for the backward
                        uint32_t zg[16], zu[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            zg[i] = pack_bf16x2(f32(gv[2 * i]), f32(gv[2 * i + 1]));
                            zu[i] = pack_bf16x2(f32(uv[2 * i]), f32(uv[2 * i + 1]));
                        }
                        uint4* dg = reinterpret_cast<uint4*>(g.out_z + (size_t)row * g.z_cols + col);
                        uint4* du = reinterpret_cast<uint4*>(g.out_z + (size_t)row * g.z_cols + g.out_cols + col);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            dg[v] = make_uint4(zg[4 * v], zg[4 * v + 1], zg[4 * v + 2], zg[4 * v + 3]);
                            du[v] = make_uint4(zu[4 * v], zu[4 * v + 1], zu[4 * v + 2], zu[4 * v + 3]);
                        }
                    }
                    if (rv && col < g.out_cols) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(silu_f32(f32(gv[2 * i])) * f32(uv[2 * i]),
                                                silu_f32(f32(gv[2 * i + 1])) * f32(uv[2 * i + 1]));
                        uint4* dst = reinterpret_cast<uint4*>(g.out + (size_t)row * g.out_cols + col);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
            } else {
                const float gate = gate_pre;
                // a half unit: BN/2 columns from accumulator column 0
                const int ncols = hv < 0 ? BN : BN / 2;
                const int col0 = n * BN + (hv > 0 ? BN / 2 : 0);
#pragma unroll 1
                for (int c = 0; c < ncols; c += 32) {
                    uint32_t av[32];
                    ptx::tmem_ld32(tb + c, av);
                    const int col = col0 + c;
                    if (EPI == EPI_DGELU || EPI == EPI_DSWIGLU) {
                        // z loads issued before the TMEM wait; 32 columns of this row
                        uint4 zg[4], zu[4];
                        const bool live = rv && col < g.out_cols;
                        const uint16_t* zr = g.in_z + (size_t)row * g.z_cols + col;
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            zg[v] = live ? ldg_nc_v4(zr + 8 * v) : make_uint4(0, 0, 0, 0);
                            if (EPI == EPI_DSWIGLU)
                                zu[v] = live ? ldg_nc_v4(zr + g.out_cols + 8 * v) : make_uint4(0, 0, 0, 0);
                        }
                        ptx::tmem_ld_wait();
                        if (live) {
                            uint32_t pg[16], pu[16];
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                float a[8], u[8];
                                unpack_bf16x8(zg[v], a);
                                if (EPI == EPI_DSWIGLU) unpack_bf16x8(zu[v], u);
#pragma unroll
                                for (int i = 0; i < 8; i += 2) {
                                    float o[2], ou[2];
#pragma unroll
                                    for (int h = 0; h < 2; ++h) {
                                        const float da = f32(av[8 * v + i + h]), z = a[i + h];
                                        if (EPI == EPI_DGELU) {
                                            const float cdf = 0.5f * (1.0f + erff(z * 0.70710678118654752f));
                                            const float pdf = 0.39894228040143268f * expf(-0.5f * z * z);
                                            o[h] = da * (cdf + z * pdf);
                                        } else {
                                            const float sg = 1.0f / (1.0f + expf(-z));
                                            o[h] = da * u[i + h] * (sg * (1.0f + z * (1.0f - sg)));
                                            ou[h] = da * (z * sg);
                                        }
                                    }
                                    pg[4 * v + i / 2] = pack_bf16x2(o[0], o[1]);
                                    if (EPI == EPI_DSWIGLU) pu[4 * v + i / 2] = pack_bf16x2(ou[0], ou[1]);
                                }
                            }
                            uint4* dg = reinterpret_cast<uint4*>(g.out + (size_t)row * g.z_cols + col);
#pragma unroll
                            for (int v = 0; v < 4; ++v) dg[v] = make_uint4(pg[4 * v], pg[4 * v + 1], pg[4 * v + 2], pg[4 * v + 3]);
                            if (EPI == EPI_DSWIGLU) {
                                uint4* du = reinterpret_cast<uint4*>(g.out + (size_t)row * g.z_cols + g.out_cols + col);
#pragma unroll
                                for (int v = 0; v < 4; ++v)
                                    du[v] = make_uint4(pu[4 * v], pu[4 * v + 1], pu[4 * v + 2], pu[4 * v + 3]);
                            }
                        }
                        continue;
                    }
                    ptx::tmem_ld_wait();
                    if (EPI != EPI_GATE && rv && col < g.out_cols && g.out_z) {
                        uint32_t zk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) zk[i] = pack_bf16x2(f32(av[2 * i]), f32(av[2 * i + 1]));
                        uint4* dz = reinterpret_cast<uint4*>(g.out_z + (size_t)row * g.z_cols + col);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dz[v] = make_uint4(zk[4 * v], zk[4 * v + 1], zk[4 * v + 2], zk[4 * v + 3]);
                    }
                    if (EPI == EPI_IDENT && g.out_f32) {   // fp32 output, no rounding
                        if (rv && col < g.out_cols) {
                            float4* dst = reinterpret_cast<float4*>(g.out_f32 + (size_t)row * g.out_cols + col);
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                dst[v] = make_float4(f32(av[4 * v]), f32(av[4 * v + 1]), f32(av[4 * v + 2]),
                                                     f32(av[4 * v + 3]));
                        }
                        continue;
                    }
                    if (rv && col < g.out_cols) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float z0 = f32(av[2 * i]), z1 = f32(av[2 * i + 1]);
                            if (EPI == EPI_GELU) {
                                z0 = gelu_f32(z0);
                                z1 = gelu_f32(z1);
                            } else if (EPI == EPI_GATE) {
                                z0 *= gate;
                                z1 *= gate;
                            }
                            pk[i] = pack_bf16x2(z0, z1);
                        }
                        uint4* dst = reinterpret_cast<uint4*>(g.out + (size_t)row * g.out_cols + col);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_u32(&tempty_bar[acc]));
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
        }
        if ((TMA_OUT_OK || FWD_TMA_SW) &&
            (WGRAD || g.out_f32 != nullptr || ((FWD_TMA || FWD_TMA_SW || BMN_TMA) && tma_rows)) && lane == 0)
            ptx::bulk_wait_group<0>();   // every output store has completed
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace tcg
