// bf16 grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2), weights on
// the 256-row side ("swap-AB").
//
// Same operation as ffn_tc.cuh (expert-parallelism tutorial
// "专家并行：混合专家模型的分布式训练方案" §2.1 step 4, with the d -> d_ff -> d
// expert of the ETP page "ETP专家并行加速MoE模型：ms-swift中稀疏架构的极致优化"), laid
// out for two SMs per tile:
//
//   D[256 weight rows, N tokens] = W[256 rows, K] . X[N tokens, K]^T
//
// Each CTA of a pair stages 128 weight rows and N/2 token rows per K block
// (32 KB), so a 6-stage ring fits and every SM loads 1/3 fewer bytes per
// tensor-core cycle than a 1-SM 128x256 tile.  N is the token count of the
// tile rounded up to 32 (at most 256), so a ragged expert segment costs no
// tensor work beyond its last 32 tokens.  Tiles run token-tile fastest inside
// (expert, weight tile), so the pairs working at the same time share one
// weight tile through L2.
//
// Roles (6 warps per CTA, in both CTAs of the pair):
//   warp 0     TMA producer: its CTA's weight rows (two 64-row boxes) and
//              token rows (one 128-row box); completion is counted on the
//              leader CTA's full barrier, which expects both CTAs' bytes
//   warp 1     (leader CTA only) single-thread tcgen05.mma M=256 N=tile;
//              commits free each ring stage and publish each accumulator in
//              both CTAs; two 256-column accumulators per CTA
//   warps 2-5  epilogue: TMEM lane = weight row, column = token; values go
//              through a small shared-memory transpose so every store is a
//              run of 16-byte vectors along one token's output row
// SwiGLU: each CTA's 128 weight rows are 64 gate rows and the 64 matching up
// rows, so gate and up of one output meet in the same CTA (lanes r and r+64).
//
// Waits on mbarriers are bounded (error flag + orderly exit).  The only
// unbounded waits are the two cluster barriers at entry and exit, which both
// CTAs of the pair always reach.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"
#include "tiles.cuh"

namespace tc2 {

constexpr int BMW = 256;                       // weight rows per pair tile
constexpr int BNT = 256;                       // max tokens per tile
constexpr int BK = 64;
constexpr int A_BYTES = 128 * BK * 2;          // 16 KB: this CTA's weight rows
constexpr int B_BYTES = 128 * BK * 2;          // 16 KB: one 128-row token box
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STAGES = 6;
constexpr int THREADS = 192;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int XPOSE_FLOATS = 32 * 33;          // per epilogue warp
constexpr int UP_FLOATS = 64 * 33;             // SwiGLU up values of one chunk
constexpr int SMEM_DYN = STAGES * STAGE_BYTES + (4 * XPOSE_FLOATS + UP_FLOATS) * 4 + BNT * 4 + 1024;

enum { EPI_GELU = 0, EPI_SWIGLU = 1, EPI_IDENT = 2, EPI_GATE = 3 };

struct Args {
    const int32_t* offsets;
    const int32_t* kept;
    int E;
    int K;             // reduction length (d for up, F for down)
    int n_wtiles;      // weight tiles per expert
    int w_rows;        // rows of one expert's weight in the 2-D view [E*w_rows, K]
    int F;             // SwiGLU: row offset of the up half
    int out_cols;      // columns of the output (F for up, d for down)
    uint16_t* out;     // bf16 [rows_max, out_cols]
    const float* row_gate;
    unsigned long long wait_limit;
};

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// Tile p -> expert, token tile, weight tile (token tile fastest).
__device__ __forceinline__ void decode(const int* tstart, int E, int n_wtiles, int p, int& e, int& nt, int& mw)
{
    e = find_expert(tstart, E, p / n_wtiles);
    const int local = p - tstart[e] * n_wtiles;
    const int ntok = tstart[e + 1] - tstart[e];
    mw = local / ntok;
    nt = local - mw * ntok;
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const Args g)
{
    extern __shared__ uint8_t dsmem[];
    __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int tstart[257];
    __shared__ int epi_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx2::cluster_rank();
    const bool leader = rank == 0;
    const uint32_t smem0 = (ptx::smem_u32(dsmem) + 1023u) & ~1023u;
    uint8_t* smem0_ptr = dsmem + (smem0 - ptx::smem_u32(dsmem));
    float* xpose = reinterpret_cast<float*>(smem0_ptr + STAGES * STAGE_BYTES);
    float* upbuf = xpose + 4 * XPOSE_FLOATS;
    float* gates = upbuf + UP_FLOATS;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_u32(&tfull_bar[a]), 1);
            ptx::mbar_init(ptx::smem_u32(&tempty_bar[a]), 8);   // 4 epilogue warps x 2 CTAs
        }
        ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
        epi_abort = 0;
        ptx::fence_mbar_init();
        ptx::tma_prefetch_desc(&tmW);
        ptx::tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        ptx2::tmem_alloc(ptx::smem_u32(&tmem_base_sh), TMEM_COLS);
        ptx2::tmem_relinquish();
    }
    if (warp == 2) build_mtile_prefix<BNT>(g.kept, g.E, tstart, lane);
    __syncwarp();
    ptx::tc_fence_before();
    ptx2::cluster_sync();   // barriers of both CTAs initialised before any remote use
    ptx::tc_fence_after();

    const uint32_t tmem_base = tmem_base_sh;
    const int total = tstart[g.E] * g.n_wtiles;
    const int nk = (g.K + BK - 1) / BK;
    const uint64_t limit = g.wait_limit;
    const int pair = (int)ptx2::cluster_id_x(), npairs = (int)ptx2::nclusters_x();

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            for (int p = pair; ok && p < total; p += npairs) {
                int e, nt, mw;
                decode(tstart, g.E, g.n_wtiles, p, e, nt, mw);
                const int kept_e = __ldg(g.kept + e);
                const int nvalid = min(BNT, kept_e - nt * BNT);
                const int n32 = (nvalid + 31) & ~31;
                const int tok_row = __ldg(g.offsets + e) + nt * BNT + (int)rank * (n32 / 2);
                int wrow0, wrow1;
                if (EPI == EPI_SWIGLU) {
                    const int f0 = mw * 128 + (int)rank * 64;
                    wrow0 = e * g.w_rows + f0;
                    wrow1 = wrow0 + g.F;
                } else {
                    wrow0 = e * g.w_rows + mw * BMW + (int)rank * 128;
                    wrow1 = wrow0 + 64;
                }
                for (int kb = 0; kb < nk; ++kb) {
                    if (!ptx2::mbar_wait_cluster(ptx::smem_u32(&empty_bar[stage]), phase ^ 1u, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = ptx::smem_u32(&full_bar[stage]);
                    const uint32_t fb = ptx2::mapa(fb_local, 0);
                    if (leader) ptx::mbar_arrive_expect_tx(fb_local, 2 * STAGE_BYTES);
                    const uint32_t sa = smem0 + stage * STAGE_BYTES;
                    ptx2::tma_load_2d_pair(sa, &tmW, fb, kb * BK, wrow0);
                    ptx2::tma_load_2d_pair(sa + A_BYTES / 2, &tmW, fb, kb * BK, wrow1);
                    ptx2::tma_load_2d_pair(sa + A_BYTES, &tmX, fb, kb * BK, tok_row);
                    ++fills;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            // the last fill of each stage is known to have landed once the MMA that
            // read it freed the stage
            for (long long f = fills - 1; f >= 0 && f >= fills - STAGES; --f) {
                const int s = (int)(f % STAGES);
                const uint32_t par = (uint32_t)((f / STAGES) & 1);
                if (!ptx2::mbar_wait_cluster(ptx::smem_u32(&empty_bar[s]), par, limit)) {
                    moe_flag(MOE_DEV_TIMEOUT);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            for (int p = pair; ok && p < total; p += npairs) {
                int e, nt, mw;
                decode(tstart, g.E, g.n_wtiles, p, e, nt, mw);
                const int nvalid = min(BNT, __ldg(g.kept + e) - nt * BNT);
                const int n32 = (nvalid + 31) & ~31;
                const uint32_t idesc = ptx::idesc_bf16_f32(256, n32);
                if (!ptx2::mbar_wait_cluster(ptx::smem_u32(&tempty_bar[acc]), aphase ^ 1u, limit)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!ptx2::mbar_wait_cluster(ptx::smem_u32(&full_bar[stage]), phase, limit)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = smem0 + stage * STAGE_BYTES, sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        ptx2::mma_bf16(d_tmem, ptx::sdesc_kmajor_sw128(sa + kk * 32), ptx::sdesc_kmajor_sw128(sb + kk * 32),
                                       idesc, (kb | kk) != 0);
                    ptx2::mma_commit_multicast(ptx::smem_u32(&empty_bar[stage]), 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx2::mma_commit_multicast(ptx::smem_u32(&tfull_bar[acc]), 0x3);
                acc ^= 1;
                if (acc == 0) aphase ^= 1u;
            }
            if (!ok) moe_flag(MOE_DEV_TIMEOUT);
            // no MMA may still write TMEM when the pair frees it
            ptx2::mma_commit_multicast(ptx::smem_u32(&drain_bar), 0x1);
            if (!ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, limit)) moe_flag(MOE_DEV_TIMEOUT);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;              // TMEM lane quarter of this warp
        const int ew = warp - 2;             // epilogue warp index 0..3
        float* xp = xpose + ew * XPOSE_FLOATS;
        int acc = 0;
        uint32_t aphase = 0;
        for (int p = pair; p < total; p += npairs) {
            int e, nt, mw;
            decode(tstart, g.E, g.n_wtiles, p, e, nt, mw);
            const int nvalid = min(BNT, __ldg(g.kept + e) - nt * BNT);
            const int tok0 = __ldg(g.offsets + e) + nt * BNT;
            // previous tile's readers of `gates` / `upbuf` are done before they change
            ptx::named_bar_sync(1, 128);
            if (EPI == EPI_GATE)
                for (int j = threadIdx.x - 64; j < nvalid; j += 128) gates[j] = __ldg(g.row_gate + tok0 + j);
            const bool waited = ptx2::mbar_wait_cluster(ptx::smem_u32(&tfull_bar[acc]), aphase, limit);
            if (!__all_sync(0xffffffffu, waited) && lane == 0) epi_abort = 1;
            // every epilogue warp reaches this barrier, so the decision below is uniform
            ptx::named_bar_sync(1, 128);
            if (epi_abort) {
                moe_flag(MOE_DEV_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            // output features of this warp's 32 rows (SwiGLU: rows 0-63 gate, 64-127 up)
            int fbase;
            if (EPI == EPI_SWIGLU) fbase = mw * 128 + (int)rank * 64 + (q & 1) * 32;
            else fbase = mw * BMW + (int)rank * 128 + q * 32;
            const bool fvalid = fbase < g.out_cols;
            for (int c = 0; c < nvalid; c += 32) {
                uint32_t v[32];
                ptx::tmem_ld32(tb + c, v);
                ptx::tmem_ld_wait();
                if (EPI == EPI_SWIGLU) {
                    if (q >= 2)
#pragma unroll
                        for (int j = 0; j < 32; ++j) upbuf[((q - 2) * 32 + lane) * 33 + j] = f32(v[j]);
                    ptx::named_bar_sync(1, 128);
                    if (q < 2) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            xp[j * 33 + lane] = silu_f32(f32(v[j])) * upbuf[(q * 32 + lane) * 33 + j];
                    }
                    ptx::named_bar_sync(1, 128);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        float z = f32(v[j]);
                        if (EPI == EPI_GELU) z = gelu_f32(z);
                        else if (EPI == EPI_GATE) z *= (c + j < nvalid) ? gates[c + j] : 0.f;
                        xp[j * 33 + lane] = z;
                    }
                    __syncwarp();
                }
                // lane j writes token c+j: 32 consecutive outputs = 4 x 16 B
                if ((EPI != EPI_SWIGLU || q < 2) && fvalid && c + lane < nvalid) {
                    const float* src = xp + lane * 33;
                    uint4* dst = reinterpret_cast<uint4*>(g.out + (size_t)(tok0 + c + lane) * g.out_cols + fbase);
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4)
                        dst[v4] = make_uint4(pack_bf16x2(src[8 * v4 + 0], src[8 * v4 + 1]),
                                             pack_bf16x2(src[8 * v4 + 2], src[8 * v4 + 3]),
                                             pack_bf16x2(src[8 * v4 + 4], src[8 * v4 + 5]),
                                             pack_bf16x2(src[8 * v4 + 6], src[8 * v4 + 7]));
                }
                __syncwarp();
            }
            ptx::tc_fence_before();
            if (lane == 0) ptx2::mbar_arrive_remote(ptx2::mapa(ptx::smem_u32(&tempty_bar[acc]), 0));
            acc ^= 1;
            if (acc == 0) aphase ^= 1u;
        }
    }

    ptx::tc_fence_before();
    ptx2::cluster_sync();   // neither CTA leaves while the pair's MMAs or arrivals may touch it
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx2::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace tc2
