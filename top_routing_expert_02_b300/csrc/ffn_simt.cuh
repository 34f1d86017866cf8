// True-fp32 expert FFN on CUDA cores (the fp32 layer: no TF32, no bf16).
//
// Expert-parallelism tutorial "专家并行：混合专家模型的分布式训练方案" §2.1 step 4:
// each expert runs its FFN on the rows it received.  Up:  h = act(x_perm
// w1[e]^T); down: y_perm = row_gate * (h w2[e]^T).  32x32 output tiles, one
// expert per tile; every output is one fp32 FMA chain over K in order.
#pragma once
#include "common.cuh"
#include "tiles.cuh"

namespace simt {

constexpr int BM = 32, BN = 32, BK = 32, THREADS = 256;
enum { ACT_GELU = 0, ACT_SWIGLU = 1, ACT_IDENT = 2, ACT_GATE = 3 };

// ACT_GATE is the down-projection (K = F, N = d, output scaled by row_gate).
template <int ACT>
__global__ void __launch_bounds__(THREADS)
ffn_simt_kernel(const float* __restrict__ A, const int32_t* __restrict__ offsets,
                const int32_t* __restrict__ kept, int E, int K, int N, int F,
                const float* __restrict__ Wt, const float* __restrict__ row_gate, float* __restrict__ out)
{
    __shared__ int mstart[257];
    __shared__ float As[BK][BM + 1], Bg[BK][BN + 1], Bu[BK][BN + 1];
    const int tid = threadIdx.x, tx = tid & 31, ty = tid >> 5;
    if (tid < 32) build_mtile_prefix<BM>(kept, E, mstart, tid);
    __syncthreads();
    const int mt = blockIdx.y;
    if (mt >= mstart[E]) return;
    const int e = find_expert(mstart, E, mt);
    const int m = mt - mstart[e];
    const int rows_valid = __ldg(kept + e) - m * BM;
    const int row0 = __ldg(offsets + e) + m * BM;
    const int n0 = blockIdx.x * BN;
    // rows of this expert's weight matrix in [rows, K] layout
    const int wrows = (ACT == ACT_SWIGLU) ? 2 * F : N;
    const float* W = Wt + (size_t)e * wrows * K;

    float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int v = tid; v < BM * BK; v += THREADS) {
            const int r = v / BK, kk = v % BK;
            As[kk][r] = (r < rows_valid) ? __ldg(A + (size_t)(row0 + r) * K + k0 + kk) : 0.f;
            Bg[kk][r] = __ldg(W + (size_t)(n0 + r) * K + k0 + kk);
            if (ACT == ACT_SWIGLU) Bu[kk][r] = __ldg(W + (size_t)(F + n0 + r) * K + k0 + kk);
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            const float bg = Bg[kk][tx];
            const float bu = (ACT == ACT_SWIGLU) ? Bu[kk][tx] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float a = As[kk][ty + 8 * i];
                ag[i] = fmaf(a, bg, ag[i]);
                if (ACT == ACT_SWIGLU) au[i] = fmaf(a, bu, au[i]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty + 8 * i;
        if (r >= rows_valid) continue;
        const float z = ag[i];
        float o;
        if (ACT == ACT_GELU) o = gelu_f32(z);
        else if (ACT == ACT_SWIGLU) o = silu_f32(z) * au[i];
        else if (ACT == ACT_IDENT) o = z;
        else o = __ldg(row_gate + row0 + r) * z;
        out[(size_t)(row0 + r) * N + n0 + tx] = o;
    }
}

}  // namespace simt
