// C ABI of the MoE-layer forward (see include/moe_b300.h for the contract).
//
// One translation unit: the kernels live in the headers included below and
// share the device status word defined in common.cuh.  This file validates
// arguments, encodes TMA tensor maps, picks launch shapes and enqueues the
// kernels; it allocates nothing.
#include <atomic>
#include <initializer_list>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "backward.cuh"
#include "combine.cuh"
#include "dispatch.cuh"
#include "ffn_simt.cuh"
#include "ffn_tc.cuh"
#include "ffn_tc2.cuh"
#include "route.cuh"
#include "route_fused.cuh"
#include "route_small.cuh"

namespace {

constexpr int MAX_E = 256;
constexpr int MAX_K = 16;
constexpr unsigned long long DEFAULT_WAIT_LIMIT = 4000000000ull;   // ~2 s of SM cycles
std::atomic<unsigned long long> g_wait_limit{DEFAULT_WAIT_LIMIT};
std::atomic<int> g_forced_bn{0};   // 0: pick the GEMM tile width per call
std::atomic<int> g_wgrad_order{0};  // weight-gradient tile order: 0 automatic, 1 M-fastest, 2 N-fastest
std::atomic<int> g_gemm_order{0};   // forward / data-gradient tile order: 0 automatic (M-fastest), 1 M-fastest, 2 N-fastest
std::atomic<int> g_gemm_tail{1};    // a short last wave of forward tiles runs as half-width units: 1 on, 0 off
std::atomic<int> g_gemm_tma_store{1};   // down-projection output tiles by TMA stores: 1 on, 0 per-thread stores

// Weight-gradient tile order.  N-fastest (the blocks running together share
// the A tile and write neighbouring column blocks of the same output rows)
// measured 3-7% faster for dw1 on the e8 and e128 layers and for dw2 on e8,
// 2-4% slower for dw2 on e128; it is the automatic choice.
inline int wgrad_n_fastest(int, int)
{
    return g_wgrad_order.load() == 1 ? 0 : 1;
}
std::atomic<int> g_gemm_kind{0};   // 0 auto, 1 one-SM tiles, 2 CTA-pair tiles

inline bool dtype_ok(int dt) { return dt == MOE_F32 || dt == MOE_BF16; }
inline int esize(moe_dtype dt) { return dt == MOE_BF16 ? 2 : 4; }

inline moe_status launch_status()
{
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        std::fprintf(stderr, "moe_b300: CUDA error: %s\n", cudaGetErrorString(e));
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

// Status of a cudaLaunchKernelEx call (its error is also cleared from the
// runtime's last-error slot).
inline moe_status launch_ex_status(cudaError_t e)
{
    if (e != cudaSuccess) {
        std::fprintf(stderr, "moe_b300: CUDA launch error: %s\n", cudaGetErrorString(e));
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    return launch_status();
}

// Launch configuration of a kernel that is a programmatic dependent of the
// kernel before it in the stream (it may start once that kernel has called
// griddepcontrol.launch_dependents; it calls griddepcontrol.wait before it
// reads that kernel's results).
std::atomic<int> g_pdl{1};   // programmatic dependent launches: 1 on, 0 plain stream order
std::atomic<int> g_router_kind{0};   // bf16 router: 0 automatic (tensor cores), 1 tensor cores, 2 CUDA cores for E <= 8
struct PdlLaunch {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg;
    PdlLaunch(int grid, int threads, cudaStream_t stream, size_t smem = 0)
    {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = g_pdl.load();
        cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3((unsigned)threads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    PdlLaunch(const PdlLaunch&) = delete;
};

// Blocks of `kern` that fit on one SM at once (at least 1).
template <typename K>
int resident_blocks(K kern, int threads, size_t dyn_smem = 0)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, dyn_smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    return n > 0 ? n : 1;
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

// Every buffer moved with 16-byte vectors or TMA must start on a 16-byte
// boundary; a misaligned pointer is refused before anything is enqueued.
static bool all_aligned16(std::initializer_list<const void*> ps)
{
    for (const void* p : ps)
        if (p && ((uintptr_t)p & 15u)) return false;
    return true;
}

// Router block shape: experts per lane and tokens per warp.
inline int route_epl(int E) { return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : 8; }
inline int route_tw(int E) { return route_epl(E) == 1 ? 2 : 4; }
inline int route_tokens_per_block(int E) { return route::WARPS * route_tw(E); }
inline size_t route_ws_bytes_simt(long long T, int E)
{
    const long long nblk = (T + route_tokens_per_block(E) - 1) / route_tokens_per_block(E);
    return (size_t)nblk * E * sizeof(float);
}

// Fused tensor-core router (bf16 x, E <= 128): launch shape.
struct RouteFuShape {
    int E_pad, emax, TPB, S, xstages, wstages, smem, ngroups, grid;
    uint32_t tmem_cols;
};
inline bool route_fu_shape(long long T, int d, int E, RouteFuShape* s)
{
    if (E > rfu::MAX_EPAD || T <= 0 || d % rfu::BK) return false;
    s->E_pad = (E + 15) / 16 * 16;
    s->emax = s->E_pad <= 16 ? 16 : s->E_pad <= 32 ? 32 : s->E_pad <= 64 ? 64 : 128;
    // E_pad <= 32: one MMA per tile and K step for the three stacked parts
    const bool fused_parts = s->emax <= 32;
    const long long ntiles = (T + rfu::BM - 1) / rfu::BM;
    const int tcols = rfu::tile_tmem_cols(fused_parts, s->E_pad);
    const int nk = d / rfu::BK;
    const long long sms = (long long)sm_count();
    // CTAs of one launch for TPB tiles per CTA: clusters of S CTAs split d
    // while the CTAs still fit on the GPU at once (one CTA per SM)
    auto splits = [&](long long groups) {
        int S = 1;
        while (S < rfu::MAX_SPLITS && 2 * S <= nk && groups * S * 2 <= sms) S *= 2;
        return S;
    };
    // two 128-token tiles per CTA (one weight block serves both) when their
    // TMEM columns fit and the launch still fills the GPU as well
    const long long g1 = ntiles, g2 = (ntiles + 1) / 2;
    const long long c1 = g1 * splits(g1), c2 = g2 * splits(g2);
    s->TPB = (2 * tcols <= 512 && ntiles >= 2 && (c2 >= c1 || c2 >= sms * 3 / 4)) ? 2 : 1;
    uint32_t c = 32;
    while (c < (uint32_t)(s->TPB * tcols)) c <<= 1;
    s->tmem_cols = c;
    // one CTA per SM: x and weight rings of the same depth in K blocks, as
    // deep as the 227 KB (less alignment and static use) allow.  (A shorter
    // weight ring with a deeper x ring measured slower: at small E the
    // weight boxes' L2 latency then shows, and at E = 128 it gained nothing.)
    const int xbytes = s->TPB * rfu::X_BYTES, wbytes = 3 * s->E_pad * 128;
    int st = (232448 - 1024 - 1536) / (xbytes + wbytes);
    if (st > rfu::MAX_XSTAGES) st = rfu::MAX_XSTAGES;
    if (st < 2) st = 2;
    s->xstages = s->wstages = st;
    const int ring = st * (xbytes + wbytes);
    const int fin = rfu::finish_smem_bytes(s->TPB, s->E_pad);
    s->smem = (ring > fin ? ring : fin) + 1024;
    s->ngroups = (int)((ntiles + s->TPB - 1) / s->TPB);
    s->S = splits(s->ngroups);
    s->grid = s->ngroups * s->S;
    return true;
}
inline size_t align256(size_t n) { return (n + 255) / 256 * 256; }
// Workspace of the tensor-core router: the three bf16 parts of the weight
// [3 E_pad, d], the fp32 logits [T, E] (E > 64), one row of E probability
// sums per finishing block (E > 64; space for one per CTA at E <= 64), and
// the E fixed-point probability-sum accumulators with the count of finished
// CTAs (E <= 64).
inline size_t route_parts_bytes(int d, const RouteFuShape& sh) { return align256((size_t)3 * sh.E_pad * d * 2); }
inline long long route_fin_blocks(long long T) { return (T + rfu::FIN_TOKENS - 1) / rfu::FIN_TOKENS; }
// E <= 64: the logits kernel finishes its own tokens (one probability-sum row
// per CTA); larger E: fp32 logits [T, E] for route_finish_kernel (one row per
// finishing block)
inline bool route_finish_here(const RouteFuShape& sh) { return sh.emax <= 64; }
inline size_t route_logits_bytes(long long T, int E, const RouteFuShape& sh)
{
    return route_finish_here(sh) ? 0 : align256((size_t)T * E * sizeof(float));
}
inline size_t route_ws_bytes_tc(long long T, int d, int E)
{
    RouteFuShape sh;
    if (!route_fu_shape(T, d, E, &sh)) return 0;
    const long long rows = route_finish_here(sh) ? sh.grid : route_fin_blocks(T);
    // + the fixed-point probability-sum accumulators [E] and the count of finished CTAs
    return route_parts_bytes(d, sh) + route_logits_bytes(T, E, sh) + align256((size_t)rows * E * sizeof(float)) +
           align256((size_t)E * 8 + 4);
}
// CUDA-core router for E <= 8 (bf16 x): d / 8 threads per block (whole
// warps, at most 512), tokens spread evenly over one wave of blocks, at most
// TPC_MAX per block (an even count: tokens go through the butterfly in pairs).
struct RouteSmShape {
    int tpc, grid, threads;
    size_t smem;
};
inline bool route_small_shape(long long T, int d, int E, RouteSmShape* s)
{
    if (E > rsm::EMAX || T <= 0 || d % 256 || d < 256 || d > 8 * rsm::MAX_THREADS) return false;
    const long long sms = (long long)sm_count();
    long long tpc = (T + sms - 1) / sms;
    tpc = (tpc + rsm::NT - 1) / rsm::NT * rsm::NT;
    if (tpc > rsm::TPC_MAX) tpc = rsm::TPC_MAX;
    s->tpc = (int)tpc;
    s->grid = (int)((T + tpc - 1) / tpc);
    s->threads = d / 8;
    s->smem = rsm::smem_bytes(d, s->tpc);
    return s->smem <= 227 * 1024;
}
inline size_t route_ws_bytes_small(long long T, int d, int E)
{
    RouteSmShape sh;
    return route_small_shape(T, d, E, &sh) ? (size_t)sh.grid * E * sizeof(float) : 0;
}
inline size_t route_ws_bytes(long long T, int d, int E)
{
    const size_t a = route_ws_bytes_simt(T, E), b = route_ws_bytes_tc(T, d, E), c = route_ws_bytes_small(T, d, E);
    return a > b ? (a > c ? a : c) : (b > c ? b : c);
}
inline long long dispatch_chunks(long long T, int k)
{
    const int ch = dispatch::chunk_size(T * k);
    return (T * k + ch - 1) / ch;
}
// Per-chunk expert histograms of the ranking.
inline size_t dispatch_ws_bytes(long long T, int k, int E) { return (size_t)dispatch_chunks(T, k) * E * sizeof(int); }


// Opt a kernel into `bytes` of dynamic shared memory once per device (the
// attribute is per device; setting it again on every launch is wasted host time).
bool ensure_dyn_smem(const void* kernel, int bytes)
{
    struct Entry {
        const void* k;
        int dev;
        int bytes;
    };
    static std::mutex mu;
    static Entry done[256];
    static int n_done = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].k == kernel && done[i].dev == dev && done[i].bytes >= bytes) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    for (int i = 0; i < n_done; ++i)
        if (done[i].k == kernel && done[i].dev == dev) {
            done[i].bytes = bytes;
            return true;
        }
    if (n_done < 256) done[n_done++] = Entry{kernel, dev, bytes};
    return true;
}

// ---------------------------------------------------------- TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// bf16 matrix [rows, cols] (cols contiguous), boxes of 64 columns x box_rows
// rows, 128-byte swizzle, zero fill outside.
bool make_tmap_bf16_box(CUtensorMap* m, const void* base, unsigned long long rows, unsigned long long cols,
                        unsigned box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows, cols] with a row stride of ld elements (ld >= cols), 64x64 boxes.
bool make_tmap_bf16_box_ld(CUtensorMap* m, const void* base, unsigned long long rows, unsigned long long cols,
                           unsigned long long ld)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows, cols] with a 32x32 box and the 128-byte swizzle (the output
// tiles of the weight-gradient GEMM, stored by TMA).
bool make_tmap_f32_out(CUtensorMap* m, const void* base, unsigned long long rows, unsigned long long cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A_rows: rows of the A tensor (default rows_max; T of x when gathering; M in
// the weight-gradient mode, where K is the packed column count ld).
template <int EPI, int BN, int MODE = tcg::MODE_ROWS>
moe_status launch_tc_bn(const void* A, long long rows_max, int K, const void* W, long long w_rows_total,
                        tcg::Args args, cudaStream_t stream, long long A_rows = -1)
{
    using SH = tcg::Shape<BN>;
    constexpr bool wg = MODE == tcg::MODE_WGRAD || MODE == tcg::MODE_WGRAD_ROWS;
    CUtensorMap ta, tb;
    if (MODE == tcg::MODE_WGRAD_ROWS) {
        // A [rows_max, M] and B [rows_max, N], both read as 64x64 boxes (rows = K)
        const unsigned long long lda = (unsigned long long)(args.lda > 0 ? args.lda : args.m_rows);
        if (!make_tmap_bf16_box_ld(&ta, A, (unsigned long long)rows_max, (unsigned long long)args.m_rows, lda) ||
            !make_tmap_bf16_box(&tb, W, (unsigned long long)rows_max, (unsigned long long)args.out_cols, 64))
            return MOE_ERR_CUDA;
    } else if (!make_tmap_bf16_box(&ta, A, (unsigned long long)(A_rows >= 0 ? A_rows : rows_max),
                                   (unsigned long long)K, MODE == tcg::MODE_GATHER ? 1 : 128)) {
        return MOE_ERR_CUDA;
    }
    if (MODE == tcg::MODE_BMN) {   // B [E*K rows, N cols], N contiguous: 64x64 boxes
        if (!make_tmap_bf16_box(&tb, W, (unsigned long long)w_rows_total, (unsigned long long)args.out_cols, 64))
            return MOE_ERR_CUDA;
    } else if (MODE != tcg::MODE_WGRAD_ROWS &&
               !make_tmap_bf16_box(&tb, W, (unsigned long long)w_rows_total, (unsigned long long)K, BN / 2)) {
        return MOE_ERR_CUDA;
    }
    CUtensorMap tc;
    memset(&tc, 0, sizeof tc);
    if (wg) {
        const unsigned long long rows = (unsigned long long)args.E * args.m_rows, cols = args.out_cols;
        if (args.out_f32 ? !make_tmap_f32_out(&tc, args.out_f32, rows, cols)
                         : !make_tmap_bf16_box(&tc, args.out, rows, cols, 32))
            return MOE_ERR_CUDA;
    } else if (MODE == tcg::MODE_BMN && EPI == tcg::EPI_IDENT && args.out_f32) {   // fp32 [rows_max, N] by TMA
        if (!make_tmap_f32_out(&tc, args.out_f32, (unsigned long long)rows_max, (unsigned long long)args.out_cols))
            return MOE_ERR_CUDA;
    }
    // the forward projections: bf16 [rows_max, out_cols] 32-row x 64-column output blocks by TMA
    // stores (not while the up projection also keeps the pre-activation z for the backward)
    constexpr bool fwd_tma = (MODE == tcg::MODE_ROWS &&
                              (EPI == tcg::EPI_GATE || EPI == tcg::EPI_GELU || EPI == tcg::EPI_IDENT ||
                               (EPI == tcg::EPI_SWIGLU && BN % 128 == 0))) ||
                             (MODE == tcg::MODE_BMN && EPI == tcg::EPI_IDENT);   // + dx_perm (bf16 out)
    args.tma_store = (fwd_tma && args.out_z == nullptr && args.out_f32 == nullptr) ? g_gemm_tma_store.load() : 0;
    if (fwd_tma && args.tma_store &&
        !make_tmap_bf16_box(&tc, args.out, (unsigned long long)rows_max, (unsigned long long)args.out_cols, 32))
        return MOE_ERR_CUDA;
    const int smem = (wg || MODE == tcg::MODE_BMN || fwd_tma) ? SH::WG_SMEM_DYN : SH::SMEM_DYN;
    if (!ensure_dyn_smem((const void*)tcg::grouped_gemm_kernel<EPI, BN, MODE>, smem)) return launch_status();
    const long long max_tiles = wg
                                    ? (long long)args.E * args.m_tiles * args.n_tiles
                                    : ((rows_max + tcg::BM - 1) / tcg::BM + args.E) * args.n_tiles;
    const int grid = (int)(max_tiles < sm_count() ? max_tiles : sm_count());
    if (grid <= 0) return MOE_OK;
    if (!wg) args.n_fastest = g_gemm_order.load() == 2;
    args.tail_halves = g_gemm_tail.load();
    // a programmatic dependent of the kernel before it: launch and set-up overlap that kernel's end
    PdlLaunch gl(grid, tcg::THREADS, stream, (size_t)smem);
    return launch_ex_status(cudaLaunchKernelEx(&gl.cfg, tcg::grouped_gemm_kernel<EPI, BN, MODE>, ta, tb, tc, args));
}

// Output-tile width of the tensor-core GEMMs.  Measured in SM cycles on the
// B300 for the e8 / e16 / e128 layers, 256 columns beats 192 and 128 on
// every GEMM, even where narrower tiles balance the waves better: the wider
// tile reuses each A row block over more output columns per byte loaded.
int choose_bn(long long, int, bool) { return 256; }

template <int EPI>
moe_status launch_tc(const void* A, long long rows_max, int K, const void* W, long long w_rows_total, tcg::Args a,
                     int n_out, cudaStream_t stream)
{
    const bool sw = EPI == tcg::EPI_SWIGLU;
    const int forced = g_forced_bn.load();
    const int bn = forced ? forced : choose_bn(rows_max, n_out, sw);
    a.n_step = sw ? bn / 2 : bn;
    a.half_off = sw ? n_out : bn / 2;
    a.n_tiles = (n_out + a.n_step - 1) / a.n_step;
    switch (bn) {
    case 128: return launch_tc_bn<EPI, 128>(A, rows_max, K, W, w_rows_total, a, stream);
    case 192: return launch_tc_bn<EPI, 192>(A, rows_max, K, W, w_rows_total, a, stream);
    default: return launch_tc_bn<EPI, 256>(A, rows_max, K, W, w_rows_total, a, stream);
    }
}

// CTA-pair (2-SM) grouped GEMM, weights on the 256-row side.
template <int EPI>
moe_status launch_tc2(const void* W, long long w_rows_total, const void* X, long long rows_max, int K, tc2::Args a,
                      cudaStream_t stream)
{
    CUtensorMap tw, tx;
    if (!make_tmap_bf16_box(&tw, W, (unsigned long long)w_rows_total, (unsigned long long)K, 64)) return MOE_ERR_CUDA;
    if (!make_tmap_bf16_box(&tx, X, (unsigned long long)rows_max, (unsigned long long)K, 128)) return MOE_ERR_CUDA;
    if (!ensure_dyn_smem((const void*)tc2::grouped_gemm_2sm_kernel<EPI>, tc2::SMEM_DYN)) return launch_status();
    const long long max_tok_tiles = (rows_max + tc2::BNT - 1) / tc2::BNT + a.E;
    const long long max_pairs = max_tok_tiles * a.n_wtiles;
    long long npairs = sm_count() / 2;
    if (npairs > max_pairs) npairs = max_pairs;
    if (npairs <= 0) return MOE_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * npairs), 1, 1);
    cfg.blockDim = dim3(tc2::THREADS, 1, 1);
    cfg.dynamicSmemBytes = tc2::SMEM_DYN;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, tc2::grouped_gemm_2sm_kernel<EPI>, tw, tx, a) != cudaSuccess) return launch_status();
    return launch_status();
}

// 1-SM or CTA-pair kernel for this call.
bool use_pair_kernel()
{
    const int kind = g_gemm_kind.load();
    return kind == 2;
}

template <int ACT>
moe_status launch_simt(const float* A, const int32_t* offsets, const int32_t* kept, int E, int K, int N, int F,
                       const float* W, const float* gate, float* out, long long rows_max, cudaStream_t stream)
{
    const long long max_mtiles = (rows_max + simt::BM - 1) / simt::BM + E;
    if (max_mtiles > 65535) return MOE_ERR_UNSUPPORTED;
    dim3 grid(N / simt::BN, (unsigned)max_mtiles);
    simt::ffn_simt_kernel<ACT><<<grid, simt::THREADS, 0, stream>>>(A, offsets, kept, E, K, N, F, W, gate, out);
    return launch_status();
}

template <int EPL, int TW>
void launch_route(bool bf16, int nblk, const void* x, const float* W, const float* b, int T, int d, int E, int k,
                  int renorm, int32_t* idx, float* gate, float* partial, RouteSel sel, cudaStream_t s)
{
    if (bf16)
        route::route_kernel<EPL, TW, true><<<nblk, route::THREADS, 0, s>>>(x, W, b, T, d, E, k, renorm, idx, gate,
                                                                           partial, sel);
    else
        route::route_kernel<EPL, TW, false><<<nblk, route::THREADS, 0, s>>>(x, W, b, T, d, E, k, renorm, idx, gate,
                                                                            partial, sel);
}

__global__ void selftest_wait_kernel(unsigned long long limit)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        ptx::fence_mbar_init();
        // nothing ever arrives on this barrier: the wait must run out
        if (!ptx::mbar_wait(ptx::smem_u32(&bar), 0, limit)) moe_flag(MOE_DEV_TIMEOUT);
    }
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status s)
{
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int64_t moe_capacity(int64_t T, int E, double cf)
{
    if (T < 0 || E < 1) return -1;
    if (cf <= 0.0) return T;
    return (int64_t)llround(((double)T / (double)E) * cf);
}

int64_t moe_perm_rows_max(int64_t T, int k, int E, int64_t cap)
{
    if (T < 0 || k < 1 || E < 1 || cap < 0) return -1;
    const int64_t all = T * k, lim = (int64_t)E * cap;
    return all < lim ? all : lim;
}

namespace {
// Token splits of the router weight gradient: enough blocks for two waves
// (at most 64 splits, at least 32 tokens each).
int router_wgrad_splits(int64_t T, int E, int d)
{
    const int base = ceil_div_i(d, bwd::RW_COLS) * ceil_div_i(E, bwd::RW_EXP);
    int S = ceil_div_i(2 * 148, base);
    if (S > 64) S = 64;
    const int maxS = ceil_div_i(T, 32);
    if (S > maxS) S = maxS;
    return S < 1 ? 1 : S;
}
}  // namespace

namespace {
// Router gradients on the tensor cores: Ep = E rounded up to 64, S token
// splits of the weight-gradient GEMM (enough tiles for two waves, >= 256 rows each).
struct RouterGradsLayout {
    int Ep, S;
    size_t dl3, W3, zr, P, seg1, segS, total;   // byte offsets in the workspace
};

RouterGradsLayout router_grads_layout(int64_t T, int E, int d)
{
    RouterGradsLayout L{};
    L.Ep = (E + 63) / 64 * 64;
    const int tiles = ceil_div_i(2 * L.Ep, 128) * ceil_div_i(d, 256);
    int S = ceil_div_i(2 * 148, tiles);
    const int maxS = (int)(T / 256 > 0 ? T / 256 : 1);
    if (S > maxS) S = maxS;
    if (S > 64) S = 64;
    L.S = S < 1 ? 1 : S;
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    size_t o = 0;
    L.dl3 = o;  o += up((size_t)T * 3 * L.Ep * 2);
    L.W3 = o;   o += up((size_t)3 * L.Ep * d * 2);
    L.zr = o;   o += up((size_t)T * d * 4);
    L.P = o;    o += up((size_t)L.S * 2 * L.Ep * d * 4);
    L.seg1 = o; o += 256;
    L.segS = o; o += up((size_t)(2 * L.S + 1) * 4);
    L.total = o;
    return L;
}
}  // namespace

size_t moe_workspace_bytes(moe_call call, int64_t T, int d, int E, int k, int F, moe_act act, moe_dtype dtype)
{
    (void)F;
    (void)act;
    (void)dtype;
    if (T < 0 || E < 1 || E > MAX_E || k < 1 || d < 0) return 0;
    switch (call) {
    case MOE_CALL_ROUTE: return route_ws_bytes(T, d, E);
    case MOE_CALL_DISPATCH: return dispatch_ws_bytes(T, k, E);
    case MOE_CALL_FFN: return 0;
    case MOE_CALL_ROUTER_WGRAD:
        return T < 1 || d < 1 ? 0 : (size_t)router_wgrad_splits(T, E, d) * E * d * sizeof(float);
    case MOE_CALL_ROUTER_GRADS:
        return T < 1 || d < 1 ? 0 : router_grads_layout(T, E, d).total;
    }
    return 0;
}

static moe_status route_impl(const void* x, moe_dtype xdt, const float* w_router, const float* b_router, int64_t T,
                             int d, int E, int k, int renorm, int32_t* topk_idx, float* topk_gate, float* prob_sum,
                             RouteSel sel, void* ws, size_t ws_bytes, cudaStream_t stream)
{
    if (T < 0 || d <= 0 || E < 1 || E > MAX_E || k < 1 || k > MAX_K || k > E || !dtype_ok(xdt))
        return MOE_ERR_INVALID_ARG;
    if (T * k >= INT_MAX || (long long)T * d >= (1LL << 40)) return MOE_ERR_INVALID_ARG;
    if (!prob_sum || (T > 0 && (!x || !w_router || !topk_idx || !topk_gate))) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({x, w_router, ws})) return MOE_ERR_UNSUPPORTED;
    if (d % 64) return MOE_ERR_UNSUPPORTED;
    const size_t need = route_ws_bytes(T, d, E);
    if (need && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
    const int rk = g_router_kind.load();
    RouteSmShape ss;
    if (xdt == MOE_BF16 && rk == 2 && route_small_shape(T, d, E, &ss)) {
        // on request, few experts: one CUDA-core kernel (logits, softmax,
        // top-k, per-block probability sums), then prob_sum_kernel adds the
        // blocks' rows.  On the B300 it takes as long as the tensor-core
        // router at E = 8 (its FMAs and butterflies are issue-bound), so the
        // automatic choice stays with the tensor cores.
        const int kmax = k <= 2 ? 2 : k <= 4 ? 4 : 8;
        void (*kern)(const rsm::Args) = kmax == 2 ? rsm::route_small_kernel<2>
                                        : kmax == 4 ? rsm::route_small_kernel<4> : rsm::route_small_kernel<8>;
        if (!ensure_dyn_smem((const void*)kern, (int)ss.smem)) return launch_status();
        rsm::Args a{};
        a.x = (const uint16_t*)x;
        a.W = w_router;
        a.bias = b_router;
        a.T = (int)T;
        a.d = d;
        a.E = E;
        a.k = k;
        a.renorm = renorm;
        a.tpc = ss.tpc;
        a.idx = topk_idx;
        a.gate = topk_gate;
        a.psum = (float*)ws;
        a.sel = sel;
        PdlLaunch rl(ss.grid, ss.threads, stream, ss.smem);
        moe_status st = launch_ex_status(cudaLaunchKernelEx(&rl.cfg, kern, a));
        if (st != MOE_OK) return st;
        PdlLaunch pl(E, 256, stream);
        return launch_ex_status(cudaLaunchKernelEx(&pl.cfg, rfu::prob_sum_kernel, (const float*)ws, ss.grid, E,
                                                   prob_sum));
    }
    RouteFuShape sh;
    if (xdt == MOE_BF16 && rk != 2 && route_fu_shape(T, d, E, &sh)) {
        // the weight split into three bf16 parts; the tensor-core logits
        // kernel, which for E <= 64 also takes the softmax, top-k and
        // probability sums (its last CTA writes prob_sum); for larger E the
        // finishing kernel does that and prob_sum_kernel adds its per-block
        // rows.  Each launch after the first is a programmatic dependent of
        // the one before, so its set-up overlaps that kernel's tail.
        const bool here = route_finish_here(sh);
        uint4* parts = (uint4*)ws;
        float* logits = here ? nullptr
                             : (sel.logits ? sel.logits : (float*)((char*)ws + route_parts_bytes(d, sh)));
        float* psum = (float*)((char*)ws + route_parts_bytes(d, sh) + route_logits_bytes(T, E, sh));
        const int kmax = k <= 2 ? 2 : k <= 4 ? 4 : k <= 8 ? 8 : 16;
        void (*kern)(const CUtensorMap, const CUtensorMap, const rfu::Args) = nullptr;
        void (*fin)(const rfu::FinArgs) = nullptr;
#define MOE_RFU(EM)                                                                                       \
        kern = kmax == 2 ? rfu::route_fused_kernel<EM, 2> : kmax == 4 ? rfu::route_fused_kernel<EM, 4> :       \
               kmax == 8 ? rfu::route_fused_kernel<EM, 8> : rfu::route_fused_kernel<EM, 16>
        if (sh.emax == 16) MOE_RFU(16);
        else if (sh.emax == 32) MOE_RFU(32);
        else if (sh.emax == 64) MOE_RFU(64);
        else {
            kern = rfu::route_fused_kernel<128, 2>;   // finishing is left to route_finish_kernel
            fin = kmax == 2 ? rfu::route_finish_kernel<128, 2> : kmax == 4 ? rfu::route_finish_kernel<128, 4> :
                  kmax == 8 ? rfu::route_finish_kernel<128, 8> : rfu::route_finish_kernel<128, 16>;
        }
#undef MOE_RFU
        if (!ensure_dyn_smem((const void*)kern, sh.smem)) return launch_status();
        CUtensorMap tx, tw;
        if (!make_tmap_bf16_box(&tx, x, (unsigned long long)T, (unsigned long long)d, rfu::BM)) return MOE_ERR_CUDA;
        if (!make_tmap_bf16_box(&tw, parts, (unsigned long long)(3 * sh.E_pad), (unsigned long long)d,
                                (unsigned)(3 * sh.E_pad <= 256 ? 3 * sh.E_pad : sh.E_pad)))
            return MOE_ERR_CUDA;
        rfu::Args a{};
        a.T = (int)T;
        a.d = d;
        a.E = E;
        a.E_pad = sh.E_pad;
        a.k = k;
        a.renorm = renorm;
        a.nk = d / rfu::BK;
        a.S = sh.S;
        a.TPB = sh.TPB;
        a.xstages = sh.xstages;
        a.wstages = sh.wstages;
        a.tmem_cols = sh.tmem_cols;
        a.bias = b_router;
        a.idx = topk_idx;
        a.gate = topk_gate;
        a.psum = psum;
        a.sel = sel;
        a.logits = logits;
        a.wait_limit = g_wait_limit.load();
        const int rows = here ? sh.grid : (int)route_fin_blocks(T);
        unsigned long long* psum_fx =
            (unsigned long long*)((char*)psum + align256((size_t)rows * E * sizeof(float)));
        unsigned* done = (unsigned*)(psum_fx + E);
        a.psum_fx = psum_fx;
        a.done = done;
        a.prob_sum = prob_sum;
        rfu::FinArgs f{};
        f.T = (int)T;
        f.E = E;
        f.k = k;
        f.renorm = renorm;
        f.logits = logits;
        f.idx = topk_idx;
        f.gate = topk_gate;
        f.psum = psum;
        f.sel = sel;

        const long long n8 = (long long)sh.E_pad * (d / 8);
        long long sg = (n8 + 255) / 256;
        if (sg > 4LL * sm_count()) sg = 4LL * sm_count();
        rfu::split_weight_kernel<<<(int)sg, 256, 0, stream>>>(w_router, E, sh.E_pad, d, parts,
                                                               here ? psum_fx : nullptr, done);
        moe_status st = launch_status();
        if (st != MOE_OK) return st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = g_pdl.load();
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)sh.S;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)sh.grid);
        cfg.blockDim = dim3(rfu::THREADS);
        cfg.dynamicSmemBytes = (size_t)sh.smem;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = sh.S > 1 ? 2 : 1;
        st = launch_ex_status(cudaLaunchKernelEx(&cfg, kern, tx, tw, a));
        if (st != MOE_OK) return st;
        if (!here) {
            cudaLaunchConfig_t fcfg = {};
            fcfg.gridDim = dim3((unsigned)rows);
            fcfg.blockDim = dim3(rfu::FIN_THREADS);
            fcfg.stream = stream;
            fcfg.attrs = attr;
            fcfg.numAttrs = 1;
            st = launch_ex_status(cudaLaunchKernelEx(&fcfg, fin, f));
            if (st != MOE_OK) return st;
        }
        if (here) return MOE_OK;   // prob_sum: written by the logits kernel's last CTA
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3((unsigned)E);
        pcfg.blockDim = dim3(256);
        pcfg.stream = stream;
        pcfg.attrs = attr;
        pcfg.numAttrs = 1;
        return launch_ex_status(cudaLaunchKernelEx(&pcfg, rfu::prob_sum_kernel, (const float*)psum, rows, E,
                                                   prob_sum));
    }
    const int tpb = route_tokens_per_block(E);
    const int nblk = (int)((T + tpb - 1) / tpb);
    float* partial = (float*)ws;
    if (nblk > 0) {
        const bool bf = xdt == MOE_BF16;
        const int Ti = (int)T;
        switch (route_epl(E)) {
        case 1: launch_route<1, 2>(bf, nblk, x, w_router, b_router, Ti, d, E, k, renorm, topk_idx, topk_gate, partial, sel, stream); break;
        case 2: launch_route<2, 4>(bf, nblk, x, w_router, b_router, Ti, d, E, k, renorm, topk_idx, topk_gate, partial, sel, stream); break;
        case 4: launch_route<4, 4>(bf, nblk, x, w_router, b_router, Ti, d, E, k, renorm, topk_idx, topk_gate, partial, sel, stream); break;
        default: launch_route<8, 4>(bf, nblk, x, w_router, b_router, Ti, d, E, k, renorm, topk_idx, topk_gate, partial, sel, stream); break;
        }
        const moe_status st = launch_status();
        if (st != MOE_OK) return st;
    }
    route::route_finalize<<<1, route::FIN_THREADS, 0, stream>>>(partial, nblk, E, prob_sum);
    return launch_status();
}

moe_status moe_route(const void* x, moe_dtype xdt, const float* w_router, const float* b_router, int64_t T, int d,
                     int E, int k, int renorm, int32_t* topk_idx, float* topk_gate, float* prob_sum, void* ws,
                     size_t ws_bytes, moe_stream_t stream)
{
    const RouteSel plain{1, E > 0 ? E : 1, 1, nullptr, nullptr};
    return route_impl(x, xdt, w_router, b_router, T, d, E, k, renorm, topk_idx, topk_gate, prob_sum, plain, ws,
                      ws_bytes, (cudaStream_t)stream);
}

moe_status moe_route_ex(const void* x, moe_dtype xdt, const float* w_router, const float* b_router, int64_t T, int d,
                        int E, int k, int renorm, int n_group, int topk_group, int32_t* topk_idx, float* topk_gate,
                        float* prob_sum, float* lse, float* logits, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (n_group < 1 || n_group > 32 || E < 1 || E % n_group || topk_group < 1 || topk_group > n_group)
        return MOE_ERR_INVALID_ARG;
    if ((long long)k > (long long)topk_group * (E / n_group)) return MOE_ERR_INVALID_ARG;
    const RouteSel sel{n_group, E / n_group, topk_group, T > 0 ? lse : nullptr, T > 0 ? logits : nullptr};
    return route_impl(x, xdt, w_router, b_router, T, d, E, k, renorm, topk_idx, topk_gate, prob_sum, sel, ws,
                      ws_bytes, (cudaStream_t)stream);
}

moe_status moe_z_loss(const float* lse, int64_t T, float beta, float* loss, moe_stream_t stream)
{
    if (T <= 0 || !lse || !loss) return MOE_ERR_INVALID_ARG;
    combine::z_loss_kernel<<<1, combine::ZL_THREADS, 0, (cudaStream_t)stream>>>(lse, (long long)T, beta, loss);
    return launch_status();
}

moe_status moe_dispatch(const int32_t* topk_idx, const float* topk_gate, int64_t T, int k, int E, int64_t cap,
                        const void* x, moe_dtype xdt, int d, int32_t* counts, int32_t* kept, int32_t* offsets,
                        int32_t* slot_row, int32_t* row_token, float* row_gate, void* x_perm, int32_t* n_dropped,
                        void* ws, size_t ws_bytes, moe_stream_t stream_)
{
    cudaStream_t stream = (cudaStream_t)stream_;
    if (T < 0 || k < 1 || k > MAX_K || E < 1 || E > MAX_E || k > E || cap < 0 || d <= 0 || !dtype_ok(xdt))
        return MOE_ERR_INVALID_ARG;
    if (T * k >= INT_MAX) return MOE_ERR_INVALID_ARG;
    if (!counts || !kept || !offsets || !n_dropped) return MOE_ERR_INVALID_ARG;
    const int64_t rows_max = moe_perm_rows_max(T, k, E, cap);
    if (T > 0 && (!topk_idx || !topk_gate || !x || !slot_row)) return MOE_ERR_INVALID_ARG;
    if (rows_max > 0 && (!row_token || !row_gate)) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({x, x_perm})) return MOE_ERR_UNSUPPORTED;
    if (d % 64) return MOE_ERR_UNSUPPORTED;
    const size_t need = dispatch_ws_bytes(T, k, E);
    if (need && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
    const int nchunk = (int)dispatch_chunks(T, k);
    const int cap32 = cap > INT_MAX ? INT_MAX : (int)cap;
    int* hist = (int*)ws;
    // hist -> (scan) -> rank -> scatter, each a programmatic dependent of the one before
    // (T = 0: no histograms; one rank block writes the zero counts)
    const bool small = dispatch::chunk_size(T * k) == dispatch::SMALL_CHUNK;
    const bool scanned = nchunk > 0 && dispatch::use_chunk_scan(nchunk, E, !small);
    if (nchunk > 0) {
        PdlLaunch hl(nchunk, dispatch::THREADS, stream);   // waits for the router's last kernel
        const moe_status st0 = launch_ex_status(cudaLaunchKernelEx(
            &hl.cfg, small ? dispatch::hist_kernel<dispatch::SMALL_CHUNK> : dispatch::hist_kernel<dispatch::LARGE_CHUNK>,
            topk_idx, (int)T, k, E, hist));
        if (st0 != MOE_OK) return st0;
        if (scanned) {   // per-expert prefix over the chunks, and counts
            PdlLaunch sl((E + dispatch::WARPS - 1) / dispatch::WARPS, dispatch::THREADS, stream);
            const moe_status st_s = launch_ex_status(
                cudaLaunchKernelEx(&sl.cfg, dispatch::scan_kernel, hist, nchunk, E, counts));
            if (st_s != MOE_OK) return st_s;
        }
    }
    {
        PdlLaunch rl(nchunk > 0 ? nchunk : 1, dispatch::THREADS, stream);
        const moe_status st1 = launch_ex_status(cudaLaunchKernelEx(
            &rl.cfg, small ? dispatch::rank_kernel<dispatch::SMALL_CHUNK> : dispatch::rank_kernel<dispatch::LARGE_CHUNK>,
            topk_idx, topk_gate, (int)T, k, E, cap32, (const int*)hist, nchunk, (int)scanned, counts, kept, offsets,
            slot_row, row_token, row_gate, n_dropped));
        if (st1 != MOE_OK) return st1;
    }
    moe_status st = launch_status();
    if (st != MOE_OK || rows_max == 0 || !x_perm) return st;   // x_perm NULL: the up GEMM gathers from x
    const int vec16 = d * esize(xdt) / 16;
    const long long tasks = T * ((vec16 + dispatch::CHUNK_VEC - 1) / dispatch::CHUNK_VEC);
    long long grid = (tasks + dispatch::WARPS - 1) / dispatch::WARPS;
    if (!ensure_dyn_smem((const void*)dispatch::scatter_tokens_kernel, dispatch::SCATTER_SMEM)) return launch_status();
    // only resident blocks stage x before the ranking ends: one wave of them, grid-striding
    static const int per_sm = resident_blocks(dispatch::scatter_tokens_kernel, dispatch::THREADS,
                                              (size_t)dispatch::SCATTER_SMEM);
    if (grid > (long long)sm_count() * per_sm) grid = (long long)sm_count() * per_sm;
    // a programmatic dependent of the ranking: x copies start before slot_row is final
    PdlLaunch sl((int)grid, dispatch::THREADS, stream, (size_t)dispatch::SCATTER_SMEM);
    return launch_ex_status(cudaLaunchKernelEx(&sl.cfg, dispatch::scatter_tokens_kernel, slot_row, (int)T, k,
                                               (const uint4*)x, (uint4*)x_perm, vec16, g_wait_limit.load()));
}

moe_status moe_permute_rows(const void* src, const int32_t* index, int64_t n, int d, moe_dtype dtype, void* dst,
                            moe_stream_t stream)
{
    if (n < 0 || d <= 0 || !dtype_ok(dtype) || (n > 0 && (!src || !index || !dst))) return MOE_ERR_INVALID_ARG;
    const int row_bytes = d * esize(dtype);
    if (row_bytes % 16 || ((uintptr_t)src & 15u) || ((uintptr_t)dst & 15u)) return MOE_ERR_UNSUPPORTED;
    if (n == 0) return MOE_OK;
    long long grid = (n + dispatch::WARPS - 1) / dispatch::WARPS;
    if (grid > (long long)sm_count() * 8) grid = (long long)sm_count() * 8;
    dispatch::permute_rows_kernel<<<(int)grid, dispatch::THREADS, 0, (cudaStream_t)stream>>>(
        (const uint4*)src, index, (long long)n, row_bytes / 16, (uint4*)dst);
    return launch_status();
}

static moe_status ffn_common_checks(const int32_t* offsets, const int32_t* kept, int E, int d, int F,
                                    moe_dtype dtype, int64_t rows_max)
{
    if (E < 1 || E > MAX_E || d <= 0 || F <= 0 || rows_max < 0 || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
    if (!offsets || !kept) return MOE_ERR_INVALID_ARG;
    if (d % 64 || F % 64) return MOE_ERR_UNSUPPORTED;
    if (rows_max >= INT_MAX) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

static moe_status expert_up_impl(const void* x_perm, const int32_t* offsets, const int32_t* kept, int E, int d,
                                 int F, moe_act act, moe_dtype dtype, const void* w1, int64_t rows_max, void* h,
                                 void* z, cudaStream_t stream)
{
    moe_status st = ffn_common_checks(offsets, kept, E, d, F, dtype, rows_max);
    if (st != MOE_OK) return st;
    if (act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU && act != MOE_ACT_IDENTITY) return MOE_ERR_INVALID_ARG;
    if (!w1 || (rows_max > 0 && (!x_perm || !h))) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({x_perm, w1, h, z})) return MOE_ERR_UNSUPPORTED;
    if (rows_max == 0) return MOE_OK;
    const int N1 = act == MOE_ACT_SWIGLU ? 2 * F : F;
    if (dtype == MOE_F32) {
        const float* A = (const float*)x_perm;
        const float* W = (const float*)w1;
        float* out = (float*)h;
        switch (act) {
        case MOE_ACT_GELU: return launch_simt<simt::ACT_GELU>(A, offsets, kept, E, d, F, F, W, nullptr, out, rows_max, stream);
        case MOE_ACT_SWIGLU: return launch_simt<simt::ACT_SWIGLU>(A, offsets, kept, E, d, F, F, W, nullptr, out, rows_max, stream);
        default: return launch_simt<simt::ACT_IDENT>(A, offsets, kept, E, d, F, F, W, nullptr, out, rows_max, stream);
        }
    }
    if (use_pair_kernel() && !z) {
        tc2::Args b{};
        b.offsets = offsets;
        b.kept = kept;
        b.E = E;
        b.K = d;
        b.w_rows = N1;
        b.F = F;
        b.out_cols = F;
        b.out = (uint16_t*)h;
        b.row_gate = nullptr;
        b.wait_limit = g_wait_limit.load();
        b.n_wtiles = act == MOE_ACT_SWIGLU ? (F + 127) / 128 : (F + 255) / 256;
        const long long wr = (long long)E * N1;
        if (act == MOE_ACT_SWIGLU) return launch_tc2<tc2::EPI_SWIGLU>(w1, wr, x_perm, rows_max, d, b, stream);
        if (act == MOE_ACT_GELU) return launch_tc2<tc2::EPI_GELU>(w1, wr, x_perm, rows_max, d, b, stream);
        return launch_tc2<tc2::EPI_IDENT>(w1, wr, x_perm, rows_max, d, b, stream);
    }
    tcg::Args a{};
    a.offsets = offsets;
    a.kept = kept;
    a.E = E;
    a.K = d;
    a.b_rows = N1;
    a.out_cols = F;
    a.out = (uint16_t*)h;
    a.row_gate = nullptr;
    a.out_z = (uint16_t*)z;
    a.z_cols = N1;
    a.wait_limit = g_wait_limit.load();
    if (act == MOE_ACT_SWIGLU)
        return launch_tc<tcg::EPI_SWIGLU>(x_perm, rows_max, d, w1, (long long)E * N1, a, F, stream);
    if (act == MOE_ACT_GELU) return launch_tc<tcg::EPI_GELU>(x_perm, rows_max, d, w1, (long long)E * N1, a, F, stream);
    return launch_tc<tcg::EPI_IDENT>(x_perm, rows_max, d, w1, (long long)E * N1, a, F, stream);
}

moe_status moe_expert_up(const void* x_perm, const int32_t* offsets, const int32_t* kept, int E, int d, int F,
                         moe_act act, moe_dtype dtype, const void* w1, int64_t rows_max, void* h, moe_stream_t stream)
{
    return expert_up_impl(x_perm, offsets, kept, E, d, F, act, dtype, w1, rows_max, h, nullptr,
                          (cudaStream_t)stream);
}

moe_status moe_expert_up_z(const void* x_perm, const int32_t* offsets, const int32_t* kept, int E, int d, int F,
                           moe_act act, moe_dtype dtype, const void* w1, int64_t rows_max, void* h, void* z,
                           moe_stream_t stream)
{
    if (dtype != MOE_BF16) return dtype_ok(dtype) ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
    if (rows_max > 0 && !z) return MOE_ERR_INVALID_ARG;
    return expert_up_impl(x_perm, offsets, kept, E, d, F, act, dtype, w1, rows_max, h, z, (cudaStream_t)stream);
}

moe_status moe_expert_up_gathered(const void* x, int64_t T, const int32_t* row_token, const int32_t* offsets,
                                  const int32_t* kept, int E, int d, int F, moe_act act, moe_dtype dtype,
                                  const void* w1, int64_t rows_max, void* h, moe_stream_t stream_)
{
    cudaStream_t stream = (cudaStream_t)stream_;
    moe_status st = ffn_common_checks(offsets, kept, E, d, F, dtype, rows_max);
    if (st != MOE_OK) return st;
    if (act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU && act != MOE_ACT_IDENTITY) return MOE_ERR_INVALID_ARG;
    if (T < 0 || T >= INT_MAX || !w1 || (rows_max > 0 && (!x || !row_token || !h))) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({x, w1, h})) return MOE_ERR_UNSUPPORTED;
    if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (rows_max == 0 || T == 0) return MOE_OK;
    // the copies address x with 32-bit row offsets and 16-byte vectors
    if ((unsigned long long)T * (unsigned long long)d * 2ull >= (1ull << 32) || ((uintptr_t)x & 15u))
        return MOE_ERR_UNSUPPORTED;
    const int N1 = act == MOE_ACT_SWIGLU ? 2 * F : F;
    tcg::Args a{};
    a.offsets = offsets;
    a.kept = kept;
    a.E = E;
    a.K = d;
    a.b_rows = N1;
    a.out_cols = F;
    a.out = (uint16_t*)h;
    a.row_gate = nullptr;
    a.row_token = row_token;
    a.a_base = (const uint8_t*)x;
    a.a_row_bytes = (uint32_t)d * 2u;
    a.wait_limit = g_wait_limit.load();
    const bool sw = act == MOE_ACT_SWIGLU;
    a.n_step = sw ? 128 : 256;
    a.half_off = sw ? F : 128;
    a.n_tiles = (F + a.n_step - 1) / a.n_step;
    const long long wr = (long long)E * N1;
    constexpr int G = tcg::MODE_GATHER;
    if (sw) return launch_tc_bn<tcg::EPI_SWIGLU, 256, G>(x, rows_max, d, w1, wr, a, stream, T);
    if (act == MOE_ACT_GELU) return launch_tc_bn<tcg::EPI_GELU, 256, G>(x, rows_max, d, w1, wr, a, stream, T);
    return launch_tc_bn<tcg::EPI_IDENT, 256, G>(x, rows_max, d, w1, wr, a, stream, T);
}

moe_status moe_expert_down(const void* h, const int32_t* offsets, const int32_t* kept, int E, int d, int F,
                           moe_dtype dtype, const void* w2, const float* row_gate, int64_t rows_max, void* y_perm,
                           moe_stream_t stream_)
{
    cudaStream_t stream = (cudaStream_t)stream_;
    moe_status st = ffn_common_checks(offsets, kept, E, d, F, dtype, rows_max);
    if (st != MOE_OK) return st;
    if (!w2 || (rows_max > 0 && (!h || !row_gate || !y_perm))) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({h, w2, y_perm})) return MOE_ERR_UNSUPPORTED;
    if (rows_max == 0) return MOE_OK;
    if (dtype == MOE_F32)
        return launch_simt<simt::ACT_GATE>((const float*)h, offsets, kept, E, F, d, F, (const float*)w2, row_gate,
                                           (float*)y_perm, rows_max, stream);
    if (use_pair_kernel()) {
        tc2::Args b{};
        b.offsets = offsets;
        b.kept = kept;
        b.E = E;
        b.K = F;
        b.w_rows = d;
        b.F = F;
        b.out_cols = d;
        b.out = (uint16_t*)y_perm;
        b.row_gate = row_gate;
        b.wait_limit = g_wait_limit.load();
        b.n_wtiles = (d + 255) / 256;
        return launch_tc2<tc2::EPI_GATE>(w2, (long long)E * d, h, rows_max, F, b, stream);
    }
    tcg::Args a{};
    a.offsets = offsets;
    a.kept = kept;
    a.E = E;
    a.K = F;
    a.b_rows = d;
    a.out_cols = d;
    a.out = (uint16_t*)y_perm;
    a.row_gate = row_gate;
    a.wait_limit = g_wait_limit.load();
    return launch_tc<tcg::EPI_GATE>(h, rows_max, F, w2, (long long)E * d, a, d, stream);
}

moe_status moe_expert_ffn(const void* x_perm, const int32_t* offsets, const int32_t* kept, int E, int d, int F,
                          moe_act act, moe_dtype dtype, const void* w1, const void* w2, const float* row_gate,
                          int64_t rows_max, void* h, void* y_perm, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    (void)ws;
    (void)ws_bytes;
    moe_status st = moe_expert_up(x_perm, offsets, kept, E, d, F, act, dtype, w1, rows_max, h, stream);
    if (st != MOE_OK) return st;
    return moe_expert_down(h, offsets, kept, E, d, F, dtype, w2, row_gate, rows_max, y_perm, stream);
}

namespace {
moe_status combine_impl(const void* y_perm, const int32_t* slot_row, int64_t T, int k, int d, moe_dtype dtype, void* y,
                        combine::AuxArgs aux, cudaStream_t stream)
{
    if (T < 0 || k < 1 || k > MAX_K || d <= 0 || !dtype_ok(dtype) || T * k >= INT_MAX) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!slot_row || !y || !y_perm)) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({y_perm, y})) return MOE_ERR_UNSUPPORTED;
    if (d % 64) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    const int vec16 = d * esize(dtype) / 16;
    const long long tasks = T * ((vec16 + combine::CHUNK_VEC - 1) / combine::CHUNK_VEC);
    long long grid = (tasks + combine::WARPS - 1) / combine::WARPS;
    // one wave of resident blocks, grid-striding over the (token, chunk) tasks
    static const int per_sm_bf16 = resident_blocks(combine::combine_kernel<true>, combine::THREADS);
    static const int per_sm_f32 = resident_blocks(combine::combine_kernel<false>, combine::THREADS);
    const long long wave = (long long)sm_count() * (dtype == MOE_BF16 ? per_sm_bf16 : per_sm_f32);
    if (grid > wave) grid = wave;
    // a programmatic dependent of the kernel writing y_perm: it launches while that kernel's last blocks
    // run and waits (griddepcontrol.wait) before reading y_perm
    PdlLaunch cl((int)grid, combine::THREADS, stream);
    if (dtype == MOE_BF16)
        return launch_ex_status(cudaLaunchKernelEx(&cl.cfg, combine::combine_kernel<true>, (const uint4*)y_perm,
                                                   slot_row, (int)T, k, vec16, (uint4*)y, aux));
    return launch_ex_status(cudaLaunchKernelEx(&cl.cfg, combine::combine_kernel<false>, (const uint4*)y_perm,
                                               slot_row, (int)T, k, vec16, (uint4*)y, aux));
}
}  // namespace

moe_status moe_combine(const void* y_perm, const int32_t* slot_row, int64_t T, int k, int d, moe_dtype dtype, void* y,
                       moe_stream_t stream)
{
    return combine_impl(y_perm, slot_row, T, k, d, dtype, y, combine::AuxArgs{}, (cudaStream_t)stream);
}

moe_status moe_combine_aux(const void* y_perm, const int32_t* slot_row, int64_t T, int k, int d, moe_dtype dtype,
                           void* y, const int32_t* counts, const float* prob_sum, int E, float alpha, float* loss,
                           moe_stream_t stream)
{
    if (T < 1 || E < 1 || E > MAX_E || !counts || !prob_sum || !loss) return MOE_ERR_INVALID_ARG;
    return combine_impl(y_perm, slot_row, T, k, d, dtype, y, combine::AuxArgs{counts, prob_sum, (long long)T, E, alpha, loss},
                        (cudaStream_t)stream);
}

moe_status moe_aux_loss(const int32_t* counts, const float* prob_sum, int64_t T, int E, float alpha, float* loss,
                        moe_stream_t stream_)
{
    cudaStream_t stream = (cudaStream_t)stream_;
    if (T < 1 || E < 1 || E > MAX_E || !counts || !prob_sum || !loss) return MOE_ERR_INVALID_ARG;
    combine::aux_loss_kernel<<<1, 32, 0, stream>>>(counts, prob_sum, (long long)T, E, alpha, loss);
    return launch_status();
}

moe_status moe_check(moe_stream_t stream_)
{
    cudaStream_t stream = (cudaStream_t)stream_;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
    }
    unsigned int st = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&st, g_moe_status, sizeof st) != cudaSuccess) return MOE_ERR_CUDA;
    if (st && cudaMemcpyToSymbol(g_moe_status, &zero, sizeof zero) != cudaSuccess) return MOE_ERR_CUDA;
    if (st & MOE_DEV_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (st & MOE_DEV_BAD_EXPERT) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

void moe_set_wait_limit(uint64_t cycles) { g_wait_limit.store(cycles ? cycles : DEFAULT_WAIT_LIMIT); }

moe_status moe_set_gemm_kernel(int kind)
{
    if (kind < 0 || kind > 2) return MOE_ERR_INVALID_ARG;
    g_gemm_kind.store(kind);
    return MOE_OK;
}

moe_status moe_set_wgrad_order(int order)
{
    if (order < 0 || order > 2) return MOE_ERR_INVALID_ARG;
    g_wgrad_order.store(order);
    return MOE_OK;
}

moe_status moe_set_gemm_order(int order)
{
    if (order < 0 || order > 2) return MOE_ERR_INVALID_ARG;
    g_gemm_order.store(order);
    return MOE_OK;
}

moe_status moe_set_router_kernel(int kind)
{
    if (kind < 0 || kind > 2) return MOE_ERR_INVALID_ARG;
    g_router_kind.store(kind);
    return MOE_OK;
}

moe_status moe_set_gemm_tma_store(int on)
{
    if (on != 0 && on != 1) return MOE_ERR_INVALID_ARG;
    g_gemm_tma_store.store(on);
    return MOE_OK;
}

moe_status moe_set_launch_overlap(int on)
{
    if (on != 0 && on != 1) return MOE_ERR_INVALID_ARG;
    g_pdl.store(on);
    return MOE_OK;
}

moe_status moe_set_gemm_tail_halves(int on)
{
    if (on != 0 && on != 1) return MOE_ERR_INVALID_ARG;
    g_gemm_tail.store(on);
    return MOE_OK;
}

moe_status moe_set_gemm_tile_n(int bn)
{
    if (bn != 0 && bn != 128 && bn != 192 && bn != 256) return MOE_ERR_INVALID_ARG;
    g_forced_bn.store(bn);
    return MOE_OK;
}

moe_status moe_selftest_wait_timeout(moe_stream_t stream_)
{
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream_>>>(g_wait_limit.load());
    return launch_status();
}

}  // extern "C"

// ------------------------------------------------- dispatch without allocation
// Some callers cannot allocate device memory at the point where they run the
// layer: an inference engine's plugin enqueue callback that must not call
// cudaMalloc, a process whose device memory is handed out entirely by its
// own pool, or a latency-critical loop that cannot afford the device-wide
// synchronisation cudaMalloc may cause.  moe_dispatch_noalloc gives them the
// dispatch step with its scratch (the per-chunk expert histograms) in the
// fixed array below instead of a caller-provided workspace.
namespace {
constexpr size_t NOALLOC_SCRATCH_BYTES = 256u * 1024u;   // 64 Ki int32 histogram cells
constexpr int NOALLOC_MAX_DEVICES = 64;
// Every GPU that loads this library holds these 256 KiB until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES];

// Device address of the array on the current device, looked up once per device
// with that device current.  (In host code the array's name is only a host-side
// stand-in, not a device address.)
moe_status noalloc_scratch(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return launch_status();
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            std::fprintf(stderr, "moe_dispatch_noalloc: cudaGetSymbolAddress failed: %s\n", cudaGetErrorString(e));
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return MOE_OK;
}
}  // namespace

// ============================================================== backward ===

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

moe_status moe_transpose_experts(const void* w, int E, int R, int C, moe_dtype dtype, void* wt, moe_stream_t stream)
{
    if (E < 1 || R <= 0 || C <= 0 || !w || !wt || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 || R % 64 || C % 64 || R / 64 > 65535 || E > 65535 || !aligned16(w) || !aligned16(wt))
        return MOE_ERR_UNSUPPORTED;
    bwd::transpose_experts_kernel<<<dim3(C / 64, R / 64, E), 256, 0, (cudaStream_t)stream>>>(
        (const uint16_t*)w, R, C, (uint16_t*)wt);
    return launch_status();
}

moe_status moe_combine_bwd(const void* dy, const int32_t* slot_row, const float* row_gate, const void* y_perm,
                           int64_t T, int k, int d, moe_dtype dtype, void* do_perm, float* dgate, moe_stream_t stream)
{
    if (T < 0 || k < 1 || k > MAX_K || d <= 0 || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!dy || !slot_row || !row_gate || !y_perm || !do_perm || !dgate)) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({dy, y_perm, do_perm})) return MOE_ERR_UNSUPPORTED;
    if (dtype != MOE_BF16 || d % 64) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    int grid = ceil_div_i(T, bwd::CB_THREADS / 32);
    if (grid > sm_count() * 8) grid = sm_count() * 8;
    bwd::combine_bwd_kernel<<<grid, bwd::CB_THREADS, 0, (cudaStream_t)stream>>>(
        (const uint4*)dy, slot_row, row_gate, (const uint4*)y_perm, (int)T, k, d / 8, (uint4*)do_perm, dgate);
    return launch_status();
}

moe_status moe_act_bwd(const void* z, const void* da, const int32_t* offsets, int E, int F, moe_act act,
                       moe_dtype dtype, int64_t rows_max, void* dz, moe_stream_t stream)
{
    if (E < 1 || E > MAX_E || F <= 0 || rows_max < 0 || !offsets || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
    if (act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU && act != MOE_ACT_IDENTITY) return MOE_ERR_INVALID_ARG;
    if (rows_max > 0 && (!z || !da || !dz)) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({z, da, dz})) return MOE_ERR_UNSUPPORTED;
    if (dtype != MOE_BF16 || F % 64) return MOE_ERR_UNSUPPORTED;
    if (rows_max == 0) return MOE_OK;
    const int grid = sm_count() * 8;
    cudaStream_t st = (cudaStream_t)stream;
    const uint16_t *zp = (const uint16_t*)z, *ap = (const uint16_t*)da;
    if (act == MOE_ACT_SWIGLU)
        bwd::act_bwd_kernel<MOE_ACT_SWIGLU><<<grid, 256, 0, st>>>(zp, ap, offsets, E, F, (uint16_t*)dz);
    else if (act == MOE_ACT_GELU)
        bwd::act_bwd_kernel<MOE_ACT_GELU><<<grid, 256, 0, st>>>(zp, ap, offsets, E, F, (uint16_t*)dz);
    else
        bwd::act_bwd_kernel<MOE_ACT_IDENTITY><<<grid, 256, 0, st>>>(zp, ap, offsets, E, F, (uint16_t*)dz);
    return launch_status();
}

int64_t moe_wgrad_cols(int64_t rows_max, int E)
{
    if (rows_max < 0 || E < 1) return -1;
    return (rows_max + 64LL * E + 63) / 64 * 64;
}

moe_status moe_expert_dgrad(const void* a, const int32_t* offsets, const int32_t* kept, int E, int K, int N,
                            moe_dtype dtype, const void* w, int64_t rows_max, void* out, moe_stream_t stream)
{
    moe_status st = ffn_common_checks(offsets, kept, E, K, N, dtype, rows_max);
    if (st != MOE_OK) return st;
    if (!w || (rows_max > 0 && (!a || !out))) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({a, w, out})) return MOE_ERR_UNSUPPORTED;
    if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (rows_max == 0) return MOE_OK;
    tcg::Args g{};
    g.offsets = offsets;
    g.kept = kept;
    g.E = E;
    g.K = K;
    g.n_step = 256;
    g.half_off = 128;
    g.n_tiles = (N + 255) / 256;
    g.out_cols = N;
    g.out = (uint16_t*)out;
    g.wait_limit = g_wait_limit.load();
    return launch_tc_bn<tcg::EPI_IDENT, 256, tcg::MODE_BMN>(a, rows_max, K, w, (long long)E * K, g,
                                                             (cudaStream_t)stream);
}

moe_status moe_expert_dgrad_act(const void* do_perm, const int32_t* offsets, const int32_t* kept, int E, int d,
                                int F, moe_act act, moe_dtype dtype, const void* w2, const void* z, int64_t rows_max,
                                void* dz, moe_stream_t stream)
{
    moe_status st = ffn_common_checks(offsets, kept, E, d, F, dtype, rows_max);
    if (st != MOE_OK) return st;
    if (act != MOE_ACT_GELU && act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
    if (!w2 || (rows_max > 0 && (!do_perm || !z || !dz))) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({do_perm, w2, z, dz})) return MOE_ERR_UNSUPPORTED;
    if (dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (rows_max == 0) return MOE_OK;
    tcg::Args g{};
    g.offsets = offsets;
    g.kept = kept;
    g.E = E;
    g.K = d;
    g.n_step = 256;
    g.half_off = 128;
    g.n_tiles = (F + 255) / 256;
    g.out_cols = F;
    g.out = (uint16_t*)dz;
    g.in_z = (const uint16_t*)z;
    g.z_cols = act == MOE_ACT_SWIGLU ? 2 * F : F;
    g.wait_limit = g_wait_limit.load();
    cudaStream_t s = (cudaStream_t)stream;
    if (act == MOE_ACT_SWIGLU)
        return launch_tc_bn<tcg::EPI_DSWIGLU, 256, tcg::MODE_BMN>(do_perm, rows_max, d, w2, (long long)E * d, g, s);
    return launch_tc_bn<tcg::EPI_DGELU, 256, tcg::MODE_BMN>(do_perm, rows_max, d, w2, (long long)E * d, g, s);
}

moe_status moe_pack_segments_t(const void* src, const int32_t* offsets, const int32_t* kept, int E, int C,
                               int64_t rows_max, int64_t ld, moe_dtype dtype, void* dst, moe_stream_t stream)
{
    if (E < 1 || E > MAX_E || C <= 0 || rows_max < 0 || !offsets || !kept || !dtype_ok(dtype))
        return MOE_ERR_INVALID_ARG;
    if (ld < moe_wgrad_cols(rows_max, E) || ld % 64) return MOE_ERR_INVALID_ARG;
    if (rows_max > 0 && (!src || !dst)) return MOE_ERR_INVALID_ARG;
    if (!all_aligned16({src, dst})) return MOE_ERR_UNSUPPORTED;
    if (dtype != MOE_BF16 || C % 64 || ld / 64 > 65535) return MOE_ERR_UNSUPPORTED;
    if (rows_max == 0) return MOE_OK;
    bwd::pack_segments_t_kernel<<<dim3(C / 64, (unsigned)(ld / 64)), 256, 0, (cudaStream_t)stream>>>(
        (const uint16_t*)src, offsets, kept, E, C, (long long)ld, (uint16_t*)dst);
    return launch_status();
}

moe_status moe_expert_wgrad(const void* at, const void* bt, const int32_t* kept, int E, int M, int N, int64_t ld,
                            moe_dtype dtype, void* dw, moe_dtype dw_dtype, moe_stream_t stream)
{
    if (E < 1 || E > MAX_E || M <= 0 || N <= 0 || ld <= 0 || !kept || !at || !bt || !dw || !dtype_ok(dtype) ||
        !dtype_ok(dw_dtype))
        return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 || M % 64 || N % 64 || ld % 64 || ld >= INT_MAX) return MOE_ERR_UNSUPPORTED;
    if (!all_aligned16({at, bt, dw})) return MOE_ERR_UNSUPPORTED;
    tcg::Args a{};
    a.kept = kept;
    a.E = E;
    a.K = (int)ld;
    a.m_tiles = (M + 127) / 128;
    a.m_rows = M;
    a.n_step = 256;
    a.half_off = 128;
    a.n_tiles = (N + 255) / 256;
    a.out_cols = N;
    a.out_f32 = dw_dtype == MOE_F32 ? (float*)dw : nullptr;
    a.out = dw_dtype == MOE_BF16 ? (uint16_t*)dw : nullptr;
    a.n_fastest = wgrad_n_fastest(M, N);
    a.wait_limit = g_wait_limit.load();
    return launch_tc_bn<tcg::EPI_IDENT, 256, tcg::MODE_WGRAD>(at, 0, (int)ld, bt, N, a, (cudaStream_t)stream, M);
}

moe_status moe_expert_wgrad_rows(const void* a, const void* b, const int32_t* offsets, const int32_t* kept, int E,
                                 int M, int N, int64_t rows_max, moe_dtype dtype, void* dw, moe_dtype dw_dtype,
                                 moe_stream_t stream)
{
    if (E < 1 || E > MAX_E || M <= 0 || N <= 0 || rows_max < 0 || !offsets || !kept || !dw || !dtype_ok(dtype) ||
        !dtype_ok(dw_dtype))
        return MOE_ERR_INVALID_ARG;
    if (rows_max > 0 && (!a || !b)) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 || M % 64 || N % 64 || rows_max >= INT_MAX)
        return MOE_ERR_UNSUPPORTED;
    if (!all_aligned16({a, b, dw})) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    if (rows_max == 0) {   // no rows: every expert's gradient is zero
        const size_t bytes = (size_t)E * M * N * (dw_dtype == MOE_F32 ? 4 : 2);
        return cudaMemsetAsync(dw, 0, bytes, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
    }
    tcg::Args g{};
    g.offsets = offsets;
    g.kept = kept;
    g.E = E;
    g.K = 0;
    g.m_tiles = (M + 127) / 128;
    g.m_rows = M;
    g.n_step = 256;
    g.half_off = 128;
    g.n_tiles = (N + 255) / 256;
    g.out_cols = N;
    g.out_f32 = dw_dtype == MOE_F32 ? (float*)dw : nullptr;
    g.out = dw_dtype == MOE_BF16 ? (uint16_t*)dw : nullptr;
    g.n_fastest = wgrad_n_fastest(M, N);
    g.wait_limit = g_wait_limit.load();
    return launch_tc_bn<tcg::EPI_IDENT, 256, tcg::MODE_WGRAD_ROWS>(a, rows_max, 0, b, 0, g, st);
}

moe_status moe_route_bwd(const float* logits, const int32_t* topk_idx, const float* dgate, const int32_t* counts,
                         int64_t T, int E, int k, int renorm, float aux_coef, float z_coef, float* dl,
                         moe_stream_t stream)
{
    if (T < 0 || E < 1 || E > MAX_E || k < 1 || k > MAX_K || k > E || !counts) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_idx || !dgate || !dl)) return MOE_ERR_INVALID_ARG;
    if (T * k >= INT_MAX || T * E >= ((int64_t)1 << 40)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    int grid = ceil_div_i(T, 8);
    if (grid > sm_count() * 8) grid = sm_count() * 8;
    cudaStream_t st = (cudaStream_t)stream;
    const int Ti = (int)T;
#define MOE_RB(EP) bwd::route_bwd_kernel<EP><<<grid, 256, 0, st>>>(logits, topk_idx, dgate, counts, Ti, E, k, renorm, \
                                                                  aux_coef, z_coef, dl)
    if (E <= 32) MOE_RB(1);
    else if (E <= 64) MOE_RB(2);
    else if (E <= 128) MOE_RB(4);
    else MOE_RB(8);
#undef MOE_RB
    return launch_status();
}

moe_status moe_grad_x(const void* dx_perm, const int32_t* slot_row, const float* dl, const float* w_router,
                      int64_t T, int k, int E, int d, moe_dtype dtype, void* dx, moe_stream_t stream)
{
    if (T < 0 || k < 1 || k > MAX_K || E < 1 || E > MAX_E || d <= 0 || !dtype_ok(dtype)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!dx_perm || !slot_row || !dl || !w_router || !dx)) return MOE_ERR_INVALID_ARG;
    if (T / bwd::GX_TOK >= 65535 || d % 64) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!aligned16(dx_perm) || !aligned16(w_router) || !aligned16(dx))) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    const dim3 grid(ceil_div_i(d, bwd::GX_COLS), ceil_div_i(T, bwd::GX_TOK));
    cudaStream_t st = (cudaStream_t)stream;
    if (dtype == MOE_BF16)
        bwd::grad_x_kernel<true><<<grid, 256, 0, st>>>(dx_perm, slot_row, dl, w_router, (int)T, k, E, d, dx);
    else
        bwd::grad_x_kernel<false><<<grid, 256, 0, st>>>(dx_perm, slot_row, dl, w_router, (int)T, k, E, d, dx);
    return launch_status();
}

moe_status moe_router_wgrad(const float* dl, const void* x, moe_dtype xdt, int64_t T, int E, int d, float* dW,
                            float* db, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (T < 1 || E < 1 || E > MAX_E || d <= 0 || !dl || !x || !dW || !dtype_ok(xdt)) return MOE_ERR_INVALID_ARG;
    if (d % 64 || !all_aligned16({x, ws})) return MOE_ERR_UNSUPPORTED;
    const int S = router_wgrad_splits(T, E, d);
    const size_t need = (size_t)S * E * d * sizeof(float);
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const int per = ceil_div_i(ceil_div_i(T, S), 32) * 32;
    const dim3 grid(ceil_div_i(d, bwd::RW_COLS), ceil_div_i(E, bwd::RW_EXP), S);
    float* part = (float*)ws;
    if (xdt == MOE_BF16)
        bwd::router_wgrad_kernel<true><<<grid, 256, 0, st>>>(dl, x, (int)T, E, d, per, part);
    else
        bwd::router_wgrad_kernel<false><<<grid, 256, 0, st>>>(dl, x, (int)T, E, d, per, part);
    moe_status s = launch_status();
    if (s != MOE_OK) return s;
    const long long n = (long long)E * d;
    int g2 = ceil_div_i(n, 256);
    if (g2 > sm_count() * 8) g2 = sm_count() * 8;
    bwd::router_wgrad_sum_kernel<<<g2, 256, 0, st>>>(part, S, n, dW);
    s = launch_status();
    if (s != MOE_OK || !db) return s;
    rfu::prob_sum_kernel<<<E, 256, 0, st>>>(dl, (int)T, E, db);
    return launch_status();
}

moe_status moe_router_grads(const void* dx_perm, const int32_t* slot_row, const float* dl, const float* w_router,
                            const void* x, int64_t T, int k, int E, int d, moe_dtype dtype, void* dx, float* dW,
                            float* db, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    if (T < 0 || k < 1 || k > MAX_K || E < 1 || E > MAX_E || d <= 0 || !dtype_ok(dtype) || !dW || !db)
        return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!dx_perm || !slot_row || !dl || !w_router || !x || !dx)) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 || d % 64 || T >= INT_MAX) return MOE_ERR_UNSUPPORTED;
    if (!all_aligned16({dx_perm, w_router, x, dx, dW, ws})) return MOE_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    if (T == 0) {   // no tokens: the router gets no gradient
        if (cudaMemsetAsync(dW, 0, (size_t)E * d * sizeof(float), st) != cudaSuccess ||
            cudaMemsetAsync(db, 0, (size_t)E * sizeof(float), st) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    const RouterGradsLayout L = router_grads_layout(T, E, d);
    if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    uint8_t* w = (uint8_t*)ws;
    uint16_t* dl3 = (uint16_t*)(w + L.dl3);
    uint16_t* W3 = (uint16_t*)(w + L.W3);
    float* zr = (float*)(w + L.zr);
    float* P = (float*)(w + L.P);
    int32_t* seg1 = (int32_t*)(w + L.seg1);
    int32_t* segS = (int32_t*)(w + L.segS);
    const int Ep = L.Ep, K3 = 3 * Ep;

    // 1. bf16 parts of dl and W, row segments
    {
        const long long n = (long long)T * Ep + (long long)Ep * d;
        long long g1 = (n + 255) / 256;
        if (g1 > sm_count() * 8LL) g1 = sm_count() * 8LL;
        bwd::router_grads_prep_kernel<<<(int)g1, 256, 0, st>>>(dl, w_router, (int)T, E, Ep, d, L.S, dl3, W3, seg1,
                                                              segS);
        moe_status s = launch_status();
        if (s != MOE_OK) return s;
    }
    // 2. zr = dl3 . W3  [T, d] fp32 (one segment of T rows, B MN-major)
    {
        tcg::Args g{};
        g.offsets = seg1;
        g.kept = seg1 + 2;
        g.E = 1;
        g.K = K3;
        g.n_step = 256;
        g.half_off = 128;
        g.n_tiles = (d + 255) / 256;
        g.out_cols = d;
        g.out_f32 = zr;
        g.wait_limit = g_wait_limit.load();
        moe_status s = launch_tc_bn<tcg::EPI_IDENT, 256, tcg::MODE_BMN>(dl3, T, K3, W3, K3, g, st);
        if (s != MOE_OK) return s;
    }
    // 3. dx = zr + sum over the kept slots of dx_perm, one rounding
    {
        const int vec16 = d / 8;
        long long g3 = (T + 7) / 8;
        if (g3 > sm_count() * 16LL) g3 = sm_count() * 16LL;
        bwd::grad_x_gather_kernel<<<(int)g3, 256, 0, st>>>((const uint4*)dx_perm, slot_row, (const float4*)zr, (int)T,
                                                          k, vec16, (uint4*)dx);
        moe_status s = launch_status();
        if (s != MOE_OK) return s;
    }
    // 4. P[s] = [hi | lo](rows of split s)^T x[rows of split s]  [S, 2 Ep, d] fp32
    //    (the first 2 Ep columns of dl3, row stride 3 Ep)
    {
        tcg::Args g{};
        g.offsets = segS;
        g.kept = segS + L.S + 1;
        g.E = L.S;
        g.m_tiles = (2 * Ep + 127) / 128;
        g.m_rows = 2 * Ep;
        g.lda = K3;
        g.n_step = 256;
        g.half_off = 128;
        g.n_tiles = (d + 255) / 256;
        g.out_cols = d;
        g.out_f32 = P;
        g.wait_limit = g_wait_limit.load();
        moe_status s = launch_tc_bn<tcg::EPI_IDENT, 256, tcg::MODE_WGRAD_ROWS>(dl3, T, 0, x, 0, g, st);
        if (s != MOE_OK) return s;
    }
    // 5. dW = hi part + lo part over the splits; db = sum_t dl (fixed-order fp64 tree)
    {
        const long long n4 = (long long)E * d / 4;
        long long g5 = (n4 + 255) / 256;
        if (g5 > sm_count() * 8LL) g5 = sm_count() * 8LL;
        bwd::router_grads_reduce_kernel<<<(int)g5, 256, 0, st>>>((const float4*)P, L.S, E, Ep, d / 4, (float4*)dW);
        moe_status s = launch_status();
        if (s != MOE_OK) return s;
        rfu::prob_sum_kernel<<<E, 256, 0, st>>>(dl, (int)T, E, db);
        return launch_status();
    }
}

extern "C" moe_status moe_dispatch_noalloc(const int32_t* topk_idx, const float* topk_gate, int64_t T, int k, int E,
                                           int64_t cap, const void* x, moe_dtype xdt, int d, int32_t* counts,
                                           int32_t* kept, int32_t* offsets, int32_t* slot_row, int32_t* row_token,
                                           float* row_gate, void* x_perm, int32_t* n_dropped, moe_stream_t stream)
{
    if (T < 0 || T > INT_MAX || k < 1 || k > MAX_K || E < 1 || E > MAX_E) return MOE_ERR_INVALID_ARG;
    const size_t need = dispatch_ws_bytes(T, k, E);
    if (need > NOALLOC_SCRATCH_BYTES) {
        std::fprintf(stderr,
                     "moe_dispatch_noalloc: T*k = %lld assignments over E = %d experts need %zu bytes of "
                     "scratch; the built-in scratch holds %zu bytes (use moe_dispatch with a workspace)\n",
                     (long long)T * k, E, need, NOALLOC_SCRATCH_BYTES);
        return MOE_ERR_WORKSPACE;
    }
    void* scratch = nullptr;   // an empty batch (T*k = 0) reads no histogram
    if (need > 0) {
        const moe_status st = noalloc_scratch(&scratch);
        if (st != MOE_OK) return st;
    }
    return moe_dispatch(topk_idx, topk_gate, T, k, E, cap, x, xdt, d, counts, kept, offsets, slot_row, row_token,
                        row_gate, x_perm, n_dropped, scratch, NOALLOC_SCRATCH_BYTES, stream);
}
