/*
 * CPU oracle of the MoE-layer forward -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU-baseline
 * leg load this library.  The product path (the CUDA library and its Python
 * binding) never calls, links or imports it, and this file shares no source
 * with it.
 *
 * Plain, slow, obviously correct: every quantity is computed in double
 * precision with straightforward loops, in the order the method is stated.
 * Inputs stored as bf16 are widened exactly (the 16 bits become the top half
 * of an IEEE single).  OpenMP splits only independent tokens or output rows;
 * each dot product is summed serially in index order.
 *
 * Sources (the two pages that state the forward pass):
 *   [EP-tutorial]  "专家并行：混合专家模型的分布式训练方案" (expert-parallelism
 *                  tutorial): §1.1 router / experts / sparse top-K,
 *                  §2.1 steps 1-5 of the forward pass, §2.2 capacity formula
 *                  and token dropping, §5.1 auxiliary load-balance loss.
 *   [EP-guide]     "细粒度专家并行部署实践与优化指南" (fine-grained EP
 *                  deployment guide): §七 forward pseudo-code (top-k of the
 *                  gate probabilities, dispatch, per-expert compute, return).
 * and, for the routing variants:
 *   [swift-EP]     "ms-swift MoE模型加速：Megatron并行实测提速10倍" §3.2, the
 *                  EP bullet: route a token to an expert group, then Top-k
 *                  inside the group (16 experts split into 2 groups of 8).
 *   [swift-ETP]    "ETP专家并行加速MoE模型：ms-swift中稀疏架构的极致优化",
 *                  section on dynamic routing: a routing z-loss spreads the
 *                  router's choices.  The page gives no formula; the one
 *                  used is the router z-loss of Zoph et al., "ST-MoE:
 *                  Designing Stable and Transferable Sparse Expert Models"
 *                  (2022), eq. 5: mean over tokens of (log sum_e exp l[t,e])^2.
 *
 * Readings where the pages are silent (each is stated where it is used):
 *   softmax over all E experts, then top-k; ties -> lower expert index;
 *   k-rank = position in (logit desc, index asc) order; optional division of
 *   the k gates by their sum; capacity uses T (tokens), rounded half away
 *   from zero, no minimum; slots granted to all first choices in token order,
 *   then all second choices, ...; a dropped slot contributes nothing;
 *   f_i counts every choice before drops; P_i is the mean full softmax;
 *   GELU is the exact erf form; SwiGLU takes gate rows 0..F-1 and up rows
 *   F..2F-1 of w1[e].
 *
 * Every function is pinned by the CPU tests: brute-force top-k with exact
 * ties, the capacity table, the drop-count identity, a brute-force queue
 * simulation, identity experts, the dense-FFN and dense-mixture special cases
 * against library routines, and the closed forms of the aux loss.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_GELU = 0, ORC_SWIGLU = 1, ORC_IDENTITY = 2 };

/* Exact widening of element i of an f32 or bf16 array. */
static double elem(const void* p, int dt, int64_t i)
{
    if (dt == ORC_F32) return (double)((const float*)p)[i];
    uint32_t u = (uint32_t)((const uint16_t*)p)[i] << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* [EP-tutorial] §2.2: expert capacity = round((total tokens / experts) x cf).
 * "total tokens" is read as T; round() is half away from zero; no minimum.
 * cf <= 0 selects the dropless mode: every expert can hold all T tokens. */
int64_t orc_capacity(int64_t T, int E, double cf)
{
    if (cf <= 0.0) return T;
    return (int64_t)llround(((double)T / (double)E) * cf);
}

/* [EP-tutorial] §1.1 / §2.1 step 1: the router is a linear layer.
 * L[t,e] = sum_c x[t,c] * W[e,c] + b[e]   (b may be NULL). */
void orc_router_logits(const void* x, int xdt, const float* W, const float* b,
                       int64_t T, int d, int E, double* L)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int c = 0; c < d; ++c)
                s += elem(x, xdt, t * (int64_t)d + c) * (double)W[(int64_t)e * d + c];
            if (b) s += (double)b[e];
            L[t * E + e] = s;
        }
    }
}

/* [EP-tutorial] §2.1 step 1 and [EP-guide] §七: gate probabilities are a
 * softmax over all E experts; each token keeps the K experts of highest
 * probability.  Selection is on the logits (softmax is monotone), ordered by
 * (logit descending, expert index ascending): j = 0 is the first choice.
 *   idx[t,j]   chosen expert of rank j
 *   gate[t,j]  p[t, idx[t,j]], divided by sum_j p[t, idx[t,j]] when renorm
 *   prob[t,e]  full softmax (optional, may be NULL)
 *   prob_sum[e] = sum_t p[t,e]                                           */
void orc_route_grouped(const double* L, int64_t T, int E, int k, int renorm, int n_group, int topk_group,
                       int32_t* idx, double* gate, double* prob, double* prob_sum);

void orc_route(const double* L, int64_t T, int E, int k, int renorm,
               int32_t* idx, double* gate, double* prob, double* prob_sum)
{
    /* one group holding every expert: the choice is unrestricted */
    orc_route_grouped(L, T, E, k, renorm, 1, 1, idx, gate, prob, prob_sum);
}

/* [swift-EP] §3.2: group-limited routing.  The page says only that the
 * router picks the token's expert group and then runs Top-k inside it.
 * Readings: the E experts form n_group contiguous groups of E/n_group (the
 * placement the same section describes); a group's score is the largest
 * logit among its experts; the topk_group groups of highest score are kept
 * (equal scores: lower group index first); then the k experts are chosen
 * among the kept groups' experts in (logit desc, index asc) order.  The
 * softmax, the gates and prob_sum are those of orc_route (over all E
 * experts): only the choice is restricted.  n_group = 1 is orc_route.     */
void orc_route_grouped(const double* L, int64_t T, int E, int k, int renorm, int n_group, int topk_group,
                       int32_t* idx, double* gate, double* prob, double* prob_sum)
{
    double* P = prob ? prob : (double*)malloc(sizeof(double) * (size_t)(T * E));
    const int gsz = E / n_group;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* l = L + t * E;
        double* p = P + t * E;
        double mx = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > mx) mx = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = exp(l[e] - mx);
            z += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] /= z;

        /* group scores, and the groups in (score desc, group asc) order */
        double score[256];
        int gorder[256];
        for (int g = 0; g < n_group; ++g) {
            score[g] = l[g * gsz];
            for (int e = g * gsz + 1; e < (g + 1) * gsz; ++e)
                if (l[e] > score[g]) score[g] = l[e];
        }
        for (int g = 0; g < n_group; ++g) {
            int pos = g;
            while (pos > 0 && score[gorder[pos - 1]] < score[g]) {
                gorder[pos] = gorder[pos - 1];
                --pos;
            }
            gorder[pos] = g;
        }
        int allowed[256];
        for (int g = 0; g < n_group; ++g) allowed[g] = 0;
        for (int r = 0; r < topk_group; ++r) allowed[gorder[r]] = 1;

        /* k-rank order: insertion sort of the kept groups' experts by
         * (l desc, e asc); the insertion is stable, so equal logits keep
         * ascending indices. */
        int order[1024];
        int n = 0;
        for (int e = 0; e < E; ++e) {
            if (!allowed[e / gsz]) continue;
            int pos = n++;
            while (pos > 0 && l[order[pos - 1]] < l[e]) {
                order[pos] = order[pos - 1];
                --pos;
            }
            order[pos] = e;
        }
        double chosen = 0.0;
        for (int j = 0; j < k; ++j) chosen += p[order[j]];
        for (int j = 0; j < k; ++j) {
            idx[t * k + j] = order[j];
            gate[t * k + j] = renorm ? p[order[j]] / chosen : p[order[j]];
        }
    }
    for (int e = 0; e < E; ++e) prob_sum[e] = 0.0;
    for (int64_t t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) prob_sum[e] += P[t * E + e];
    if (!prob) free(P);
}

/* lse[t] = log sum_e exp(L[t,e]), evaluated as m + log sum_e exp(L[t,e] - m)
 * with m the row maximum (the same value, without overflow). */
void orc_logsumexp(const double* L, int64_t T, int E, double* lse)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* l = L + t * E;
        double mx = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > mx) mx = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp(l[e] - mx);
        lse[t] = mx + log(z);
    }
}

/* [swift-ETP] routing z-loss, in the ST-MoE form:
 * L_z = beta * (1/T) * sum_t lse[t]^2. */
double orc_z_loss(const double* lse, int64_t T, double beta)
{
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t) s += lse[t] * lse[t];
    return beta * s / (double)T;
}

/* [EP-tutorial] §2.1 step 2 (dispatch plan) and §2.2 (capacity, dropping).
 * Slots are granted in k-rank-then-token order: all first choices in token
 * order, then all second choices, and so on.  pos[t,j] is the place of the
 * assignment (t,j) in its expert's queue, or -1 when that place is at or
 * beyond the capacity (the slot is dropped).
 *   counts[e]  every assignment to e, before drops
 *   kept[e]    min(counts[e], cap)
 *   *n_dropped number of dropped assignments                              */
void orc_dispatch(const int32_t* idx, int64_t T, int k, int E, int64_t cap,
                  int32_t* counts, int32_t* kept, int32_t* pos, int64_t* n_dropped)
{
    int64_t* fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
    for (int j = 0; j < k; ++j)
        for (int64_t t = 0; t < T; ++t) {
            int e = idx[t * k + j];
            int64_t p = fill[e]++;
            pos[t * k + j] = (p < cap) ? (int32_t)p : -1;
        }
    int64_t dropped = 0;
    for (int e = 0; e < E; ++e) {
        counts[e] = (int32_t)fill[e];
        kept[e] = (int32_t)(fill[e] < cap ? fill[e] : cap);
        dropped += fill[e] - kept[e];
    }
    *n_dropped = dropped;
    free(fill);
}

static double act_gelu(double z) { return z * 0.5 * (1.0 + erf(z / sqrt(2.0))); }
static double act_silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert FFN applied to one row v[d] ([EP-tutorial] §2.1 step 4; the
 * two-matrix expert of the ETP page: w1 projects d -> N1, w2 projects F -> d).
 *   z[n]   = sum_c w1[e,n,c] * v[c],            n < N1
 *   a[n]   = GELU(z[n]) | silu(z[n]) * z[F+n] | z[n],   n < F
 *   out[o] = sum_n w2[e,o,n] * a[n],            o < d
 * a (length F) is returned too when not NULL.  par != 0 splits the rows of
 * each projection over threads. */
static void ffn_row(const double* v, const void* w1, const void* w2, int wdt,
                    int e, int d, int F, int act, double* a_out, double* out, int par)
{
    const int N1 = (act == ORC_SWIGLU) ? 2 * F : F;
    double* z = (double*)malloc(sizeof(double) * (size_t)N1);
    double* a = (double*)malloc(sizeof(double) * (size_t)F);
    const int64_t w1e = (int64_t)e * N1 * d, w2e = (int64_t)e * d * F;
#pragma omp parallel for schedule(static) if (par)
    for (int n = 0; n < N1; ++n) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += elem(w1, wdt, w1e + (int64_t)n * d + c) * v[c];
        z[n] = s;
    }
    for (int n = 0; n < F; ++n) {
        if (act == ORC_GELU) a[n] = act_gelu(z[n]);
        else if (act == ORC_SWIGLU) a[n] = act_silu(z[n]) * z[F + n];
        else a[n] = z[n];
    }
#pragma omp parallel for schedule(static) if (par)
    for (int o = 0; o < d; ++o) {
        double s = 0.0;
        for (int n = 0; n < F; ++n) s += elem(w2, wdt, w2e + (int64_t)o * F + n) * a[n];
        out[o] = s;
    }
    if (a_out) memcpy(a_out, a, sizeof(double) * (size_t)F);
    free(z);
    free(a);
}

/* Public single-row FFN (used by tests to look at one expert in isolation). */
void orc_expert_ffn_row(const void* v_in, int vdt, const void* w1, const void* w2, int wdt,
                        int e, int d, int F, int act, double* a_out, double* out)
{
    double* v = (double*)malloc(sizeof(double) * (size_t)d);
    for (int c = 0; c < d; ++c) v[c] = elem(v_in, vdt, c);
    ffn_row(v, w1, w2, wdt, e, d, F, act, a_out, out, 1);
    free(v);
}

/* [EP-tutorial] §2.1 steps 3-5 with the gate weighting of the layer output:
 * for each listed token t,
 *   y[t] = sum over j with pos[t,j] >= 0 of gate[t,j] * FFN_{idx[t,j]}(x[t])
 * summed in j order; a token whose every slot was dropped gets a zero row
 * (it bypasses the layer through the residual, §2.2).
 * tokens: n_tok token ids (rows of y follow this list).                    */
void orc_combine(const void* x, int xdt, const int32_t* tokens, int64_t n_tok,
                 const int32_t* idx, const double* gate, const int32_t* pos, int k,
                 const void* w1, const void* w2, int wdt, int d, int F, int act, double* y)
{
    const int outer = n_tok >= orc_num_threads();
#pragma omp parallel for schedule(dynamic, 1) if (outer)
    for (int64_t i = 0; i < n_tok; ++i) {
        const int64_t t = tokens[i];
        double* v = (double*)malloc(sizeof(double) * (size_t)d);
        double* f = (double*)malloc(sizeof(double) * (size_t)d);
        for (int c = 0; c < d; ++c) v[c] = elem(x, xdt, t * (int64_t)d + c);
        double* yt = y + i * (int64_t)d;
        for (int o = 0; o < d; ++o) yt[o] = 0.0;
        for (int j = 0; j < k; ++j) {
            if (pos[t * k + j] < 0) continue;
            ffn_row(v, w1, w2, wdt, idx[t * k + j], d, F, act, NULL, f, !outer);
            for (int o = 0; o < d; ++o) yt[o] += gate[t * k + j] * f[o];
        }
        free(v);
        free(f);
    }
}

/* [EP-tutorial] §5.1: L_aux = alpha * num_experts * sum_i f_i * P_i with
 * f_i = counts[i] / T (fraction of tokens sent to expert i, every choice,
 * before drops) and P_i = prob_sum[i] / T (mean gate probability).
 * The post-drop variant of f_i (only the slots that survived the capacity
 * cut) is the same formula with kept[] passed as counts. */
double orc_aux_loss(const int32_t* counts, const double* prob_sum, int64_t T, int E, double alpha)
{
    double s = 0.0;
    for (int e = 0; e < E; ++e) s += ((double)counts[e] / (double)T) * (prob_sum[e] / (double)T);
    return alpha * (double)E * s;
}
