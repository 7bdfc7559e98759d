/*
 * Float64 CPU oracle for one offloading-aware MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the CUDA path is
 * compared against; the library itself never links, loads or calls it.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * Every step is the plain definition from the source pages, in double
 * precision, with no blocking, fusion or reordering:
 *   - router softmax / top-k          : APEX (Adaptive Expert Prefetching for
 *     Edge MoE Inference) blog, §1 and §4.3 (alpha = softmax(q_r));
 *     SPICE write-up, section on the MoE I/O bottleneck (top-6 of 64).
 *   - prefetch router                 : APEX §4.1 (linear + softmax).
 *   - oracle budget delta*            : APEX §4.2, definition of delta*.
 *   - ordinal-logistic CDF delta_hat  : APEX §4.2, p_delta(x) and the
 *     inference rule delta_hat = min{delta : p_delta >= tau}.
 *   - stall-free substitution         : APEX §4.3, the stall-free
 *     selection of the correctness-preserving mode.
 *   - SwiGLU expert FFN, FloE sparsity: FloE (On-the-Fly MoE Inference on
 *     Memory-constrained GPU), method §1, the contextual-sparsity forward
 *     a^S(x) = (SiLU(x W_gate) (.) S_t(x W_up)) W_down.
 *   - LoRE surrogate                  : SPICE write-up, section "LoRE low-rank
 *     surrogate" (y_e ~ y_shared + B_e A_e h).
 *   - shared experts, combine         : SPICE write-up, LoRE section (the
 *     always-active shared expert) and the gate-weighted MoE sum.
 *   - look-ahead prefetch depth       : SPICE write-up, confidence-aware
 *     adaptive prefetch (top-K mass confidence, stop below the threshold,
 *     minimum depth).
 *   - bit-sliced expert weights       : ELMoE-3D (CSDN post), bit-slicing
 *     section (INT8 bit planes, top-b planes combined, shared scale) and the
 *     layout note (an expert's planes stored contiguously).
 *   - CPU-GPU orchestration           : SPICE write-up, section on CPU-GPU
 *     collaboration for prefetch misses (Fig. 6 and the per-miss cost
 *     model: fetch cost W_e/B + T_gpu against CPU cost T_cpu + 2H/B).
 *   - persistent expert cache         : ELMoE-3D (CSDN post), expert-axis
 *     elasticity: heat statistics, top-K subset, dynamic update, and the
 *     practice note on heat decay (multiply every heat by a factor just
 *     below 1 each step).
 *
 * Inputs are float32 arrays whose values are the layer's exact parameters
 * (bf16-representable for bf16 layers); each element is converted to double
 * where it is read.  Ties are broken towards the lowest index everywhere.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { POL_EXACT = 0, POL_SUBSTITUTE = 1, POL_LORE = 2, POL_HYBRID = 3, POL_HETERO = 4 };
enum { KIND_COMPUTE = 0, KIND_FETCH = 1, KIND_LORE = 2, KIND_CPU = 3 };
enum {
    M_TOPK = 0, M_PREFETCH = 1, M_THETA = 2, M_DSTAR = 3, M_SUBST = 4,
    M_GAMMA = 5, M_FLOE = 6, M_COST = 7, M_COUNT = 8
};

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the calling thread's later parallel regions (n >= 1). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Does value a (index ia) rank above value b (index ib)?  Larger first,
 * equal values ordered by the lower index. */
static int ranks_above(double a, int ia, double b, int ib) {
    return a > b || (a == b && ia < ib);
}

typedef struct { double v; int i; } orc_keyed;

/* qsort comparator: larger value first, then lower index. */
static int cmp_desc(const void* pa, const void* pb) {
    const orc_keyed* a = (const orc_keyed*)pa;
    const orc_keyed* b = (const orc_keyed*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

/* Router logits: l[t,e] = sum_j x[t,j] W[e,j] (+ bias[e]). */
void orc_logits(int T, int d, int N, const float* x, const float* W,
                const float* bias, double* l) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < N; ++e) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j)
                acc += (double)x[(size_t)t * d + j] * (double)W[(size_t)e * d + j];
            if (bias) acc += (double)bias[e];
            l[(size_t)t * N + e] = acc;
        }
}

/* Softmax over the N logits of one token. */
void orc_softmax(int N, const double* l, double* p) {
    double mx = l[0];
    for (int e = 1; e < N; ++e) if (l[e] > mx) mx = l[e];
    double s = 0.0;
    for (int e = 0; e < N; ++e) { p[e] = exp(l[e] - mx); s += p[e]; }
    for (int e = 0; e < N; ++e) p[e] /= s;
}

/* The k largest of v[0..n-1], largest first: k passes, each taking the
 * largest value not yet taken (lowest index among equals). */
void orc_topk(int n, int k, const double* v, int* idx) {
    unsigned char* taken = (unsigned char*)calloc((size_t)n, 1);
    for (int s = 0; s < k; ++s) {
        int best = -1;
        for (int i = 0; i < n; ++i)
            if (!taken[i] && (best < 0 || ranks_above(v[i], i, v[best], best))) best = i;
        idx[s] = best;
        taken[best] = 1;
    }
    free(taken);
}

/* Position of every entry in the descending order of v (0 = largest). */
static void rank_of(int n, const double* v, int* rank) {
    for (int i = 0; i < n; ++i) {
        int r = 0;
        for (int j = 0; j < n; ++j) if (j != i && ranks_above(v[j], j, v[i], i)) ++r;
        rank[i] = r;
    }
}

/* Ordinal-logistic CDF budget (APEX §4.2): s = w.x_pre,
 * p_delta = sigmoid(theta_delta - s), delta_hat = the smallest delta in
 * 0..delta_max with p_delta >= tau; delta_max when none reaches tau
 * (prefetch everything, the conservative reading of a case the page leaves
 * open).  *s_out receives s. */
int orc_delta_hat(int d, int delta_max, const float* w, const float* xpre,
                  const float* theta, double tau, double* s_out) {
    double s = 0.0;
    for (int j = 0; j < d; ++j) s += (double)w[j] * (double)xpre[j];
    if (s_out) *s_out = s;
    for (int delta = 0; delta <= delta_max; ++delta) {
        double p = 1.0 / (1.0 + exp(-((double)theta[delta] - s)));
        if (p >= tau) return delta;
    }
    return delta_max;
}

/* Prefetch set (APEX §4.2): the top-(k + delta_hat) experts of the prefetch
 * router's logits, as a bitmask. */
uint64_t orc_prefetch_set(int N, int k, int delta_hat, const double* lp) {
    int m = k + delta_hat;
    if (m > N) m = N;
    int* idx = (int*)malloc(sizeof(int) * (size_t)m);
    orc_topk(N, m, lp, idx);
    uint64_t mask = 0;
    for (int i = 0; i < m; ++i) mask |= (uint64_t)1 << idx[i];
    free(idx);
    return mask;
}

/* Oracle budget (APEX §4.2): the smallest delta in 0..N-k for which the
 * routed set is a subset of the prefetch router's top-(k+delta). */
int orc_delta_star(int N, int k, const int* routed, const double* lp) {
    for (int delta = 0; delta <= N - k; ++delta) {
        uint64_t p = orc_prefetch_set(N, k, delta, lp);
        int all = 1;
        for (int i = 0; i < k; ++i) if (!((p >> routed[i]) & 1)) { all = 0; break; }
        if (all) return delta;
    }
    return N - k;
}

/* Stall-free selection (APEX §4.3, the stall-free expert selection of its
 * correctness-preserving mode).  Meaning of the rule: the layer runs only on
 * experts that are already available, with as many experts as it routed.
 * Every routed expert that is available stays; each routed expert that is
 * not is replaced, and the replacements are the available non-routed experts
 * that the ORIGINAL router rates highest.  Written as a definition: with
 * m = |routed \ available| and pool = available \ routed, the result is
 *   (routed ∩ available)  ∪  { e ∈ pool : fewer than m members of pool rank
 *                                          above e by alpha }
 * (larger alpha ranks above; equal alpha: the lower index ranks above).
 * Sets are bitmasks over N <= 64 experts.  Returns the selected set, or
 * all-ones when the pool holds fewer than m experts. */
uint64_t orc_stall_free_select(int N, uint64_t routed, const double* alpha,
                               uint64_t available) {
    const uint64_t pool = available & ~routed;
    int m = 0, pool_size = 0;
    for (int e = 0; e < N; ++e) {
        m += (int)(((routed & ~available) >> e) & 1);
        pool_size += (int)((pool >> e) & 1);
    }
    if (pool_size < m) return ~(uint64_t)0;
    uint64_t chosen = routed & available;
    for (int e = 0; e < N; ++e) {
        if (!((pool >> e) & 1)) continue;
        int above = 0;
        for (int f = 0; f < N; ++f)
            if (f != e && ((pool >> f) & 1) && ranks_above(alpha[f], f, alpha[e], e)) ++above;
        if (above < m) chosen |= (uint64_t)1 << e;
    }
    return chosen;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One SwiGLU expert on one token (FloE method §1 with S_t = identity):
 * y[:] += sum_i SiLU(x.Wg[i]) * (x.Wu[i]) * Wd[i,:], with Wg, Wu, Wd all
 * [I, d] (row i belongs to intermediate channel i). */
void orc_expert_ffn(int d, int I, const float* x, const float* Wg, const float* Wu,
                    const float* Wd, double* y) {
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int j = 0; j < d; ++j) {
            g += (double)x[j] * (double)Wg[(size_t)i * d + j];
            u += (double)x[j] * (double)Wu[(size_t)i * d + j];
        }
        double h = silu(g) * u;
        for (int j = 0; j < d; ++j) y[j] += h * (double)Wd[(size_t)i * d + j];
    }
}

/* FloE contextual sparsity (method §1): u = x W_up; S_t keeps the m channels
 * with the largest |u| (lowest channel index among equals); gate and down
 * only for kept channels: y += sum_{i in S_t} SiLU(x.Wg[i]) u_i Wd[i,:].
 * kept[0..m-1] receives the kept channels in ascending order; *gap receives
 * the |u| gap between the m-th and (m+1)-th largest, divided by max |u|. */
void orc_expert_ffn_floe(int d, int I, int m, const float* x, const float* Wg,
                         const float* Wu, const float* Wd, double* y, int* kept,
                         double* gap) {
    double* u = (double*)malloc(sizeof(double) * (size_t)I);
    double* au = (double*)malloc(sizeof(double) * (size_t)I);
    int* order = (int*)malloc(sizeof(int) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += (double)x[j] * (double)Wu[(size_t)i * d + j];
        u[i] = acc;
        au[i] = fabs(acc);
    }
    /* Descending order of |u| by a library sort; equal magnitudes keep the
     * lower channel index first. */
    orc_keyed* kv = (orc_keyed*)malloc(sizeof(orc_keyed) * (size_t)I);
    for (int i = 0; i < I; ++i) { kv[i].v = au[i]; kv[i].i = i; }
    qsort(kv, (size_t)I, sizeof(orc_keyed), cmp_desc);
    int* rank = (int*)malloc(sizeof(int) * (size_t)I);
    for (int i = 0; i < I; ++i) { order[i] = kv[i].i; rank[kv[i].i] = i; }
    free(kv);
    double mx = I > 0 ? au[order[0]] : 0.0;
    if (gap) *gap = (m < I && mx > 0) ? (au[order[m - 1]] - au[order[m]]) / mx : INFINITY;
    int n = 0;
    for (int i = 0; i < I; ++i) {
        if (rank[i] >= m) continue;
        if (kept) kept[n] = i;
        ++n;
        double g = 0.0;
        for (int j = 0; j < d; ++j) g += (double)x[j] * (double)Wg[(size_t)i * d + j];
        double h = silu(g) * u[i];
        for (int j = 0; j < d; ++j) y[j] += h * (double)Wd[(size_t)i * d + j];
    }
    free(u); free(au); free(order); free(rank);
}

/* LoRE surrogate residual (SPICE write-up, LoRE section): v += B (A x),
 * A [r, d], B [d, r]. */
void orc_lore(int d, int r, const float* x, const float* A, const float* B, double* v) {
    for (int q = 0; q < r; ++q) {
        double z = 0.0;
        for (int j = 0; j < d; ++j) z += (double)A[(size_t)q * d + j] * (double)x[j];
        for (int j = 0; j < d; ++j) v[j] += (double)B[(size_t)j * r + q] * z;
    }
}

/* Batch-level resident set: the n_res experts with the largest prefetch
 * probability summed over the batch, sum_t softmax(l_p[t,:]).  *gap receives
 * the gap between the n_res-th and (n_res+1)-th sums. */
uint64_t orc_batch_resident(int T, int N, const double* lp, int n_res, double* gap) {
    double* sum = (double*)calloc((size_t)N, sizeof(double));
    double* q = (double*)malloc(sizeof(double) * (size_t)N);
    for (int t = 0; t < T; ++t) {
        orc_softmax(N, lp + (size_t)t * N, q);
        for (int e = 0; e < N; ++e) sum[e] += q[e];
    }
    int* idx = (int*)malloc(sizeof(int) * (size_t)N);
    orc_topk(N, N, sum, idx);
    uint64_t mask = 0;
    for (int i = 0; i < n_res && i < N; ++i) mask |= (uint64_t)1 << idx[i];
    if (gap) *gap = (n_res < N) ? sum[idx[n_res - 1]] - sum[idx[n_res]] : INFINITY;
    free(sum); free(q); free(idx);
    return mask;
}

/* Persistent expert cache, one decode step (ELMoE-3D, expert-axis
 * elasticity: "heat" statistics of the experts the routing function selects,
 * the most frequently activated top-K kept, updated as the activation pattern
 * changes; heat decay per time step from the practice note).
 *   routed[n_slots]: the experts the router selected this step (-1: none).
 *   heat[N] (in/out): heat_e <- decay * heat_e + #{slots routed to e}.
 *   Returns the new cache: the C experts of largest heat, lowest index on
 *   ties (all N if C >= N).  *gap = heat of the C-th minus the (C+1)-th.
 *   *hits = routed slots whose expert is in old_cache (the cache the step
 *   ran with). */
uint64_t orc_cache_update(int N, int n_slots, const int* routed, double decay, int C, double* heat,
                          uint64_t old_cache, int* hits, double* gap) {
    int h = 0;
    int* count = (int*)calloc((size_t)N, sizeof(int));
    for (int i = 0; i < n_slots; ++i) {
        const int e = routed[i];
        if (e < 0 || e >= N) continue;
        count[e] += 1;
        if ((old_cache >> e) & 1) h += 1;
    }
    for (int e = 0; e < N; ++e) heat[e] = decay * heat[e] + (double)count[e];
    int* idx = (int*)malloc(sizeof(int) * (size_t)N);
    orc_topk(N, N, heat, idx);
    uint64_t cache = 0;
    for (int i = 0; i < C && i < N; ++i) cache |= (uint64_t)1 << idx[i];
    if (gap) *gap = (C > 0 && C < N) ? heat[idx[C - 1]] - heat[idx[C]] : INFINITY;
    if (hits) *hits = h;
    free(count); free(idx);
    return cache;
}

/* Confidence-aware prefetch depth (SPICE write-up, section on
 * confidence-aware adaptive prefetch): a draft predicts, from the current
 * hidden state, the expert distribution of each of the next J layers; its
 * confidence C is the probability mass on the predicted top-K experts;
 * prediction goes one layer deeper while C stays at or above tau and stops
 * at the first layer below it; the depth is never below the minimum depth
 * D_min that lets a transfer finish within the layers it runs ahead of.
 * The draft's prediction head is the identity here: layer l+j's router
 * applied to the current x (the trained head is not given).
 *   x[T,d]; W[j] = router of look-ahead layer j [N,d]; bias[j] [N] or NULL.
 *   conf[T,J] = sum of the K largest of softmax(x W[j]^T + bias[j]).
 *   depth[T]  = min(J, max(d_min, c)), c = number of leading layers
 *               j = 0, 1, ... whose conf >= tau (the scan stops at the first
 *               below tau).
 *   tok_masks[T,J] = the top-K set of layer j when j < depth[t], else 0.
 *   layer_masks[J] = OR over tokens of tok_masks[., j].
 *   margin[T] (optional): the smallest |conf - tau| over the layers the scan
 *               reads, and the logit gap at position K over the layers kept. */
void orc_prefetch_depth(int T, int d, int N, int K, int J, const float* x, const float* const* W,
                        const float* const* bias, double tau, int d_min, double* conf, int* depth,
                        uint64_t* tok_masks, uint64_t* layer_masks, double* margin) {
    double* l = (double*)malloc(sizeof(double) * (size_t)N);
    double* p = (double*)malloc(sizeof(double) * (size_t)N);
    int* idx = (int*)malloc(sizeof(int) * (size_t)N);
    for (int j = 0; j < J; ++j) layer_masks[j] = 0;
    for (int t = 0; t < T; ++t) {
        double m = INFINITY;
        int c = 0, scanning = 1;
        uint64_t set[64];
        double gap[64];
        for (int j = 0; j < J; ++j) {
            orc_logits(1, d, N, x + (size_t)t * d, W[j], bias ? bias[j] : 0, l);
            orc_softmax(N, l, p);
            orc_topk(N, N, l, idx);
            double mass = 0.0;
            set[j] = 0;
            for (int i = 0; i < K; ++i) {
                mass += p[idx[i]];
                set[j] |= (uint64_t)1 << idx[i];
            }
            gap[j] = K < N ? l[idx[K - 1]] - l[idx[K]] : INFINITY;
            conf[(size_t)t * J + j] = mass;
            if (scanning) {
                const double dm = fabs(mass - tau);
                if (dm < m) m = dm;
                if (mass >= tau) c += 1;
                else scanning = 0;
            }
        }
        int dep = c > d_min ? c : d_min;
        if (dep > J) dep = J;
        depth[t] = dep;
        for (int j = 0; j < J; ++j) {
            const uint64_t s_j = j < dep ? set[j] : 0;
            tok_masks[(size_t)t * J + j] = s_j;
            layer_masks[j] |= s_j;
            if (j < dep && gap[j] < m) m = gap[j];
        }
        if (margin) margin[t] = m;
    }
    free(l); free(p); free(idx);
}

/* Bit-sliced expert weights (ELMoE-3D, CSDN post, bit-slicing section and
 * the data-layout note): each weight is an INT8 value with a scale shared
 * across precisions; its 8 bits are stored as 8 binary planes, and a b-bit
 * representation combines the top b planes (MSB-only: the lower planes are
 * dropped; the learned LSB-enhancement scale is not used).
 * Quantisation (the pages leave it open; symmetric per output row): for row
 * r of the matrix the kernel reads (W itself, or W^T when transpose is set):
 *   s_r = max_k |W[r,k]| / 127            (float32 arithmetic)
 *   q[r,k] = clamp(rint(W[r,k] / s_r), -127, 127)   (float32 division,
 *            round half to even; s_r = 0 gives q = 0)
 * W is [rows_in, cols_in] row-major; the output is [R, C] with (R, C) =
 * (rows_in, cols_in), or (cols_in, rows_in) when transpose != 0. */
void orc_bitslice_quantize(int rows_in, int cols_in, const float* W, int transpose, signed char* q,
                           float* scale) {
    const int R = transpose ? cols_in : rows_in, Cc = transpose ? rows_in : cols_in;
    for (int r = 0; r < R; ++r) {
        float mx = 0.0f;
        for (int c = 0; c < Cc; ++c) {
            const float w = transpose ? W[(size_t)c * cols_in + r] : W[(size_t)r * cols_in + c];
            const float a = fabsf(w);
            if (a > mx) mx = a;
        }
        const float sr = mx / 127.0f;
        scale[r] = sr;
        for (int c = 0; c < Cc; ++c) {
            const float w = transpose ? W[(size_t)c * cols_in + r] : W[(size_t)r * cols_in + c];
            int v = 0;
            if (sr > 0.0f) {
                const float t = w / sr;
                v = (int)rintf(t);
                if (v > 127) v = 127;
                if (v < -127) v = -127;
            }
            q[(size_t)r * Cc + c] = (signed char)v;
        }
    }
}

/* The b-bit value of an INT8 weight: decompose its two's-complement byte
 * into the 8 bit planes, keep the top b (planes 7 .. 8-b) and recombine them
 * with their place values (plane 7 carries -128, plane p < 7 carries 2^p). */
int orc_bitslice_value(int q, int b) {
    const unsigned byte = (unsigned)(unsigned char)(signed char)q;
    int v = 0;
    for (int p = 7; p >= 8 - b && p >= 0; --p) {
        const int bit = (int)((byte >> p) & 1u);
        v += bit * (p == 7 ? -128 : (1 << p));
    }
    return v;
}

/* One expert's SwiGLU FFN on one token with b-bit weights (FloE method §1
 * form of the expert, ELMoE-3D bit-sliced weights):
 *   g_c = sg[c] sum_k x_k v_b(qg[c,k]),  u_c = su[c] sum_k x_k v_b(qu[c,k])
 *   h_c = SiLU(g_c) u_c,  y_j = sd[j] sum_c h_c v_b(qdT[j,c])
 * qg, qu [I, d]; qdT [d, I] (the down projection quantised per output j). */
void orc_bitslice_ffn(int d, int I, int b, const float* x, const signed char* qg, const float* sg,
                      const signed char* qu, const float* su, const signed char* qdT, const float* sd,
                      double* y) {
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    for (int c = 0; c < I; ++c) {
        double g = 0.0, u = 0.0;
        for (int k = 0; k < d; ++k) {
            g += (double)x[k] * (double)orc_bitslice_value(qg[(size_t)c * d + k], b);
            u += (double)x[k] * (double)orc_bitslice_value(qu[(size_t)c * d + k], b);
        }
        g *= (double)sg[c];
        u *= (double)su[c];
        h[c] = g / (1.0 + exp(-g)) * u;
    }
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int c = 0; c < I; ++c) acc += h[c] * (double)orc_bitslice_value(qdT[(size_t)j * I + c], b);
        y[j] = acc * (double)sd[j];
    }
    free(h);
}

/* SPICE's per-miss cost model (CPU-GPU collaboration section): a missing
 * expert that must be computed exactly is either fetched, at a cost of its
 * weight bytes over the link plus its FFN time on the GPU, or run on the
 * CPU, at a cost of the CPU FFN time plus one hidden state down and one
 * result up the link.  Here the CPU time and the hidden state grow with the
 * n token rows that need the expert in this batch:
 *   fetch = W_e / B + T_gpu        cpu = n t_cpu + 2 (n H) / B
 * Returns 1 (fetch) when fetch < cpu, else 0 (the CPU; equal costs go to the
 * CPU).  *margin = |fetch - cpu| / max(fetch, cpu). */
int orc_hetero_fetch(int n, double link_bps, double expert_bytes, double gpu_expert_s, double cpu_row_s,
                     double hidden_bytes, double* margin) {
    const double fetch = expert_bytes / link_bps + gpu_expert_s;
    const double cpu = (double)n * cpu_row_s + 2.0 * ((double)n * hidden_bytes) / link_bps;
    const double big = fetch > cpu ? fetch : cpu;
    if (margin) *margin = big > 0.0 ? fabs(fetch - cpu) / big : 0.0;
    return fetch < cpu;
}

typedef struct {
    int T, d, N, k, I, n_shared, I_shared, r, delta_max;
    int renorm;            /* 1: gates renormalised over the final set */
    int policy;            /* POL_* */
    int use_prefetch;      /* available set includes the per-token prefetch set */
    int m_keep;            /* FloE channels kept per token (== I: dense) */
    int has_prefetch;      /* prefetch router present */
    int route_only;        /* stop after the routing decisions (no expert math) */
    double tau, gamma;
    uint64_t resident;     /* batch-level resident mask */
    /* HETERO cost model (link bytes/s, expert bytes, GPU expert seconds,
     * CPU seconds per token row, hidden-state bytes per token) */
    double link_bps, expert_bytes, gpu_expert_s, cpu_row_s, hidden_bytes;
} orc_cfg;

typedef struct {
    const float *x, *x_pre, *w_router, *router_bias, *w_prefetch, *w_ord, *theta;
    const float *w_gate, *w_up, *w_down;       /* [N, I, d] */
    const float *sh_gate, *sh_up, *sh_down;    /* [n_shared, I_shared, d] */
    const float *lore_a, *lore_b;              /* [N, r, d], [N, d, r] */
} orc_inputs;

typedef struct {
    double *logits, *prob, *logits_p;          /* [T, N] */
    int* topk_idx; double* topk_gate;          /* [T, k] */
    int* delta_hat; double* score;             /* [T] */
    uint64_t* prefetch;                        /* [T] */
    int* delta_star;                           /* [T] */
    int* final_idx; double* final_gate; int* final_kind;   /* [T, k] */
    double* y_shared;                          /* [T, d] */
    double* out;                               /* [T, d] */
    double* margin;                            /* [T, M_COUNT] */
    int* kept;                                 /* [T, k, m_keep] or NULL */
    int* status;                               /* [T] 0 ok, 1 available set too small */
} orc_outputs;

static void one_token(const orc_cfg* c, const orc_inputs* in, const orc_outputs* o, int t) {
    const int N = c->N, k = c->k, d = c->d;
    const float* x = in->x + (size_t)t * d;
    const float* xp = (in->x_pre ? in->x_pre : in->x) + (size_t)t * d;
    double* l = o->logits + (size_t)t * N;
    double* a = o->prob + (size_t)t * N;
    double* lp = o->logits_p + (size_t)t * N;
    double* mg = o->margin + (size_t)t * M_COUNT;
    for (int i = 0; i < M_COUNT; ++i) mg[i] = INFINITY;

    /* 1. router: l = x W_r^T (+b), alpha = softmax(l), K_r = top-k of l */
    orc_logits(1, d, N, x, in->w_router, in->router_bias, l);
    orc_softmax(N, l, a);
    int routed[64];
    orc_topk(N, k, l, routed);
    uint64_t rmask = 0;
    for (int i = 0; i < k; ++i) {
        rmask |= (uint64_t)1 << routed[i];
        o->topk_idx[(size_t)t * k + i] = routed[i];
        o->topk_gate[(size_t)t * k + i] = a[routed[i]];
    }
    if (k < N) {
        int sorted[64];
        orc_topk(N, k + 1, l, sorted);
        mg[M_TOPK] = l[sorted[k - 1]] - l[sorted[k]];
    }

    /* 2-4. prefetch router, delta_hat, prefetch set, delta* */
    uint64_t pmask = ~(uint64_t)0;
    if (c->has_prefetch) {
        orc_logits(1, d, N, xp, in->w_prefetch, NULL, lp);
        double s;
        int dh = orc_delta_hat(d, c->delta_max, in->w_ord, xp, in->theta, c->tau, &s);
        o->delta_hat[t] = dh;
        o->score[t] = s;
        pmask = orc_prefetch_set(N, k, dh, lp);
        o->prefetch[t] = pmask;
        o->delta_star[t] = orc_delta_star(N, k, routed, lp);
        /* decisive margins: the CDF test at delta_hat and delta_hat-1, in
         * logit units (sigmoid is monotone), the l_p gap at k+delta_hat, and
         * the l_p gaps around the lowest-ranked routed expert (delta*). */
        double lt = log(c->tau / (1.0 - c->tau));
        for (int dd = dh - 1; dd <= dh; ++dd)
            if (dd >= 0) {
                double m = fabs((double)in->theta[dd] - s - lt);
                if (m < mg[M_THETA]) mg[M_THETA] = m;
            }
        int rank[64];
        rank_of(N, lp, rank);
        int order[64];
        for (int e = 0; e < N; ++e) order[rank[e]] = e;
        int m = k + dh;
        if (m < N) mg[M_PREFETCH] = lp[order[m - 1]] - lp[order[m]];
        int worst = 0;
        for (int i = 0; i < k; ++i) if (rank[routed[i]] > worst) worst = rank[routed[i]];
        double g1 = worst > 0 ? lp[order[worst - 1]] - lp[order[worst]] : INFINITY;
        double g2 = worst + 1 < N ? lp[order[worst]] - lp[order[worst + 1]] : INFINITY;
        mg[M_DSTAR] = g1 < g2 ? g1 : g2;
    } else {
        o->delta_hat[t] = 0;
        o->score[t] = 0.0;
        o->prefetch[t] = pmask;
        o->delta_star[t] = 0;
    }

    /* 5. miss policy over the available set A_t */
    uint64_t avail = c->resident & (c->use_prefetch ? pmask : ~(uint64_t)0);
    uint64_t missing = rmask & ~avail;
    uint64_t lore_set = 0, subst_routed = 0, fetch_set = 0;
    for (int i = 0; i < k; ++i) {
        int e = routed[i];
        if (!((missing >> e) & 1)) continue;
        uint64_t bit = (uint64_t)1 << e;
        switch (c->policy) {
            case POL_EXACT: fetch_set |= bit; break;
            case POL_LORE: lore_set |= bit; break;
            case POL_SUBSTITUTE: subst_routed |= bit; break;
            case POL_HETERO: {
                /* a low-confidence miss goes to LoRE, the others are computed
                 * exactly (fetched or on the CPU: decided over the batch) */
                double dist = fabs(a[e] - c->gamma);
                if (dist < mg[M_GAMMA]) mg[M_GAMMA] = dist;
                if (a[e] < c->gamma) lore_set |= bit; else fetch_set |= bit;
                break;
            }
            default: {
                /* HYBRID: a low-confidence miss (alpha < gamma) goes to LoRE,
                 * the others are substituted */
                double dist = fabs(a[e] - c->gamma);
                if (dist < mg[M_GAMMA]) mg[M_GAMMA] = dist;
                if (a[e] < c->gamma) lore_set |= bit; else subst_routed |= bit;
            }
        }
    }
    /* Substitution only for the misses chosen for it: the stall-free selection applied to
     * the routed experts that are not sent to LoRE. */
    uint64_t final_set = rmask;
    o->status[t] = 0;
    if (subst_routed) {
        uint64_t sel = orc_stall_free_select(N, rmask & ~lore_set, a, avail);
        if (sel == ~(uint64_t)0) {
            /* fewer available experts than slots to fill */
            o->status[t] = 1;
            sel = rmask & ~lore_set & avail;
        }
        final_set = sel | lore_set;
        /* boundary gap among the substitution candidates (logit units) */
        uint64_t pool = avail & ~rmask;
        int n_sub = 0;
        for (int e = 0; e < N; ++e) n_sub += (int)((subst_routed >> e) & 1);
        double cand[64];
        int nc = 0;
        for (int e = 0; e < N; ++e) if ((pool >> e) & 1) cand[nc++] = l[e];
        if (nc > n_sub) {
            int top[64];
            orc_topk(nc, n_sub + 1, cand, top);
            mg[M_SUBST] = cand[top[n_sub - 1]] - cand[top[n_sub]];
        }
    }

    /* final slots in canonical order: descending logit, lowest index first */
    double fl[64];
    int fidx[64], nf = 0;
    for (int e = 0; e < N; ++e) if ((final_set >> e) & 1) { fl[nf] = l[e]; fidx[nf] = e; ++nf; }
    int ford[64];
    orc_topk(nf, nf, fl, ford);
    double gsum = 0.0;
    for (int i = 0; i < nf; ++i) gsum += a[fidx[ford[i]]];
    for (int i = 0; i < k; ++i) {
        int e = i < nf ? fidx[ford[i]] : -1;
        size_t s = (size_t)t * k + i;
        o->final_idx[s] = e;
        if (e < 0) { o->final_gate[s] = 0.0; o->final_kind[s] = KIND_COMPUTE; continue; }
        o->final_gate[s] = c->renorm ? a[e] / gsum : a[e];
        uint64_t bit = (uint64_t)1 << e;
        o->final_kind[s] = (lore_set & bit) ? KIND_LORE : (fetch_set & bit) ? KIND_FETCH : KIND_COMPUTE;
    }

    /* 6-7. experts, shared experts, LoRE, combine */
    if (c->route_only) return;
    double* ysh = o->y_shared + (size_t)t * d;
    double* out = o->out + (size_t)t * d;
    for (int j = 0; j < d; ++j) { ysh[j] = 0.0; out[j] = 0.0; }
    const size_t Isd = (size_t)c->I_shared * d;
    for (int s = 0; s < c->n_shared; ++s)
        orc_expert_ffn(d, c->I_shared, x, in->sh_gate + s * Isd, in->sh_up + s * Isd,
                       in->sh_down + s * Isd, ysh);
    double lore_g = 0.0;
    double* ye = (double*)malloc(sizeof(double) * (size_t)d);
    const size_t Id = (size_t)c->I * d;
    for (int i = 0; i < k; ++i) {
        size_t sl = (size_t)t * k + i;
        int e = o->final_idx[sl];
        if (e < 0) continue;
        double g = o->final_gate[sl];
        for (int j = 0; j < d; ++j) ye[j] = 0.0;
        if (o->final_kind[sl] == KIND_LORE) {
            /* y_e ~ y_shared + B_e A_e x: the shared part is added once below */
            lore_g += g;
            orc_lore(d, c->r, x, in->lore_a + (size_t)e * c->r * d,
                     in->lore_b + (size_t)e * d * c->r, ye);
        } else if (c->m_keep < c->I) {
            double gap;
            orc_expert_ffn_floe(d, c->I, c->m_keep, x, in->w_gate + e * Id, in->w_up + e * Id,
                                in->w_down + e * Id, ye,
                                o->kept ? o->kept + sl * (size_t)c->m_keep : NULL, &gap);
            if (gap < mg[M_FLOE]) mg[M_FLOE] = gap;
        } else {
            orc_expert_ffn(d, c->I, x, in->w_gate + e * Id, in->w_up + e * Id,
                           in->w_down + e * Id, ye);
        }
        for (int j = 0; j < d; ++j) out[j] += g * ye[j];
    }
    for (int j = 0; j < d; ++j) out[j] += (1.0 + lore_g) * ysh[j];
    free(ye);
}

/* Whole layer, token by token (tokens are independent).  Under HETERO the
 * exact misses are then split between fetch and CPU per expert, by the cost
 * model over the n rows of the batch that need that expert; both are exact,
 * so the outputs do not change, only the slot kinds. */
void orc_layer_forward(const orc_cfg* c, const orc_inputs* in, const orc_outputs* o) {
    int T = c->T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) one_token(c, in, o, t);
    if (c->policy != POL_HETERO) return;
    int rows[64] = {0};
    for (size_t s = 0; s < (size_t)T * c->k; ++s)
        if (o->final_kind[s] == KIND_FETCH && o->final_idx[s] >= 0) rows[o->final_idx[s]] += 1;
    int fetch[64];
    double gap[64];
    for (int e = 0; e < c->N; ++e)
        fetch[e] = rows[e] > 0 ? orc_hetero_fetch(rows[e], c->link_bps, c->expert_bytes, c->gpu_expert_s,
                                                  c->cpu_row_s, c->hidden_bytes, &gap[e])
                               : 1;
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < c->k; ++i) {
            const size_t s = (size_t)t * c->k + i;
            const int e = o->final_idx[s];
            if (o->final_kind[s] != KIND_FETCH || e < 0) continue;
            if (!fetch[e]) o->final_kind[s] = KIND_CPU;
            double* mg = o->margin + (size_t)t * M_COUNT;
            if (gap[e] < mg[M_COST]) mg[M_COST] = gap[e];
        }
}
