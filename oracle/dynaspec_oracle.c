/*
 * DynaSpec draft head + speculative-sampling verification: the CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the CPU-baseline leg of
 * the benchmark call this file; the product library never includes, links or runs it, and
 * it includes nothing of the product.  It is plain C99 with fp64 accumulation and plain
 * loops: no SIMD intrinsics, no BLAS, no blocking or reordering beyond what each step's
 * definition states.  OpenMP only splits independent rows / sequences across threads.
 *
 * What it follows (DynaSpec, arXiv 2510.13847; pages: the arXiv abstract on
 * mlsanity.com/paper/2510.13847 and the summary "DynaSpec: Context-aware Dynamic
 * Speculative Sampling for Large-Vocabulary Language Models" on papers.lunadong.com):
 *   - router: a 2-layer MLP scoring vocabulary clusters from the drafter hidden state
 *     (summary, Technical Details > System Modules "Router"; Key Hyperparameters: two
 *     layers with a ReLU between them);
 *   - position-aware budget: k_c(t) clusters kept at draft position t (summary, Key Novelty;
 *     Key Hyperparameters "shortlist_budget_decay");
 *   - shortlist: the tokens of the best-scoring clusters taken together (abstract; summary,
 *     Problem Definition, whose output is the shortlist V_S);
 *   - gathered head: logits only for the shortlisted LM-head rows (summary, System Modules
 *     "Gathered LM Head"; Novel Architectural Elements "Dynamic Vocabulary Head");
 *   - verification over the full vocabulary by rejection sampling (abstract; summary,
 *     Pipeline Flow "Rejection Sampling Verification"), i.e. the speculative sampling of
 *     Leviathan et al. 2023 ("Fast Inference from Transformers via Speculative Decoding")
 *     and Chen et al. 2023 ("Accelerating Large Language Model Decoding with Speculative
 *     Sampling"), both in the pages' reference list.  The pages do not print the algorithm;
 *     the standard statement of it is used.
 *
 * Where the pages leave a step open the plainest reading is taken and stated at the
 * function.  Decisions that turn floating point into an integer (top-k membership, the
 * greedy / Gumbel argmax, accept-or-reject, the inverse-CDF crossing) compare values
 * rounded to fp32, the precision the CUDA path decides in; every value is computed in fp64
 * first.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------ */
/* Threads (the CPU baseline reports how many it used)                                  */
/* ------------------------------------------------------------------------------------ */
void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp32 view of an fp64 value: the precision decisions are taken in. */
static float f32(double x) { return (float)x; }

/* ------------------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2,  */
/* 3", SC'11).  Each round multiplies words 0 and 2 by the two Philox constants, swaps    */
/* the halves of the 64-bit products across the lanes and xors in the round key; the key */
/* is advanced by the two Weyl constants between rounds.                                  */
/* ------------------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t MUL0 = 0xD2511F53u, MUL1 = 0xCD9E8D57u;
    const uint32_t WEYL0 = 0x9E3779B9u, WEYL1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)MUL0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)MUL1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += WEYL0;
        k1 += WEYL1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The drafter's Gumbel uniform for entry j of the shortlist (its index in the list's order:
 * selected clusters ascending, each cluster's tokens in CSR order) at draft position pos, head
 * row `row` (the pages name no generator; reading): counter (j >> 2, pos, row, 0), key = the
 * two 32-bit halves of `seed`, word j & 3, mapped to (2*(w >> 9) + 1) * 2^-24, which lies
 * strictly inside (0, 1) and is exact in fp32.  Four consecutive entries share one Philox
 * block; the list's order is fixed, so the same list always gets the same draws. */
double orc_gumbel_uniform(uint64_t seed, int64_t j, int pos, int row)
{
    uint32_t ctr[4] = {(uint32_t)((uint64_t)j >> 2), (uint32_t)pos, (uint32_t)row, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    uint32_t x = w[j & 3];
    return (2.0 * (double)(x >> 9) + 1.0) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------------------ */
/* Router (2-layer MLP): u = act(W1 h + b1), s = W2 u + b2.                              */
/* act 0 = ReLU (the summary's Key Hyperparameters); act 1 = GELU in its exact erf form,  */
/* 0.5 x (1 + erf(x / sqrt 2)), which the Tiny workload names.  No sigmoid follows: the  */
/* router is trained with BCE (summary, Objective Functions), but a sigmoid is monotone  */
/* and leaves the top-k unchanged, so the scores are the pre-sigmoid logits.              */
/* H [B, d], W1 [Hr, d], b1 [Hr], W2 [M, Hr], b2 [M] bf16 bits; u [B, Hr] (may be NULL),  */
/* scores [B, M] fp64.                                                                    */
/* ------------------------------------------------------------------------------------ */
static double act_fn(double x, int act)
{
    if (act == 0) return x > 0.0 ? x : 0.0;
    return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
}

int orc_router(const uint16_t *H, int B, int d, const uint16_t *W1, const uint16_t *b1,
               int Hr, const uint16_t *W2, const uint16_t *b2, int M, int act,
               double *u_out, double *scores)
{
    if (B < 0 || d <= 0 || Hr <= 0 || M <= 0 || (act != 0 && act != 1)) return 1;
    double *u = (double *)malloc(sizeof(double) * (size_t)B * (size_t)Hr);
    if (!u) return 2;
    #pragma omp parallel for schedule(static)
    for (long long bi = 0; bi < (long long)B * Hr; ++bi) {
        int b = (int)(bi / Hr), i = (int)(bi % Hr);
        double acc = 0.0;
        for (int k = 0; k < d; ++k)
            acc += bf16_to_f64(W1[(size_t)i * d + k]) * bf16_to_f64(H[(size_t)b * d + k]);
        u[bi] = act_fn(acc + bf16_to_f64(b1[i]), act);
    }
    #pragma omp parallel for schedule(static)
    for (long long bc = 0; bc < (long long)B * M; ++bc) {
        int b = (int)(bc / M), c = (int)(bc % M);
        double acc = 0.0;
        for (int i = 0; i < Hr; ++i)
            acc += bf16_to_f64(W2[(size_t)c * Hr + i]) * u[(size_t)b * Hr + i];
        scores[bc] = acc + bf16_to_f64(b2[c]);
    }
    if (u_out) memcpy(u_out, u, sizeof(double) * (size_t)B * (size_t)Hr);
    free(u);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Position-aware budget + top-k (abstract: the shortlist comes from the best clusters;   */
/* summary, Key Hyperparameters: k_c(t) decays with draft position t).  The decay law has */
/* no stated form; the caller passes k = the budget table's entry for the position.       */
/* Keeps the k clusters with the largest score, ties to the lower cluster id, and lists   */
/* them in ascending cluster id.  scores [B, M] fp64 -> ids [B, k].                        */
/* ------------------------------------------------------------------------------------ */
typedef struct { float s; int id; } scored_t;

static int cmp_scored_desc(const void *a, const void *b)
{
    const scored_t *x = (const scored_t *)a, *y = (const scored_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id);
}

static int cmp_int_asc(const void *a, const void *b)
{
    int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

int orc_topk(const double *scores, int B, int M, int k, int32_t *ids)
{
    if (k < 1 || k > M || B < 0) return 1;
    scored_t *buf = (scored_t *)malloc(sizeof(scored_t) * (size_t)M);
    int *sel = (int *)malloc(sizeof(int) * (size_t)k);
    if (!buf || !sel) { free(buf); free(sel); return 2; }
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < M; ++c) { buf[c].s = f32(scores[(size_t)b * M + c]); buf[c].id = c; }
        qsort(buf, (size_t)M, sizeof(scored_t), cmp_scored_desc);
        for (int i = 0; i < k; ++i) sel[i] = buf[i].id;
        qsort(sel, (size_t)k, sizeof(int), cmp_int_asc);
        for (int i = 0; i < k; ++i) ids[(size_t)b * k + i] = sel[i];
    }
    free(buf); free(sel);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Shortlist V_S = union of the selected clusters.  Clusters partition the vocabulary, so  */
/* the union needs no de-duplication.  The pages fix the set, not an order; reading: the  */
/* selected clusters in ascending id, each cluster's tokens in its CSR order.  Returns    */
/* |V_S|.  csr_off [M+1], csr_tok [V]; ids [k] ascending -> S [|V_S|].                      */
/* ------------------------------------------------------------------------------------ */
int64_t orc_shortlist(const int32_t *csr_off, const int32_t *csr_tok, int M,
                      const int32_t *ids, int k, int32_t *S)
{
    int64_t n = 0;
    for (int i = 0; i < k; ++i) {
        int c = ids[i];
        if (c < 0 || c >= M) return -1;
        for (int32_t p = csr_off[c]; p < csr_off[c + 1]; ++p) S[n++] = csr_tok[p];
    }
    return n;
}

/* ------------------------------------------------------------------------------------ */
/* Gathered head: l_j = h . W[S_j] for every shortlisted token (summary, System Modules   */
/* "Gathered LM Head": logits for the selected part of the vocabulary).  rows of H [R, d] */
/* share the list S [n]; l [R, n] fp64.                                                    */
/* ------------------------------------------------------------------------------------ */
void orc_head(const uint16_t *H, int R, int d, const uint16_t *W, const int32_t *S,
              int64_t n, double *l)
{
    #pragma omp parallel for schedule(static)
    for (long long rj = 0; rj < (long long)R * n; ++rj) {
        long long r = rj / n, j = rj % n;
        const uint16_t *w = W + (size_t)S[j] * (size_t)d;
        const uint16_t *h = H + (size_t)r * (size_t)d;
        double acc = 0.0;
        for (int k = 0; k < d; ++k) acc += bf16_to_f64(h[k]) * bf16_to_f64(w[k]);
        l[rj] = acc;
    }
}

/* ------------------------------------------------------------------------------------ */
/* Draft token from the shortlist logits, mapped back to a full-vocabulary id.            */
/*   T = 0: x = S[argmax_j l_j], ties to the lower full-vocabulary id.                     */
/*   T > 0: x = S[argmax_j (l_j / T + g_j)], g_j = -log(-log u(j))  (Gumbel-max, an exact */
/*          draw from softmax(l / T) over the shortlist), ties to the lower id.            */
/* Also returns the softmax statistics of l / T_eff (T_eff = T, or 1 when T = 0):          */
/* m = max_j l_j / T_eff and s = sum_j exp(l_j / T_eff - m).  Returns the token id and     */
/* its index in S through *idx.                                                            */
/* ------------------------------------------------------------------------------------ */
int32_t orc_draft_sample(const double *l, const int32_t *S, int64_t n, double T,
                         uint64_t seed, int pos, int row, int64_t *idx, double *m_out,
                         double *s_out)
{
    double te = T > 0.0 ? T : 1.0;
    double m = -INFINITY, s = 0.0;
    for (int64_t j = 0; j < n; ++j) if (l[j] / te > m) m = l[j] / te;
    for (int64_t j = 0; j < n; ++j) s += exp(l[j] / te - m);
    int64_t best = -1;
    float best_key = 0.0f;
    for (int64_t j = 0; j < n; ++j) {
        double key = l[j];
        if (T > 0.0) {
            double u = orc_gumbel_uniform(seed, j, pos, row);
            key = l[j] / T - log(-log(u));
        }
        float k32 = f32(key);
        if (best < 0 || k32 > best_key || (k32 == best_key && S[j] < S[best])) {
            best = j;
            best_key = k32;
        }
    }
    if (idx) *idx = best;
    if (m_out) *m_out = m;
    if (s_out) *s_out = s;
    return best < 0 ? -1 : S[best];
}

/* ------------------------------------------------------------------------------------ */
/* Verification helpers.                                                                  */
/* ------------------------------------------------------------------------------------ */

/* p = softmax(z / T) over the whole row, in fp64. */
static void softmax_row(const float *z, int V, double T, double *p)
{
    double m = -INFINITY, s = 0.0;
    for (int v = 0; v < V; ++v) if ((double)z[v] / T > m) m = (double)z[v] / T;
    for (int v = 0; v < V; ++v) { p[v] = exp((double)z[v] / T - m); s += p[v]; }
    for (int v = 0; v < V; ++v) p[v] /= s;
}

/* argmax_v z[v], ties to the lower id. */
static int argmax_row(const float *z, int V)
{
    int a = 0;
    for (int v = 1; v < V; ++v) if (z[v] > z[a]) a = v;
    return a;
}

/* Inverse-CDF draw from the non-negative weights w[0..V) in ascending token id: the smallest
 * v whose cumulative weight exceeds u * sum(w) (compared in fp32).  If rounding leaves no
 * such v, the last token with positive weight. */
static int inverse_cdf(const double *w, int V, double u)
{
    double tot = 0.0;
    for (int v = 0; v < V; ++v) tot += w[v];
    float target = f32(u * tot);
    double c = 0.0;
    int last = -1;
    for (int v = 0; v < V; ++v) {
        c += w[v];
        if (w[v] > 0.0) last = v;
        if (f32(c) > target) return v;
    }
    return last;
}

/* q = softmax(l / T) over one shortlist, scattered into a dense full-vocabulary row
 * (zero outside the shortlist). */
static void dense_q(const double *l, const int32_t *S, int64_t n, double T, int V, double *qd)
{
    double m = -INFINITY, s = 0.0;
    for (int v = 0; v < V; ++v) qd[v] = 0.0;
    for (int64_t j = 0; j < n; ++j) if (l[j] / T > m) m = l[j] / T;
    for (int64_t j = 0; j < n; ++j) s += exp(l[j] / T - m);
    for (int64_t j = 0; j < n; ++j) qd[S[j]] = exp(l[j] / T - m) / s;
}

/* ------------------------------------------------------------------------------------ */
/* Chain verification (speculative sampling, Leviathan et al. / Chen et al.), per sequence */
/* over gamma draft tokens x_1..x_gamma with target rows z_1..z_{gamma+1}:                 */
/*   p_t = softmax(z_t / T) over the FULL vocabulary, q_t = softmax(l_t / T) over the      */
/*   shortlist S_t (zero elsewhere).  For t = 1..gamma in order: accept x_t iff            */
/*   u_t * q_t(x_t) < p_t(x_t).  At the first rejection the accepted length is t-1 and the */
/*   correction is drawn from norm(max(0, p_t - q_t)) by inverse CDF with u_{gamma+1}; if  */
/*   every draft is accepted the bonus token is drawn from p_{gamma+1} the same way.       */
/*   A residual with no mass (possible only by rounding) falls back to p_t.                 */
/*   T = 0 (greedy): accept while x_t = argmax z_t; the correction / bonus is that argmax. */
/* Layouts: z [B][gamma+1][V]; the draft logits and shortlist of (b, t) start at           */
/* qoff[b*gamma + t-1] in ql / S; draft_idx [B*gamma] is x_t's index in its shortlist;     */
/* u [B][gamma+1].  The gamma+1 target rows and gamma+1 uniforms per sequence are the     */
/* standard statement's; the pages do not fix them.                                        */
/* ------------------------------------------------------------------------------------ */
int orc_verify_chain(int B, int gamma, int V, double T, const float *z, const double *ql,
                     const int64_t *qoff, const int32_t *S, const int64_t *draft_idx,
                     const float *u, int32_t *accepted, int32_t *correction)
{
    if (B < 0 || gamma < 1 || V < 1 || T < 0.0) return 1;
    int err = 0;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *qd = (double *)malloc(sizeof(double) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        if (!p || !qd || !r) { free(p); free(qd); free(r); err = 2; continue; }
        const float *zb = z + (size_t)b * (size_t)(gamma + 1) * (size_t)V;
        const float *ub = u + (size_t)b * (size_t)(gamma + 1);
        int A = gamma, corr = -1;
        for (int t = 1; t <= gamma; ++t) {
            const float *zt = zb + (size_t)(t - 1) * (size_t)V;
            int64_t lo = qoff[(size_t)b * gamma + (t - 1)], hi = qoff[(size_t)b * gamma + t];
            int64_t j = draft_idx[(size_t)b * gamma + (t - 1)];
            int x = S[lo + j];
            if (T == 0.0) {
                int a = argmax_row(zt, V);
                if (x == a) continue;
                A = t - 1; corr = a;
                break;
            }
            softmax_row(zt, V, T, p);
            dense_q(ql + lo, S + lo, hi - lo, T, V, qd);
            if (f32((double)ub[t - 1] * qd[x]) < f32(p[x])) continue;
            A = t - 1;
            double R = 0.0;
            for (int v = 0; v < V; ++v) { r[v] = p[v] > qd[v] ? p[v] - qd[v] : 0.0; R += r[v]; }
            corr = inverse_cdf(R > 0.0 ? r : p, V, (double)ub[gamma]);
            break;
        }
        if (A == gamma) {
            const float *zl = zb + (size_t)gamma * (size_t)V;
            if (T == 0.0) {
                corr = argmax_row(zl, V);
            } else {
                softmax_row(zl, V, T, p);
                corr = inverse_cdf(p, V, (double)ub[gamma]);
            }
        }
        accepted[b] = A;
        correction[b] = corr;
        free(p); free(qd); free(r);
    }
    return err;
}

/* ------------------------------------------------------------------------------------ */
/* Tree verification.  The pages cite EAGLE's tree drafting but do not state a tree       */
/* verifier; reading: recursive rejection sampling over siblings (the multi-draft form of */
/* speculative sampling used by SpecInfer and EAGLE).  Node n carries its own draft row   */
/* q_n = softmax(l_n / T) over its depth's shortlist and a token x_n drawn from it.       */
/* Walk from the root with p = softmax(z_root / T):                                        */
/*   try the children of the current node in index order; child c is accepted iff         */
/*   u_c * q_c(x_c) < p(x_c); after a rejection p <- norm(max(0, p - q_c)) (kept as it was */
/*   if that has no mass) and the next sibling is tried.  On acceptance move to c with     */
/*   p = softmax(z_c / T).  When no child is accepted (or the node is a leaf) draw the     */
/*   correction from the current p by inverse CDF with u_res[depth of the current node].  */
/*   T = 0: accept the first child whose token is argmax z of the current node; the        */
/*   correction is that argmax.                                                            */
/* Each sibling step is itself an exact speculative-sampling step, so the emitted token   */
/* follows the target distribution.                                                        */
/* Layouts (N = D * Wd nodes, depth-major, node n at depth n / Wd + 1):                    */
/*   z [B][1+N][V] (row 0 root, row 1+n after node n); parent [N] (-1 = root);             */
/*   shortlist of (b, dep) at soff[b*D + dep-1] in S; node (b, n) draft logits at          */
/*   qoff[b*N + n] in ql (same length as its shortlist); draft_idx [B][N]; u_node [B][N];  */
/*   u_res [B][D+1] -> accepted [B], correction [B], path [B][D] (node ids, -1 padded).    */
/* ------------------------------------------------------------------------------------ */
int orc_verify_tree(int B, int D, int Wd, int V, double T, const float *z,
                    const int32_t *parent, const double *ql, const int64_t *qoff,
                    const int32_t *S, const int64_t *soff, const int64_t *draft_idx,
                    const float *u_node, const float *u_res, int32_t *accepted,
                    int32_t *correction, int32_t *path)
{
    if (B < 0 || D < 1 || Wd < 1 || V < 1 || T < 0.0) return 1;
    const int N = D * Wd;
    int err = 0;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *qd = (double *)malloc(sizeof(double) * (size_t)V);
        double *rn = (double *)malloc(sizeof(double) * (size_t)V);
        if (!p || !qd || !rn) { free(p); free(qd); free(rn); err = 2; continue; }
        const float *zb = z + (size_t)b * (size_t)(1 + N) * (size_t)V;
        int cur = -1, dep = 0, A = 0, corr = -1;
        for (int i = 0; i < D; ++i) path[(size_t)b * D + i] = -1;
        for (;;) {
            const float *zc = zb + (size_t)(cur + 1) * (size_t)V;
            int next = -1;
            if (T == 0.0) {
                int a = argmax_row(zc, V);
                for (int c = 0; c < N && dep < D; ++c) {
                    if (parent[c] != cur) continue;
                    int64_t lo = soff[(size_t)b * D + dep];
                    int x = S[lo + draft_idx[(size_t)b * N + c]];
                    if (x == a) { next = c; break; }
                }
                if (next < 0) { corr = a; break; }
            } else {
                softmax_row(zc, V, T, p);           /* p holds the current (normalised) residual */
                for (int c = 0; c < N && dep < D; ++c) {
                    if (parent[c] != cur) continue;
                    int64_t lo = soff[(size_t)b * D + dep], hi = soff[(size_t)b * D + dep + 1];
                    int64_t ql0 = qoff[(size_t)b * N + c];
                    dense_q(ql + ql0, S + lo, hi - lo, T, V, qd);
                    int x = S[lo + draft_idx[(size_t)b * N + c]];
                    if (f32((double)u_node[(size_t)b * N + c] * qd[x]) < f32(p[x])) { next = c; break; }
                    double R = 0.0;
                    for (int v = 0; v < V; ++v) { rn[v] = p[v] > qd[v] ? p[v] - qd[v] : 0.0; R += rn[v]; }
                    if (R > 0.0) for (int v = 0; v < V; ++v) p[v] = rn[v] / R;
                }
                if (next < 0) { corr = inverse_cdf(p, V, (double)u_res[(size_t)b * (D + 1) + dep]); break; }
            }
            path[(size_t)b * D + A] = next;
            ++A;
            cur = next;
            ++dep;
        }
        accepted[b] = A;
        correction[b] = corr;
        free(p); free(qd); free(rn);
    }
    return err;
}

/* ------------------------------------------------------------------------------------ */
/* Spherical k-means over the LM-head rows: the offline step that forms the vocabulary     */
/* clusters the router scores (summary, Key Novelty and Key Hyperparameters: clusters of the */
/* LM-head rows by spherical k-means).  The pages give no iteration details; reading: the    */
/* standard Lloyd iteration for the cosine objective J = sum_v <W_v / |W_v|, mu_c(v)>,        */
/* centroids of unit length:                                                                */
/*   assignment  c(v) = argmax_c <W_v, mu_c>  (the row's own norm does not change the argmax), */
/*               ties to the lower c;                                                       */
/*   update      mu_c = S_c / |S_c|, S_c = sum of W_v / |W_v| over the tokens of cluster c;  */
/*               an empty cluster keeps its centroid;                                       */
/*   the CSR lists clusters in ascending id, each cluster's tokens in ascending token id.    */
/* With round_bf16 the assignment scores the centroids rounded to bf16 (round to nearest     */
/* even), the operand precision of the CUDA path's tensor-core contraction; the scores are  */
/* computed in fp64 and compared rounded to fp32, the precision that path decides in.        */
/* ------------------------------------------------------------------------------------ */
static double row_norm(const uint16_t *w, int d)
{
    double s = 0.0;
    for (int k = 0; k < d; ++k) { double x = bf16_to_f64(w[k]); s += x * x; }
    return sqrt(s);
}

static double round_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Initial centroids: rows init[0..M) of W scaled to unit length.  cent [M, d]. */
int orc_kmeans_init(const uint16_t *W, int V, int d, const int32_t *init, int M, double *cent)
{
    for (int c = 0; c < M; ++c) {
        if (init[c] < 0 || init[c] >= V) return 1;
        const uint16_t *w = W + (size_t)init[c] * d;
        double n = row_norm(w, d);
        for (int k = 0; k < d; ++k) cent[(size_t)c * d + k] = n > 0.0 ? bf16_to_f64(w[k]) / n : 0.0;
    }
    return 0;
}

/* One Lloyd step.  cent [M, d] in/out; assign [V], csr_off [M+1], csr_tok [V] out; *obj = J
 * of the new assignment under the centroids it was made with (exact fp64 centroids). */
int orc_kmeans_step(const uint16_t *W, int V, int d, int M, int round, double *cent,
                    int32_t *assign, int32_t *csr_off, int32_t *csr_tok, double *obj)
{
    double *mu = (double *)malloc(sizeof(double) * (size_t)M * d);
    double *inv = (double *)malloc(sizeof(double) * (size_t)V);
    if (!mu || !inv) { free(mu); free(inv); return 2; }
    for (size_t i = 0; i < (size_t)M * d; ++i) mu[i] = round ? round_bf16(cent[i]) : cent[i];
    double J = 0.0;
    #pragma omp parallel for schedule(static) reduction(+:J)
    for (int v = 0; v < V; ++v) {
        const uint16_t *w = W + (size_t)v * d;
        double n = row_norm(w, d);
        inv[v] = n > 0.0 ? 1.0 / n : 0.0;
        int best = 0;
        float bs = 0.f;
        for (int c = 0; c < M; ++c) {
            double s = 0.0;
            for (int k = 0; k < d; ++k) s += bf16_to_f64(w[k]) * mu[(size_t)c * d + k];
            if (c == 0 || f32(s) > bs) { bs = f32(s); best = c; }
        }
        assign[v] = best;
        double e = 0.0;
        for (int k = 0; k < d; ++k) e += bf16_to_f64(w[k]) * cent[(size_t)best * d + k];
        J += e * inv[v];
    }
    *obj = J;
    /* CSR: counts, exclusive scan, tokens in ascending id within each cluster */
    for (int c = 0; c <= M; ++c) csr_off[c] = 0;
    for (int v = 0; v < V; ++v) csr_off[assign[v] + 1]++;
    for (int c = 0; c < M; ++c) csr_off[c + 1] += csr_off[c];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)M);
    if (!fill) { free(mu); free(inv); return 2; }
    for (int c = 0; c < M; ++c) fill[c] = csr_off[c];
    for (int v = 0; v < V; ++v) csr_tok[fill[assign[v]]++] = v;
    free(fill);
    /* update: normalised sum of the unit rows of each cluster, in ascending token order */
    #pragma omp parallel for schedule(dynamic)
    for (int c = 0; c < M; ++c) {
        if (csr_off[c + 1] == csr_off[c]) continue;            /* empty: keep the centroid */
        double *dst = cent + (size_t)c * d;
        for (int k = 0; k < d; ++k) dst[k] = 0.0;
        for (int r = csr_off[c]; r < csr_off[c + 1]; ++r) {
            int v = csr_tok[r];
            const uint16_t *w = W + (size_t)v * d;
            for (int k = 0; k < d; ++k) dst[k] += bf16_to_f64(w[k]) * inv[v];
        }
        double n = 0.0;
        for (int k = 0; k < d; ++k) n += dst[k] * dst[k];
        n = sqrt(n);
        if (n > 0.0) for (int k = 0; k < d; ++k) dst[k] /= n;
    }
    free(mu);
    free(inv);
    return 0;
}
