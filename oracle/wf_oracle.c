/*
 * CPU oracle for the WhiFlash verify-and-route round.  TEST INFRASTRUCTURE:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may call it; the library never does.
 *
 * Plain, slow, obviously correct: every result is the textbook definition
 * written out as loops, in double precision, from the same bf16 / fp32 /
 * int32 inputs the GPU library receives.  No blocking, fusion or
 * reordering; OpenMP only distributes independent positions / sequences
 * across host threads (each sum keeps its natural index order).
 *
 * Sources (WhiFlash: Accelerating Speculative Decoding with Token-Level
 * Cross-Paradigm Routing, arXiv 2606.07710, and the Qwen3-4B-EAGLE3 and
 * Qwen3-4B-NeuralRouter-df-e3 model cards):
 *   - greedy verification: the target's next-token choice at a verified
 *     position is the argmax of its logits (paper Sec. 3.3.1, greedy
 *     decoding; Sec. 4 "Evaluation");
 *   - the drafted chain / tree is verified in parallel and decoding resumes
 *     from the last accepted token (paper Sec. 3.2);
 *   - acceptance length = tokens accepted per verification round
 *     (paper Sec. 4 "Metrics");
 *   - neural router: h -> Linear(d, m) -> GELU -> (dropout) -> Linear(m, 1)
 *     (paper Sec. 3.3.2 and App. A "Neural Router Architecture"); route to
 *     the autoregressive drafter iff the prediction exceeds tau (paper
 *     Sec. 3.3.2 "Hardware-Aware Routing Decision");
 *   - EAGLE-3 draft head over a fixed 32K draft vocabulary with top-k and a
 *     draft-to-target id map (EAGLE3 model card, "Model Description",
 *     "Technical Specifications", "Factors").
 *
 * Every function is pinned by tests/test_oracle_pins.py against brute force,
 * closed forms and hand-built cases; none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bfloat16 bit pattern (the high half of an IEEE binary32). */
static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One logit: <h_p, W_v> = sum_k h[p,k] * W[v,k], summed for k = 0..d-1. */
static double logit(const uint16_t* hrow, const uint16_t* wrow, int64_t d) {
    double s = 0.0;
    for (int64_t k = 0; k < d; ++k) s += bf16_value(hrow[k]) * bf16_value(wrow[k]);
    return s;
}

/*
 * Target LM head + greedy choice.  For each position p:
 *   ids[p]      = the lowest v attaining max_v <h_p, W_v>
 *   maxlogit[p] = that maximum
 *   gap[p]      = maximum - (largest logit among the other ids)  (0 on a tie)
 * maxlogit / gap may be NULL.
 */
int oracle_lmhead_argmax(const uint16_t* h, const uint16_t* W, int64_t P, int64_t d, int64_t V,
                         int32_t* ids, double* maxlogit, double* gap) {
    if (!h || !W || !ids || P < 0 || d <= 0 || V <= 0) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < P; ++p) {
        double best = -INFINITY, second = -INFINITY;
        int64_t best_v = -1;
        for (int64_t v = 0; v < V; ++v) {
            double L = logit(h + p * d, W + v * d, d);
            if (L > best) {
                second = best;
                best = L;
                best_v = v;
            } else if (L > second) {
                second = L;
            }
        }
        ids[p] = (int32_t)best_v;
        if (maxlogit) maxlogit[p] = best;
        if (gap) gap[p] = best - second;
    }
    return 0;
}

/*
 * DFlash block verification for sequence-packed chains.  Sequence b owns
 * verified rows pos_off[b] .. pos_off[b+1]-1: row pos_off[b] is the last
 * committed token, row pos_off[b]+1+j holds draft token j.  The target
 * choice at row pos_off[b]+j checks draft token j.  Drafts of sequence b are
 * draft[node_off[b] .. node_off[b+1]-1] (K = node count).
 *   n_accept[b] = largest n with draft[j] == g[root + j] for all j < n
 *   last_pos[b] = root + n  (global row of the last accepted token)
 *   bonus[b]    = g[last_pos[b]]  (the target's own next token, committed too)
 *   path[b*path_stride + j] = j for j < n, -1 after (may be NULL)
 */
int oracle_verify_chain(const int32_t* g, const int32_t* draft, const int32_t* pos_off,
                        const int32_t* node_off, int B, int32_t* n_accept, int32_t* bonus,
                        int32_t* last_pos, int32_t* path, int path_stride) {
    if (!g || !draft || !pos_off || !node_off || B < 0) return 1;
    for (int b = 0; b < B; ++b) {
        int root = pos_off[b];
        int K = node_off[b + 1] - node_off[b];
        const int32_t* dr = draft + node_off[b];
        int n = 0;
        while (n < K && dr[n] == g[root + n]) n++;
        n_accept[b] = n;
        last_pos[b] = root + n;
        bonus[b] = g[root + n];
        if (path)
            for (int j = 0; j < path_stride; ++j) path[(int64_t)b * path_stride + j] = j < n ? j : -1;
    }
    return 0;
}

/*
 * EAGLE-3 tree verification.  Sequence b has nodes node_off[b] ..
 * node_off[b+1]-1 with sequence-local parent indices (-1 = root, otherwise
 * parent < node) and draft tokens tok[].  Node i of sequence b is verified
 * at row pos_off[b]+1+i; the root at row pos_off[b].
 *   node i is accepted iff its token equals the target choice at its
 *   parent's row and its parent is accepted (the root always is);
 *   depth(i) = 1 + depth(parent) with depth(root) = 0;
 *   the deepest accepted node (lowest index on a tie) ends the accepted path;
 *   n_accept = its depth (0 when no node is accepted), last_pos = its row
 *   (the root row when none), bonus = g[last_pos], path = node ids from
 *   depth 1 down to it, -1 padded (may be NULL).
 * Returns 2 if a parent index is out of range (that sequence gets -1s).
 */
int oracle_verify_tree(const int32_t* g, const int32_t* tok, const int32_t* parent,
                       const int32_t* node_off, const int32_t* pos_off, int B, int32_t* n_accept,
                       int32_t* bonus, int32_t* last_pos, int32_t* path, int path_stride) {
    if (!g || !tok || !parent || !pos_off || !node_off || B < 0) return 1;
    int rc = 0;
    for (int b = 0; b < B; ++b) {
        int root = pos_off[b];
        int N = node_off[b + 1] - node_off[b];
        const int32_t* tk = tok + node_off[b];
        const int32_t* pa = parent + node_off[b];
        char* acc = (char*)calloc((size_t)N + 1, 1);
        int* depth = (int*)calloc((size_t)N + 1, sizeof(int));
        int bad = 0, best = -1, best_depth = 0;
        for (int i = 0; i < N; ++i) {
            int p = pa[i];
            if (p < -1 || p >= i) { bad = 1; break; }
            int prow = (p < 0) ? root : root + 1 + p;
            int parent_acc = (p < 0) ? 1 : acc[p];
            acc[i] = (char)(parent_acc && tk[i] == g[prow]);
            depth[i] = 1 + ((p < 0) ? 0 : depth[p]);
            if (acc[i] && depth[i] > best_depth) { best_depth = depth[i]; best = i; }
        }
        if (bad) {
            rc = 2;
            n_accept[b] = bonus[b] = last_pos[b] = -1;
            if (path) for (int j = 0; j < path_stride; ++j) path[(int64_t)b * path_stride + j] = -1;
        } else {
            n_accept[b] = best_depth;
            last_pos[b] = best < 0 ? root : root + 1 + best;
            bonus[b] = g[last_pos[b]];
            if (path) {
                for (int j = 0; j < path_stride; ++j) path[(int64_t)b * path_stride + j] = -1;
                for (int i = best; i >= 0; i = pa[i])
                    if (depth[i] - 1 < path_stride) path[(int64_t)b * path_stride + depth[i] - 1] = i;
            }
        }
        free(acc);
        free(depth);
    }
    return rc;
}

/*
 * Runtime-informed router, WhiFlash-Entropy (paper Sec. 3.3.1): the entropy of
 * the target's next-token distribution p = softmax(logits) at row rows[b],
 *   H[b] = - sum_v p_v log p_v   (natural log),
 * and route[b] = 1 (autoregressive drafter) if H[b] > tau, else 0.
 * The softmax is written with the usual max shift (it does not change p):
 * p_v = exp(L_v - M) / sum_u exp(L_u - M), M = max_v L_v.
 */
int oracle_entropy(const uint16_t* hidden, const int32_t* rows, int B, const uint16_t* W, int64_t d, int64_t V,
                   double tau, double* H, int32_t* route) {
    if (!hidden || !rows || !W || !H || B < 0 || d <= 0 || V <= 0) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const uint16_t* h = hidden + (int64_t)rows[b] * d;
        double* L = (double*)malloc((size_t)V * sizeof(double));
        double M = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            L[v] = logit(h, W + v * d, d);
            if (L[v] > M) M = L[v];
        }
        double S = 0.0;
        for (int64_t v = 0; v < V; ++v) S += exp(L[v] - M);
        double ent = 0.0;
        for (int64_t v = 0; v < V; ++v) {
            const double p = exp(L[v] - M) / S;
            if (p > 0.0) ent -= p * log(p);
        }
        H[b] = ent;
        if (route) route[b] = ent > tau ? 1 : 0;
        free(L);
    }
    return 0;
}

/*
 * Rows kept after verification (paper Sec. 3.2: decoding continues from the
 * last accepted token, so the target states of the committed positions are
 * kept and every other drafted row is dropped).  For sequence b with
 * n = n_accept[b] accepted drafts along path[b*path_stride ..]:
 *   acc_rows[b*(path_stride+1) + 0]     = pos_off[b]                (the root row)
 *   acc_rows[b*(path_stride+1) + j]     = pos_off[b] + 1 + path[j-1], j = 1..n
 *   acc_rows[b*(path_stride+1) + j]     = -1                        for j > n
 *   acc_off[0] = 0, acc_off[b+1] = acc_off[b] + n + 1   (packed order of the kept rows)
 */
int oracle_accepted_rows(const int32_t* n_accept, const int32_t* path, int path_stride, const int32_t* pos_off,
                         int B, int32_t* acc_rows, int32_t* acc_off) {
    if (!n_accept || !pos_off || !acc_rows || !acc_off || B < 0 || path_stride < 0) return 1;
    acc_off[0] = 0;
    for (int b = 0; b < B; ++b) {
        const int n = n_accept[b];
        int32_t* out = acc_rows + (int64_t)b * (path_stride + 1);
        for (int j = 0; j <= path_stride; ++j) out[j] = -1;
        out[0] = pos_off[b];
        for (int j = 1; j <= n && j <= path_stride; ++j) out[j] = pos_off[b] + 1 + path[(int64_t)b * path_stride + j - 1];
        acc_off[b + 1] = acc_off[b] + n + 1;
    }
    return 0;
}

/*
 * EAGLE-3 draft-tree construction (the context-aware dynamic tree; paper
 * App. A / Table 7: depth 8, top-k 10, 60 draft tokens; EAGLE3 card
 * "Factors").  Step t = 0 .. D-1 expands the frontier: frontier slot j (only
 * slot 0, the root, at t = 0) proposes k children with target ids
 * tid[t][j][c] and draft log-probabilities lp[t][j][c] (<= 0).  A child's
 * score is its parent's score (0 for the root) plus its lp.  The k best
 * children of step t (score desc, creation order asc) are the frontier of
 * step t+1, slot 0 first.  Every child of every step joins the pool; the N
 * best of the pool (same order) form the tree, listed depth by depth and,
 * within a depth, in that order; parent[] indexes that list (-1 = root).
 * Scores are summed in fp32 (the precision the kernel decides in), in this
 * order, so both sides rank the same numbers.
 * Creation order: step 0 child c -> c; step t >= 1 -> k + (t-1)k^2 + j*k + c.
 * Returns 2 (and writes -1s) for a sequence with an lp > 0 or not finite.
 */
typedef struct { float s; int32_t idx; } ranked;

static int by_score_then_index(const void* a, const void* b) {
    const ranked* x = (const ranked*)a;
    const ranked* y = (const ranked*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

int oracle_build_tree(const int32_t* tid, const float* lp, int B, int D, int k, int N, int32_t* parent,
                      int32_t* token, float* score, int32_t* depth) {
    if (!tid || !lp || !parent || !token || B < 0 || D < 1 || k < 1 || N < 1) return 1;
    const int pool_n = k + (D - 1) * k * k;
    if (N > pool_n) return 1;
    int rc = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t* T = tid + (int64_t)b * D * k * k;
        const float* L = lp + (int64_t)b * D * k * k;
        float* ps = (float*)malloc(sizeof(float) * pool_n);       /* pool: score */
        int32_t* pp = (int32_t*)malloc(sizeof(int32_t) * pool_n); /* parent pool index, -1 root */
        int32_t* pt = (int32_t*)malloc(sizeof(int32_t) * pool_n); /* token */
        int32_t* pd = (int32_t*)malloc(sizeof(int32_t) * pool_n); /* depth */
        ranked* r = (ranked*)malloc(sizeof(ranked) * pool_n);
        int32_t frontier[64];
        int bad = 0, made = 0;
        for (int t = 0; t < D && !bad; ++t) {
            const int slots = t == 0 ? 1 : k;
            const int first = made;
            for (int j = 0; j < slots; ++j)
                for (int c = 0; c < k; ++c) {
                    const float l = L[((int64_t)t * k + j) * k + c];
                    if (!(l <= 0.0f)) bad = 1;
                    const int par = t == 0 ? -1 : frontier[j];
                    ps[made] = (par < 0 ? 0.0f : ps[par]) + l;
                    pp[made] = par;
                    pt[made] = T[((int64_t)t * k + j) * k + c];
                    pd[made] = t + 1;
                    made++;
                }
            /* next frontier: the k best children of this step */
            const int n_step = made - first;
            for (int i = 0; i < n_step; ++i) { r[i].s = ps[first + i]; r[i].idx = first + i; }
            qsort(r, (size_t)n_step, sizeof(ranked), by_score_then_index);
            for (int j = 0; j < k; ++j) frontier[j] = r[j].idx;
        }
        int32_t* P_ = parent + (int64_t)b * N;
        int32_t* T_ = token + (int64_t)b * N;
        if (bad) {
            rc = 2;
            for (int i = 0; i < N; ++i) {
                P_[i] = T_[i] = -1;
                if (score) score[(int64_t)b * N + i] = 0.0f;
                if (depth) depth[(int64_t)b * N + i] = -1;
            }
        } else {
            for (int i = 0; i < pool_n; ++i) { r[i].s = ps[i]; r[i].idx = i; }
            qsort(r, (size_t)pool_n, sizeof(ranked), by_score_then_index);
            /* the N best, listed depth by depth (stable within a depth) */
            int32_t* new_of = (int32_t*)malloc(sizeof(int32_t) * pool_n);
            for (int i = 0; i < pool_n; ++i) new_of[i] = -1;
            int out = 0;
            for (int dd = 1; dd <= D; ++dd)
                for (int i = 0; i < N; ++i)
                    if (pd[r[i].idx] == dd) new_of[r[i].idx] = out++;
            for (int i = 0; i < N; ++i) {
                const int q = r[i].idx, o = new_of[q];
                P_[o] = pp[q] < 0 ? -1 : new_of[pp[q]];
                T_[o] = pt[q];
                if (score) score[(int64_t)b * N + o] = ps[q];
                if (depth) depth[(int64_t)b * N + o] = pd[q];
            }
            free(new_of);
        }
        free(ps); free(pp); free(pt); free(pd); free(r);
    }
    return rc;
}

/* GELU in its exact form: x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt 2)) (paper App. A). */
double oracle_gelu(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

/*
 * Neural router f_theta and the threshold decision.  For each b, with
 * h = hidden[rows[b]] (bf16):
 *   z_j      = b1[j] + sum_k W1[j,k] * h[k]          (W1 row-major [m, d])
 *   delta[b] = b2 + sum_j w2[j] * GELU(z_j)           (dropout is the identity)
 *   route[b] = 1 (EAGLE-3) if delta[b] > tau else 0 (DFlash)
 */
int oracle_router(const uint16_t* hidden, const int32_t* rows, int B, int64_t d, int64_t m,
                  const float* W1, const float* b1, const float* w2, double b2, double tau,
                  double* delta, int32_t* route) {
    if (!hidden || !rows || !W1 || !b1 || !w2 || !delta || !route || B < 0) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const uint16_t* h = hidden + (int64_t)rows[b] * d;
        double out = b2;
        for (int64_t j = 0; j < m; ++j) {
            double z = b1[j];
            for (int64_t k = 0; k < d; ++k) z += (double)W1[j * d + k] * bf16_value(h[k]);
            out += (double)w2[j] * oracle_gelu(z);
        }
        delta[b] = out;
        route[b] = out > tau ? 1 : 0;
    }
    return 0;
}

typedef struct { double v; int32_t id; } scored_id;

/* order: higher logit first, lower id first on equal logits */
static int by_logit_desc(const void* a, const void* b) {
    const scored_id* x = (const scored_id*)a;
    const scored_id* y = (const scored_id*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->id > y->id) - (x->id < y->id);
}

/*
 * EAGLE-3 draft head + top-k + draft-to-target map.  For each b:
 *   logits over the draft vocabulary L_v = <x_b, Wd_v>, v < Vd;
 *   sort all Vd (logit desc, id asc); the first k draft ids, their logits,
 *   and their target ids d2t[id];
 *   lse[b]     = log sum_v exp(L_v)   (may be NULL)
 *   min_gap[b] = smallest difference between consecutive sorted logits among
 *                the first k+1 (may be NULL; used by the input generator).
 */
int oracle_draft_topk(const uint16_t* x, const uint16_t* Wd, const int32_t* d2t, int B, int64_t d,
                      int64_t Vd, int k, int32_t* draft_ids, int32_t* tids, double* vals, double* lse,
                      double* min_gap) {
    if (!x || !Wd || !d2t || B < 0 || k < 1 || k > Vd) return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        scored_id* s = (scored_id*)malloc((size_t)Vd * sizeof(scored_id));
        for (int64_t v = 0; v < Vd; ++v) {
            s[v].v = logit(x + (int64_t)b * d, Wd + v * d, d);
            s[v].id = (int32_t)v;
        }
        qsort(s, (size_t)Vd, sizeof(scored_id), by_logit_desc);
        for (int j = 0; j < k; ++j) {
            if (draft_ids) draft_ids[(int64_t)b * k + j] = s[j].id;
            if (tids) tids[(int64_t)b * k + j] = d2t[s[j].id];
            if (vals) vals[(int64_t)b * k + j] = s[j].v;
        }
        if (lse) {
            double mx = s[0].v, acc = 0.0;
            for (int64_t v = 0; v < Vd; ++v) acc += exp(s[v].v - mx);
            lse[b] = mx + log(acc);
        }
        if (min_gap) {
            double mg = INFINITY;
            for (int j = 0; j < k && j + 1 < Vd; ++j)
                if (s[j].v - s[j + 1].v < mg) mg = s[j].v - s[j + 1].v;
            min_gap[b] = mg;
        }
        free(s);
    }
    return 0;
}

/*
 * One verify-and-route round (paper Sec. 3.2): target argmax at every
 * verified row, acceptance per sequence (kind[b] 0 = DFlash chain,
 * 1 = EAGLE-3 tree; kind NULL = all trees), then the router on the hidden
 * state of each sequence's last accepted row.
 */
int oracle_round(const uint16_t* hidden, const uint16_t* W, int64_t d, int64_t V, const int32_t* pos_off,
                 const int32_t* node_off, const int32_t* kind, const int32_t* tok, const int32_t* parent,
                 int B, int64_t m, const float* W1, const float* b1, const float* w2, double b2, double tau,
                 int32_t* ids, int32_t* n_accept, int32_t* bonus, int32_t* last_pos, int32_t* path,
                 int path_stride, double* delta, int32_t* route) {
    int64_t P = pos_off[B];
    int rc = oracle_lmhead_argmax(hidden, W, P, d, V, ids, NULL, NULL);
    if (rc) return rc;
    for (int b = 0; b < B; ++b) {
        int32_t* pb = path ? path + (int64_t)b * path_stride : NULL;
        int one_kind = kind ? kind[b] : 1;
        /* a single sequence at a time, viewed through its own offsets */
        int32_t po[2] = {0, pos_off[b + 1] - pos_off[b]};
        int32_t no[2] = {0, node_off[b + 1] - node_off[b]};
        int32_t na, bo, lp;
        if (one_kind == 0)
            rc = oracle_verify_chain(ids + pos_off[b], tok + node_off[b], po, no, 1, &na, &bo, &lp, pb,
                                     path_stride);
        else
            rc = oracle_verify_tree(ids + pos_off[b], tok + node_off[b], parent + node_off[b], no, po, 1,
                                    &na, &bo, &lp, pb, path_stride);
        n_accept[b] = na;
        bonus[b] = bo;
        last_pos[b] = lp < 0 ? -1 : lp + pos_off[b];
        if (rc) return rc;
    }
    return oracle_router(hidden, last_pos, B, d, m, W1, b1, w2, b2, tau, delta, route);
}

/* ------------------------------------------------------------------------
 * KV-only catch-up of the autoregressive drafter (paper Sec. 3.4 "Lazy
 * Catch-up" and "KV-only Prefill"): when the router switches to the EAGLE-3
 * drafter, the tokens accepted while it was idle (the backlog) enter its KV
 * cache in one batch; for them only the attention layer's keys and values
 * are computed, and only the final backlog token runs through the layer in
 * full.  The drafter is one Llama-style decoder layer (EAGLE3 card,
 * "Technical Specifications": LlamaForCausalLMEagle3, 1 decoder layer,
 * hidden 2560, 32 attention heads, 8 KV heads).  The steps of that layer's
 * attention part, as used here:
 *   a     = RMSNorm(u) * gamma                (pre-attention norm)
 *   k     = rope(Wk a, pos),  v = Wv a         (per KV head, head size D)
 *   q     = rope(Wq a, pos)                    (final token only)
 *   o_h   = softmax_t(<q_h, K_g[t]> / sqrt D) V_g   over the whole cache,
 *           query head h reading KV head g = h / (H / G)
 *   out   = u + Wo o                           (residual; final token only)
 * The cache holds bf16 values (the drafter runs in bf16, paper Sec. 4).
 * ---------------------------------------------------------------------- */

/* Round to the nearest bf16, ties to even (through the nearest binary32). */
static uint16_t bf16_round(double x) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* RMSNorm: a[i] = u[i] / sqrt(mean_k u[k]^2 + eps) * gamma[i]. */
void oracle_rmsnorm(const uint16_t* u, int64_t din, const uint16_t* gamma, double eps, double* a) {
    double ss = 0.0;
    for (int64_t i = 0; i < din; ++i) ss += bf16_value(u[i]) * bf16_value(u[i]);
    const double r = 1.0 / sqrt(ss / (double)din + eps);
    for (int64_t i = 0; i < din; ++i) a[i] = bf16_value(u[i]) * r * bf16_value(gamma[i]);
}

/*
 * Rotary position embedding of one head vector x[D] at position pos: the
 * pair (x[i], x[i + D/2]) turns by the angle pos * theta^(-2i/D), i < D/2
 * (the "rotate half" pairing of Llama-style layers).
 */
void oracle_rope(const double* x, int D, double pos, double theta, double* y) {
    const int half = D / 2;
    for (int i = 0; i < half; ++i) {
        const double ang = pos * pow(theta, -2.0 * (double)i / (double)D);
        const double c = cos(ang), s = sin(ang);
        const double x1 = x[i], x2 = x[i + half];
        y[i] = x1 * c - x2 * s;
        y[i + half] = x2 * c + x1 * s;
    }
}

/* <W[row], a> for a bf16 weight row and a double vector, summed in index order. */
static double row_dot(const uint16_t* w, const double* a, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += bf16_value(w[i]) * a[i];
    return s;
}

/*
 * Catch-up of B sequences.  Sequence b has n_b = bl_off[b+1] - bl_off[b] >= 1
 * backlog tokens with layer inputs u[bl_off[b] + j] ([N, din] bf16) and
 * L_b = cache_len[b] entries already in its caches Kc, Vc ([B, cap, G*D] bf16,
 * KV head g at columns g*D ..).  Backlog token j sits at position L_b + j;
 * its key and value go to cache row L_b + j.  For the final token
 * (j = n_b - 1): q[b] ([B, H*D], may be NULL) after the rotation, attn[b]
 * ([B, H*D], may be NULL) the attention output over cache rows
 * 0 .. L_b + n_b - 1, and out[b] ([B, din]) = u_final + Wo attn.
 * Wq [H*D, din], Wk / Wv [G*D, din], Wo [din, H*D], gamma [din], all bf16.
 * Returns 2 if a sequence has no backlog or does not fit its cache.
 */
int oracle_catchup(const uint16_t* u, const int32_t* bl_off, const int32_t* cache_len, int B, int64_t din, int H,
                   int G, int D, const uint16_t* gamma, double eps, double theta, const uint16_t* Wq,
                   const uint16_t* Wk, const uint16_t* Wv, const uint16_t* Wo, uint16_t* Kc, uint16_t* Vc,
                   int64_t cap, double* q, double* attn, double* out) {
    if (!u || !bl_off || !cache_len || !gamma || !Wq || !Wk || !Wv || !Wo || !Kc || !Vc || !out) return 1;
    if (B < 0 || din < 1 || H < 1 || G < 1 || H % G || D < 2 || D % 2) return 1;
    for (int b = 0; b < B; ++b) {
        const int64_t n = bl_off[b + 1] - bl_off[b];
        if (n < 1 || cache_len[b] < 0 || cache_len[b] + n > cap) return 2;
    }
    const int64_t GD = (int64_t)G * D, HD = (int64_t)H * D;
    const int64_t N = bl_off[B];
    /* keys and values of every backlog token (independent rows) */
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < N; ++r) {
        int b = 0;
        while (bl_off[b + 1] <= r) ++b;
        const int64_t pos = cache_len[b] + (r - bl_off[b]);
        double* a = (double*)malloc((size_t)din * sizeof(double));
        double* kh = (double*)malloc((size_t)D * sizeof(double));
        double* kr = (double*)malloc((size_t)D * sizeof(double));
        oracle_rmsnorm(u + r * din, din, gamma, eps, a);
        uint16_t* krow = Kc + ((int64_t)b * cap + pos) * GD;
        uint16_t* vrow = Vc + ((int64_t)b * cap + pos) * GD;
        for (int g = 0; g < G; ++g) {
            for (int e = 0; e < D; ++e) kh[e] = row_dot(Wk + ((int64_t)g * D + e) * din, a, din);
            oracle_rope(kh, D, (double)pos, theta, kr);
            for (int e = 0; e < D; ++e) {
                krow[(int64_t)g * D + e] = bf16_round(kr[e]);
                vrow[(int64_t)g * D + e] = bf16_round(row_dot(Wv + ((int64_t)g * D + e) * din, a, din));
            }
        }
        free(a); free(kh); free(kr);
    }
    /* the final backlog token of each sequence, through the attention sublayer */
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int64_t f = bl_off[b + 1] - 1;
        const int64_t T = cache_len[b] + (bl_off[b + 1] - bl_off[b]);
        const double pos = (double)(T - 1);
        double* a = (double*)malloc((size_t)din * sizeof(double));
        double* qb = (double*)malloc((size_t)HD * sizeof(double));
        double* ob = (double*)malloc((size_t)HD * sizeof(double));
        double* tmp = (double*)malloc((size_t)D * sizeof(double));
        double* sc = (double*)malloc((size_t)T * sizeof(double));
        oracle_rmsnorm(u + f * din, din, gamma, eps, a);
        for (int h = 0; h < H; ++h) {
            for (int e = 0; e < D; ++e) tmp[e] = row_dot(Wq + ((int64_t)h * D + e) * din, a, din);
            oracle_rope(tmp, D, pos, theta, qb + (int64_t)h * D);
        }
        for (int h = 0; h < H; ++h) {
            const int g = h / (H / G);
            const double* qh = qb + (int64_t)h * D;
            double mx = -INFINITY;
            for (int64_t t = 0; t < T; ++t) {
                const uint16_t* kt = Kc + ((int64_t)b * cap + t) * GD + (int64_t)g * D;
                double s = 0.0;
                for (int e = 0; e < D; ++e) s += qh[e] * bf16_value(kt[e]);
                sc[t] = s / sqrt((double)D);
                if (sc[t] > mx) mx = sc[t];
            }
            double Z = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                sc[t] = exp(sc[t] - mx);
                Z += sc[t];
            }
            for (int e = 0; e < D; ++e) {
                double acc = 0.0;
                for (int64_t t = 0; t < T; ++t)
                    acc += sc[t] * bf16_value(Vc[((int64_t)b * cap + t) * GD + (int64_t)g * D + e]);
                ob[(int64_t)h * D + e] = acc / Z;
            }
        }
        for (int64_t i = 0; i < din; ++i)
            out[(int64_t)b * din + i] = bf16_value(u[f * din + i]) + row_dot(Wo + i * HD, ob, HD);
        if (q) memcpy(q + (int64_t)b * HD, qb, (size_t)HD * sizeof(double));
        if (attn) memcpy(attn + (int64_t)b * HD, ob, (size_t)HD * sizeof(double));
        free(a); free(qb); free(ob); free(tmp); free(sc);
    }
    return 0;
}
