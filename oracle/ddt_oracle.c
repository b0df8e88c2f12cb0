/*
 * ddt_oracle.c -- plain fp64 CPU oracle of one DDTree verification round.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the benchmark's
 * CPU-baseline leg; never by the product path.  It shares no code with the CUDA
 * library.  Every step is written the plain way: full sorts, linear scans, one
 * row at a time, fp64 everywhere.  OpenMP only spreads independent
 * (layer, request, head) units over cores; it changes no arithmetic.
 *
 * Citations use the page titles listed in ddt_oracle.h ([NOTES], [ARCH], [CHALL],
 * [GDN]).  Readings of points the pages leave open are marked READING.
 */
#include "ddt_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Tree build                                                                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    double v;
    int id;
} vid_t;

/* Rank order of one depth: logit descending, then token id ascending (ties go to
 * the lower id, READING of "ties to the lower token id"). */
static int cmp_rank(const void* a, const void* b) {
    const vid_t* x = (const vid_t*)a;
    const vid_t* y = (const vid_t*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id);
}

/* A tree node under consideration: the path through `parent` (index into the
 * selected list, -1 = root) extended by the token of rank `rank` at `depth`. */
typedef struct {
    double L;     /* sum of the path's logits, depth 1 first */
    double s;     /* L - sum of the path's per-depth log-sum-exp = log of the
                     product of the drafter probabilities along the path */
    int depth;    /* 1..D */
    int rank;     /* 0..k-1 within the depth's top-k */
    int parent;   /* index into sel[], -1 for the root */
    int token;
} node_t;

/* Tokens of the path of node `c` (root excluded), depth 1 first. */
static int path_of(const node_t* sel, const node_t* c, int* out) {
    int n = c->depth;
    out[n - 1] = c->token;
    int p = c->parent;
    for (int i = n - 2; i >= 0; --i) {
        out[i] = sel[p].token;
        p = sel[p].parent;
    }
    return n;
}

/* Total order of the best-first selection: higher score first; on an exact score
 * tie, the token sequence that is lexicographically smaller (lower ids first, a
 * prefix before its extensions) first.  READING of "ties to the lower token id". */
static int better(const node_t* sel, const node_t* a, const node_t* b, int* pa, int* pb) {
    if (a->s > b->s) return 1;
    if (a->s < b->s) return 0;
    int na = path_of(sel, a, pa);
    int nb = path_of(sel, b, pb);
    int n = na < nb ? na : nb;
    for (int i = 0; i < n; ++i) {
        if (pa[i] != pb[i]) return pa[i] < pb[i];
    }
    return na < nb;
}

typedef struct {
    int parent_new;
    int rank;
    int sel_index;
} bfs_key_t;

static int cmp_bfs(const void* a, const void* b) {
    const bfs_key_t* x = (const bfs_key_t*)a;
    const bfs_key_t* y = (const bfs_key_t*)b;
    if (x->parent_new != y->parent_new) return x->parent_new < y->parent_new ? -1 : 1;
    return (x->rank < y->rank) ? -1 : (x->rank > y->rank);
}

/*
 * [ARCH]: take the top-K ids and log-probabilities at every depth; seed a max-heap
 * with the most probable depth-1 token; repeatedly pop the best node, add it to the
 * tree, and push its next-ranked sibling and its best child; stop once `budget`
 * nodes are in the tree.  The heap here is a plain linear scan of the frontier.
 * [ARCH] flattening: root + nodes, positions shared per depth, ancestor-only mask.
 */
int ddto_build_tree(int B, int D, int V, int k, int budget,
                    const double* logits, const int32_t* root_token, const int32_t* prefix_len,
                    int32_t* token, int32_t* parent, int32_t* depth, int32_t* position,
                    int32_t* rank, int32_t* n_nodes, uint32_t* anc, double* score,
                    double* lse, double* margin, int32_t* margin_depth) {
    if (B < 1 || D < 1 || V < 1 || k < 1 || k > V || budget < 0) return DDTO_ERR_ARG;
    const int N = budget + 1;
    const int W = (N + 31) / 32;
    int rc = DDTO_OK;

#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        double* lse_b = lse + (long)b * D;
        int* top_id = (int*)malloc(sizeof(int) * (size_t)D * k);
        double* top_v = (double*)malloc(sizeof(double) * (size_t)D * k);
        vid_t* buf = (vid_t*)malloc(sizeof(vid_t) * (size_t)V);
        node_t* sel = (node_t*)malloc(sizeof(node_t) * (size_t)(budget > 0 ? budget : 1));
        node_t* front = (node_t*)malloc(sizeof(node_t) * (size_t)(2 * budget + 2));
        int* pa = (int*)malloc(sizeof(int) * (size_t)D);
        int* pb = (int*)malloc(sizeof(int) * (size_t)D);

        /* Per-depth log-sum-exp and rank order. */
        for (int d = 0; d < D; ++d) {
            const double* row = logits + ((long)b * D + d) * V;
            double m = row[0];
            for (int v = 1; v < V; ++v)
                if (row[v] > m) m = row[v];
            double sum = 0.0;
            for (int v = 0; v < V; ++v) sum += exp(row[v] - m);
            lse_b[d] = m + log(sum);
            for (int v = 0; v < V; ++v) {
                buf[v].v = row[v];
                buf[v].id = v;
            }
            qsort(buf, (size_t)V, sizeof(vid_t), cmp_rank);
            for (int r = 0; r < k; ++r) {
                top_id[d * k + r] = buf[r].id;
                top_v[d * k + r] = buf[r].v;
            }
        }

        /* Best-first selection. */
        int n_sel = 0, n_front = 0;
        if (budget > 0) {
            node_t s0;
            s0.depth = 1;
            s0.rank = 0;
            s0.parent = -1;
            s0.token = top_id[0];
            s0.L = 0.0 + top_v[0];
            s0.s = s0.L - lse_b[0];
            front[n_front++] = s0;
        }
        while (n_sel < budget && n_front > 0) {
            int best = 0;
            for (int i = 1; i < n_front; ++i)
                if (better(sel, &front[i], &front[best], pa, pb)) best = i;
            node_t c = front[best];
            front[best] = front[--n_front];
            int me = n_sel;
            sel[n_sel++] = c;
            /* the parent's L and the cumulative normaliser of this depth */
            double L_par = (c.parent < 0) ? 0.0 : sel[c.parent].L;
            double C_dep = 0.0;
            for (int d = 0; d < c.depth; ++d) C_dep += lse_b[d];
            if (c.rank + 1 < k) { /* next-ranked sibling */
                node_t sib = c;
                sib.rank = c.rank + 1;
                sib.token = top_id[(c.depth - 1) * k + sib.rank];
                sib.L = L_par + top_v[(c.depth - 1) * k + sib.rank];
                sib.s = sib.L - C_dep;
                front[n_front++] = sib;
            }
            if (c.depth < D) { /* best child */
                node_t ch;
                ch.depth = c.depth + 1;
                ch.rank = 0;
                ch.parent = me;
                ch.token = top_id[c.depth * k];
                ch.L = c.L + top_v[c.depth * k];
                ch.s = ch.L - (C_dep + lse_b[c.depth]);
                front[n_front++] = ch;
            }
        }

        /* Decision margin at the cut: last selected vs best left on the frontier. */
        if (n_front > 0 && n_sel > 0) {
            int best = 0;
            for (int i = 1; i < n_front; ++i)
                if (better(sel, &front[i], &front[best], pa, pb)) best = i;
            margin[b] = sel[n_sel - 1].s - front[best].s;
            margin_depth[2 * b] = sel[n_sel - 1].depth;
            margin_depth[2 * b + 1] = front[best].depth;
        } else {
            margin[b] = INFINITY;
            margin_depth[2 * b] = -1;
            margin_depth[2 * b + 1] = -1;
        }

        /* Canonical numbering (READING): breadth first -- depth ascending, then the
         * parent's new index, then the rank. */
        int* new_idx = (int*)malloc(sizeof(int) * (size_t)(n_sel > 0 ? n_sel : 1));
        bfs_key_t* keys = (bfs_key_t*)malloc(sizeof(bfs_key_t) * (size_t)(n_sel > 0 ? n_sel : 1));
        int next = 1;
        for (int dd = 1; dd <= D; ++dd) {
            int nk = 0;
            for (int i = 0; i < n_sel; ++i) {
                if (sel[i].depth != dd) continue;
                keys[nk].parent_new = sel[i].parent < 0 ? 0 : new_idx[sel[i].parent];
                keys[nk].rank = sel[i].rank;
                keys[nk].sel_index = i;
                ++nk;
            }
            qsort(keys, (size_t)nk, sizeof(bfs_key_t), cmp_bfs);
            for (int j = 0; j < nk; ++j) new_idx[keys[j].sel_index] = next++;
        }

        int32_t* tok = token + (long)b * N;
        int32_t* par = parent + (long)b * N;
        int32_t* dep = depth + (long)b * N;
        int32_t* pos = position + (long)b * N;
        int32_t* rk = rank + (long)b * N;
        double* sc = score + (long)b * N;
        uint32_t* an = anc + (long)b * N * W;
        for (int i = 0; i < N; ++i) {
            tok[i] = par[i] = dep[i] = pos[i] = rk[i] = -1;
            sc[i] = -INFINITY;
            for (int w = 0; w < W; ++w) an[(long)i * W + w] = 0u;
        }
        tok[0] = root_token[b];
        dep[0] = 0;
        pos[0] = prefix_len[b];
        sc[0] = 0.0;
        for (int i = 0; i < n_sel; ++i) {
            int r = new_idx[i];
            tok[r] = sel[i].token;
            par[r] = sel[i].parent < 0 ? 0 : new_idx[sel[i].parent];
            dep[r] = sel[i].depth;
            pos[r] = prefix_len[b] + sel[i].depth;
            rk[r] = sel[i].rank;
            sc[r] = sel[i].s;
        }
        n_nodes[b] = n_sel + 1;
        /* ancestor-or-self mask: parents precede children in the numbering */
        an[0] |= 1u;
        for (int i = 1; i <= n_sel; ++i) {
            for (int w = 0; w < W; ++w) an[(long)i * W + w] = an[(long)par[i] * W + w];
            an[(long)i * W + i / 32] |= 1u << (i % 32);
        }

        free(new_idx);
        free(keys);
        free(top_id);
        free(top_v);
        free(buf);
        free(sel);
        free(front);
        free(pa);
        free(pb);
    }
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Tree attention                                                             */
/* ------------------------------------------------------------------------- */

/* [NOTES] "Why hybrid attention makes it hard": a row sees the committed prefix and
 * its own ancestors, never its siblings.  Textbook softmax attention over that key
 * set, max-subtracted, fp64.  READING: no soft-cap, bias or window; q/k are taken
 * after any rotary embedding. */
int ddto_attn_row(int P, int n_nodes, int d, const double* q,
                  const double* k_prefix, const double* v_prefix, long ld_prefix,
                  const double* k_tree, const double* v_tree, long ld_tree,
                  const uint32_t* anc_row, double scale, double* out) {
    int nk = P + n_nodes;
    double* s = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    char* use = (char*)malloc((size_t)(nk > 0 ? nk : 1));
    double m = -INFINITY;
    for (int j = 0; j < nk; ++j) {
        const double* kr;
        if (j < P) {
            kr = k_prefix + (long)j * ld_prefix;
            use[j] = 1;
        } else {
            int t = j - P;
            kr = k_tree + (long)t * ld_tree;
            use[j] = (anc_row[t / 32] >> (t % 32)) & 1u;
        }
        if (!use[j]) continue;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += q[c] * kr[c];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    double l = 0.0;
    for (int j = 0; j < nk; ++j) {
        if (!use[j]) continue;
        double w = exp(s[j] - m);
        l += w;
        const double* vr = (j < P) ? v_prefix + (long)j * ld_prefix : v_tree + (long)(j - P) * ld_tree;
        for (int c = 0; c < d; ++c) out[c] += w * vr[c];
    }
    if (l > 0.0)
        for (int c = 0; c < d; ++c) out[c] /= l;
    free(s);
    free(use);
    return DDTO_OK;
}

int ddto_tree_attn(int L, int B, int N, int Hq, int Hkv, int d, int Pcap,
                   const double* q, const double* k_tree, const double* v_tree,
                   const double* k_cache, const double* v_cache,
                   const int32_t* prefix_len, const int32_t* n_nodes, const uint32_t* anc,
                   double scale, double* o) {
    if (L < 1 || B < 1 || N < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1) return DDTO_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (prefix_len[b] < 0 || prefix_len[b] > Pcap || n_nodes[b] < 1 || n_nodes[b] > N)
            return DDTO_ERR_ARG;
    const int W = (N + 31) / 32;
    const int G = Hq / Hkv;
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hq; ++h) {
                int g = h / G;
                const double* kp = k_cache + (((long)l * B + b) * Hkv + g) * Pcap * d;
                const double* vp = v_cache + (((long)l * B + b) * Hkv + g) * Pcap * d;
                const double* kt = k_tree + (((long)l * B + b) * N * Hkv + g) * d;
                const double* vt = v_tree + (((long)l * B + b) * N * Hkv + g) * d;
                for (int i = 0; i < N; ++i) {
                    double* out = o + ((((long)l * B + b) * N + i) * Hq + h) * d;
                    if (i >= n_nodes[b]) {
                        for (int c = 0; c < d; ++c) out[c] = 0.0;
                        continue;
                    }
                    const double* qr = q + ((((long)l * B + b) * N + i) * Hq + h) * d;
                    ddto_attn_row(prefix_len[b], n_nodes[b], d, qr, kp, vp, d, kt, vt,
                                  (long)Hkv * d, anc + ((long)b * N + i) * W, scale, out);
                }
            }
    return DDTO_OK;
}

/* ------------------------------------------------------------------------- */
/* Tree Gated DeltaNet                                                        */
/* ------------------------------------------------------------------------- */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Short causal conv + SiLU of one channel of node n ([GDN]; READING: no bias).
 * The window is the node's own ancestor path, newest last; taps that reach past the
 * root read the committed conv state (oldest row first).  anc_list[t] is the node t
 * steps up the path (anc_list[0] = n), depth = steps from n to the root. */
static double conv_channel(int c, int C, int K, const double* x, const double* w_c,
                           const double* conv_state, const int* anc_list, int dep) {
    double acc = 0.0;
    for (int j = 0; j < K; ++j) {
        int back = K - 1 - j; /* tap j looks `back` steps into the past */
        double in;
        if (back <= dep)
            in = x[(long)anc_list[back] * C + c];
        else
            in = conv_state[(long)(K - 1 - (back - dep)) * C + c];
        acc += w_c[j] * in;
    }
    return silu(acc);
}

/* [NOTES] "Why hybrid attention makes it hard": each node reads GDN and conv state
 * from its parent and writes scratch.  [GDN]: per node n with parent p,
 *   q^ = q / sqrt(|q|^2 + 1e-6) / sqrt(dk),  k^ = k / sqrt(|k|^2 + 1e-6),  v = conv(v),
 *   S_n = alpha_n S_p + k^ (beta_n (v - alpha_n S_p^T k^))^T,   o_n = S_n^T q^.
 * READING: eps 1e-6 inside the root, q scaled by 1/sqrt(dk), no output gate/norm. */
int ddto_gdn_unit(int N, int n_nodes, int Hk, int Hv, int dk, int dv, int K, int h,
                  const double* x, const double* conv_w, const double* conv_state,
                  const double* beta, const double* decay, const double* S0,
                  const int32_t* parent, double* o, double* S_node) {
    if (Hv % Hk || n_nodes < 1 || n_nodes > N || K < 1) return DDTO_ERR_ARG;
    if (parent[0] != -1) return DDTO_ERR_TREE;
    for (int i = 1; i < n_nodes; ++i)
        if (parent[i] < 0 || parent[i] >= i) return DDTO_ERR_TREE;
    const int C = 2 * Hk * dk + Hv * dv;
    const int g = h / (Hv / Hk);
    const int cq = g * dk, ck = Hk * dk + g * dk, cv = 2 * Hk * dk + h * dv;
    const long SS = (long)dk * dv;

    double* states = S_node;
    if (!states) states = (double*)malloc(sizeof(double) * (size_t)n_nodes * SS);
    double* qh = (double*)malloc(sizeof(double) * (size_t)dk);
    double* kh = (double*)malloc(sizeof(double) * (size_t)dk);
    double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
    double* u = (double*)malloc(sizeof(double) * (size_t)dv);
    int* anc_list = (int*)malloc(sizeof(int) * (size_t)(n_nodes + 1));

    for (int n = 0; n < N; ++n) {
        double* on = o + (long)n * dv;
        if (n >= n_nodes) {
            for (int j = 0; j < dv; ++j) on[j] = 0.0;
            continue;
        }
        int dep = 0;
        anc_list[0] = n;
        for (int a = parent[n]; a >= 0; a = parent[a]) anc_list[++dep] = a;

        double nq = 0.0, nk = 0.0;
        for (int i = 0; i < dk; ++i) {
            qh[i] = conv_channel(cq + i, C, K, x, conv_w + (long)(cq + i) * K, conv_state, anc_list, dep);
            kh[i] = conv_channel(ck + i, C, K, x, conv_w + (long)(ck + i) * K, conv_state, anc_list, dep);
            nq += qh[i] * qh[i];
            nk += kh[i] * kh[i];
        }
        double rq = 1.0 / sqrt(nq + 1e-6) / sqrt((double)dk);
        double rk = 1.0 / sqrt(nk + 1e-6);
        for (int i = 0; i < dk; ++i) {
            qh[i] *= rq;
            kh[i] *= rk;
        }
        for (int j = 0; j < dv; ++j)
            vv[j] = conv_channel(cv + j, C, K, x, conv_w + (long)(cv + j) * K, conv_state, anc_list, dep);

        const double a = decay[(long)n * Hv + h];
        const double bt = beta[(long)n * Hv + h];
        const double* Sp = parent[n] < 0 ? S0 : states + (long)parent[n] * SS;
        double* Sn = states + (long)n * SS;
        for (int j = 0; j < dv; ++j) {
            double pred = 0.0;
            for (int i = 0; i < dk; ++i) pred += Sp[(long)i * dv + j] * kh[i];
            u[j] = bt * (vv[j] - a * pred);
        }
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) Sn[(long)i * dv + j] = a * Sp[(long)i * dv + j] + kh[i] * u[j];
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += Sn[(long)i * dv + j] * qh[i];
            on[j] = acc;
        }
    }
    if (!S_node) free(states);
    free(qh);
    free(kh);
    free(vv);
    free(u);
    free(anc_list);
    return DDTO_OK;
}

int ddto_tree_gdn(int L, int B, int N, int Hk, int Hv, int dk, int dv, int K,
                  const double* x, const double* conv_w, const double* conv_state,
                  const double* beta, const double* decay, const double* S,
                  const int32_t* parent, const int32_t* n_nodes,
                  double* o, double* S_node) {
    if (L < 1 || B < 1 || N < 1 || Hk < 1 || Hv < 1 || Hv % Hk || dk < 1 || dv < 1 || K < 1)
        return DDTO_ERR_ARG;
    const int C = 2 * Hk * dk + Hv * dv;
    const long SS = (long)dk * dv;
    int rc = DDTO_OK;
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hv; ++h) {
                const long lb = (long)l * B + b;
                double* o_u = (double*)malloc(sizeof(double) * (size_t)N * dv);
                double* sn_u = S_node ? (double*)malloc(sizeof(double) * (size_t)N * SS) : NULL;
                double* be = (double*)malloc(sizeof(double) * (size_t)N * Hv);
                double* de = (double*)malloc(sizeof(double) * (size_t)N * Hv);
                for (long t = 0; t < (long)N * Hv; ++t) {
                    be[t] = beta[lb * N * Hv + t];
                    de[t] = decay[lb * N * Hv + t];
                }
                int r = ddto_gdn_unit(N, n_nodes[b], Hk, Hv, dk, dv, K, h, x + lb * N * C,
                                      conv_w + (long)l * C * K, conv_state + lb * (K - 1) * C, be, de,
                                      S + (lb * Hv + h) * SS, parent + (long)b * N, o_u, sn_u);
                if (r != DDTO_OK) {
#pragma omp critical
                    rc = r;
                }
                for (int n = 0; n < N; ++n)
                    for (int j = 0; j < dv; ++j) o[((lb * N + n) * Hv + h) * dv + j] = o_u[(long)n * dv + j];
                if (S_node)
                    for (int n = 0; n < N; ++n)
                        for (long e = 0; e < SS; ++e)
                            S_node[((lb * N + n) * Hv + h) * SS + e] =
                                (n < n_nodes[b]) ? sn_u[(long)n * SS + e] : 0.0;
                free(o_u);
                free(sn_u);
                free(be);
                free(de);
            }
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Tree walk                                                                  */
/* ------------------------------------------------------------------------- */

/* [ARCH] "follow_verified_tree": compare the target's token at the current node with
 * the tokens of its children; walk down while one matches.  The target token of a
 * row is its argmax (READING: ties to the lower id).  [NOTES] "What broke along the
 * way": the bonus token (the target's token at the last accepted node) is emitted but
 * is not an accepted draft. */
static int walk_impl(int B, int N, int V, int D, const double* target_logits,
                     const int32_t* target_argmax_in, const int32_t* token, const int32_t* parent,
                     const int32_t* n_nodes, int32_t* target_argmax_out, int32_t* acc_nodes,
                     int32_t* acc_len, int32_t* bonus, int32_t* emitted, int32_t* n_emitted, int flat) {
    if (B < 1 || N < 1 || V < 1 || D < 0) return DDTO_ERR_ARG;
    const int A = D + 1;
    int* t = (int*)malloc(sizeof(int) * (size_t)N);
    for (int b = 0; b < B; ++b) {
        const int nn = n_nodes[b];
        for (int i = 0; i < N; ++i) {
            if (i >= nn) {
                t[i] = -1;
            } else if (target_logits) {
                const double* row = target_logits + ((long)b * N + i) * V;
                int best = 0;
                for (int v = 1; v < V; ++v)
                    if (row[v] > row[best]) best = v;
                t[i] = best;
            } else {
                t[i] = target_argmax_in[(long)b * N + i];
            }
            if (target_argmax_out) target_argmax_out[(long)b * N + i] = t[i];
        }
        int32_t* an = acc_nodes + (long)b * A;
        int32_t* em = emitted + (long)b * A;
        for (int j = 0; j < A; ++j) an[j] = em[j] = -1;
        int cur = 0, a = 0;
        an[0] = 0;
        for (;;) {
            int next = -1;
            for (int c = 1; c < nn; ++c)
                if (parent[(long)b * N + c] == cur && (flat || token[(long)b * N + c] == t[cur])) {
                    next = c;
                    break;
                }
            /* flat: only the first child, the rank-0 one, may be taken */
            if (flat && next >= 0 && token[(long)b * N + next] != t[cur]) next = -1;
            if (next < 0 || a + 1 >= A) break;
            cur = next;
            an[++a] = cur;
        }
        acc_len[b] = a;
        bonus[b] = t[cur];
        for (int j = 1; j <= a; ++j) em[j - 1] = token[(long)b * N + an[j]];
        em[a] = t[cur];
        n_emitted[b] = a + 1;
    }
    free(t);
    return DDTO_OK;
}

int ddto_walk(int B, int N, int V, int D, const double* target_logits,
              const int32_t* target_argmax_in, const int32_t* token, const int32_t* parent,
              const int32_t* n_nodes, int32_t* target_argmax_out, int32_t* acc_nodes,
              int32_t* acc_len, int32_t* bonus, int32_t* emitted, int32_t* n_emitted) {
    return walk_impl(B, N, V, D, target_logits, target_argmax_in, token, parent, n_nodes, target_argmax_out,
                     acc_nodes, acc_len, bonus, emitted, n_emitted, 0);
}

/* [NOTES] "What broke along the way": the safe mode commits only along the flat chain,
 * i.e. the walk descends only into a node's first (rank-0) child. */
int ddto_walk_flat(int B, int N, int V, int D, const double* target_logits,
                   const int32_t* target_argmax_in, const int32_t* token, const int32_t* parent,
                   const int32_t* n_nodes, int32_t* target_argmax_out, int32_t* acc_nodes,
                   int32_t* acc_len, int32_t* bonus, int32_t* emitted, int32_t* n_emitted) {
    return walk_impl(B, N, V, D, target_logits, target_argmax_in, token, parent, n_nodes, target_argmax_out,
                     acc_nodes, acc_len, bonus, emitted, n_emitted, 1);
}

/* Tree-walk rejection sampling: see ddt_oracle.h for the READING.  p_u is formed row by
 * row in fp64 (max-shifted exponentials, their plain sum); every comparison of a
 * probability with a uniform is in fp64. */
static double min_d(double a, double b) { return a < b ? a : b; }

int ddto_walk_sample(int B, int N, int V, int D, int C, double T, const double* target_logits,
                     const double* uniforms, const int32_t* token, const int32_t* parent,
                     const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len, int32_t* bonus,
                     int32_t* emitted, int32_t* n_emitted, double* margin, int32_t* status) {
    if (B < 1 || N < 1 || V < 1 || D < 0 || C < 1 || !(T > 0.0)) return DDTO_ERR_ARG;
    const int A = D + 1;
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    char* rejected = (char*)malloc((size_t)V);
    int* kids = (int*)malloc(sizeof(int) * (size_t)N);
    for (int b = 0; b < B; ++b) {
        const int nn = n_nodes[b];
        const int32_t* tok = token + (long)b * N;
        const int32_t* par = parent + (long)b * N;
        int32_t* an = acc_nodes + (long)b * A;
        int32_t* em = emitted + (long)b * A;
        for (int j = 0; j < A; ++j) an[j] = em[j] = -1;
        acc_len[b] = 0;
        bonus[b] = -1;
        n_emitted[b] = 0;
        margin[b] = INFINITY;
        /* the tree: parents before children, tokens in range, at most C children a node,
         * no token twice among one node's children */
        int st = (nn >= 1 && nn <= N) ? DDTO_OK : DDTO_ERR_TREE;
        if (st == DDTO_OK && par[0] != -1) st = DDTO_ERR_TREE;
        for (int i = 1; st == DDTO_OK && i < nn; ++i)
            if (par[i] < 0 || par[i] >= i || tok[i] < 0 || tok[i] >= V) st = DDTO_ERR_TREE;
        for (int u = 0; st == DDTO_OK && u < nn; ++u) {
            int m = 0;
            for (int i = 1; i < nn; ++i)
                if (par[i] == u) {
                    for (int j = 0; j < m; ++j)
                        if (tok[kids[j]] == tok[i]) st = DDTO_ERR_TREE;
                    kids[m++] = i;
                }
            if (m > C) st = DDTO_ERR_TREE;
        }
        for (int i = 0; st == DDTO_OK && i < nn; ++i)
            for (int v = 0; v < V; ++v)
                if (!isfinite(target_logits[((long)b * N + i) * V + v])) {
                    st = DDTO_ERR_NONFINITE;
                    break;
                }
        status[b] = st;
        if (st != DDTO_OK) {
            margin[b] = 0.0;
            continue;
        }
        int cur = 0, a = 0;
        an[0] = 0;
        for (;;) {
            /* p_u = softmax(logits[u] / T) */
            const double* row = target_logits + ((long)b * N + cur) * V;
            double mx = row[0];
            for (int v = 1; v < V; ++v)
                if (row[v] > mx) mx = row[v];
            double Z = 0.0;
            for (int v = 0; v < V; ++v) {
                p[v] = exp((row[v] - mx) / T);
                Z += p[v];
            }
            for (int v = 0; v < V; ++v) p[v] /= Z;
            memset(rejected, 0, (size_t)V);
            const double* U = uniforms + ((long)b * A + a) * (C + 1);
            double R = 0.0;
            int next = -1;
            if (a + 1 < A) {
                int i = 0;
                for (int c = 1; c < nn; ++c) {
                    if (par[c] != cur) continue;
                    const double thr = p[tok[c]] / (1.0 - R);
                    margin[b] = min_d(margin[b], fabs(U[i] - thr));
                    if (U[i] < thr) {
                        next = c;
                        break;
                    }
                    R += p[tok[c]];
                    rejected[tok[c]] = 1;
                    ++i;
                }
            }
            if (next < 0) {
                /* bonus from the residual: rejected children removed, renormalised */
                const double target = U[C] * (1.0 - R);
                double run = 0.0;
                int t = -1;
                for (int v = 0; v < V; ++v) {
                    if (rejected[v]) continue;
                    const double before = run;
                    run += p[v];
                    if (run > target) {
                        t = v;
                        margin[b] = min_d(margin[b], min_d(target - before, run - target));
                        break;
                    }
                }
                if (t < 0) {
                    for (int v = V - 1; v >= 0; --v)
                        if (!rejected[v] && p[v] > 0.0) {
                            t = v;
                            break;
                        }
                    margin[b] = 0.0;
                }
                bonus[b] = t;
                break;
            }
            cur = next;
            an[++a] = cur;
        }
        acc_len[b] = a;
        for (int j = 1; j <= a; ++j) em[j - 1] = tok[an[j]];
        em[a] = bonus[b];
        n_emitted[b] = a + 1;
    }
    free(p);
    free(rejected);
    free(kids);
    return DDTO_OK;
}

/* ------------------------------------------------------------------------- */
/* Commit                                                                     */
/* ------------------------------------------------------------------------- */

/* [NOTES] "Why hybrid attention makes it hard" / "Where the next step is": once a
 * path is accepted, only that path is copied into the contiguous KV and recurrent
 * buffers.  [ARCH]: the KV cache keeps only the accepted path's entries.
 * KV: tree rows root..last accepted go to cache positions prefix_len.. in order.
 * GDN: the committed state becomes the state after the last accepted node, i.e. the
 * sequential recurrence run along the accepted path from the old committed state.
 * Conv: the last K-1 raw inputs of [old conv state, path inputs].  The bonus token is
 * not committed (it is the next round's root). */
int ddto_commit(int La, int B, int N, int Hkv, int d, int Pcap,
                const double* k_tree, const double* v_tree, double* k_cache, double* v_cache,
                int Lg, int Hk, int Hv, int dk, int dv, int K,
                const double* x, const double* conv_w, const double* beta, const double* decay,
                double* S, double* conv_state,
                const int32_t* acc_nodes, const int32_t* acc_len, int A,
                int32_t* prefix_len, int32_t* src_row, int32_t* dst_pos, int32_t* status) {
    if (B < 1 || N < 1 || A < 1) return DDTO_ERR_ARG;
    const int C = 2 * Hk * dk + Hv * dv;
    const long SS = (long)dk * dv;
    for (int b = 0; b < B; ++b) {
        const int a = acc_len[b];
        const int P = prefix_len[b];
        int32_t* sr = src_row + (long)b * A;
        int32_t* dp = dst_pos + (long)b * A;
        for (int j = 0; j < A; ++j) sr[j] = dp[j] = -1;
        if (a < 0 || a + 1 > A) {
            status[b] = DDTO_ERR_ARG;
            continue;
        }
        if (La > 0 && P + a + 1 > Pcap) {
            status[b] = DDTO_ERR_CAPACITY;
            continue;
        }
        status[b] = DDTO_OK;
        const int32_t* path = acc_nodes + (long)b * A;
        for (int j = 0; j <= a; ++j) {
            sr[j] = path[j];
            dp[j] = P + j;
        }
        for (int l = 0; l < La; ++l)
            for (int g = 0; g < Hkv; ++g)
                for (int j = 0; j <= a; ++j) {
                    const double* ks = k_tree + ((((long)l * B + b) * N + path[j]) * Hkv + g) * d;
                    const double* vs = v_tree + ((((long)l * B + b) * N + path[j]) * Hkv + g) * d;
                    double* kd = k_cache + ((((long)l * B + b) * Hkv + g) * Pcap + P + j) * d;
                    double* vd = v_cache + ((((long)l * B + b) * Hkv + g) * Pcap + P + j) * d;
                    for (int c = 0; c < d; ++c) {
                        kd[c] = ks[c];
                        vd[c] = vs[c];
                    }
                }
        /* GDN: the accepted path as a chain, run through the same per-node rule. */
        const int n = a + 1;
        int32_t* chain_parent = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
        double* xc = (double*)malloc(sizeof(double) * (size_t)n * C);
        double* bc = (double*)malloc(sizeof(double) * (size_t)n * Hv);
        double* dc = (double*)malloc(sizeof(double) * (size_t)n * Hv);
        double* oc = (double*)malloc(sizeof(double) * (size_t)n * dv);
        double* sc = (double*)malloc(sizeof(double) * (size_t)n * SS);
        double* cs_new = (double*)malloc(sizeof(double) * (size_t)(K > 1 ? K - 1 : 1) * C);
        for (int l = 0; l < Lg; ++l) {
            const long lb = (long)l * B + b;
            for (int j = 0; j < n; ++j) {
                chain_parent[j] = j - 1;
                for (int c = 0; c < C; ++c) xc[(long)j * C + c] = x[(lb * N + path[j]) * C + c];
                for (int h = 0; h < Hv; ++h) {
                    bc[(long)j * Hv + h] = beta[(lb * N + path[j]) * Hv + h];
                    dc[(long)j * Hv + h] = decay[(lb * N + path[j]) * Hv + h];
                }
            }
            double* cs = conv_state + lb * (K - 1) * C;
            for (int h = 0; h < Hv; ++h) {
                double* Sh = S + (lb * Hv + h) * SS;
                ddto_gdn_unit(n, n, Hk, Hv, dk, dv, K, h, xc, conv_w + (long)l * C * K, cs, bc, dc, Sh,
                              chain_parent, oc, sc);
                for (long e = 0; e < SS; ++e) Sh[e] = sc[(long)(n - 1) * SS + e];
            }
            /* conv state: the last K-1 rows of [cs ; xc] */
            for (int r = 0; r < K - 1; ++r) {
                int src = r + n; /* index into the concatenation of length K-1+n */
                for (int c = 0; c < C; ++c)
                    cs_new[(long)r * C + c] =
                        (src < K - 1) ? cs[(long)src * C + c] : xc[(long)(src - (K - 1)) * C + c];
            }
            for (long e = 0; e < (long)(K - 1) * C; ++e) cs[e] = cs_new[e];
        }
        free(chain_parent);
        free(xc);
        free(bc);
        free(dc);
        free(oc);
        free(sc);
        free(cs_new);
        prefix_len[b] = P + a + 1;
    }
    return DDTO_OK;
}

/* ------------------------------------------------------------------------- */
/* Paged KV caches                                                            */
/* ------------------------------------------------------------------------- */

/* [NOTES] "Where the next step is": the verifier must read the prefix from paged KV
 * blocks.  Row p of a request's prefix lives at row p % page of page block_table[b][p/page]. */
int ddto_gather_pages(int L, int B, int Hkv, int d, int page, int num_pages, int max_pages,
                      const double* pages, const int32_t* block_table, const int32_t* prefix_len,
                      int Pcap, double* cache) {
    if (L < 1 || B < 1 || Hkv < 1 || d < 1 || page < 1 || num_pages < 1 || max_pages < 1 || Pcap < 0)
        return DDTO_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        const int P = prefix_len[b];
        if (P < 0 || P > Pcap || P > (long)max_pages * page) return DDTO_ERR_ARG;
        for (int p = 0; p < P; ++p) {
            const int pg = block_table[(long)b * max_pages + p / page];
            if (pg < 0 || pg >= num_pages) return DDTO_ERR_ARG;
        }
    }
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < Hkv; ++g)
                for (int p = 0; p < Pcap; ++p) {
                    double* dst = cache + ((((long)l * B + b) * Hkv + g) * Pcap + p) * d;
                    if (p >= prefix_len[b]) {
                        for (int i = 0; i < d; ++i) dst[i] = 0.0;
                        continue;
                    }
                    const int pg = block_table[(long)b * max_pages + p / page];
                    const double* src = pages + ((((long)l * num_pages + pg) * Hkv + g) * page + p % page) * d;
                    for (int i = 0; i < d; ++i) dst[i] = src[i];
                }
    return DDTO_OK;
}

int ddto_scatter_pages(int L, int B, int Hkv, int d, int page, int num_pages, int max_pages,
                       const double* cache, int Pcap, const int32_t* block_table,
                       const int32_t* n_rows, double* pages) {
    if (L < 1 || B < 1 || Hkv < 1 || d < 1 || page < 1 || num_pages < 1 || max_pages < 1 || Pcap < 0)
        return DDTO_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        if (n_rows[b] < 0 || n_rows[b] > Pcap || n_rows[b] > (long)max_pages * page) return DDTO_ERR_ARG;
        for (int p = 0; p < n_rows[b]; ++p) {
            const int pg = block_table[(long)b * max_pages + p / page];
            if (pg < 0 || pg >= num_pages) return DDTO_ERR_ARG;
        }
    }
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b)
            for (int g = 0; g < Hkv; ++g)
                for (int p = 0; p < n_rows[b]; ++p) {
                    const int pg = block_table[(long)b * max_pages + p / page];
                    const double* src = cache + ((((long)l * B + b) * Hkv + g) * Pcap + p) * d;
                    double* dst = pages + ((((long)l * num_pages + pg) * Hkv + g) * page + p % page) * d;
                    for (int i = 0; i < d; ++i) dst[i] = src[i];
                }
    return DDTO_OK;
}

/* ------------------------------------------------------------------------- */
/* Rotary embedding by depth                                                  */
/* ------------------------------------------------------------------------- */

/* [NOTES] "Where the next step is" / [ARCH] positions shared per depth: every row of a
 * node is rotated by its node's position, pairs (i, i + rot/2). */
int ddto_rope_tree(int L, int B, int N, int H, int d, int rot, double theta,
                   const int32_t* position, const int32_t* n_nodes, double* x) {
    if (L < 1 || B < 1 || N < 1 || H < 1 || rot < 2 || rot > d || rot % 2 || !(theta > 1.0)) return DDTO_ERR_ARG;
    const int half = rot / 2;
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b)
            for (int n = 0; n < n_nodes[b] && n < N; ++n)
                for (int h = 0; h < H; ++h) {
                    double* row = x + ((((long)l * B + b) * N + n) * H + h) * d;
                    for (int i = 0; i < half; ++i) {
                        const double a = (double)position[(long)b * N + n] * pow(theta, -2.0 * i / rot);
                        const double x0 = row[i], x1 = row[i + half];
                        row[i] = x0 * cos(a) - x1 * sin(a);
                        row[i + half] = x1 * cos(a) + x0 * sin(a);
                    }
                }
    return DDTO_OK;
}
