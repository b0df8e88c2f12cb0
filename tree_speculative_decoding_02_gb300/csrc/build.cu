// build.cu -- ddt_build_tree: best-first draft-tree construction.
//
// "From Tree-Based Speculative Decoding to Drafter Training", section "The Architecture
// of DDTree: Tree Construction and Verification": top-K ids and log-probabilities per
// depth, a max-heap seeded with the best depth-1 token, each pop adding the node to the
// tree and pushing its next-ranked sibling and its best child, until the budget is
// spent; the tree is then flattened (root + nodes, per-depth positions, ancestor-only
// mask).
//
// GB300 layout of the work:
//   k_build_row      grid (D, B): one CTA per depth row of a request, one HBM pass plus
//                    one L2 pass over the row: log-sum-exp and the exact top-k (a
//                    threshold from the warps' lane bests, then the few entries at or
//                    above it ranked by one warp).
//   k_build_tree     grid B: per request, one warp runs the best-first selection over a
//                    shared-memory frontier, then the CTA numbers the nodes breadth first
//                    (one pass over all depths) and writes the flattened tree and its
//                    bit-packed ancestor mask.
#include <cuda.h>
#include <float.h>
#include <limits.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace ddt {

// ---------------------------------------------------------------------------- row pass
// One CTA per (depth, request) row of the drafter logits:
//   1. one streaming pass: each thread's max, a running sum of exp(v - its max) (rescaled
//      when the max grows) and a non-finite check.  The k-th largest of the 512 thread
//      maxima, tau, is reached by k entries of the row, so it is at or below the value of
//      the row's k-th best entry;
//   2. only the threads whose max reaches tau can hold such entries (usually a few in
//      the whole row): each warp re-reads those threads' entries together, and the ones
//      that reach tau (ties included) are collected in shared memory, from which one
//      warp takes the exact top-k by (value desc, id asc).
// If more entries than the buffer holds reach tau (not seen on drafter-like rows), each
// warp ranks its own entries with a warp top-k and the warp lists are merged instead.
struct BuildRow {
    double lse;  // log sum_v exp(logit_v)
    int bad;     // 1 if the row holds NaN or +-Inf
    int pad;
};

size_t build_ws_bytes(int B, int D, int V, int k) {
    (void)V;
    const long rows = (long)B * D;
    size_t bytes = rows * sizeof(BuildRow) + rows * k * (sizeof(float) + sizeof(int));
    return (bytes + 255) & ~(size_t)255;
}

namespace {
constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kCandCap = 1024;
}  // namespace

// an integer key with the order of the float (-0 just below +0); not for NaN
__device__ __forceinline__ int ord_key(float f) {
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads, 4) k_build_row(const T* __restrict__ logits, int D, int V, int k, int vec,
                                                           BuildRow* __restrict__ rows, float* __restrict__ top_v,
                                                           int* __restrict__ top_id) {
    const int d = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long r = (long)b * D + d;
    const T* x = logits + r * V;
    __shared__ float s_cv[kCandCap];
    __shared__ int s_ci[kCandCap];
    __shared__ float s_wv[kRowWarps * 32];
    __shared__ int s_wi[kRowWarps * 32];
    __shared__ float s_m[kRowWarps];
    __shared__ double s_sum[kRowWarps];
    __shared__ int s_nc, s_bad;
    const VId emp = vid_empty();
    if (tid == 0) {
        s_nc = 0;
        s_bad = 0;
    }

    // ---- pass 1.  A NaN or +inf entry makes the sum NaN (an exponential of NaN, or
    //      inf - inf) and a -inf entry the smallest entry -inf: together they flag every
    //      non-finite row.
    const float LOG2E = 1.4426950408889634f;
    float m = emp.v, acc = 0.f, lo = -emp.v;
    auto see8 = [&](const float (&t8)[8], int n) {
        float m8 = emp.v, l8 = -emp.v;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < n) {
                m8 = fmaxf(m8, t8[u]);
                l8 = fminf(l8, t8[u]);
            }
        lo = fminf(lo, l8);
        if (m8 > m) {
            acc *= exp2f((m - m8) * LOG2E);
            m = m8;
        }
        const float mb = m * LOG2E;
        float s8 = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (u < n) s8 += exp2f(fmaf(t8[u], LOG2E, -mb));
        acc += s8;
    };
    if (vec) {  // V % 8 == 0 and 16-byte aligned rows: 8 entries a load
#pragma unroll 4
        for (int e = tid * 8; e < V; e += kRowThreads * 8) {
            float t8[8];
            load8_stream(x + e, t8);
            see8(t8, 8);
        }
    } else {
        for (int e = tid * 8; e < V; e += kRowThreads * 8) {
            float t8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t8[u] = (e + u < V) ? to_f32(x[e + u]) : emp.v;
            see8(t8, min(8, V - e));
        }
    }
    int bad = !(fabsf(acc) < INFINITY) || lo == emp.v;  // a thread with no entries: acc 0, lo +inf
    // the warp's thread maxima, largest first
    float tv = m;
    int ti = lane;
    warp_sort_best_first(tv, ti);
    const float wm = warp_max(m);
    bad = warp_or(bad);
    if (lane == 0) {
        s_m[warp] = wm;
        if (bad) s_bad = 1;
    }
    s_wv[warp * 32 + lane] = tv;
    __syncthreads();
    float M = s_m[0];
#pragma unroll 1
    for (int w = 1; w < kRowWarps; ++w) M = fmaxf(M, s_m[w]);
    // tau = the k-th largest thread max of the block: k thread maxima, i.e. k entries of
    // the row, reach it, so it is at or below the row's k-th best value.  Every warp merges
    // the warps' sorted lists (lane w walks warp w's list) and pops k times.
    float tau_v = emp.v;
    {
        int pos = 0;
        float head = lane < kRowWarps ? s_wv[lane * 32] : emp.v;
#pragma unroll 1
        for (int i = 0; i < k; ++i) {
            const int key = lane < kRowWarps ? ord_key(head) : INT_MIN;
            const unsigned who = __ballot_sync(kFull, key == __reduce_max_sync(kFull, key));
            const int src = __ffs(who) - 1;
            tau_v = __shfl_sync(kFull, head, src);
            if (lane == src) head = ++pos < 32 ? s_wv[lane * 32 + pos] : emp.v;
        }
    }
    const bool row_bad = s_bad != 0;
    // the sum of exp(v - M): fp32 per thread and across the warp, fp64 across warps
    const float ws = warp_sum(m == emp.v ? 0.f : acc * exp2f((m - M) * LOG2E));
    if (lane == 0) s_sum[warp] = (double)ws;

    // ---- pass 2: the entries that reach tau, from the threads whose max reaches it; the
    //      warp re-reads one such thread's entries at a time, a load a lane
    if (!row_bad) {
        unsigned q = __ballot_sync(kFull, m >= tau_v);
        while (q) {
            const int t = warp * 32 + __ffs(q) - 1;  // the thread whose entries are re-read
            q &= q - 1;
            const int nch = t * 8 < V ? (V - t * 8 + kRowThreads * 8 - 1) / (kRowThreads * 8) : 0;
            for (int j = lane; j < nch; j += 32) {
                const int e = t * 8 + j * kRowThreads * 8;
                float t8[8];
                if (vec) {
                    load8(x + e, t8);
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u) t8[u] = (e + u < V) ? to_f32(x[e + u]) : emp.v;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (t8[u] >= tau_v) {
                        const int pos = atomicAdd(&s_nc, 1);
                        if (pos < kCandCap) {
                            s_cv[pos] = t8[u];
                            s_ci[pos] = e + u;
                        }
                    }
            }
        }
    }
    __syncthreads();
    const int nc = s_nc;
    if (nc > kCandCap && !row_bad) {
        // overflow: every warp ranks its own entries, then the warp lists are merged
        WarpTopK tk;
        tk.init(k);
        for (int e0 = warp * 32; e0 < V; e0 += kRowThreads) {
            const int e = e0 + lane;
            const float v = e < V ? to_f32(x[e]) : emp.v;
            const bool q = e < V && v >= tau_v;
            if (__any_sync(kFull, q)) tk.insert(q ? v : emp.v, q ? e : emp.id);
        }
        s_wv[warp * 32 + lane] = tk.v;
        s_wi[warp * 32 + lane] = tk.id;
        __syncthreads();
    }
    if (warp == 0) {
        WarpTopK tk;
        tk.init(k);
        if (!row_bad) {
            if (nc <= kCandCap) {
                for (int c0 = 0; c0 < nc; c0 += 32) {
                    const int c = c0 + lane;
                    tk.insert(c < nc ? s_cv[c] : emp.v, c < nc ? s_ci[c] : emp.id);
                }
            } else {
                for (int w = 0; w < kRowWarps; ++w) tk.insert(s_wv[w * 32 + lane], s_wi[w * 32 + lane]);
            }
        }
        if (lane < k) {
            top_v[r * k + lane] = tk.v;
            top_id[r * k + lane] = tk.id;
        }
        if (lane == 0) {
            double tot = 0.0;
            for (int w = 0; w < kRowWarps; ++w) tot += s_sum[w];
            const double lse = (double)M + log(tot);
            rows[r].lse = lse;
            rows[r].bad = row_bad || !isfinite(lse);
        }
    }
}

// ---------------------------------------------------------------------- selection
constexpr int kRegSlots = 3;  // frontier slots a lane holds in registers (budget <= 94)

struct Cand {
    double L;   // sum of path logits, depth 1 first (its score is L - cum LSE of its depth)
    int depth;  // 1..D
    int rank;   // within the depth's top-k
    int parent; // index into the selected list, -1 = root
    int pad;
    // the two entries a pop of this one pushes, scored ahead of time: its next-ranked
    // sibling and its best child (path sum L and score s; unused where none exists)
    double sib_L, sib_s, ch_L, ch_s;
    // the token path as a key with the path's lexicographic order (see lex_key_bits)
    unsigned long long lk;
};

struct TreeSmem {
    // per depth
    float* top_v;   // [D][k]
    double* top_vd; // [D][k] the same logits as doubles (converted once, not per push)
    int* top_id;    // [D][k]
    double* cum;    // [D+1] cumulative LSE, cum[0] = 0
    // selection: every candidate ever pushed stays in the pool, in push order; the
    // frontier and the selected list hold pool indices, so a pop moves 12 bytes
    Cand* pool;     // [2 budget + 1]
    int* fidx;      // [budget + 2] frontier entries (pool indices)
    long long* fs;  // [budget + 2] their scores as order-preserving integer keys
    unsigned long long* fl;  // [budget + 2] their token-path keys
    int* idr;       // [D][k] 1 + the token's place among its depth's k token ids
    int* sel;       // [budget] selected entries (pool indices)
    int* new_idx;   // [budget]
    int* out_par;   // [N]
};

__device__ __forceinline__ const Cand& selc(const TreeSmem& S, int i) { return S.pool[S.sel[i]]; }

__device__ __forceinline__ int cand_token(const TreeSmem& S, int k, const Cand& c) {
    return S.top_id[(c.depth - 1) * k + c.rank];
}

// Lexicographic order of the two candidates' token paths (lower ids first, a prefix
// before its extensions); only consulted on an exact score tie.  The deeper candidate is
// lifted to the other's depth (meeting it means one path is a prefix of the other), then
// both climb in step until their parents agree: the tokens below that common ancestor
// differ and decide.  No path is materialised.
__device__ bool lex_less(const TreeSmem& S, int k, const Cand& a, const Cand& b) {
    int da = a.depth, db = b.depth;
    int ta = cand_token(S, k, a), tb = cand_token(S, k, b);
    int pa = a.parent, pb = b.parent;  // rows of S.sel; -1 = the root
    while (da > db) {
        const Cand& u = selc(S, pa);
        ta = cand_token(S, k, u);
        pa = u.parent;
        --da;
    }
    if (a.depth > b.depth && pa == pb && ta == tb) return false;  // b is a prefix of a
    while (db > da) {
        const Cand& u = selc(S, pb);
        tb = cand_token(S, k, u);
        pb = u.parent;
        --db;
    }
    if (b.depth > a.depth && pa == pb && ta == tb) return true;   // a is a proper prefix of b
    while (pa != pb) {
        const Cand& u = selc(S, pa);
        const Cand& v = selc(S, pb);
        ta = cand_token(S, k, u);
        tb = cand_token(S, k, v);
        pa = u.parent;
        pb = v.parent;
    }
    return ta < tb;
}

// A score (a log-probability: strictly negative, finite) as a 64-bit key with the same
// order: flipping every bit but the sign of a negative double's pattern reverses the
// integer order into the value order, and equal doubles get equal keys.  The selection
// compares keys on the integer pipe (this chip's FP64 rate is a small fraction of its
// FP32 rate, and the argmax is a dependent chain of compares).
__device__ __forceinline__ long long score_key(double s) {
    const long long b = __double_as_longlong(s);
    return b < 0 ? (b ^ 0x7fffffffffffffffLL) : b;
}

// Token paths as integer keys.  Every token at depth d is one of that depth's k top
// tokens, so comparing two paths' tokens at a depth is comparing the tokens' places in
// the depth's id order.  A path is packed as 1 + that place for each level, depth 1 in
// the highest bits and zeros after its last level, so a prefix sorts before its
// extensions: the integer order of two keys is the lexicographic order of the paths.
// Bits a level, or 0 when D levels do not fit 64 bits (then ties climb the paths).
__device__ __forceinline__ int lex_key_bits(int D, int k) {
    int bits = 1;
    while ((1 << bits) < k + 1) ++bits;
    return bits * D <= 64 ? bits : 0;
}

// frontier entry i before entry j in the selection order (score, then token path)
__device__ __forceinline__ bool front_before(const TreeSmem& S, int k, long long si, int i, long long sj, int j) {
    if (si != sj) return si > sj;
    return i != j && lex_less(S, k, S.pool[S.fidx[i]], S.pool[S.fidx[j]]);
}

// rank-path key of selected node i: the ranks along its path from the root, `bits` bits
// a level, first level highest; within a depth its order is the breadth-first order
__device__ __forceinline__ unsigned long long rank_key(const TreeSmem& S, int i, int bits) {
    unsigned long long key = 0;
    int sh = 0;
    for (int a = i; a >= 0; a = selc(S, a).parent, sh += bits) key |= (unsigned long long)selc(S, a).rank << sh;
    return key << (64 - sh);  // root-first levels at the top; depth is compared separately
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) k_build_tree(int D, int k, int budget, const BuildRow* __restrict__ rows,
                                                          const float* __restrict__ rtv, const int* __restrict__ rti,
                                                          const int32_t* __restrict__ root_token,
                                                          const int32_t* __restrict__ prefix_len,
                                                          int32_t* __restrict__ token, int32_t* __restrict__ parent,
                                                          int32_t* __restrict__ depth, int32_t* __restrict__ position,
                                                          int32_t* __restrict__ n_nodes, uint32_t* __restrict__ anc,
                                                          double* __restrict__ score, int32_t* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = budget + 1;
    const int W = (N + 31) / 32;

    TreeSmem S;
    unsigned char* p = smem_raw;
    S.cum = reinterpret_cast<double*>(p);      p += sizeof(double) * (kMaxDepth + 1);
    S.fs = reinterpret_cast<long long*>(p);    p += sizeof(long long) * (budget + 2);
    S.fl = reinterpret_cast<unsigned long long*>(p); p += sizeof(unsigned long long) * (budget + 2);
    S.pool = reinterpret_cast<Cand*>(p);       p += sizeof(Cand) * (2 * budget + 1);
    S.top_vd = reinterpret_cast<double*>(p);   p += sizeof(double) * D * k;
    S.top_v = reinterpret_cast<float*>(p);     p += sizeof(float) * D * k;
    S.top_id = reinterpret_cast<int*>(p);      p += sizeof(int) * D * k;
    S.idr = reinterpret_cast<int*>(p);         p += sizeof(int) * D * k;
    S.fidx = reinterpret_cast<int*>(p);        p += sizeof(int) * (budget + 2);
    S.sel = reinterpret_cast<int*>(p);         p += sizeof(int) * (budget + 1);
    S.new_idx = reinterpret_cast<int*>(p);     p += sizeof(int) * (budget + 1);
    S.out_par = reinterpret_cast<int*>(p);     p += sizeof(int) * N;
    __shared__ int s_bad;
    __shared__ int s_nsel;

    // 1. the depths' top-k lists and log-sum-exps (from the row pass); the rows' records
    //    are loaded by D threads at once and staged (S.cum[d + 1], and S.idr[d] until the
    //    id places overwrite it)
    for (int e = tid; e < D * k; e += kThreads) {
        const float v = rtv[(long)b * D * k + e];
        S.top_v[e] = v;
        S.top_vd[e] = (double)v;
        S.top_id[e] = rti[(long)b * D * k + e];
    }
    for (int d = tid; d < D; d += kThreads) {
        const BuildRow rr = rows[(long)b * D + d];
        S.cum[d + 1] = rr.lse;
        S.idr[d] = rr.bad;
    }
    __syncthreads();
    if (tid == 0) {
        int bad = 0;
        double c = 0.0;
        S.cum[0] = 0.0;
        for (int d = 0; d < D; ++d) {
            bad |= S.idr[d];       // the rows' flags and log-sum-exps, staged below
            c += S.cum[d + 1];     // cumulative in depth order, as the scores are defined
            S.cum[d + 1] = c;
        }
        s_bad = bad;
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    for (int e = tid; e < D * k; e += kThreads) {
        const int* ids = S.top_id + (e / k) * k;
        const int t = S.top_id[e];
        int pl = 1;
        for (int r = 0; r < k; ++r) pl += ids[r] < t;
        S.idr[e] = pl;
    }
    __syncthreads();
    const int lbits = lex_key_bits(D, k);

    // 2. best-first selection: one warp keeps the frontier in shared memory (entries and
    //    their scores).  A pop is a warp argmax over the scores -- the token-path order is
    //    consulted only on an exact score tie -- after which the best entry moves to the
    //    selected list and its next-ranked sibling and best child enter the frontier.
    //    Their scores were formed when the popped entry itself was pushed, so a pop waits
    //    on no fp64 add: lanes 0 and 1 score the successors of the two new entries right
    //    after pushing them, and write those scores only after the next argmax, which
    //    hides the adds' latency.  Every score is the same fp64 expression as ever:
    //    L = L(parent) + logit, s = L - cum LSE of the depth.
    if (warp == 0) {
        // successors of an entry at (depth d, rank r) whose parent path sums to Lp and
        // whose own path sums to L: sibling (d, r + 1) and child (d + 1, 0); indices are
        // clamped where the successor does not exist (its score is then never used)
        auto successors = [&](int d, int r, double Lp, double L, double& sL, double& sS, double& cL, double& cS) {
            const int rs = min(r + 1, k - 1), dc = min(d + 1, D);
            sL = Lp + S.top_vd[(d - 1) * k + rs];
            sS = sL - S.cum[d];
            cL = L + S.top_vd[(dc - 1) * k];
            cS = cL - S.cum[dc];
        };
        int n_sel = 0;
        if (lbits && budget + 2 <= 32 * kRegSlots) {
            // The frontier in registers: slot j is register j / 32 of lane j % 32, holding the
            // entry's score key, token-path key and pool index.  A pop is then a lane-local
            // compare of at most kRegSlots slots, a warp argmax, and register moves; only
            // the pool records (written once, read at their pop) live in shared memory.
            long long rk[kRegSlots];
            unsigned long long rl[kRegSlots];
            int rp[kRegSlots];
#pragma unroll
            for (int r = 0; r < kRegSlots; ++r) {
                rk[r] = LLONG_MIN;
                rl[r] = ~0ull;
                rp[r] = -1;
            }
            int n_front = 0, n_pool = 0;
            if (budget > 0 && !bad) {
                Cand c0;
                c0.depth = 1;
                c0.rank = 0;
                c0.parent = -1;
                c0.pad = 0;
                c0.L = S.top_vd[0];
                successors(1, 0, 0.0, c0.L, c0.sib_L, c0.sib_s, c0.ch_L, c0.ch_s);
                c0.lk = (unsigned long long)S.idr[0] << (64 - lbits);
                if (lane == 0) {
                    S.pool[0] = c0;
                    rk[0] = score_key(c0.L - S.cum[1]);
                    rl[0] = c0.lk;
                    rp[0] = 0;
                }
                n_front = 1;
                n_pool = 1;
            }
            __syncwarp();
            int pend = -1;
            double pL = 0.0, pS = 0.0, qL = 0.0, qS = 0.0;
            while (n_sel < budget && n_front > 0) {
                // this lane's best slot by (score desc, token path asc)
                int bj = -1;
                long long bk = LLONG_MIN;
                unsigned long long bl = ~0ull;
                int bp = -1;
#pragma unroll
                for (int r = 0; r < kRegSlots; ++r) {
                    const bool live = r * 32 + lane < n_front;
                    if (live && (bj < 0 || rk[r] > bk || (rk[r] == bk && rl[r] < bl))) {
                        bj = r;
                        bk = rk[r];
                        bl = rl[r];
                        bp = rp[r];
                    }
                }
                // warp argmax of the 64-bit keys as two 32-bit warp reductions: the high
                // halves (sign bit flipped: unsigned order), then the low halves among the
                // lanes that hold the top high half
                const unsigned long long uk = (unsigned long long)bk ^ 0x8000000000000000ull;
                const unsigned khi = (unsigned)(uk >> 32), klo = (unsigned)uk;
                const unsigned mhi = __reduce_max_sync(kFull, khi);
                const unsigned mlo = __reduce_max_sync(kFull, khi == mhi ? klo : 0u);
                const bool top = bj >= 0 && khi == mhi && klo == mlo;
                const unsigned tied = __ballot_sync(kFull, top);
                int wl = __ffs(tied) - 1;
                if (__popc(tied) > 1) {  // exact score tie: the smaller token path, the same way
                    const unsigned lhi = (unsigned)(bl >> 32), llo = (unsigned)bl;
                    const unsigned nhi = __reduce_min_sync(kFull, top ? lhi : ~0u);
                    const unsigned nlo = __reduce_min_sync(kFull, top && lhi == nhi ? llo : ~0u);
                    wl = __ffs(__ballot_sync(kFull, top && lhi == nhi && llo == nlo)) - 1;
                }
                const int wr = __shfl_sync(kFull, bj, wl);
                const int pc = __shfl_sync(kFull, bp, wl);
                // the last pop's new entries get their successor scores (the adds are done)
                if (pend >= 0) {
                    Cand& u = S.pool[pend];
                    u.sib_L = pL;
                    u.sib_s = pS;
                    u.ch_L = qL;
                    u.ch_s = qS;
                }
                __syncwarp();
                const Cand& c = S.pool[pc];
                const int c_depth = c.depth, c_rank = c.rank, c_parent = c.parent;
                const unsigned long long c_lk = c.lk;
                const double c_L = c.L, c_sL = c.sib_L, c_sS = c.sib_s, c_cL = c.ch_L, c_cS = c.ch_s;
                const bool has_sib = c_rank + 1 < k, has_ch = c_depth < D;
                const int me = n_sel, nf = n_front - 1;
                // the last slot moves into the popped one
                {
                    const int ln = nf & 31, rn = nf >> 5;
                    long long mv_k = rk[0];
                    unsigned long long mv_l = rl[0];
                    int mv_p = rp[0];
#pragma unroll
                    for (int r = 1; r < kRegSlots; ++r)
                        if (r == rn) {
                            mv_k = rk[r];
                            mv_l = rl[r];
                            mv_p = rp[r];
                        }
                    mv_k = __shfl_sync(kFull, mv_k, ln);
                    mv_l = __shfl_sync(kFull, mv_l, ln);
                    mv_p = __shfl_sync(kFull, mv_p, ln);
                    if (lane == wl) {
#pragma unroll
                        for (int r = 0; r < kRegSlots; ++r)
                            if (r == wr) {
                                rk[r] = mv_k;
                                rl[r] = mv_l;
                                rp[r] = mv_p;
                            }
                    }
                }
                // the new entries (every lane forms the same keys; the slot's owner keeps them)
                const int sh_s = 64 - lbits * c_depth, sh_c = 64 - lbits * (c_depth + 1);
                const unsigned long long fmask = (((unsigned long long)1 << lbits) - 1) << sh_s;
                const unsigned long long lk_s =
                    (c_lk & ~fmask) | ((unsigned long long)S.idr[(c_depth - 1) * k + min(c_rank + 1, k - 1)] << sh_s);
                const unsigned long long lk_c =
                    has_ch ? (c_lk | ((unsigned long long)S.idr[min(c_depth, D - 1) * k] << sh_c)) : 0ull;
                const int slot_s = nf, slot_c = nf + (int)has_sib;
#pragma unroll
                for (int r = 0; r < kRegSlots; ++r) {
                    if (has_sib && slot_s == r * 32 + lane) {
                        rk[r] = score_key(c_sS);
                        rl[r] = lk_s;
                        rp[r] = n_pool;
                    }
                    if (has_ch && slot_c == r * 32 + lane) {
                        rk[r] = score_key(c_cS);
                        rl[r] = lk_c;
                        rp[r] = n_pool + (int)has_sib;
                    }
                }
                // their pool records: lane 0 the sibling, lane 1 the child, each with its own
                // successors' scores started now and stored after the next argmax
                pend = -1;
                if (lane < 2 && (lane == 0 ? has_sib : has_ch)) {
                    Cand e;
                    e.depth = lane == 0 ? c_depth : c_depth + 1;
                    e.rank = lane == 0 ? c_rank + 1 : 0;
                    e.parent = lane == 0 ? c_parent : me;
                    e.pad = 0;
                    e.L = lane == 0 ? c_sL : c_cL;
                    e.lk = lane == 0 ? lk_s : lk_c;
                    e.sib_L = e.sib_s = e.ch_L = e.ch_s = 0.0;
                    pend = n_pool + (lane == 0 ? 0 : (int)has_sib);
                    const double Lp = lane == 0 ? (c_parent < 0 ? 0.0 : selc(S, c_parent).L) : c_L;
                    successors(e.depth, e.rank, Lp, e.L, pL, pS, qL, qS);
                    S.pool[pend] = e;
                }
                if (lane == 0) S.sel[me] = pc;
                n_front = nf + has_sib + has_ch;
                n_pool += has_sib + has_ch;
                ++n_sel;
                __syncwarp();
            }
        } else {
            int n_front = 0, n_pool = 0;
            if (budget > 0 && !bad) {
                if (lane == 0) {
                    Cand c0;
                    c0.depth = 1;
                    c0.rank = 0;
                    c0.parent = -1;
                    c0.pad = 0;
                    c0.L = S.top_vd[0];
                    successors(1, 0, 0.0, c0.L, c0.sib_L, c0.sib_s, c0.ch_L, c0.ch_s);
                    c0.lk = lbits ? (unsigned long long)S.idr[0] << (64 - lbits) : 0ull;
                    S.pool[0] = c0;
                    S.fidx[0] = 0;
                    S.fs[0] = score_key(c0.L - S.cum[1]);
                    S.fl[0] = c0.lk;
                }
                n_front = 1;
                n_pool = 1;
            }
            __syncwarp();
            // lanes 0 and 1: the pool entry pushed last pop whose successor scores are still in
            // registers (-1: none)
            int pend = -1;
            double pL = 0.0, pS = 0.0, qL = 0.0, qS = 0.0;
            while (n_sel < budget && n_front > 0) {
                int best = -1;
                long long bs = 0;
                unsigned long long bl = 0;
                for (int i = lane; i < n_front; i += 32) {
                    const long long si = S.fs[i];
                    const unsigned long long li = S.fl[i];
                    const bool before = lbits ? (si > bs || (si == bs && li < bl)) : front_before(S, k, si, i, bs, best);
                    if (best < 0 || before) {
                        best = i;
                        bs = si;
                        bl = li;
                    }
                }
                // warp argmax on the score keys; the token-path order decides only between
                // lanes that hold the same top score (exact ties, which bf16 logits make
                // common: every pair of nodes below two tied siblings ties too)
                long long mk = best >= 0 ? bs : LLONG_MIN;
    #pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const long long om = __shfl_xor_sync(kFull, mk, o);
                    mk = om > mk ? om : mk;
                }
                const bool top = best >= 0 && bs == mk;
                const unsigned tied = __ballot_sync(kFull, top);
                if (__popc(tied) == 1) {
                    best = __shfl_sync(kFull, best, __ffs(tied) - 1);
                } else if (lbits) {
                    unsigned long long ml = top ? bl : ~0ull;
    #pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const unsigned long long om = __shfl_xor_sync(kFull, ml, o);
                        ml = om < ml ? om : ml;
                    }
                    best = __shfl_sync(kFull, best, __ffs(__ballot_sync(kFull, top && bl == ml)) - 1);
                } else {
                    int w = -1;
                    for (unsigned t = tied; t; t &= t - 1) {
                        const int idx = __shfl_sync(kFull, best, __ffs(t) - 1);
                        if (w < 0 || lex_less(S, k, S.pool[S.fidx[idx]], S.pool[S.fidx[w]])) w = idx;
                    }
                    best = w;
                }
                // the last pop's new entries get their successor scores (the adds are done by now)
                if (pend >= 0) {
                    Cand& u = S.pool[pend];
                    u.sib_L = pL;
                    u.sib_s = pS;
                    u.ch_L = qL;
                    u.ch_s = qS;
                }
                __syncwarp();
                // the popped entry leaves the frontier (its slot takes the last entry) and joins
                // the selected list; lane 0 pushes its next-ranked sibling, lane 1 its best child
                const int pc = S.fidx[best];
                const Cand& c = S.pool[pc];
                const int c_depth = c.depth, c_rank = c.rank, c_parent = c.parent;
                const unsigned long long c_lk = c.lk;
                const bool has_sib = c_rank + 1 < k, has_ch = c_depth < D;
                const int me = n_sel, nf = n_front - 1;
                const bool push = lane < 2 && (lane == 0 ? has_sib : has_ch);
                double eL = 0.0, eS = 0.0, Lp = 0.0;
                if (push) {
                    eL = lane == 0 ? c.sib_L : c.ch_L;
                    eS = lane == 0 ? c.sib_s : c.ch_s;
                    Lp = lane == 0 ? (c_parent < 0 ? 0.0 : selc(S, c_parent).L) : c.L;
                }
                __syncwarp();
                if (lane == 0) {
                    S.fidx[best] = S.fidx[nf];
                    S.fs[best] = S.fs[nf];
                    S.fl[best] = S.fl[nf];
                    S.sel[me] = pc;
                }
                __syncwarp();
                pend = -1;
                if (push) {
                    Cand e;
                    e.depth = lane == 0 ? c_depth : c_depth + 1;
                    e.rank = lane == 0 ? c_rank + 1 : 0;
                    e.parent = lane == 0 ? c_parent : me;
                    e.pad = 0;
                    e.L = eL;
                    e.lk = 0ull;
                    if (lbits) {
                        // the sibling replaces the last level of the popped entry's path, the
                        // child appends a level
                        const int sh = 64 - lbits * e.depth;
                        const unsigned long long field = (unsigned long long)S.idr[(e.depth - 1) * k + e.rank] << sh;
                        e.lk = lane == 0 ? ((c_lk & ~((((unsigned long long)1 << lbits) - 1) << sh)) | field) : (c_lk | field);
                    }
                    pend = n_pool + (lane == 0 ? 0 : (int)has_sib);
                    const int slot = nf + (lane == 0 ? 0 : (int)has_sib);
                    // its own successors: the sibling's parent path is the popped entry's, the
                    // child's parent is the popped entry itself
                    successors(e.depth, e.rank, Lp, e.L, pL, pS, qL, qS);
                    e.sib_L = e.sib_s = e.ch_L = e.ch_s = 0.0;
                    S.pool[pend] = e;
                    S.fidx[slot] = pend;
                    S.fs[slot] = score_key(eS);
                    S.fl[slot] = e.lk;
                }
                n_front = nf + has_sib + has_ch;
                n_pool += has_sib + has_ch;
                ++n_sel;
                __syncwarp();
            }
        }
        if (lane == 0) s_nsel = n_sel;
    }
    __syncthreads();
    const int n_sel = s_nsel;

    // 3. canonical breadth-first numbering (depth, then parent's row, then rank), all depths
    //    in one pass: within a depth that order is the lexicographic order of the nodes'
    //    rank paths from the root.  When the path fits 64 bits (ceil(log2 k) bits a level)
    //    it is packed into a key; otherwise two nodes climb to where their parents agree.
    {
        int bits = 1;
        while ((1 << bits) < k) ++bits;
        const bool packed = bits * D <= 64;
        unsigned long long* key = reinterpret_cast<unsigned long long*>(S.fs);  // free now
        int* dep = S.out_par;                                                  // free until step 4
        for (int i = tid; i < n_sel; i += kThreads) {
            if (packed) key[i] = rank_key(S, i, bits);
            dep[i] = selc(S, i).depth;
        }
        __syncthreads();
        for (int i = tid; i < n_sel; i += kThreads) {
            const int di = dep[i];
            const unsigned long long ki = packed ? key[i] : 0ull;
            int r = 1;
            if (packed) {
                // every thread reads the same j: broadcast loads, no branches
#pragma unroll 8
                for (int j = 0; j < n_sel; ++j) {
                    const int dj = dep[j];
                    r += (dj < di) | ((dj == di) & (key[j] < ki));
                }
                S.new_idx[i] = r;
                continue;
            }
            for (int j = 0; j < n_sel; ++j) {
                const int dj = dep[j];
                if (dj < di) {
                    ++r;
                } else if (dj == di && j != i) {
                    {
                        int a = i, c = j;
                        while (selc(S, a).parent != selc(S, c).parent) {
                            a = selc(S, a).parent;
                            c = selc(S, c).parent;
                        }
                        r += selc(S, c).rank < selc(S, a).rank;
                    }
                }
            }
            S.new_idx[i] = r;
        }
    }
    __syncthreads();

    // 4. flattened outputs
    const long ob = (long)b * N;
    for (int r = tid; r < N; r += kThreads) S.out_par[r] = -1;
    __syncthreads();
    for (int i = tid; i < n_sel; i += kThreads) {
        const Cand& c = selc(S, i);
        const int r = S.new_idx[i];
        S.out_par[r] = c.parent < 0 ? 0 : S.new_idx[c.parent];
        token[ob + r] = cand_token(S, k, c);
        parent[ob + r] = S.out_par[r];
        depth[ob + r] = c.depth;
        position[ob + r] = prefix_len[b] + c.depth;
        if (score) score[ob + r] = c.L - S.cum[c.depth];  // the same fp64 expression it was ranked by
    }
    for (int r = n_sel + 1 + tid; r < N; r += kThreads) {
        token[ob + r] = -1;
        parent[ob + r] = -1;
        depth[ob + r] = -1;
        position[ob + r] = -1;
        if (score) score[ob + r] = -INFINITY;
    }
    if (tid == 0) {
        token[ob] = root_token[b];
        parent[ob] = -1;
        depth[ob] = 0;
        position[ob] = prefix_len[b];
        if (score) score[ob] = 0.0;
        n_nodes[b] = n_sel + 1;
        status[b] = bad ? DDT_ERR_NONFINITE : DDT_OK;
    }
    __syncthreads();
    // ancestor-or-self mask, one row per thread and word
    for (int e = tid; e < N * W; e += kThreads) {
        const int r = e / W, w = e % W;
        uint32_t bits = 0;
        if (r <= n_sel) {
            for (int a = r; a >= 0; a = (a == 0) ? -1 : S.out_par[a])
                if (a / 32 == w) bits |= 1u << (a % 32);
        }
        anc[(ob + r) * W + w] = bits;
    }
}

size_t build_tree_smem(int D, int k, int budget) {
    const int N = budget + 1;
    size_t b = sizeof(double) * (kMaxDepth + 1) + 2 * sizeof(long long) * (budget + 2) +
               sizeof(Cand) * (2 * budget + 1) + sizeof(double) * D * k + sizeof(float) * D * k +
               2 * sizeof(int) * D * k + sizeof(int) * (budget + 2) + sizeof(int) * (budget + 1) +
               sizeof(int) * (budget + 1) + sizeof(int) * N;
    return (b + 15) & ~(size_t)15;
}

cudaError_t launch_build_tree(int B, int D, int V, int k, int budget, ddt_dtype dtype, const void* logits,
                              const int32_t* root_token, const int32_t* prefix_len, int32_t* token,
                              int32_t* parent, int32_t* depth, int32_t* position, int32_t* n_nodes,
                              uint32_t* anc, double* score, int32_t* status, void* ws, cudaStream_t st) {
    const long nrows = (long)B * D;
    unsigned char* w = static_cast<unsigned char*>(ws);
    BuildRow* rows = reinterpret_cast<BuildRow*>(w);
    float* tv = reinterpret_cast<float*>(w + nrows * sizeof(BuildRow));
    int* ti = reinterpret_cast<int*>(w + nrows * sizeof(BuildRow) + nrows * k * sizeof(float));
    if (B > 65535) return cudaErrorInvalidValue;
    const dim3 g1(D, B);
    const int vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    if (dtype == DDT_BF16)
        k_build_row<__nv_bfloat16><<<counted(g1), kRowThreads, 0, st>>>(static_cast<const __nv_bfloat16*>(logits), D, V,
                                                                          k, vec, rows, tv, ti);
    else
        k_build_row<float><<<counted(g1), kRowThreads, 0, st>>>(static_cast<const float*>(logits), D, V, k, vec, rows,
                                                                  tv, ti);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t sm = build_tree_smem(D, k, budget);
    if (sm > 48 * 1024) {
        e = cudaFuncSetAttribute(k_build_tree<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
    }
    k_build_tree<512><<<counted(B), 512, sm, st>>>(D, k, budget, rows, tv, ti, root_token, prefix_len, token, parent,
                                                   depth, position, n_nodes, anc, score, status);
    return cudaGetLastError();
}

}  // namespace ddt

// ---------------------------------------------------------------------------------
// ddt_build_tree_noalloc: the same tree build for callers that cannot allocate device
// memory.  Some hosts of this library have no device allocator of their own (a plain C
// program, or a plugin living inside a process whose GPU memory is owned by another
// runtime), and some must not call cudaMalloc/cudaFree in their decode loop because
// those calls synchronise the device.  For them the build's per-row results (the
// log-sum-exp and top-k list of every depth row) live in one file-scope device array
// instead of a caller-supplied workspace.
//
// The array is a fixed kStaticScratchBytes (4 MiB) on every GPU that loads this library,
// held until the process exits.  Its device address is looked up with
// cudaGetSymbolAddress (on the host the symbol is only a stand-in, never a device
// pointer) once per device and context: the address is cached with the id of the CUDA
// context it was looked up in, and looked up again when the device's current context is
// another one (after cudaDeviceReset, or once the primary context was released and made
// again, the old address would point into an unloaded module).  The first call in each
// context does that lookup, so make it before any stream capture.  All calls on a device
// share the array: calls whose kernels overlap on the GPU (different streams, or
// different host threads without ordering) race on it and must be serialised by the
// caller.  The partial kernel writes every record the tree kernel reads, so nothing in
// the array has to start at zero.
namespace ddt {
namespace {
constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;
__device__ __align__(256) unsigned char g_build_scratch[kStaticScratchBytes];
struct ScratchAddr {
    unsigned long long ctx_id;  // 0: not looked up yet
    void* ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Id of the calling thread's current CUDA context (0 if none, or if the driver cannot
// tell); ids are never reused within a process, unlike context handles.
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_cur || !get_id || get_cur(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_build_scratch in the current device's current context.
cudaError_t static_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    const unsigned long long id = current_ctx_id();
    ScratchAddr& c = g_scratch_addr[dev];
    if (id == 0 || c.ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_build_scratch);  // makes the primary context current if none is
        if (e != cudaSuccess) return e;
        c.ptr = p;
        c.ctx_id = current_ctx_id();  // 0 when the driver cannot tell: look up again next time
    }
    *out = c.ptr;
    return cudaSuccess;
}
}  // namespace

}  // namespace ddt

extern "C" ddt_status ddt_build_tree_noalloc(int B, int D, int V, int top_k, int budget, ddt_dtype dtype,
                                             const void* draft_logits, const int32_t* root_token,
                                             const int32_t* prefix_len, int32_t* token, int32_t* parent,
                                             int32_t* depth, int32_t* position, int32_t* n_nodes, uint32_t* anc,
                                             double* score, int32_t* status, ddt_stream_t stream) {
    using namespace ddt;
    if (B < 1 || D < 1 || V < 1 || top_k < 1 || budget < 0 || (dtype != DDT_F32 && dtype != DDT_BF16))
        return DDT_ERR_INVALID_ARG;
    if (D > kMaxDepth || top_k > kMaxTopK || top_k > V || budget > kMaxBudget) return DDT_ERR_UNSUPPORTED;
    if (!draft_logits || !root_token || !prefix_len || !token || !parent || !depth || !position || !n_nodes || !anc ||
        !status)
        return DDT_ERR_INVALID_ARG;
    // the per-row results of this call must fit the static array
    if (build_ws_bytes(B, D, V, top_k) > kStaticScratchBytes) return DDT_ERR_CAPACITY;
    if (build_tree_smem(D, top_k, budget) > 200 * 1024) return DDT_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (static_scratch(&scratch) != cudaSuccess) return DDT_ERR_CUDA;
    const cudaError_t e = launch_build_tree(B, D, V, top_k, budget, dtype, draft_logits, root_token, prefix_len, token,
                                           parent, depth, position, n_nodes, anc, score, status, scratch,
                                           reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return DDT_OK;
    return e == cudaErrorInvalidValue ? DDT_ERR_UNSUPPORTED : DDT_ERR_CUDA;
}

