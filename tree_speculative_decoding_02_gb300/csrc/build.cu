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
//   k_build_partial  grid (chunks, D, B): one HBM pass over the logits.  Each CTA
//                    reduces one 8192-token chunk of one depth row to (max, sum of
//                    exp(v - max), top-k list): a threshold from the lane bests, one
//                    bitonic sort per warp, bitonic merges of the warp lists.
//   k_build_tree     grid B: per request, warp-per-depth merge of the chunk partials
//                    (LSE and top-k), then one warp runs the best-first selection over a
//                    shared-memory frontier, then the CTA renumbers breadth first and
//                    writes the flattened tree and its bit-packed ancestor mask.
#include <cuda.h>
#include <float.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace ddt {

// ------------------------------------------------------------------------------ partial
struct BuildPartial {
    float m;        // chunk max
    int nonfinite;  // 1 if the chunk holds NaN/Inf
    double s;       // sum over the chunk of exp(v - m)
};

size_t build_ws_bytes(int B, int D, int V, int k) {
    const long nch = (V + kBuildChunk - 1) / kBuildChunk;
    const long parts = (long)B * D * nch;
    size_t bytes = parts * sizeof(BuildPartial);
    bytes += parts * k * (sizeof(float) + sizeof(int));
    return (bytes + 255) & ~(size_t)255;
}

template <typename T>
__global__ void __launch_bounds__(256, 4) k_build_partial(const T* __restrict__ logits, int D, int V, int k,
                                                        int nch, int vec, BuildPartial* __restrict__ part,
                                                        float* __restrict__ pv, int* __restrict__ pid) {
    constexpr int kPer = kBuildChunk / 256;  // elements per thread (32)
    const int c = blockIdx.x, d = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long row = ((long)b * D + d) * V;
    const int start = c * kBuildChunk;
    const int len = min(kBuildChunk, V - start);

    float v[kPer];
    int bad = 0;
    if (vec) {
        // 8-wide vector loads: thread t covers elements [t*8 + j*2048, +8)
#pragma unroll
        for (int j = 0; j < kPer / 8; ++j) {
            const int e = tid * 8 + j * 2048;
            float t8[8];
            if (e + 8 <= len) {
                load8_stream(logits + row + start + e, t8);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) t8[u] = (e + u < len) ? to_f32(logits[row + start + e + u]) : vid_empty().v;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) v[j * 8 + u] = t8[u];
        }
    } else {
#pragma unroll
        for (int j = 0; j < kPer / 8; ++j)
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = tid * 8 + j * 2048 + u;
                v[j * 8 + u] = (e < len) ? to_f32(logits[row + start + e]) : vid_empty().v;
            }
    }
#pragma unroll
    for (int j = 0; j < kPer / 8; ++j)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = tid * 8 + j * 2048 + u;
            if (e < len && !finite_f32(v[j * 8 + u])) bad = 1;
        }

    // warp top-k.  The k-th best of the 32 lane bests is beaten or equalled by at least k
    // entries, so every entry of the warp's top k is at or above it: only those entries
    // are kept.  When at most 32 qualify (the usual case) they are sorted in one bitonic
    // pass; otherwise they are inserted one at a time.
    __shared__ float s_v[8][32];
    __shared__ int s_id[8][32];
    __shared__ float s_max[8];
    __shared__ double s_sum[8];
    __shared__ int s_bad[8];
    const VId emp = vid_empty();
    float bv = emp.v;
    int bid = emp.id;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = tid * 8 + (j >> 3) * 2048 + (j & 7);
        if (e < len && beats(v[j], start + e, bv, bid)) {
            bv = v[j];
            bid = start + e;
        }
    }
    warp_sort_best_first(bv, bid);
    const float thv = __shfl_sync(kFull, bv, k - 1);
    const int thid = __shfl_sync(kFull, bid, k - 1);
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = tid * 8 + (j >> 3) * 2048 + (j & 7);
        cnt += (e < len && !beats(thv, thid, v[j], start + e)) ? 1 : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += nb;
    }
    const int total = __shfl_sync(kFull, incl, 31);
    float wv;
    int wid;
    if (total <= 32) {
        int pos = incl - cnt;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int e = tid * 8 + (j >> 3) * 2048 + (j & 7);
            if (e < len && !beats(thv, thid, v[j], start + e)) {
                s_v[warp][pos] = v[j];
                s_id[warp][pos] = start + e;
                ++pos;
            }
        }
        __syncwarp();
        wv = lane < total ? s_v[warp][lane] : emp.v;
        wid = lane < total ? s_id[warp][lane] : emp.id;
        warp_sort_best_first(wv, wid);
    } else {
        WarpTopK tk;
        tk.init(k);
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int e = tid * 8 + (j >> 3) * 2048 + (j & 7);
            const bool q = e < len && !beats(thv, thid, v[j], start + e);
            if (__any_sync(kFull, q)) tk.insert(q ? v[j] : emp.v, q ? start + e : emp.id);
        }
        wv = tk.v;
        wid = tk.id;
    }
    if (lane >= k) {
        wv = emp.v;
        wid = emp.id;
    }
    __syncwarp();
    s_v[warp][lane] = wv;
    s_id[warp][lane] = wid;
    const float wmax = __shfl_sync(kFull, wv, 0);
    if (lane == 0) s_max[warp] = wmax;
    const int wbad = __any_sync(kFull, bad);
    if (lane == 0) s_bad[warp] = wbad;
    __syncthreads();
    float m = s_max[0];
    int anybad = s_bad[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
        m = fmaxf(m, s_max[w]);
        anybad |= s_bad[w];
    }

    // sum of exp(v - m): fp32 over the thread's 32 terms, fp64 across threads
    const float LOG2E = 1.4426950408889634f;
    const float mb = m * LOG2E;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = tid * 8 + (j >> 3) * 2048 + (j & 7);
        if (e < len) acc += exp2f(fmaf(v[j], LOG2E, -mb));
    }
    double dacc = warp_sum((double)acc);
    if (lane == 0) s_sum[warp] = dacc;

    // merge the eight warp lists in warp 0
    __syncthreads();
    if (warp == 0) {
        float fv = s_v[0][lane];
        int fid = s_id[0][lane];
        for (int w = 1; w < 8; ++w) warp_merge_best_first(fv, fid, s_v[w][lane], s_id[w][lane]);
        const long p = ((long)b * D + d) * nch + c;
        if (lane < k) {
            pv[p * k + lane] = fv;
            pid[p * k + lane] = fid;
        }
        if (lane == 0) {
            double tot = 0.0;
            for (int w = 0; w < 8; ++w) tot += s_sum[w];
            part[p].m = m;
            part[p].nonfinite = anybad;
            part[p].s = tot;
        }
    }
}

// ---------------------------------------------------------------------- selection
struct Cand {
    double L;   // sum of path logits, depth 1 first
    double s;   // L - cum LSE of its depth
    int depth;  // 1..D
    int rank;   // within the depth's top-k
    int parent; // index into the selected list, -1 = root
    int pad;
};

struct TreeSmem {
    // per depth
    float* top_v;   // [D][k]
    int* top_id;    // [D][k]
    double* cum;    // [D+1] cumulative LSE, cum[0] = 0
    // selection
    Cand* sel;      // [budget]
    Cand* front;    // [budget + 2]
    int* new_idx;   // [budget]
    int* out_par;   // [N]
    int* depth_cnt; // [D + 2]
};

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
        const Cand& u = S.sel[pa];
        ta = cand_token(S, k, u);
        pa = u.parent;
        --da;
    }
    if (a.depth > b.depth && pa == pb && ta == tb) return false;  // b is a prefix of a
    while (db > da) {
        const Cand& u = S.sel[pb];
        tb = cand_token(S, k, u);
        pb = u.parent;
        --db;
    }
    if (b.depth > a.depth && pa == pb && ta == tb) return true;   // a is a proper prefix of b
    while (pa != pb) {
        const Cand& u = S.sel[pa];
        const Cand& v = S.sel[pb];
        ta = cand_token(S, k, u);
        tb = cand_token(S, k, v);
        pa = u.parent;
        pb = v.parent;
    }
    return ta < tb;
}

__device__ __forceinline__ bool cand_better(const TreeSmem& S, int k, const Cand& a, const Cand& b) {
    if (a.s != b.s) return a.s > b.s;
    return lex_less(S, k, a, b);
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) k_build_tree(int D, int V, int k, int budget, int nch,
                                                          const BuildPartial* __restrict__ part,
                                                          const float* __restrict__ pv,
                                                          const int* __restrict__ pid,
                                                          const int32_t* __restrict__ root_token,
                                                          const int32_t* __restrict__ prefix_len,
                                                          int32_t* __restrict__ token, int32_t* __restrict__ parent,
                                                          int32_t* __restrict__ depth, int32_t* __restrict__ position,
                                                          int32_t* __restrict__ n_nodes, uint32_t* __restrict__ anc,
                                                          double* __restrict__ score, int32_t* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kThreads / 32;
    const int N = budget + 1;
    const int W = (N + 31) / 32;

    TreeSmem S;
    unsigned char* p = smem_raw;
    S.cum = reinterpret_cast<double*>(p);      p += sizeof(double) * (kMaxDepth + 1);
    S.sel = reinterpret_cast<Cand*>(p);        p += sizeof(Cand) * (budget + 1);
    S.front = reinterpret_cast<Cand*>(p);      p += sizeof(Cand) * (budget + 2);
    S.top_v = reinterpret_cast<float*>(p);     p += sizeof(float) * D * k;
    S.top_id = reinterpret_cast<int*>(p);      p += sizeof(int) * D * k;
    S.new_idx = reinterpret_cast<int*>(p);     p += sizeof(int) * (budget + 1);
    S.out_par = reinterpret_cast<int*>(p);     p += sizeof(int) * N;
    S.depth_cnt = reinterpret_cast<int*>(p);   p += sizeof(int) * (kMaxDepth + 2);
    __shared__ double s_lse[kMaxDepth];
    __shared__ int s_bad;
    __shared__ int s_nsel;

    if (tid == 0) s_bad = 0;
    __syncthreads();

    // 1. per depth: merge the chunk partials into LSE and the depth's top-k
    for (int d = warp; d < D; d += kWarps) {
        const long base = ((long)b * D + d) * nch;
        float M = vid_empty().v;
        int bad = 0;
        for (int c = lane; c < nch; c += 32) {
            M = fmaxf(M, part[base + c].m);
            bad |= part[base + c].nonfinite;
        }
        M = warp_max(M);
        bad = warp_or(bad);
        double sum = 0.0;
        for (int c = lane; c < nch; c += 32) sum += part[base + c].s * exp((double)part[base + c].m - (double)M);
        sum = warp_sum(sum);
        WarpTopK tk;
        tk.init(k);
        for (int c0 = 0; c0 < nch * k; c0 += 32) {
            const int e = c0 + lane;
            const bool ok = e < nch * k;
            tk.insert(ok ? pv[base * k + e] : vid_empty().v, ok ? pid[base * k + e] : 0x7fffffff);
        }
        if (lane < k) {
            S.top_v[d * k + lane] = tk.v;
            S.top_id[d * k + lane] = tk.id;
        }
        if (lane == 0) {
            s_lse[d] = (double)M + log(sum);
            if (bad || !isfinite(s_lse[d])) atomicOr(&s_bad, 1);
        }
    }
    __syncthreads();
    const bool bad = s_bad != 0;
    if (tid == 0) {
        double c = 0.0;
        S.cum[0] = 0.0;
        for (int d = 0; d < D; ++d) {
            c += s_lse[d];
            S.cum[d + 1] = c;
        }
    }
    __syncthreads();

    // 2. best-first selection (one warp; the frontier lives in shared memory)
    if (warp == 0) {
        int n_sel = 0, n_front = 0;
        if (budget > 0 && !bad) {
            if (lane == 0) {
                Cand c0;
                c0.depth = 1;
                c0.rank = 0;
                c0.parent = -1;
                c0.L = 0.0 + (double)S.top_v[0];
                c0.s = c0.L - S.cum[1];
                S.front[0] = c0;
            }
            n_front = 1;
        }
        __syncwarp();
        while (n_sel < budget && n_front > 0) {
            int best = -1;
            for (int i = lane; i < n_front; i += 32)
                if (best < 0 || cand_better(S, k, S.front[i], S.front[best])) best = i;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                // lanes that already agree skip the compare: on equal scores it walks both
                // token paths, which for an entry against itself is the whole path
                const int other = __shfl_xor_sync(kFull, best, o);
                if (other >= 0 && other != best && (best < 0 || cand_better(S, k, S.front[other], S.front[best])))
                    best = other;
            }
            best = __shfl_sync(kFull, best, 0);
            int nf = 0;
            if (lane == 0) {
                const Cand c = S.front[best];
                S.front[best] = S.front[n_front - 1];
                nf = n_front - 1;
                const int me = n_sel;
                S.sel[me] = c;
                const double L_par = (c.parent < 0) ? 0.0 : S.sel[c.parent].L;
                if (c.rank + 1 < k) {  // next-ranked sibling: same parent, same depth
                    Cand sib = c;
                    sib.rank = c.rank + 1;
                    sib.L = L_par + (double)S.top_v[(c.depth - 1) * k + sib.rank];
                    sib.s = sib.L - S.cum[c.depth];
                    S.front[nf++] = sib;
                }
                if (c.depth < D) {  // best child
                    Cand ch;
                    ch.depth = c.depth + 1;
                    ch.rank = 0;
                    ch.parent = me;
                    ch.L = c.L + (double)S.top_v[c.depth * k];
                    ch.s = ch.L - S.cum[c.depth + 1];
                    S.front[nf++] = ch;
                }
            }
            n_front = __shfl_sync(kFull, nf, 0);
            ++n_sel;
            __syncwarp();
        }
        if (lane == 0) s_nsel = n_sel;
    }
    __syncthreads();
    const int n_sel = s_nsel;

    // 3. canonical breadth-first numbering: depth, then parent's new row, then rank
    for (int i = tid; i < kMaxDepth + 2; i += kThreads) S.depth_cnt[i] = 0;
    __syncthreads();
    for (int i = tid; i < n_sel; i += kThreads) atomicAdd(&S.depth_cnt[S.sel[i].depth], 1);
    __syncthreads();
    int base = 1;
    for (int dd = 1; dd <= D; ++dd) {
        const int cnt = S.depth_cnt[dd];
        if (cnt == 0) break;
        for (int i = tid; i < n_sel; i += kThreads) {
            const Cand& ci = S.sel[i];
            if (ci.depth != dd) continue;
            const int pi = ci.parent < 0 ? 0 : S.new_idx[ci.parent];
            int r = 0;
            for (int j = 0; j < n_sel; ++j) {
                const Cand& cj = S.sel[j];
                if (cj.depth != dd) continue;
                const int pj = cj.parent < 0 ? 0 : S.new_idx[cj.parent];
                r += (pj < pi) || (pj == pi && cj.rank < ci.rank);
            }
            S.new_idx[i] = base + r;
        }
        base += cnt;
        __syncthreads();
    }

    // 4. flattened outputs
    const long ob = (long)b * N;
    for (int r = tid; r < N; r += kThreads) S.out_par[r] = -1;
    __syncthreads();
    for (int i = tid; i < n_sel; i += kThreads) {
        const Cand& c = S.sel[i];
        const int r = S.new_idx[i];
        S.out_par[r] = c.parent < 0 ? 0 : S.new_idx[c.parent];
        token[ob + r] = cand_token(S, k, c);
        parent[ob + r] = S.out_par[r];
        depth[ob + r] = c.depth;
        position[ob + r] = prefix_len[b] + c.depth;
        if (score) score[ob + r] = c.s;
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
    size_t b = sizeof(double) * (kMaxDepth + 1) + sizeof(Cand) * (budget + 1) + sizeof(Cand) * (budget + 2) +
               sizeof(float) * D * k + sizeof(int) * D * k + sizeof(int) * (budget + 1) + sizeof(int) * N +
               sizeof(int) * (kMaxDepth + 2);
    return (b + 15) & ~(size_t)15;
}

cudaError_t launch_build_tree(int B, int D, int V, int k, int budget, ddt_dtype dtype, const void* logits,
                              const int32_t* root_token, const int32_t* prefix_len, int32_t* token,
                              int32_t* parent, int32_t* depth, int32_t* position, int32_t* n_nodes,
                              uint32_t* anc, double* score, int32_t* status, void* ws, cudaStream_t st) {
    const int nch = (V + kBuildChunk - 1) / kBuildChunk;
    const long parts = (long)B * D * nch;
    unsigned char* w = static_cast<unsigned char*>(ws);
    BuildPartial* part = reinterpret_cast<BuildPartial*>(w);
    float* pv = reinterpret_cast<float*>(w + parts * sizeof(BuildPartial));
    int* pid = reinterpret_cast<int*>(w + parts * sizeof(BuildPartial) + parts * k * sizeof(float));
    dim3 g1(nch, D, B);
    const int vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    if (dtype == DDT_BF16)
        k_build_partial<__nv_bfloat16><<<counted(g1), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(logits), D, V, k, nch,
                                                          vec, part, pv, pid);
    else
        k_build_partial<float><<<counted(g1), 256, 0, st>>>(static_cast<const float*>(logits), D, V, k, nch, vec, part, pv,
                                                  pid);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t sm = build_tree_smem(D, k, budget);
    if (sm > 48 * 1024) {
        e = cudaFuncSetAttribute(k_build_tree<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
    }
    k_build_tree<512><<<counted(B), 512, sm, st>>>(D, V, k, budget, nch, part, pv, pid, root_token, prefix_len, token,
                                          parent, depth, position, n_nodes, anc, score, status);
    return cudaGetLastError();
}

}  // namespace ddt

// ---------------------------------------------------------------------------------
// ddt_build_tree_noalloc: the same tree build for callers that cannot allocate device
// memory.  Some hosts of this library have no device allocator of their own (a plain C
// program, or a plugin living inside a process whose GPU memory is owned by another
// runtime), and some must not call cudaMalloc/cudaFree in their decode loop because
// those calls synchronise the device.  For them the build's per-chunk partials live in
// one file-scope device array instead of a caller-supplied workspace.
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
    // the partials of this call must fit the static array
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

