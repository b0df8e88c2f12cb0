// walk_sample.cu -- ddt_walk_accept_sample: tree-walk rejection sampling.
//
// "The Moment of Truth: Validating DDTree Speculative Decoding on Qwen3.6-27B", section
// "The Path to This Message": the serving stack's sampler is a linear-chain rejection
// sampler, and verifying a tree at a temperature needs a walk of its own.  The pages give
// no algorithm; the rule used is speculative sampling's (Leviathan, Kalman and Matias,
// ICML 2023; Chen et al., 2023) over each visited node's children, whose draft is a point
// mass (SpecInfer, Miao et al., ASPLOS 2024):
//   p_u = softmax(logits[u] / T); children tried in row order; R = mass of the children
//   already rejected; child i is accepted iff U[step][i] < p_u(x_i) / (1 - R); when none
//   is, the bonus is the smallest id whose running sum of p_u (rejected ids skipped)
//   exceeds U[step][C] * (1 - R).
//
//   k_walk_lse     grid (chunks, N, B): one HBM pass over the target logits; each CTA
//                  reduces a 16384-token chunk of one row to its max m_c and
//                  sum_v exp((l_v - m_c) / T) (fp32 terms in groups of 8, fp64 across
//                  threads).
//   k_walk_sample  grid B: tree checks; warp 0 walks down, merging the visited row's
//                  chunk partials and deciding each tried child in fp64; then the CTA
//                  draws the bonus: a warp scan of the residual chunk masses picks the
//                  chunk, a block scan over that chunk's 16384 terms picks the token.
#include "common.cuh"
#include "kernels.h"

namespace ddt {

constexpr int kSampleChunk = 16384;                         // vocabulary entries a k_walk_lse CTA reduces
constexpr int kSampleThreads = 256;
constexpr int kSamplePer = kSampleChunk / kSampleThreads;  // 64 entries a thread

struct LsePartial {
    float m;        // largest raw logit of the chunk
    int nonfinite;  // a NaN or +-inf logit in the chunk
    double s;       // sum over the chunk of exp((l - m) * inv_t)
};

size_t walk_sample_ws_bytes(int B, int N, int V) {
    const long nch = (V + kSampleChunk - 1) / kSampleChunk;
    return (((size_t)B * N * nch * sizeof(LsePartial)) + 255) & ~(size_t)255;
}

// One tempered term: exp((l - m) / T) with the division taken as a product by the fp32
// reciprocal inv_t.  -inf (an entry past the row's end) gives 0.
__device__ __forceinline__ float tempered(float l, float m, float inv_t) { return expf((l - m) * inv_t); }

template <typename T>
__global__ void __launch_bounds__(kSampleThreads) k_walk_lse(const T* __restrict__ logits, int N, int V, int nch,
                                                             int vec, float inv_t,
                                                             const int32_t* __restrict__ n_nodes,
                                                             LsePartial* __restrict__ part) {
    const int c = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
    const int nn = n_nodes[b];
    if (i >= nn || nn > N) return;  // rows past the tree are not needed
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T* row = logits + ((long)b * N + i) * V + (long)c * kSampleChunk;
    const int len = min(kSampleChunk, V - c * kSampleChunk);
    float x[kSamplePer];
    float mx = -INFINITY;
    int bad = 0;
#pragma unroll
    for (int j = 0; j < kSamplePer / 8; ++j) {
        const int e = tid * 8 + j * (kSampleThreads * 8);
        float t8[8];
        if (vec && e + 8 <= len) {
            load8_stream(row + e, t8);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) t8[u] = (e + u < len) ? to_f32(row[e + u]) : -INFINITY;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            x[j * 8 + u] = t8[u];
            if (e + u < len) {
                if (!finite_f32(t8[u])) bad = 1;
                mx = fmaxf(mx, t8[u]);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    bad = __any_sync(kFull, bad);
    __shared__ float s_mx[kSampleThreads / 32];
    __shared__ int s_bad[kSampleThreads / 32];
    __shared__ double s_sum[kSampleThreads / 32];
    if (lane == 0) {
        s_mx[warp] = mx;
        s_bad[warp] = bad;
    }
    __syncthreads();
    float m = s_mx[0];
#pragma unroll
    for (int w = 1; w < kSampleThreads / 32; ++w) m = fmaxf(m, s_mx[w]);
    float g[kSamplePer / 8];
#pragma unroll
    for (int j = 0; j < kSamplePer / 8; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += tempered(x[j * 8 + u], m, inv_t);
        g[j] = acc;
    }
    double ds = (double)(((g[0] + g[1]) + (g[2] + g[3])) + ((g[4] + g[5]) + (g[6] + g[7])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ds += __shfl_down_sync(kFull, ds, o);
    if (lane == 0) s_sum[warp] = ds;
    __syncthreads();
    if (tid == 0) {
        double s = 0.0;
        int anybad = 0;
        for (int w = 0; w < kSampleThreads / 32; ++w) {
            s += s_sum[w];
            anybad |= s_bad[w];
        }
        LsePartial pp;
        pp.m = m;
        pp.nonfinite = anybad;
        pp.s = s;
        part[((long)b * N + i) * nch + c] = pp;
    }
}

// Warp-wide: the row's max and Z = sum_v exp((l_v - m) / T) from its chunk partials.  Every
// lane returns lane 0's values, so decisions taken on them are uniform across the warp.
__device__ __forceinline__ void row_stats(const LsePartial* __restrict__ P, int nch, float inv_t, int lane, float& m,
                                          double& z) {
    float mm = -INFINITY;
    for (int c = lane; c < nch; c += 32) mm = fmaxf(mm, P[c].m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, o));
    double zz = 0.0;
    for (int c = lane; c < nch; c += 32) zz += P[c].s * (double)tempered(P[c].m, mm, inv_t);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zz += __shfl_down_sync(kFull, zz, o);
    m = mm;
    z = __shfl_sync(kFull, zz, 0);
}

template <typename T>
__global__ void __launch_bounds__(kSampleThreads) k_walk_sample(
    const T* __restrict__ logits, int N, int V, int A, int C, int nch, int vec, float inv_t,
    const LsePartial* __restrict__ part, const float* __restrict__ uniforms, const int32_t* __restrict__ token,
    const int32_t* __restrict__ parent, const int32_t* __restrict__ n_nodes, int32_t* __restrict__ acc_nodes,
    int32_t* __restrict__ acc_len, int32_t* __restrict__ bonus, int32_t* __restrict__ emitted,
    int32_t* __restrict__ n_emitted, int32_t* __restrict__ status) {
    __shared__ int s_tok[kMaxRows], s_par[kMaxRows], s_cnt[kMaxRows];
    __shared__ float s_lc[kMaxRows];  // logit of node i's token in its parent's row
    __shared__ double s_incl[kSampleThreads];
    __shared__ double s_wsum[kSampleThreads / 32];
    __shared__ uint32_t s_rejbits[kSampleChunk / 32];
    __shared__ int s_rejtok[kMaxTopK];
    __shared__ float s_rejterm[kMaxTopK];
    __shared__ int s_path[kMaxAccept + 1];
    __shared__ int s_err, s_cur, s_a, s_nrej, s_chunk, s_pick, s_last, s_bonus;
    __shared__ float s_m;
    __shared__ double s_local;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nn = n_nodes[b];
    const long ob = (long)b * N;
    int32_t* an = acc_nodes + (long)b * A;
    int32_t* em = emitted + (long)b * A;
    // every thread takes this branch on its own copy of n_nodes: s_err changes inside it
    const bool nn_ok = nn >= 1 && nn <= N;
    if (tid == 0) s_err = nn_ok ? DDT_OK : DDT_ERR_TREE;
    __syncthreads();
    if (nn_ok) {
        for (int i = tid; i < nn; i += kSampleThreads) {
            s_tok[i] = token[ob + i];
            s_par[i] = parent[ob + i];
            s_cnt[i] = 0;
        }
        __syncthreads();
        // the tree: parents before children, tokens in range, distinct sibling tokens,
        // at most C children a node; each node's token logit in its parent's row
        for (int i = tid; i < nn; i += kSampleThreads) {
            const int p = s_par[i], t = s_tok[i];
            const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i && t >= 0 && t < V);
            if (!ok) {
                atomicMax(&s_err, DDT_ERR_TREE);
                continue;
            }
            if (i == 0) continue;
            atomicAdd(&s_cnt[p], 1);
            s_lc[i] = to_f32(logits[(ob + p) * V + t]);
            for (int j = 1; j < i; ++j)
                if (s_par[j] == p && s_tok[j] == t) {
                    atomicMax(&s_err, DDT_ERR_TREE);
                    break;
                }
        }
        for (int j = tid; j < nn * nch; j += kSampleThreads)
            if (part[ob * nch + j].nonfinite) atomicMax(&s_err, DDT_ERR_NONFINITE);  // a tree error outranks it
        __syncthreads();
        for (int i = tid; i < nn; i += kSampleThreads)
            if (s_cnt[i] > C) atomicMax(&s_err, DDT_ERR_TREE);
        __syncthreads();
    }
    if (s_err != DDT_OK) {
        for (int j = tid; j < A; j += kSampleThreads) {
            an[j] = -1;
            em[j] = -1;
        }
        if (tid == 0) {
            acc_len[b] = 0;
            bonus[b] = -1;
            n_emitted[b] = 0;
            status[b] = s_err;
        }
        return;
    }

    // ---- the walk (warp 0): one uniform per tried child, decisions in fp64
    if (warp == 0) {
        int cur = 0, a = 0, nrej = 0;
        float m = 0.f;
        double zr = 0.0;
        if (lane == 0) s_path[0] = 0;
        for (;;) {
            row_stats(part + (ob + cur) * nch, nch, inv_t, lane, m, zr);
            const float* U = uniforms + ((long)b * A + a) * (C + 1);
            nrej = 0;
            int next = -1;
            if (a + 1 < A) {
                for (int base = 1; base < nn && next < 0; base += 32) {
                    const int c = base + lane;
                    unsigned mask = __ballot_sync(kFull, c < nn && s_par[c] == cur);
                    while (mask != 0u && next < 0) {
                        const int cc = base + __ffs(mask) - 1;
                        mask &= mask - 1u;
                        const float term = tempered(s_lc[cc], m, inv_t);
                        // p(x) / (1 - R) with both taken relative to Z: term / (Z - rejected terms)
                        if ((double)U[nrej] < (double)term / zr) {
                            next = cc;
                        } else {
                            if (lane == 0) {
                                s_rejtok[nrej] = s_tok[cc];
                                s_rejterm[nrej] = term;
                            }
                            zr -= (double)term;
                            ++nrej;
                        }
                    }
                }
            }
            if (next < 0) {
                if (lane == 0) {
                    s_cur = cur;
                    s_a = a;
                    s_nrej = nrej;
                    s_m = m;
                    s_local = (double)U[C] * zr;  // the bonus draw's target in units of the terms
                }
                break;
            }
            cur = next;
            ++a;
            if (lane == 0) s_path[a] = cur;
        }
    }
    __syncthreads();

    // ---- the bonus chunk (warp 0): residual chunk masses in id order, inclusive scan
    const int cur = s_cur, nrej = s_nrej;
    const float m = s_m;
    if (warp == 0) {
        const LsePartial* P = part + (ob + cur) * nch;
        const double target = s_local;
        double carry = 0.0;
        int pick = -1, last = -1;
        double before = 0.0;
        for (int base = 0; base < nch; base += 32) {
            const int c = base + lane;
            double mc = 0.0;
            if (c < nch) {
                mc = P[c].s * (double)tempered(P[c].m, m, inv_t);
                for (int r = 0; r < nrej; ++r)
                    if (s_rejtok[r] / kSampleChunk == c) mc -= (double)s_rejterm[r];
            }
            double incl = mc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            incl += carry;
            const unsigned over = __ballot_sync(kFull, c < nch && incl > target);
            const unsigned pos = __ballot_sync(kFull, c < nch && mc > 0.0);
            if (pick < 0 && over != 0u) {
                const int l = __ffs(over) - 1;
                pick = base + l;
                before = __shfl_sync(kFull, incl - mc, l);
            }
            if (pos != 0u) last = base + 31 - __clz(pos);
            carry = __shfl_sync(kFull, incl, 31);
        }
        if (lane == 0) {
            // rounding left the target past the residual mass: the last chunk that has some,
            // and in it the largest id with a positive term (an infinite local target)
            s_chunk = (pick >= 0) ? pick : last;
            s_local = (pick >= 0) ? target - before : INFINITY;
            s_pick = 0x7fffffff;
            s_last = -1;
        }
    }
    for (int j = tid; j < kSampleChunk / 32; j += kSampleThreads) s_rejbits[j] = 0u;
    __syncthreads();
    const int chunk = s_chunk;
    if (chunk >= 0) {
        const int start = chunk * kSampleChunk;
        if (tid < nrej) {
            const int t = s_rejtok[tid] - start;
            if (t >= 0 && t < kSampleChunk) atomicOr(&s_rejbits[t >> 5], 1u << (t & 31));
        }
        __syncthreads();
        // ---- the bonus token: block scan of this chunk's residual terms in id order
        const int len = min(kSampleChunk, V - start);
        const T* row = logits + (ob + cur) * V + start;
        const int e0 = tid * kSamplePer;
        float g[kSamplePer / 8];
        int lastpos = -1;
#pragma unroll
        for (int j = 0; j < kSamplePer / 8; ++j) {
            const int e = e0 + j * 8;
            float t8[8];
            if (vec && e + 8 <= len) {
                load8(row + e, t8);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) t8[u] = (e + u < len) ? to_f32(row[e + u]) : -INFINITY;
            }
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool rej = (s_rejbits[(e + u) >> 5] >> ((e + u) & 31)) & 1u;
                const float tv = (e + u < len && !rej) ? tempered(t8[u], m, inv_t) : 0.f;
                if (tv > 0.f) lastpos = e + u;
                acc += tv;
            }
            g[j] = acc;
        }
        double incl = (double)(((g[0] + g[1]) + (g[2] + g[3])) + ((g[4] + g[5]) + (g[6] + g[7])));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_wsum[warp] = incl;
        if (lastpos >= 0) atomicMax(&s_last, lastpos);
        __syncthreads();
        double wbefore = 0.0;
        for (int w = 0; w < warp; ++w) wbefore += s_wsum[w];
        incl += wbefore;
        s_incl[tid] = incl;
        const double target = s_local;
        if (incl > target) atomicMin(&s_pick, tid);
        __syncthreads();
        if (tid == s_pick) {
            // the smallest thread whose inclusive sum passes the target walks its own ids
            double run = (tid == 0) ? 0.0 : s_incl[tid - 1];
            int pickid = (lastpos >= 0) ? lastpos : s_last;  // if rounding runs the scan dry
            bool done = false;
            for (int j = 0; j < kSamplePer / 8 && !done; ++j) {
                if (run + (double)g[j] <= target) {
                    run += (double)g[j];
                    continue;
                }
                const int e = e0 + j * 8;
                for (int u = 0; u < 8 && !done; ++u) {
                    const bool rej = (s_rejbits[(e + u) >> 5] >> ((e + u) & 31)) & 1u;
                    if (e + u >= len || rej) continue;
                    run += (double)tempered(to_f32(row[e + u]), m, inv_t);
                    if (run > target) {
                        pickid = e + u;
                        done = true;
                    }
                }
            }
            s_bonus = (pickid >= 0) ? start + pickid : -1;
        }
        if (tid == 0 && s_pick == 0x7fffffff) s_bonus = (s_last >= 0) ? start + s_last : -1;
    } else if (tid == 0) {
        s_bonus = -1;  // no residual mass at all
    }
    __syncthreads();

    // ---- outputs: rows root..a, emitted = accepted tokens then the bonus
    const int a = s_a;
    for (int j = tid; j < A; j += kSampleThreads) {
        an[j] = (j <= a) ? s_path[j] : -1;
        em[j] = (j < a) ? s_tok[s_path[j + 1]] : ((j == a) ? s_bonus : -1);
    }
    if (tid == 0) {
        acc_len[b] = a;
        bonus[b] = s_bonus;
        n_emitted[b] = a + 1;
        status[b] = DDT_OK;
    }
}

cudaError_t launch_walk_sample(int B, int N, int V, int A, int C, float temperature, ddt_dtype dtype,
                               const void* logits, const float* uniforms, const int32_t* token,
                               const int32_t* parent, const int32_t* n_nodes, int32_t* acc_nodes, int32_t* acc_len,
                               int32_t* bonus, int32_t* emitted, int32_t* n_emitted, int32_t* status, void* ws,
                               cudaStream_t st) {
    const int nch = (V + kSampleChunk - 1) / kSampleChunk;
    const float inv_t = 1.0f / temperature;
    LsePartial* part = static_cast<LsePartial*>(ws);
    const int vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    dim3 g(nch, N, B);
    if (dtype == DDT_BF16) {
        const __nv_bfloat16* l = static_cast<const __nv_bfloat16*>(logits);
        k_walk_lse<__nv_bfloat16><<<counted(g), kSampleThreads, 0, st>>>(l, N, V, nch, vec, inv_t, n_nodes, part);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        k_walk_sample<__nv_bfloat16><<<counted(B), kSampleThreads, 0, st>>>(
            l, N, V, A, C, nch, vec, inv_t, part, uniforms, token, parent, n_nodes, acc_nodes, acc_len, bonus,
            emitted, n_emitted, status);
    } else {
        const float* l = static_cast<const float*>(logits);
        k_walk_lse<float><<<counted(g), kSampleThreads, 0, st>>>(l, N, V, nch, vec, inv_t, n_nodes, part);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        k_walk_sample<float><<<counted(B), kSampleThreads, 0, st>>>(l, N, V, A, C, nch, vec, inv_t, part, uniforms,
                                                                    token, parent, n_nodes, acc_nodes, acc_len,
                                                                    bonus, emitted, n_emitted, status);
    }
    return cudaGetLastError();
}

}  // namespace ddt
