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
//   k_walk_lse     grid (units / 8, N, B): one HBM pass over the target logits; each warp
//                  reduces a 2048-token unit of one row to its max m_u and
//                  sum_v 2^((l_v - m_u) * s2), s2 = log2(e) / T (fp32: groups of 8 terms,
//                  pairwise above them, a shuffle tree across the warp).  A full bf16 unit
//                  takes its max and its finiteness check two entries at a time on the
//                  packed pairs.  No block barrier and no fp64, so loads of the next warp's
//                  unit overlap this one's math.
//   k_walk_sample  grid B: tree checks; warp 0 walks down, merging the visited row's unit
//                  partials in fp64 and deciding each tried child in fp64; then the CTA
//                  draws the bonus: a warp scan of the residual unit masses picks the unit,
//                  a block scan over that unit's 2048 terms picks the token.
#include "common.cuh"
#include "kernels.h"

namespace ddt {

constexpr int kSampleUnit = 2048;                         // vocabulary entries one warp reduces
constexpr int kSampleThreads = 256;
constexpr int kUnitsPerCta = kSampleThreads / 32;
constexpr int kLanePer = kSampleUnit / 32;                // 64 entries a lane
constexpr int kScanPer = kSampleUnit / kSampleThreads;    // 8 entries a thread in the bonus scan

// One unit's partial: m = the largest raw logit, s = sum of 2^((l - m) * s2) over the
// unit; s = -1 flags a NaN or +-inf logit in it; an empty unit has m = -inf, s = 0.
struct LsePartial {
    float m;
    float s;
};

static inline int units_of(int V) { return (V + kSampleUnit - 1) / kSampleUnit; }

size_t walk_sample_ws_bytes(int B, int N, int V) {
    return (((size_t)B * N * units_of(V) * sizeof(LsePartial)) + 255) & ~(size_t)255;
}

// One tempered term: exp((l - m) / T) = 2^((l - m) * s2) with s2 = log2(e) / T rounded to
// fp32, by the hardware base-2 exponential (ex2.approx.ftz: relative error about 2^-22;
// terms below 2^-126 of the row's largest flush to zero).  -inf (an entry past the row's
// end, or the empty max) gives 0.  Every term of both kernels comes from this one function.
__device__ __forceinline__ float tempered(float l, float m, float s2) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"((l - m) * s2));
    return y;
}

// Eight consecutive entries kept in their storage format until used (bf16: one 16-byte
// word, so a lane holds its 64 entries in 32 registers); entries at or past `len` read
// as -inf.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
    uint4 w;
    __device__ __forceinline__ void load(const __nv_bfloat16* __restrict__ p, int e, int len, int vec) {
        if (vec && e + 8 <= len) {
            w = ld_stream_u4(p + e);
        } else {
            uint32_t h[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) h[q] = (e + q < len) ? (uint32_t)__bfloat16_as_ushort(p[e + q]) : 0xff80u;
            w = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
        }
    }
    __device__ __forceinline__ float at(int q) const {
        const uint32_t v = q < 2 ? w.x : (q < 4 ? w.y : (q < 6 ? w.z : w.w));
        return __uint_as_float((q & 1) ? (v & 0xffff0000u) : (v << 16));
    }
};
template <>
struct Raw8<float> {
    float v[8];
    __device__ __forceinline__ void load(const float* __restrict__ p, int e, int len, int vec) {
        if (vec && e + 8 <= len) {
            load8_stream(p + e, v);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = (e + q < len) ? p[e + q] : -INFINITY;
        }
    }
    __device__ __forceinline__ float at(int q) const { return v[q]; }
};

template <typename T>
__global__ void __launch_bounds__(kSampleThreads) k_walk_lse(const T* __restrict__ logits, int N, int V, int nunits,
                                                             int vec, float s2, const int32_t* __restrict__ n_nodes,
                                                             LsePartial* __restrict__ part) {
    const int i = blockIdx.y, b = blockIdx.z;
    const int lane = threadIdx.x & 31;
    const int u = blockIdx.x * kUnitsPerCta + (threadIdx.x >> 5);
    const int nn = n_nodes[b];
    if (i >= nn || nn > N || u >= nunits) return;  // rows past the tree are not needed
    const T* row = logits + ((long)b * N + i) * V + (long)u * kSampleUnit;
    const int len = min(kSampleUnit, V - u * kSampleUnit);
    Raw8<T> r[kLanePer / 8];
#pragma unroll
    for (int j = 0; j < kLanePer / 8; ++j) r[j].load(row, lane * 8 + j * 256, len, vec);
    float mt = -INFINITY;
    int bad = 0;
    if constexpr (sizeof(T) == 2) {
        if (len == kSampleUnit) {
            // a full bf16 unit: packed maxima two entries at a time, and the largest exponent
            // field of each half (0x7f80 marks Inf or NaN)
            __nv_bfloat162 m2 = __float2bfloat162_rn(-INFINITY);
            uint32_t ex = 0;
#pragma unroll
            for (int j = 0; j < kLanePer / 8; ++j) {
                const uint32_t ww[4] = {r[j].w.x, r[j].w.y, r[j].w.z, r[j].w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    ex = __vmaxu2(ex, ww[q] & 0x7f807f80u);
                    m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&ww[q]));
                }
            }
            bad = (ex & 0xffffu) == 0x7f80u || (ex >> 16) == 0x7f80u;
            mt = fmaxf(__low2float(m2), __high2float(m2));
        }
    }
    if (sizeof(T) != 2 || len != kSampleUnit) {
#pragma unroll
        for (int j = 0; j < kLanePer / 8; ++j)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float x = r[j].at(q);
                if (lane * 8 + j * 256 + q < len) {
                    if (!finite_f32(x)) bad = 1;
                    mt = fmaxf(mt, x);
                }
            }
    }
    float g[kLanePer / 8];
#pragma unroll
    for (int j = 0; j < kLanePer / 8; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) acc += tempered(r[j].at(q), mt, s2);
        g[j] = acc;
    }
    float st = mt == -INFINITY ? 0.f : ((g[0] + g[1]) + (g[2] + g[3])) + ((g[4] + g[5]) + (g[6] + g[7]));
    float mw = mt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(kFull, mw, o));
    if (mt != -INFINITY) st *= tempered(mt, mw, s2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) st += __shfl_down_sync(kFull, st, o);
    bad = __any_sync(kFull, bad);
    if (lane == 0) {
        LsePartial pp;
        pp.m = mw;
        pp.s = bad ? -1.f : st;
        part[((long)b * N + i) * nunits + u] = pp;
    }
}

// Warp-wide: the row's max and Z = sum_v exp((l_v - m) / T) from its unit partials, the
// sum in fp64.  Every lane returns lane 0's values, so decisions taken on them are
// uniform across the warp.
__device__ __forceinline__ void row_stats(const LsePartial* __restrict__ P, int nunits, float s2, int lane, float& m,
                                          double& z) {
    float mm = -INFINITY;
    for (int c = lane; c < nunits; c += 32) mm = fmaxf(mm, P[c].m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, o));
    double zz = 0.0;
    for (int c = lane; c < nunits; c += 32) {
        const LsePartial pp = P[c];
        if (pp.s > 0.f) zz += (double)pp.s * (double)tempered(pp.m, mm, s2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zz += __shfl_down_sync(kFull, zz, o);
    m = mm;
    z = __shfl_sync(kFull, zz, 0);
}

template <typename T>
__global__ void __launch_bounds__(kSampleThreads) k_walk_sample(
    const T* __restrict__ logits, int N, int V, int A, int C, int nunits, int vec, float s2,
    const LsePartial* __restrict__ part, const float* __restrict__ uniforms, const int32_t* __restrict__ token,
    const int32_t* __restrict__ parent, const int32_t* __restrict__ n_nodes, int32_t* __restrict__ acc_nodes,
    int32_t* __restrict__ acc_len, int32_t* __restrict__ bonus, int32_t* __restrict__ emitted,
    int32_t* __restrict__ n_emitted, int32_t* __restrict__ status) {
    __shared__ int s_tok[kMaxRows], s_par[kMaxRows], s_cnt[kMaxRows];
    __shared__ float s_lc[kMaxRows];  // logit of node i's token in its parent's row
    __shared__ double s_incl[kSampleThreads];
    __shared__ double s_wsum[kSampleThreads / 32];
    __shared__ uint32_t s_rejbits[kSampleUnit / 32];
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
        for (int j = tid; j < nn * nunits; j += kSampleThreads)
            if (part[ob * nunits + j].s < 0.f) atomicMax(&s_err, DDT_ERR_NONFINITE);  // a tree error outranks it
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
            row_stats(part + (ob + cur) * nunits, nunits, s2, lane, m, zr);
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
                        const float term = tempered(s_lc[cc], m, s2);
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

    // ---- the bonus unit (warp 0): residual unit masses in id order, inclusive scan
    const int cur = s_cur, nrej = s_nrej;
    const float m = s_m;
    if (warp == 0) {
        const LsePartial* P = part + (ob + cur) * nunits;
        const double target = s_local;
        double carry = 0.0;
        int pick = -1, last = -1;
        double before = 0.0;
        for (int base = 0; base < nunits; base += 32) {
            const int c = base + lane;
            double mc = 0.0;
            if (c < nunits) {
                const LsePartial pp = P[c];
                mc = (double)pp.s * (double)tempered(pp.m, m, s2);
                for (int r = 0; r < nrej; ++r)
                    if (s_rejtok[r] / kSampleUnit == c) mc -= (double)s_rejterm[r];
            }
            double incl = mc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            incl += carry;
            const unsigned over = __ballot_sync(kFull, c < nunits && incl > target);
            const unsigned pos = __ballot_sync(kFull, c < nunits && mc > 0.0);
            if (pick < 0 && over != 0u) {
                const int l = __ffs(over) - 1;
                pick = base + l;
                before = __shfl_sync(kFull, incl - mc, l);
            }
            if (pos != 0u) last = base + 31 - __clz(pos);
            carry = __shfl_sync(kFull, incl, 31);
        }
        if (lane == 0) {
            // rounding left the target past the residual mass: the last unit that has some,
            // and in it the largest id with a positive term (an infinite local target)
            s_chunk = (pick >= 0) ? pick : last;
            s_local = (pick >= 0) ? target - before : INFINITY;
            s_pick = 0x7fffffff;
            s_last = -1;
        }
    }
    for (int j = tid; j < kSampleUnit / 32; j += kSampleThreads) s_rejbits[j] = 0u;
    __syncthreads();
    const int unit = s_chunk;
    if (unit >= 0) {
        const int start = unit * kSampleUnit;
        if (tid < nrej) {
            const int t = s_rejtok[tid] - start;
            if (t >= 0 && t < kSampleUnit) atomicOr(&s_rejbits[t >> 5], 1u << (t & 31));
        }
        __syncthreads();
        // ---- the bonus token: block scan of this unit's residual terms in id order
        const int len = min(kSampleUnit, V - start);
        const T* row = logits + (ob + cur) * V + start;
        const int e0 = tid * kScanPer;
        float t8[kScanPer];
        if (vec && e0 + kScanPer <= len) {
            load8(row + e0, t8);
        } else {
#pragma unroll
            for (int q = 0; q < kScanPer; ++q) t8[q] = (e0 + q < len) ? to_f32(row[e0 + q]) : -INFINITY;
        }
        const uint32_t rejw = (s_rejbits[e0 >> 5] >> (e0 & 31)) & 0xffu;  // 8 entries share a word
        float tv[kScanPer];
        int lastpos = -1;
        float acc = 0.f;
#pragma unroll
        for (int q = 0; q < kScanPer; ++q) {
            tv[q] = (e0 + q < len && !((rejw >> q) & 1u)) ? tempered(t8[q], m, s2) : 0.f;
            if (tv[q] > 0.f) lastpos = e0 + q;
            acc += tv[q];
        }
        double incl = (double)acc;
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
            for (int q = 0; q < kScanPer; ++q) {
                if (tv[q] <= 0.f) continue;
                run += (double)tv[q];
                if (run > target) {
                    pickid = e0 + q;
                    break;
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
    const int nunits = units_of(V);
    const float s2 = (float)(1.4426950408889634 / (double)temperature);  // log2(e) / T
    LsePartial* part = static_cast<LsePartial*>(ws);
    const int vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
    dim3 g((nunits + kUnitsPerCta - 1) / kUnitsPerCta, N, B);
    if (dtype == DDT_BF16) {
        const __nv_bfloat16* l = static_cast<const __nv_bfloat16*>(logits);
        k_walk_lse<__nv_bfloat16><<<counted(g), kSampleThreads, 0, st>>>(l, N, V, nunits, vec, s2, n_nodes, part);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        k_walk_sample<__nv_bfloat16><<<counted(B), kSampleThreads, 0, st>>>(
            l, N, V, A, C, nunits, vec, s2, part, uniforms, token, parent, n_nodes, acc_nodes, acc_len, bonus,
            emitted, n_emitted, status);
    } else {
        const float* l = static_cast<const float*>(logits);
        k_walk_lse<float><<<counted(g), kSampleThreads, 0, st>>>(l, N, V, nunits, vec, s2, n_nodes, part);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        k_walk_sample<float><<<counted(B), kSampleThreads, 0, st>>>(l, N, V, A, C, nunits, vec, s2, part, uniforms,
                                                                    token, parent, n_nodes, acc_nodes, acc_len,
                                                                    bonus, emitted, n_emitted, status);
    }
    return cudaGetLastError();
}

}  // namespace ddt
