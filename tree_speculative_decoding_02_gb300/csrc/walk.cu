// walk.cu -- ddt_walk_accept: greedy tree walk against the target's argmax.
//
// "From Tree-Based Speculative Decoding to Drafter Training", section "The Architecture
// of DDTree: Tree Construction and Verification": follow_verified_tree compares the
// target model's tokens against the tree and walks down while a child matches.
// "DDTree on vLLM: candid research notes", section "What broke along the way": the
// target's bonus token is emitted but must not be fed back as an accepted draft.
//
//   k_walk_argmax   grid (chunks, N, B): one HBM pass over the target logits; each CTA
//                   reduces a 16384-token chunk of one row to (max, lowest argmax id)
//                   (k_walk_argmax_bf16 for bf16 rows: packed maxima, then the id).
//   k_walk_descend  grid B: warp-per-row merge of the chunk partials, tree check, then
//                   one warp walks down with a ballot over the rows per step.
#include "common.cuh"
#include "kernels.h"

namespace ddt {

// vocabulary entries one argmax CTA reduces (eight 16-byte loads a thread in flight)
constexpr int kWalkChunk = 16384;

struct ArgPartial {
    float v;
    int id;
    int nonfinite;
    int pad;
};

size_t walk_ws_bytes(int B, int N, int V) {
    const long nch = (V + kWalkChunk - 1) / kWalkChunk;
    return (((size_t)B * N * nch * sizeof(ArgPartial)) + 255) & ~(size_t)255;
}

template <typename T>
__global__ void __launch_bounds__(256) k_walk_argmax(const T* __restrict__ logits, int N, int V, int nch, int vec,
                                                      const int32_t* __restrict__ n_nodes,
                                                      ArgPartial* __restrict__ part) {
    const int c = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
    const int nn = n_nodes[b];
    if (i >= nn || nn > N) return;  // rows past the tree are not needed
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long row = ((long)b * N + i) * V;
    const int start = c * kWalkChunk;
    const int len = min(kWalkChunk, V - start);
    float bv = vid_empty().v;
    int bid = 0x7fffffff;
    int bad = 0;
#pragma unroll
    for (int j = 0; j < kWalkChunk / 2048; ++j) {
        const int e = tid * 8 + j * 2048;
        float t8[8];
        if (vec && e + 8 <= len) {
            load8_stream(logits + row + start + e, t8);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) t8[u] = (e + u < len) ? to_f32(logits[row + start + e + u]) : vid_empty().v;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (e + u < len) {
                if (!finite_f32(t8[u])) bad = 1;
                if (beats(t8[u], start + e + u, bv, bid)) {
                    bv = t8[u];
                    bid = start + e + u;
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, o);
        const int oid = __shfl_xor_sync(kFull, bid, o);
        if (beats(ov, oid, bv, bid)) {
            bv = ov;
            bid = oid;
        }
    }
    bad = __any_sync(kFull, bad);
    __shared__ float s_v[8];
    __shared__ int s_id[8], s_bad[8];
    if (lane == 0) {
        s_v[warp] = bv;
        s_id[warp] = bid;
        s_bad[warp] = bad;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < 8; ++w) {
            if (beats(s_v[w], s_id[w], bv, bid)) {
                bv = s_v[w];
                bid = s_id[w];
            }
            bad |= s_bad[w];
        }
        ArgPartial pp;
        pp.v = bv;
        pp.id = bid;
        pp.nonfinite = bad;
        pp.pad = 0;
        part[((long)b * N + i) * nch + c] = pp;
    }
}

// bf16 logits: the chunk's maximum on packed bf16 pairs (one max per two entries), the
// non-finite check as the largest exponent field seen, then the lowest id holding that
// maximum from the few threads whose own maximum it is.  Same output as k_walk_argmax.
__global__ void __launch_bounds__(256) k_walk_argmax_bf16(const __nv_bfloat16* __restrict__ logits, int N, int V,
                                                           int nch, int vec, const int32_t* __restrict__ n_nodes,
                                                           ArgPartial* __restrict__ part) {
    const int c = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
    const int nn = n_nodes[b];
    if (i >= nn || nn > N) return;  // rows past the tree are not needed
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16* row = logits + ((long)b * N + i) * V + (long)c * kWalkChunk;
    const int len = min(kWalkChunk, V - c * kWalkChunk);
    // entries past the row's end read as the lowest finite bf16 (never non-finite, and
    // never taken: the id search below stops at the row's end)
    constexpr uint32_t kLow = 0xff7fff7fu;
    uint4 w[kWalkChunk / 2048];
#pragma unroll
    for (int j = 0; j < kWalkChunk / 2048; ++j) {
        const int e = tid * 8 + j * 2048;
        if (vec && e + 8 <= len) {
            w[j] = ld_stream_u4(row + e);
        } else {
            uint32_t h[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) h[u] = (e + u < len) ? (uint32_t)__bfloat16_as_ushort(row[e + u]) : 0xff7fu;
            w[j] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
        }
    }
    __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&kLow);
    uint32_t ex = 0;  // largest exponent field per half: 0x7f80 marks Inf or NaN
#pragma unroll
    for (int j = 0; j < kWalkChunk / 2048; ++j) {
        const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            ex = __vmaxu2(ex, ww[q] & 0x7f807f80u);
            m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&ww[q]));
        }
    }
    int bad = (ex & 0xffffu) == 0x7f80u || (ex >> 16) == 0x7f80u;
    float mt = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o));
    bad = __any_sync(kFull, bad);
    __shared__ float s_v[8];
    __shared__ int s_id[8], s_bad[8];
    if (lane == 0) {
        s_v[warp] = mt;
        s_bad[warp] = bad;
    }
    __syncthreads();
    float M = s_v[0];
#pragma unroll
    for (int q = 1; q < 8; ++q) M = fmaxf(M, s_v[q]);
    // the lowest id holding M: a thread's ids rise with j, then u
    int bid = 0x7fffffff;
    const float mine = fmaxf(__low2float(m2), __high2float(m2));
    if (mine == M) {
        for (int j = 0; j < kWalkChunk / 2048 && bid == 0x7fffffff; ++j) {
            const uint32_t ww[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = tid * 8 + j * 2048 + u;
                const uint32_t h = (ww[u >> 1] >> ((u & 1) * 16)) << 16;
                if (e < len && __uint_as_float(h) == M && bid == 0x7fffffff) bid = c * kWalkChunk + e;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bid = min(bid, __shfl_xor_sync(kFull, bid, o));
    if (lane == 0) s_id[warp] = bid;
    __syncthreads();
    if (tid == 0) {
        int id = s_id[0], anybad = s_bad[0];
        for (int q = 1; q < 8; ++q) {
            id = min(id, s_id[q]);
            anybad |= s_bad[q];
        }
        ArgPartial pp;
        pp.v = M;
        pp.id = id;
        pp.nonfinite = anybad;
        pp.pad = 0;
        part[((long)b * N + i) * nch + c] = pp;
    }
}

__global__ void __launch_bounds__(256) k_walk_descend(int N, int V, int A, int nch, int have_logits, int flat,
                                                       const ArgPartial* __restrict__ part,
                                                       int32_t* __restrict__ targ, const int32_t* __restrict__ token,
                                                       const int32_t* __restrict__ parent,
                                                       const int32_t* __restrict__ n_nodes,
                                                       int32_t* __restrict__ acc_nodes, int32_t* __restrict__ acc_len,
                                                       int32_t* __restrict__ bonus, int32_t* __restrict__ emitted,
                                                       int32_t* __restrict__ n_emitted, int32_t* __restrict__ status) {
    __shared__ int s_t[kMaxRows], s_tok[kMaxRows], s_par[kMaxRows];
    __shared__ int s_err;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nn = n_nodes[b];
    const long ob = (long)b * N;
    // decided on each thread's own copy of n_nodes: the checks below write s_err, and a
    // thread that read it late would leave while the others go on to the barriers
    const bool nn_ok = nn >= 1 && nn <= N;
    if (tid == 0) s_err = nn_ok ? DDT_OK : DDT_ERR_TREE;
    __syncthreads();
    if (!nn_ok) {
        for (int j = tid; j < A; j += blockDim.x) {
            acc_nodes[(long)b * A + j] = -1;
            emitted[(long)b * A + j] = -1;
        }
        if (tid == 0) {
            acc_len[b] = 0;
            bonus[b] = -1;
            n_emitted[b] = 0;
            status[b] = s_err;
        }
        return;
    }
    for (int i = tid; i < nn; i += blockDim.x) {
        s_tok[i] = token[ob + i];
        s_par[i] = parent[ob + i];
        const bool ok = (i == 0) ? (s_par[i] == -1) : (s_par[i] >= 0 && s_par[i] < i);
        if (!ok) atomicExch(&s_err, DDT_ERR_TREE);
    }
    // target token per row
    for (int i = warp; i < N; i += blockDim.x / 32) {
        int t = -1;
        if (i < nn) {
            if (have_logits) {
                float bv = vid_empty().v;
                int bid = 0x7fffffff, bad = 0;
                for (int c = lane; c < nch; c += 32) {
                    const ArgPartial pp = part[(ob + i) * nch + c];
                    bad |= pp.nonfinite;
                    if (beats(pp.v, pp.id, bv, bid)) {
                        bv = pp.v;
                        bid = pp.id;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(kFull, bv, o);
                    const int oid = __shfl_xor_sync(kFull, bid, o);
                    if (beats(ov, oid, bv, bid)) {
                        bv = ov;
                        bid = oid;
                    }
                }
                bad = __any_sync(kFull, bad);
                if (bad && lane == 0) atomicExch(&s_err, DDT_ERR_NONFINITE);
                t = bid;
            } else {
                t = targ[ob + i];
            }
        }
        if (lane == 0) {
            if (i < nn) s_t[i] = t;
            if (have_logits) targ[ob + i] = t;
        }
    }
    __syncthreads();
    if (warp != 0) return;
    int32_t* an = acc_nodes + (long)b * A;
    int32_t* em = emitted + (long)b * A;
    int cur = 0, a = 0;
    if (s_err == DDT_OK) {
        for (;;) {
            const int want = s_t[cur];
            int found = 0x7fffffff;
            // flat: only the first child (the rank-0 one: children are numbered by rank)
            for (int c = 1 + lane; c < nn; c += 32)
                if (s_par[c] == cur && (flat || s_tok[c] == want)) found = min(found, c);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) found = min(found, __shfl_xor_sync(kFull, found, o));
            if (flat && found != 0x7fffffff && s_tok[found] != want) found = 0x7fffffff;
            if (found == 0x7fffffff || a + 1 >= A) break;
            if (lane == 0) an[a + 1] = found;
            cur = found;
            ++a;
        }
    }
    __syncwarp();
    // rows root..a, then padding; emitted = accepted tokens then the bonus token
    for (int j = lane; j < A; j += 32) {
        if (j == 0) an[0] = 0;
        if (j > a) an[j] = -1;
    }
    __syncwarp();
    for (int j = lane; j < A; j += 32) {
        int e = -1;
        if (s_err == DDT_OK) {
            if (j < a) e = s_tok[an[j + 1]];
            else if (j == a) e = s_t[cur];
        }
        em[j] = e;
    }
    if (lane == 0) {
        acc_len[b] = (s_err == DDT_OK) ? a : 0;
        bonus[b] = (s_err == DDT_OK) ? s_t[cur] : -1;
        n_emitted[b] = (s_err == DDT_OK) ? a + 1 : 0;
        status[b] = s_err;
    }
}

cudaError_t launch_walk(int B, int N, int V, int A, ddt_dtype dtype, const void* logits, int32_t* targ,
                        const int32_t* token, const int32_t* parent, const int32_t* n_nodes, int32_t* acc_nodes,
                        int32_t* acc_len, int32_t* bonus, int32_t* emitted, int32_t* n_emitted, int32_t* status,
                        void* ws, int flat, cudaStream_t st) {
    const int nch = (V + kWalkChunk - 1) / kWalkChunk;
    ArgPartial* part = static_cast<ArgPartial*>(ws);
    if (logits) {
        dim3 g(nch, N, B);
        const int vec = (V % 8 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
        if (dtype == DDT_BF16)
            k_walk_argmax_bf16<<<counted(g), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(logits), N, V, nch, vec,
                                                            n_nodes, part);
        else
            k_walk_argmax<float><<<counted(g), 256, 0, st>>>(static_cast<const float*>(logits), N, V, nch, vec, n_nodes, part);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    k_walk_descend<<<counted(B), 256, 0, st>>>(N, V, A, nch, logits != nullptr, flat, part, targ, token, parent, n_nodes, acc_nodes,
                                      acc_len, bonus, emitted, n_emitted, status);
    return cudaGetLastError();
}

}  // namespace ddt
