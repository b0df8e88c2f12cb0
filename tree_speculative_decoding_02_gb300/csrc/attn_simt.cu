// attn_simt.cu -- ddt_tree_attn, CUDA-core version (fp32 arithmetic throughout).
//
// "DDTree on vLLM: candid research notes", section "Why hybrid attention makes it hard":
// each candidate row sees the committed prefix plus its own ancestors and never its
// siblings.  "From Tree-Based Speculative Decoding to Drafter Training", section "The
// Architecture of DDTree: Tree Construction and Verification": one target pass over the
// flattened tree with an ancestor-only mask.
//
// One CTA takes 32 query rows of one (layer, request, kv head): rows are (node, head)
// pairs of the GQA group, so all of them share the kv head's keys.  Keys stream through
// shared memory in tiles of 32 (prefix rows first, then tree rows); each lane scores
// one key of the tile for four rows, the warp keeps an online softmax per row, and
// lanes own d/32 output channels.  Prefix rows >= prefix_len and tree rows >= n_nodes
// are never loaded.  This kernel serves fp32 inputs and any head size the tensor-core
// kernel does not take.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace ddt {

namespace {
constexpr int kRows = 32;  // query rows per CTA (4 per warp)
constexpr int kKeys = 32;  // keys per shared-memory tile
}  // namespace

template <typename Tin, typename Tout, int D>
__global__ void __launch_bounds__(256) k_attn_simt(int B, int N, int Hq, int Hkv, int Pcap,
                                                    const Tin* __restrict__ q, const Tin* __restrict__ k_tree,
                                                    const Tin* __restrict__ v_tree, const Tin* __restrict__ k_cache,
                                                    const Tin* __restrict__ v_cache,
                                                    const int32_t* __restrict__ prefix_len,
                                                    const int32_t* __restrict__ n_nodes,
                                                    const uint32_t* __restrict__ anc, float scale,
                                                    Tout* __restrict__ o, int32_t* __restrict__ status) {
    constexpr int E = D / 32;
    extern __shared__ float sm[];
    float* sq = sm;                       // [kRows][D]
    float* sk = sq + kRows * D;           // [kKeys][D + 1]
    float* sv = sk + kKeys * (D + 1);     // [kKeys][D]
    const int G = Hq / Hkv;
    const int rows_total = N * G;
    const int row0 = blockIdx.x * kRows;
    const int g = blockIdx.y;
    const int l = blockIdx.z / B, b = blockIdx.z % B;
    const int W = (N + 31) / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = prefix_len[b], nn = n_nodes[b];
    const bool bad = (P < 0 || P > Pcap || nn < 1 || nn > N);
    if (blockIdx.x == 0 && g == 0 && l == 0 && tid == 0)
        status[b] = (P < 0 || P > Pcap) ? DDT_ERR_CAPACITY : (bad ? DDT_ERR_TREE : DDT_OK);

    const long lb = (long)l * B + b;
    // rows of this warp
    int node_r[4], head_r[4];
    bool live_r[4], in_r[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int R = row0 + warp * 4 + rr;
        in_r[rr] = R < rows_total;
        node_r[rr] = in_r[rr] ? R / G : 0;
        head_r[rr] = g * G + (in_r[rr] ? R % G : 0);
        live_r[rr] = in_r[rr] && !bad && node_r[rr] < nn;
    }
    if (bad) {
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
            if (in_r[rr]) {
                Tout* orow = o + ((lb * N + node_r[rr]) * Hq + head_r[rr]) * D;
#pragma unroll
                for (int e = 0; e < E; ++e) orow[lane + 32 * e] = from_f32<Tout>(0.f);
            }
        return;
    }
    for (int e = tid; e < kRows * D; e += 256) {
        const int r = e / D, c = e % D;
        const int R = row0 + r;
        float val = 0.f;
        if (R < rows_total) {
            const int node = R / G, h = g * G + R % G;
            if (node < nn) val = to_f32(q[((lb * N + node) * Hq + h) * D + c]);
        }
        sq[r * D + c] = val;
    }

    float m[4], lsum[4], acc[4][E];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        m[rr] = -INFINITY;
        lsum[rr] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[rr][e] = 0.f;
    }
    const float sl2 = scale * 1.4426950408889634f;  // softmax in base 2
    const int n_pre = (P + kKeys - 1) / kKeys;
    const int n_tree = (nn + kKeys - 1) / kKeys;
    const Tin* kc = k_cache + (lb * Hkv + g) * (long)Pcap * D;
    const Tin* vc = v_cache + (lb * Hkv + g) * (long)Pcap * D;
    for (int t = 0; t < n_pre + n_tree; ++t) {
        const bool tree = t >= n_pre;
        const int base = tree ? (t - n_pre) * kKeys : t * kKeys;
        const int lim = tree ? nn : P;
        __syncthreads();
        for (int e = tid; e < kKeys * D; e += 256) {
            const int kr = e / D, c = e % D;
            const int key = base + kr;
            float kv = 0.f, vv = 0.f;
            if (key < lim) {
                if (tree) {
                    const long off = ((lb * N + key) * Hkv + g) * D + c;
                    kv = to_f32(k_tree[off]);
                    vv = to_f32(v_tree[off]);
                } else {
                    kv = to_f32(kc[(long)key * D + c]);
                    vv = to_f32(vc[(long)key * D + c]);
                }
            }
            sk[kr * (D + 1) + c] = kv;
            sv[kr * D + c] = vv;
        }
        __syncthreads();
        const int key = base + lane;
        float s[4];
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) s[rr] = 0.f;
        const float* krow = sk + lane * (D + 1);
        const float* q0 = sq + (warp * 4) * D;
#pragma unroll 8
        for (int c = 0; c < D; ++c) {
            const float kx = krow[c];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) s[rr] = fmaf(q0[rr * D + c], kx, s[rr]);
        }
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            bool vis = live_r[rr] && key < lim;
            if (vis && tree) vis = (anc[((long)b * N + node_r[rr]) * W + key / 32] >> (key % 32)) & 1u;
            const float sc = vis ? s[rr] * sl2 : -INFINITY;
            const float mt = warp_max(sc);
            const float mn = fmaxf(m[rr], mt);
            const float corr = (mn == -INFINITY) ? 1.f : exp2f(m[rr] - mn);
            const float p = vis ? exp2f(sc - mn) : 0.f;
            lsum[rr] = lsum[rr] * corr + warp_sum(p);
            m[rr] = mn;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[rr][e] *= corr;
#pragma unroll 4
            for (int kk = 0; kk < kKeys; ++kk) {
                const float pk = __shfl_sync(kFull, p, kk);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[rr][e] = fmaf(pk, sv[kk * D + lane + 32 * e], acc[rr][e]);
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        if (!in_r[rr]) continue;
        Tout* orow = o + ((lb * N + node_r[rr]) * Hq + head_r[rr]) * D;
        const float inv = (live_r[rr] && lsum[rr] > 0.f) ? 1.f / lsum[rr] : 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) orow[lane + 32 * e] = from_f32<Tout>(live_r[rr] ? acc[rr][e] * inv : 0.f);
    }
}

template <typename Tin, typename Tout, int D>
static cudaError_t attn_simt_go(int L, int B, int N, int Hq, int Hkv, int Pcap, const void* q, const void* kt,
                                const void* vt, const void* kc, const void* vc, const int32_t* pl,
                                const int32_t* nn, const uint32_t* anc, float scale, void* o, int32_t* status,
                                cudaStream_t st) {
    const size_t smem = sizeof(float) * (kRows * D + kKeys * (D + 1) + kKeys * D);
    cudaError_t e = cudaFuncSetAttribute(k_attn_simt<Tin, Tout, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int G = Hq / Hkv;
    dim3 grid((N * G + kRows - 1) / kRows, Hkv, L * B);
    k_attn_simt<Tin, Tout, D><<<counted(grid), 256, smem, st>>>(
        B, N, Hq, Hkv, Pcap, static_cast<const Tin*>(q), static_cast<const Tin*>(kt), static_cast<const Tin*>(vt),
        static_cast<const Tin*>(kc), static_cast<const Tin*>(vc), pl, nn, anc, scale, static_cast<Tout*>(o), status);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t attn_simt_d(int d, int L, int B, int N, int Hq, int Hkv, int Pcap, const void* q, const void* kt,
                               const void* vt, const void* kc, const void* vc, const int32_t* pl, const int32_t* nn,
                               const uint32_t* anc, float scale, void* o, int32_t* status, cudaStream_t st) {
    switch (d) {
        case 64: return attn_simt_go<Tin, Tout, 64>(L, B, N, Hq, Hkv, Pcap, q, kt, vt, kc, vc, pl, nn, anc, scale, o, status, st);
        case 128: return attn_simt_go<Tin, Tout, 128>(L, B, N, Hq, Hkv, Pcap, q, kt, vt, kc, vc, pl, nn, anc, scale, o, status, st);
        case 256: return attn_simt_go<Tin, Tout, 256>(L, B, N, Hq, Hkv, Pcap, q, kt, vt, kc, vc, pl, nn, anc, scale, o, status, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_simt(int L, int B, int N, int Hq, int Hkv, int d, int Pcap, ddt_dtype in, ddt_dtype out,
                             const void* q, const void* k_tree, const void* v_tree, const void* k_cache,
                             const void* v_cache, const int32_t* prefix_len, const int32_t* n_nodes,
                             const uint32_t* anc, float scale, void* o, int32_t* status, cudaStream_t st) {
    if (in == DDT_F32 && out == DDT_F32)
        return attn_simt_d<float, float>(d, L, B, N, Hq, Hkv, Pcap, q, k_tree, v_tree, k_cache, v_cache, prefix_len,
                                         n_nodes, anc, scale, o, status, st);
    if (in == DDT_F32 && out == DDT_BF16)
        return attn_simt_d<float, __nv_bfloat16>(d, L, B, N, Hq, Hkv, Pcap, q, k_tree, v_tree, k_cache, v_cache,
                                                 prefix_len, n_nodes, anc, scale, o, status, st);
    if (in == DDT_BF16 && out == DDT_F32)
        return attn_simt_d<__nv_bfloat16, float>(d, L, B, N, Hq, Hkv, Pcap, q, k_tree, v_tree, k_cache, v_cache,
                                                 prefix_len, n_nodes, anc, scale, o, status, st);
    return attn_simt_d<__nv_bfloat16, __nv_bfloat16>(d, L, B, N, Hq, Hkv, Pcap, q, k_tree, v_tree, k_cache, v_cache,
                                                     prefix_len, n_nodes, anc, scale, o, status, st);
}

}  // namespace ddt
