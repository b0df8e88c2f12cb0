// gdn_tc.cu -- ddt_tree_gdn with the dense part on the tensor cores (kind::tf32).
//
// "DDTree on vLLM: candid research notes", sections "Why hybrid attention makes it hard"
// and "Where the next step is": each node reads its parent's GDN and conv state and
// writes scratch, never the committed state.  Rule: gated delta rule of Yang, Kautz and
// Hatamizadeh, "Gated Delta Networks" (ICLR 2025), in the tree-masked "WY" form
// described in gdn.cu (every term runs over the node's own ancestors only):
//   u_t = b_t (v_t - g_t S0 k_t) - sum_{s in anc(t)} b_t G_ts (k_s . k_t) u_s
//   o_t = g_t S0 q_t + sum_{s in anc(t)+t} G_ts (k_s . q_t) u_s
// One CTA owns a (layer, request, key head) and the Hv/Hk value heads that read it:
//   thread 0    TMA: the key head's q and k channel rows (node rows, then conv-state
//               rows) at the start, and each value head's v channel rows one head ahead.
//   all warps   conv + SiLU + L2 norm of q and k for every node, written once as a tf32
//               K-major tile [k rows | q rows] (128-byte swizzle); the (k_s . k_t) and
//               (k_s . q_t) dot products along every ancestor chain.
//   warp 0      TMA: each value head's committed state S0 (dv x dk fp32, key channel
//               contiguous) into shared memory.
//   warp 1      tcgen05.mma kind::tf32: D = S0 [k | q]^T, i.e. S0 k_t and S0 q_t for every
//               node, into one of two TMEM buffers (lane = value channel).
//   all warps   per value channel (= TMEM lane; the warps of a lane quarter take
//               interleaved 8-node chunks): v_t by the conv along the path, the chain
//               coefficients by back substitution, o_t; written to global.
// S0 is read once from HBM; no node state ever exists.  Waits are bounded.
#include <cuda.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace ddt {

namespace {

constexpr int kDK = 128, kDV = 128;  // head sizes of this path
constexpr int kMD = 16;              // deepest tree this path takes (drafter depth <= 16)
// threads a CTA: 16 warps for conv width 4 (registers allow it), 12 for the generic width;
// lane 0 of warp 0 loads S0, lane 0 of warp 1 issues the MMAs, every warp runs the
// epilogue (the warps of a TMEM lane quarter take interleaved node chunks)
__host__ __device__ constexpr int gdn_threads(int kt) { return kt == 4 ? 512 : 384; }
constexpr int kMaxK = 8;    // widest short conv

struct GdnTcParams {
    int L, B, N, Hk, Hv, R, K, C, QOFF, NPAD;
    int wvec;  // conv_w is 16-byte aligned: width-4 taps are read as vectors
    const void* x;
    const void* conv_w;
    const void* conv_state;
    const float* beta;
    const float* decay;
    const int32_t* parent;
    const int32_t* n_nodes;
    void* o;
    int32_t* status;
};

struct GdnSmem {
    size_t s0, kq, u, sk, kk, qk, ca, cb, tr, alist, small, sv, bars, total;
};

// esz = bytes per input element (the staged v rows keep the input type)
__host__ __device__ GdnSmem gdn_tc_layout(int N, int NPAD, int K, int esz) {
    GdnSmem L;
    size_t off = 0;
    // [k | q] tile (tf32 high parts): NPAD rows in four 32-column chunks; the Gram MMA
    // reads 128 rows of every chunk, so the last chunk's reads reach 128 rows past its start
    const size_t kq_bytes = (size_t)(3 * NPAD + (NPAD > 128 ? NPAD : 128)) * 128;
    L.kq = off;
    off += kq_bytes;
    // S0 tile (64 KiB) followed by R.  Until the Gram MMA has finished, the same bytes
    // hold the low parts of the [k | q] tile (same layout as the high parts).
    L.s0 = off;
    off += (size_t)kDV * kDK * 4;
    L.u = off;
    // R (one column per value channel), first used for the Gram rows [N][2N + 1]
    size_t ub = (size_t)N * (kDV > 2 * N + 1 ? kDV : 2 * N + 1) * 4;
    if (L.u + ub < L.s0 + kq_bytes) ub = L.s0 + kq_bytes - L.u;
    // during the conv stage the k channels' input rows are staged past the low parts
    L.sk = (L.s0 + kq_bytes > L.u ? L.s0 + kq_bytes - L.u : 0);
    L.sk = L.u + ((L.sk + 127) & ~(size_t)127);  // a TMA destination: 128-byte aligned
    const size_t skb = (size_t)(N + K - 1) * kDK * esz;
    if (L.u + ub < L.sk + skb) ub = L.sk + skb - L.u;
    off += (ub + 15) & ~(size_t)15;
    L.kk = off;
    off += (size_t)N * kMD * 4;
    L.qk = off;
    off += (size_t)N * kMD * 4;
    L.ca = off;
    off += (size_t)N * kMD * 4;
    L.cb = off;
    off += (size_t)2 * N * kMD * 4;          // two heads' buffers
    off = (off + 15) & ~(size_t)15;
    L.tr = off;                              // 16-byte aligned: four taps load as one int4
    off += (size_t)N * kMaxK * 4;            // conv input rows as staging-row indices
    L.alist = off;
    off += (size_t)N * kMD * 4;
    L.small = off;
    off += (size_t)N * 4 * 9;                // dep, par, qself, gcum[2], beta[2], decay[2]
    off = (off + 127) & ~(size_t)127;
    L.sv = off;                              // one value head's v channels: node rows, then conv-state rows (TMA)
    off += (size_t)(N + K - 1) * kDV * esz;
    off = (off + 7) & ~(size_t)7;
    L.bars = off;
    off += 128;
    L.total = off + 1024;                    // alignment slack
    return L;
}

__device__ __forceinline__ float silu_g(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// byte offset of element (row, col) of a K-major fp32 tile with 128-byte swizzle whose
// column blocks of 32 elements are `rows * 128` bytes apart
__device__ __forceinline__ uint32_t sw_off(int row, int col, int rows) {
    const int blk = col >> 5, chunk = (col & 31) >> 2;
    return blk * (rows * 128) + row * 128 + ((chunk ^ (row & 7)) << 4) + (col & 3) * 4;
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }

// four consecutive channels of a staged row (shared memory) as floats
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    v[0] = a.x;
    v[1] = a.y;
    v[2] = a.z;
    v[3] = a.w;
}


}  // namespace

// KT: compile-time conv width (K == KT), or kMaxK for any K <= kMaxK given at run time
template <typename Tin, typename Tout, int KT>
__global__ void __launch_bounds__(gdn_threads(KT), 1) k_gdn_tc(const GdnTcParams p, const __grid_constant__ CUtensorMap tm_s,
                                                    const __grid_constant__ CUtensorMap tm_x,
                                                    const __grid_constant__ CUtensorMap tm_cs) {
    constexpr int kThr = gdn_threads(KT), kEpi = kThr, kQuads = kThr / 128;
    extern __shared__ unsigned char smem_raw[];
    // align to 1024 B by pointer arithmetic on the shared array (keeps the address space)
    unsigned char* base = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int N = p.N;
    const GdnSmem lay = gdn_tc_layout(N, p.NPAD, p.K, (int)sizeof(Tin));
    unsigned char* sS0 = base + lay.s0;
    unsigned char* sKQ = base + lay.kq;
    unsigned char* sLO = sS0;  // low parts of [k | q], until the Gram MMA is done
    float* ubuf = reinterpret_cast<float*>(base + lay.u);
    float* skk = reinterpret_cast<float*>(base + lay.kk);
    float* sqk = reinterpret_cast<float*>(base + lay.qk);
    float* sca = reinterpret_cast<float*>(base + lay.ca);
    float* scb = reinterpret_cast<float*>(base + lay.cb);
    int* trow = reinterpret_cast<int*>(base + lay.tr);                // [N][K] the same rows in sv
    Tin* sv = reinterpret_cast<Tin*>(base + lay.sv);                  // [N + K - 1][kDV]
    // the per-node chain arrays (alist, skk, sqk, sca, scb) are level-major, [level][N]:
    // threads that each take a node touch consecutive words
    int* alist = reinterpret_cast<int*>(base + lay.alist);
    int* sdep = reinterpret_cast<int*>(base + lay.small);
    int* spar = sdep + N;
    float* sqself = reinterpret_cast<float*>(spar + N);
    float* sg = sqself + N;     // [2][N] (two heads' buffers, as sbeta, sdec and scb)
    float* sbeta = sg + 2 * N;
    float* sdec = sbeta + 2 * N;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + lay.bars);
    uint64_t* full = bars;        // S0 landed
    uint64_t* s_free = bars + 1;  // MMA done reading S0
    uint64_t* d_full = bars + 2;  // [2] D ready
    uint64_t* d_free = bars + 4;  // [2] epilogue done with D (kEpi arrivals)
    uint64_t* drain = bars + 6;
    uint64_t* g_done = bars + 7;  // Gram-matrix MMA done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    int* err = abort_flag + 1;
    uint64_t* qk_full = bars + 10;  // q and k rows staged
    uint64_t* v_full = bars + 11;   // a value head's v rows staged (one phase a head)

    const int g = blockIdx.x, b = blockIdx.y, l = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long lb = (long)l * p.B + b;
    const int C = p.C, K = KT < kMaxK ? KT : p.K;
    const int nn = p.n_nodes[b];
    const Tin* xb = static_cast<const Tin*>(p.x) + lb * N * C;
    const Tin* csb = static_cast<const Tin*>(p.conv_state) + lb * (K - 1) * C;
    const Tin* wl = static_cast<const Tin*>(p.conv_w) + (long)l * C * K;

    Tin* sk = reinterpret_cast<Tin*>(base + lay.sk);  // [N + K - 1][kDK], like sv
    // rows of one 128-channel group (x channels cb) into a staging buffer by TMA: the N
    // node rows of this (layer, request), then its K - 1 conv-state rows at row N
    const uint32_t stage_bytes = (uint32_t)((N + K - 1) * 128 * (int)sizeof(Tin));
    auto stage_rows = [&](Tin* dst, uint64_t* bar, int cb) {
        tc::tma_load_2d(dst, &tm_x, bar, cb, (int)(lb * N));
        if (K > 1) tc::tma_load_2d(dst + (long)N * 128, &tm_cs, bar, cb, (int)(lb * (K - 1)));
    };
    if (tid == 0) {
        *err = (nn < 1 || nn > N) ? DDT_ERR_TREE : DDT_OK;
        *abort_flag = 0;
        tc::mbar_init(full, 1);
        tc::mbar_init(s_free, 1);
        tc::mbar_init(d_full, 1);
        tc::mbar_init(d_full + 1, 1);
        tc::mbar_init(d_free, kEpi);
        tc::mbar_init(d_free + 1, kEpi);
        tc::mbar_init(drain, 1);
        tc::mbar_init(g_done, 1);
        tc::mbar_init(qk_full, 1);
        tc::mbar_init(v_full, 1);
        tc::fence_mbar_init();
        // ---- the group's q and k channel rows (node rows and conv-state rows) into shared
        //      memory, issued first so that they land while the tree is parsed
        tc::prefetch_tmap(&tm_x);
        if (K > 1) tc::prefetch_tmap(&tm_cs);
        tc::mbar_expect_tx(qk_full, 2 * stage_bytes);
        stage_rows(sv, qk_full, g * kDK);
        stage_rows(sk, qk_full, (p.Hk + g) * kDK);
    }
    // the conv weights of the group's q and k channels (four channels a lane), and the
    // first value head's gates and v-channel conv weights, all loaded early and kept in
    // the input type until they are used (so that no conversion waits on the loads here);
    // taps past K repeat the last one and are never used
    const int c4 = 4 * lane;
    Tin w_in[2][4][KT];
    {
        const int cbq = g * kDK, cbk = (p.Hk + g) * kDK;
        if (KT == 4 && p.wvec) {
            // width 4: a lane's four channels are 16 consecutive weights (16-byte vectors)
            constexpr int kV = 16 * (int)sizeof(Tin) / 16;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint4 buf[kV];
                const uint4* src = reinterpret_cast<const uint4*>(wl + (long)((part ? cbk : cbq) + c4) * 4);
#pragma unroll
                for (int i = 0; i < kV; ++i) buf[i] = src[i];
                const Tin* vals = reinterpret_cast<const Tin*>(buf);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                    for (int q = 0; q < KT; ++q) w_in[part][ch][q] = vals[ch * 4 + (q & 3)];
            }
        } else {
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                    for (int q = 0; q < KT; ++q)
                        w_in[part][ch][q] = wl[(long)((part ? cbk : cbq) + c4 + ch) * K + min(q, K - 1)];
        }
    }
    float dec_nx = 0.f, beta_nx = 0.f;
    if (tid < nn && nn <= N) {
        dec_nx = p.decay[(lb * N + tid) * p.Hv + g * p.R];
        beta_nx = p.beta[(lb * N + tid) * p.Hv + g * p.R];
    }
    Tin wv_nx[KT];
    {
        const int cv = 2 * p.Hk * kDK + g * p.R * kDV + (tid & (kDV - 1));
#pragma unroll
        for (int q = 0; q < KT; ++q) wv_nx[q] = wl[(long)cv * K + min(q, K - 1)];
    }
    // warm L2 with the v channels of the later value heads and with their gates
    {
        const int nr = min(max(nn, 0), N);
        const int lv = (kDV * (int)sizeof(Tin) + 127) / 128, step = 128 / (int)sizeof(Tin);
        const int per = (p.R - 1) * lv;
        for (int e = tid; e < (nr + K - 1) * per; e += kThr) {
            const int r = e / per, sgm = e % per;
            const Tin* row = r < nr ? xb + (long)r * C : csb + (long)(r - nr) * C;
            prefetch_l2(row + 2L * p.Hk * kDK + (long)(g * p.R + 1) * kDV + (long)sgm * step);
        }
        for (int n = tid; n < nr; n += kThr) {
            prefetch_l2(p.beta + (lb * N + n) * p.Hv + (long)g * p.R);
            prefetch_l2(p.decay + (lb * N + n) * p.Hv + (long)g * p.R);
        }
    }
    __syncthreads();
    const int nv = (*err == DDT_OK) ? nn : 0;
    // ---- tree check, ancestor lists, conv input rows (the node's path, newest last,
    //      continued by the committed conv state past the root)
    for (int n = tid; n < nv; n += kThr) {
        const int pr = p.parent[(long)b * N + n];
        spar[n] = pr;
        if ((n == 0 && pr != -1) || (n > 0 && (pr < 0 || pr >= n))) atomicExch(err, DDT_ERR_TREE);
    }
    __syncthreads();
    if (*err == DDT_OK) {
        for (int n = tid; n < nn; n += kThr) {
            int d = 0;
            for (int a = spar[n]; a >= 0; a = spar[a]) {
                if (d >= kMD) {
                    atomicExch(err, DDT_ERR_UNSUPPORTED);
                    break;
                }
                alist[d++ * N + n] = a;  // level-major: [level][node]
            }
            sdep[n] = d;
            for (int q = 0; q < K; ++q) {
                const int back = K - 1 - q;
                const int r = back == 0 ? n : (back <= d ? alist[(back - 1) * N + n] : N + (K - 1 - (back - d)));
                trow[n * K + q] = r;
            }
        }
    }
    __syncthreads();
    Tout* obase = static_cast<Tout*>(p.o) + lb * N * p.Hv * kDV;
    if (*err != DDT_OK) {
        tc::mbar_wait(qk_full, 0, abort_flag);  // no copy may still be landing when the CTA leaves
        if (tid == 0 && g == 0 && l == 0) p.status[b] = *err;
        for (int hi = 0; hi < p.R; ++hi) {
            const int h = g * p.R + hi;
            for (int e = tid; e < N * kDV; e += kThr)
                obase[((long)(e / kDV) * p.Hv + h) * kDV + e % kDV] = from_f32<Tout>(0.f);
        }
        return;
    }

    // ---- setup: TMEM, first S0 load
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    __syncthreads();
    const int srow0 = (int)((lb * p.Hv + (long)g * p.R) * kDV);
    if (tid == 0) tc::prefetch_tmap(&tm_s);

    // ---- conv + SiLU + L2 norm of q and k from the staged rows: a warp takes a node (three
    //      at a time, so their load, SiLU and reduction chains overlap) and a lane four
    //      channels of q and of k, so each norm is one warp reduction and each 16-byte store
    //      of the swizzled tile is conflict-free
    {
        float w[2][4][KT];
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                for (int q = 0; q < KT; ++q) w[part][ch][q] = (q < K) ? to_f32(w_in[part][ch][q]) : 0.f;
        tc::mbar_wait(qk_full, 0, abort_flag);
#pragma unroll 3
        for (int n = warp; n < N; n += kThr / 32) {
            float y[2][4] = {};
            if (n < nn) {
#pragma unroll
                for (int q = 0; q < KT; ++q) {
                    if (q < K) {
                        const int rs = trow[n * K + q];
                        float in[2][4];
                        load4(sv + (long)rs * kDK + c4, in[0]);
                        load4(sk + (long)rs * kDK + c4, in[1]);
#pragma unroll
                        for (int part = 0; part < 2; ++part)
#pragma unroll
                            for (int ch = 0; ch < 4; ++ch) y[part][ch] = fmaf(w[part][ch][q], in[part][ch], y[part][ch]);
                    }
                }
                float ss[2] = {0.f, 0.f};
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        y[part][ch] = silu_g(y[part][ch]);
                        ss[part] = fmaf(y[part][ch], y[part][ch], ss[part]);
                    }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    ss[0] += __shfl_xor_sync(kFull, ss[0], o);
                    ss[1] += __shfl_xor_sync(kFull, ss[1], o);
                }
                const float sc[2] = {rsqrtf(ss[0] + 1e-6f) * rsqrtf((float)kDK), rsqrtf(ss[1] + 1e-6f)};
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) y[part][ch] *= sc[part];
            }
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const int row = part == 0 ? p.QOFF + n : n;
                // y = hi + lo, hi rounded to tf32: the dense MMAs read hi, the Gram reads both
                float hv[4], lo[4];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    hv[ch] = tc::tf32_rn(y[part][ch]);
                    lo[ch] = y[part][ch] - hv[ch];
                }
                *reinterpret_cast<float4*>(sKQ + sw_off(row, c4, p.NPAD)) = make_float4(hv[0], hv[1], hv[2], hv[3]);
                *reinterpret_cast<float4*>(sLO + sw_off(row, c4, p.NPAD)) = make_float4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        // padding rows of the tile: [N, QOFF) and [QOFF + N, NPAD)
        const int gap = p.QOFF - N;
        for (int e = tid; e < (p.NPAD - 2 * N) * (kDK / 4); e += kThr) {
            const int pr = e / (kDK / 4), col = (e % (kDK / 4)) * 4;
            const int row = pr < gap ? N + pr : p.QOFF + N + (pr - gap);
            *reinterpret_cast<float4*>(sKQ + sw_off(row, col, p.NPAD)) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(sLO + sw_off(row, col, p.NPAD)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    tc::fence_proxy_async();
    __syncthreads();
    // the q rows are consumed: the first value head's v rows go into their buffer
    const int cv0 = 2 * p.Hk * kDK + g * p.R * kDV;  // x channel of the first value head
    if (tid == 0) {
        tc::mbar_expect_tx(v_full, stage_bytes);
        stage_rows(sv, v_full, cv0);
    }

    // ---- dot products along ancestor chains: the Gram matrix G[t][c] = k_t . kq_c for tile
    //      rows t < 128 and every [k | q] column c holds all k_s . k_t and k_s . q_t.  It is
    //      taken as three tf32 MMAs, hi.hi + lo.hi + hi.lo, which keeps it near fp32 accuracy
    //      (one tf32 product loses too much in the chains of the delta rule).  The lanes of
    //      rows t < n_nodes copy [k.k | k.q] to shared memory, then each node gathers the
    //      entries of its own ancestor chain.
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t gcol = 0;           // D buffer 0, free until the first head's MMA
    float* gram = ubuf;                // [N][2N + 1]: k_t.k_s | k_t.q_s, odd stride (no bank conflicts)
    const int gs = 2 * N + 1;
    if (tid == 32) {
        const uint32_t idesc = tc::idesc_tf32(128, p.NPAD, false, false);
        const uint64_t dh = tc::desc_sw128(tc::smem_u32(sKQ), 16, 1024);
        const uint64_t dl = tc::desc_sw128(tc::smem_u32(sLO), 16, 1024);
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
            const uint64_t da = pass == 1 ? dl : dh, db = pass == 2 ? dl : dh;
#pragma unroll
            for (int kk = 0; kk < kDK / 8; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * (p.NPAD * 128) + (kk & 3) * 32) >> 4);
                tc::mma_tf32_ss(tmem + gcol, da + off, db + off, idesc, (pass | kk) ? 1u : 0u);
            }
        }
        tc::mma_commit(g_done);
    }
    if (tid == 0) {
        // the low parts are dead once the Gram MMAs are done: load the first S0 over them
        if (tc::mbar_wait(g_done, 0, abort_flag)) {
            tc::mbar_expect_tx(full, kDV * kDK * 4);
            for (int blk = 0; blk < kDK / 32; ++blk)
                tc::tma_load_2d(sS0 + blk * (kDV * 128), &tm_s, full, blk * 32, srow0);
        }
    }
    if (warp >= 4 && warp < 12) {
        const int t = (tid & 127);  // tile row = TMEM lane
        const bool gok = __all_sync(kFull, tc::mbar_wait(g_done, 0, abort_flag));
        if (gok) {
            tc::tc_fence_after();
            const uint32_t rowaddr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + gcol;
            // warps 4-7 the k columns [0, N), warps 8-11 the q columns [QOFF, QOFF + N), 32 at a time
            {
                const int part = warp >= 8;
                const int cb = part ? p.QOFF : 0, ob = part ? N : 0;
                for (int c0 = 0; c0 < N; c0 += 32) {
                    uint32_t v0[16], v1[16];
                    const bool two = c0 + 16 < N;
                    tmem_ld16(rowaddr + cb + c0, v0);
                    if (two) tmem_ld16(rowaddr + cb + c0 + 16, v1);
                    tc::tmem_wait_ld();
                    if (t < nn) {
                        float* gr = gram + t * gs + ob + c0;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < N) gr[i] = __uint_as_float(v0[i]);
                        if (two) {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (c0 + 16 + i < N) gr[16 + i] = __uint_as_float(v1[i]);
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < nn * (kMD + 1); e += kThr) {
        const int m = e / nn, t = e % nn;
        const int dep = sdep[t];
        if (m > dep) continue;
        if (m == dep) {
            sqself[t] = gram[t * gs + N + t];  // k_t . q_t
        } else {
            const int s = alist[m * N + t];
            skk[m * N + t] = gram[t * gs + s];      // k_t . k_s
            sqk[m * N + t] = gram[s * gs + N + t];  // k_s . q_t
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();

    // ---- per value head, all 12 warps run the epilogue (each TMEM lane quarter has three
    //      warps, which take every third 8-node chunk).  Lane 0 of warp 0 loads the next
    //      head's S0 once the MMA has read the current one; lane 0 of warp 1 issues the next
    //      head's S0 . [k | q] MMA after the R pass, while the S0 load has long landed.
    const uint32_t mma_idesc = tc::idesc_tf32(128, p.NPAD, false, false);
    const uint32_t sSa = tc::smem_u32(sS0), sKa = tc::smem_u32(sKQ);
    auto issue_mma = [&](int hi) {  // warp 1 lane 0: D[hi & 1] = S0 . [k | q]^T
        const int db = hi & 1;
        if (!tc::mbar_wait(full, hi & 1, abort_flag)) return;
        if (hi >= 2 && !tc::mbar_wait(d_free + db, ((hi - 2) >> 1) & 1, abort_flag)) return;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kDK / 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * (kDV * 128) + (kk & 3) * 32;
            const uint32_t boff = (kk >> 2) * (p.NPAD * 128) + (kk & 3) * 32;
            tc::mma_tf32_ss(tmem + db * p.NPAD, tc::desc_sw128(sSa + aoff, 16, 1024),
                            tc::desc_sw128(sKa + boff, 16, 1024), mma_idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(s_free);
        tc::mma_commit(d_full + db);
    };
    if (warp == 1 && lane == 0) issue_mma(0);
    __syncwarp();
    {
        // --------------------------------------------------------------- epilogue (12 warps)
        const int e = tid;
        const int j = e & (kDV - 1);  // value channel = TMEM lane
        const int quad = e >> 7;      // which of the kQuads interleaved sets of node chunks
        const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        bool dead = false;
        // Per-head arrays come in two buffers (head hi uses buffer hi & 1), so that the
        // gates, chain coefficients and back substitution of head hi + 1 overlap the R and
        // output passes of head hi: two barriers a head.
        //   top of head hi:  back substitution (hi); v rows (hi) landed; R pass (hi);
        //                    gates (hi + 1)
        //   barrier 1:       R rows, M rows (hi) and gates (hi + 1) visible; v rows free:
        //                    one thread stages v rows (hi + 1) by TMA; chain coefficients
        //                    (hi + 1); output pass (hi)
        //   barrier 2:       coefficients (hi + 1) visible; R rows free
        // gates of head hi (already in registers) into buffer hi & 1; next head's into registers
        auto gates = [&](int hi) {
            if (e < nn) {
                sdec[(hi & 1) * N + e] = dec_nx;
                sbeta[(hi & 1) * N + e] = beta_nx;
                if (hi + 1 < p.R) {
                    dec_nx = p.decay[(lb * N + e) * p.Hv + g * p.R + hi + 1];
                    beta_nx = p.beta[(lb * N + e) * p.Hv + g * p.R + hi + 1];
                }
            }
        };
        // chain coefficients A(t, s_m) = b_t G(t, s_m) (k_s.k_t), B(t, s_m) = G(t, s_m) (k_s.q_t)
        // and the path decay g_t of head hi (node e's own row)
        auto coefs = [&](int hi) {
            if (e < nn) {
                const float* dec = sdec + (hi & 1) * N;
                const int dep = sdep[e];
                float gam = dec[e];
                const float bt = sbeta[(hi & 1) * N + e];
                float* cb = scb + (hi & 1) * N * kMD;
                for (int m = 0; m < dep; ++m) {
                    const int s = alist[m * N + e];
                    sca[m * N + e] = bt * gam * skk[m * N + e];
                    cb[m * N + e] = gam * sqk[m * N + e];
                    gam *= dec[s];
                }
                sg[(hi & 1) * N + e] = gam;
            }
        };
        // M = B (I + A)^-1 one row per node, by back substitution along the node's own path
        // p_0 = t, p_k = k-th ancestor:  M(t, p_k) = B(t, p_k) - sum_{i<k} M(t, p_i) A(p_i, p_k),
        // M(t, t) = q_t.k_t.  Then o_t = g_t S0 q_t + sum_k M(t, p_k) R_{p_k}.
        auto backsub = [&](int hi) {
            if (e < nn) {
                const int dep = sdep[e];
                float* cb = scb + (hi & 1) * N * kMD;
                float mrow[kMD + 1];
                mrow[0] = sqself[e];
#pragma unroll
                for (int k = 1; k <= kMD; ++k) {
                    if (k > dep) break;
                    float acc = cb[(k - 1) * N + e];
                    acc = fmaf(-mrow[0], sca[(k - 1) * N + e], acc);
#pragma unroll
                    for (int i = 1; i < k; ++i) {
                        const int pi = alist[(i - 1) * N + e];
                        acc = fmaf(-mrow[i], sca[(k - i - 1) * N + pi], acc);
                    }
                    mrow[k] = acc;
                }
#pragma unroll
                for (int k = 1; k <= kMD; ++k) {
                    if (k > dep) break;
                    cb[(k - 1) * N + e] = mrow[k];  // own row only: B(t, .) is not read by others
                }
            }
        };
        gates(0);
        named_bar(1, kEpi);
        coefs(0);
        named_bar(1, kEpi);
        for (int hi = 0; hi < p.R; ++hi) {
            const int h = g * p.R + hi, db = hi & 1, cur = hi & 1;
            // conv weights of this head's v channel (used by the R pass), loaded a head ahead
            float wv[KT];
#pragma unroll
            for (int q = 0; q < KT; ++q) wv[q] = (q < K) ? to_f32(wv_nx[q]) : 0.f;
            if (warp == 0 && lane == 0 && hi + 1 < p.R && tc::mbar_wait(s_free, hi & 1, abort_flag)) {
                tc::mbar_expect_tx(full, kDV * kDK * 4);  // S0 of the next head over the read one
                for (int blk = 0; blk < kDK / 32; ++blk)
                    tc::tma_load_2d(sS0 + blk * (kDV * 128), &tm_s, full, blk * 32, srow0 + (hi + 1) * kDV);
            }
            __syncwarp();
            // the sca entries read here were written before the last barrier; the next
            // head's coefficients overwrite them only after the next one
            backsub(hi);
            // after a timeout the warp keeps meeting the named barriers but does no work
            if (!dead) dead = !__all_sync(kFull, tc::mbar_wait(d_full + db, (hi >> 1) & 1, abort_flag));
            if (!dead) dead = !__all_sync(kFull, tc::mbar_wait(v_full, hi & 1, abort_flag));
            const float* sbc = sbeta + cur * N;
            const float* sgc = sg + cur * N;
            const float* scbc = scb + cur * N * kMD;
            const uint32_t dcol = tmem + lane_base + db * p.NPAD;
            if (!dead) {
                tc::tc_fence_after();
                // pass A: R_t = b_t (v_t - g_t (S0 k_t)); v_t by the conv along the node's path.
                // Each thread takes whole 8-node chunks (the three warps of a lane quarter
                // take every third chunk), so every loaded column is used and 8 nodes are in
                // flight.
                for (int c = quad; c * 8 < nn; c += kQuads) {
                    const int t0 = c * 8;
                    uint32_t ks[8];
                    tmem_ld8(dcol + t0, ks);
                    float vin[8][KT];
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu) {
                        const int t = min(t0 + uu, nn - 1);
                        if constexpr (KT == 4) {
                            const int4 r4 = *reinterpret_cast<const int4*>(trow + t * 4);
                            vin[uu][0] = to_f32(sv[r4.x * kDV + j]);
                            vin[uu][1] = to_f32(sv[r4.y * kDV + j]);
                            vin[uu][2] = to_f32(sv[r4.z * kDV + j]);
                            vin[uu][3] = to_f32(sv[r4.w * kDV + j]);
                        } else {
#pragma unroll
                            for (int q = 0; q < KT; ++q)
                                vin[uu][q] = (q < K) ? to_f32(sv[trow[t * K + q] * kDV + j]) : 0.f;
                        }
                    }
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu) {
                        const int t = t0 + uu;
                        float acc = 0.f;
#pragma unroll
                        for (int q = 0; q < KT; ++q) acc = fmaf(wv[q], vin[uu][q], acc);
                        if (t < nn) ubuf[t * kDV + j] = sbc[t] * (silu_g(acc) - sgc[t] * __uint_as_float(ks[uu]));
                    }
                }
            }
            if (hi + 1 < p.R) gates(hi + 1);
            named_bar(1, kEpi);
            if (warp == 1 && lane == 0 && hi + 1 < p.R && !dead) issue_mma(hi + 1);
            __syncwarp();
            if (hi + 1 < p.R) {
                if (tid == 0) {  // the R pass is done with the v rows
                    tc::mbar_expect_tx(v_full, stage_bytes);
                    stage_rows(sv, v_full, cv0 + (hi + 1) * kDV);
                }
                const int cv = cv0 + (hi + 1) * kDV + j;
#pragma unroll
                for (int q = 0; q < KT; ++q) wv_nx[q] = wl[(long)cv * K + min(q, K - 1)];
                coefs(hi + 1);
            }
            if (!dead) {
                // pass C: outputs as independent sums over each node's own path; the 8 nodes
                // of a chunk advance one ancestor level at a time, so their loads overlap
                for (int c = quad; c * 8 < N; c += kQuads) {
                    const int t0 = c * 8;
                    uint32_t qs[8];
                    if (t0 < nn) {
                        tmem_ld8(dcol + p.QOFF + t0, qs);
                        tc::tmem_wait_ld();
                    }
                    float ot[8];
                    int dp[8];
                    int md = 0;
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu) {
                        const int t = t0 + uu;
                        dp[uu] = 0;
                        ot[uu] = 0.f;
                        if (t < nn) {
                            dp[uu] = sdep[t];
                            ot[uu] = fmaf(sgc[t], __uint_as_float(qs[uu]), sqself[t] * ubuf[t * kDV + j]);
                        }
                        md = max(md, dp[uu]);
                    }
                    for (int a = 0; a < md; ++a) {
#pragma unroll
                        for (int uu = 0; uu < 8; ++uu) {
                            const int t = t0 + uu;
                            if (a < dp[uu]) ot[uu] = fmaf(scbc[a * N + t], ubuf[alist[a * N + t] * kDV + j], ot[uu]);
                        }
                    }
#pragma unroll
                    for (int uu = 0; uu < 8; ++uu) {
                        const int t = t0 + uu;
                        if (t < N) obase[((long)t * p.Hv + h) * kDV + j] = from_f32<Tout>(ot[uu]);
                    }
                }
                tc::tc_fence_before();
                tc::mbar_arrive(d_free + db);
            }
            named_bar(1, kEpi);  // coefficients of the next head visible; R rows free
        }
    }
    if (warp == 1 && lane == 0) {  // every MMA has completed before TMEM is freed
        tc::mma_commit(drain);
        const long long t0 = clock64();
        while (!tc::mbar_try(drain, 0) && clock64() - t0 < tc::kWaitCycles) {
        }
    }
    __syncwarp();

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && *abort_flag) atomicExch(p.status + b, (int)DDT_ERR_TIMEOUT);
}

// ------------------------------------------------------------------------------ host
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn_gdn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

int qoff_of(int N) { return (N + 15) / 16 * 16; }
int npad_of(int N) { return (qoff_of(N) + N + 15) / 16 * 16; }

}  // namespace

bool gdn_tc_supported(int N, int Hk, int Hv, int dk, int dv, int K, ddt_dtype in) {
    if (dk != kDK || dv != kDV || K < 1 || K > kMaxK || Hv % Hk != 0 || N > gdn_threads(kMaxK)) return false;
    if (npad_of(N) > 256) return false;
    return gdn_tc_layout(N, npad_of(N), K, in == DDT_BF16 ? 2 : 4).total <= 227 * 1024;
}

template <typename Tin, typename Tout, int KT>
static cudaError_t gdn_tc_go_k(const GdnTcParams& prm, const CUtensorMap* maps, cudaStream_t st) {
    const size_t smem = gdn_tc_layout(prm.N, prm.NPAD, prm.K, (int)sizeof(Tin)).total;
    cudaError_t e = cudaFuncSetAttribute(k_gdn_tc<Tin, Tout, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_gdn_tc<Tin, Tout, KT><<<counted(dim3(prm.Hk, prm.B, prm.L)), gdn_threads(KT), smem, st>>>(prm, maps[0], maps[1], maps[2]);
    return cudaGetLastError();
}

// the common conv width 4 gets its own instance; any other width up to kMaxK the generic one
template <typename Tin, typename Tout>
static cudaError_t gdn_tc_go(const GdnTcParams& prm, const CUtensorMap* maps, cudaStream_t st) {
    return prm.K == 4 ? gdn_tc_go_k<Tin, Tout, 4>(prm, maps, st) : gdn_tc_go_k<Tin, Tout, kMaxK>(prm, maps, st);
}

cudaError_t launch_gdn_tc(int L, int B, int N, int Hk, int Hv, int K, ddt_dtype in, ddt_dtype out, const void* x,
                          const void* conv_w, const void* conv_state, const float* beta, const float* decay,
                          const float* S, const int32_t* parent, const int32_t* n_nodes, void* o, int32_t* status,
                          cudaStream_t st) {
    EncodeTiledFn enc = encode_fn_gdn();
    if (!enc) return cudaErrorNotSupported;
    GdnTcParams prm;
    prm.L = L;
    prm.B = B;
    prm.N = N;
    prm.Hk = Hk;
    prm.Hv = Hv;
    prm.R = Hv / Hk;
    prm.K = K;
    prm.C = 2 * Hk * kDK + Hv * kDV;
    prm.QOFF = qoff_of(N);
    prm.NPAD = npad_of(N);
    prm.x = x;
    prm.conv_w = conv_w;
    prm.wvec = (reinterpret_cast<uintptr_t>(conv_w) & 15) == 0;
    prm.conv_state = conv_state;
    prm.beta = beta;
    prm.decay = decay;
    prm.parent = parent;
    prm.n_nodes = n_nodes;
    prm.o = o;
    prm.status = status;
    // committed states as a 2-D fp32 tensor: rows (layer, request, value head, value
    // channel), columns the key channel; boxes of 32 columns x 128 rows
    CUtensorMap maps[3];
    const cuuint64_t dims[2] = {(cuuint64_t)kDK, (cuuint64_t)L * B * Hv * kDV};
    const cuuint64_t strides[1] = {(cuuint64_t)kDK * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)kDV};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&maps[0], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(S), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // x rows (layer, request, node) and conv-state rows (layer, request, tap) as 2-D tensors
    // of C channels; boxes of 128 channels x all N node rows (or the K - 1 state rows),
    // unswizzled, so a box lands as the [rows][128] staging layout
    const size_t esz = in == DDT_BF16 ? 2 : 4;
    const CUtensorMapDataType dt = in == DDT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const cuuint64_t cstride[1] = {(cuuint64_t)prm.C * esz};
    const cuuint64_t xdims[2] = {(cuuint64_t)prm.C, (cuuint64_t)L * B * N};
    const cuuint32_t xbox[2] = {128, (cuuint32_t)N};
    if (enc(&maps[1], dt, 2, const_cast<void*>(x), xdims, cstride, xbox, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    maps[2] = maps[1];  // (no conv-state rows to stage when K == 1)
    if (K > 1) {
        const cuuint64_t cdims[2] = {(cuuint64_t)prm.C, (cuuint64_t)L * B * (K - 1)};
        const cuuint32_t cbox[2] = {128, (cuuint32_t)(K - 1)};
        if (enc(&maps[2], dt, 2, const_cast<void*>(conv_state), cdims, cstride, cbox, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // status words start at DDT_OK; CTAs only ever write errors into them
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t) * B, st);
    if (e != cudaSuccess) return e;
    const bool ib = in == DDT_BF16, ob = out == DDT_BF16;
    if (ib && ob) return gdn_tc_go<__nv_bfloat16, __nv_bfloat16>(prm, maps, st);
    if (ib) return gdn_tc_go<__nv_bfloat16, float>(prm, maps, st);
    if (ob) return gdn_tc_go<float, __nv_bfloat16>(prm, maps, st);
    return gdn_tc_go<float, float>(prm, maps, st);
}

}  // namespace ddt
