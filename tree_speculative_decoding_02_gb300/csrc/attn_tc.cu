// attn_tc.cu -- ddt_tree_attn on the 5th-generation tensor cores (bf16 in, fp32 accumulate).
//
// "DDTree on vLLM: candid research notes", section "Why hybrid attention makes it hard":
// each candidate row sees the committed prefix plus its own ancestors, never its
// siblings.  "From Tree-Based Speculative Decoding to Drafter Training", section "The
// Architecture of DDTree": one target pass over the flattened tree with an
// ancestor-only mask.
//
// Work unit (one CTA): a layer, a request, a kv head g, a 128-row M-tile of that head's
// query rows (row = node * G + head-in-group, G = Hq/Hkv, so the whole GQA group shares
// one K/V stream), and a chunk of the prefix.  The chunk holding the prefix's end also
// takes the tree rows as keys.  Keys stream in tiles of 64:
//   warp 0      TMA producer: K and V tiles into a shared-memory ring of 6 (d = 256) or
//               8 stages (128-byte swizzle).  Prefix tiles come from a 3-D map (d, position, layer*B*Hkv);
//               the ragged last tile is shifted to end exactly at prefix_len, so no row
//               past the prefix is ever read (positions < 0 are zero-filled by TMA).
//               Tree tiles come from a 4-D map (d, kv head, node, layer*B).
//   warp 1      MMA issuer: S_j = Q K_j^T into one of two TMEM buffers (Q is the A operand,
//               kept in TMEM); O += P_j V_j with P_j read back from TMEM (written over S_j)
//               and V_j MN-major in shared memory.  P_j is stored as two bf16 parts,
//               P = P_hi + P_lo, and both are applied (two MMAs): bf16 P alone would leave
//               ~3e-3 relative error in O, the pair ~1e-5.  This thread bounds the kernel:
//               a 64-key tile is 16 QK MMAs of N = 64 (which run at about half the tensor
//               rate) and 8 P.V MMAs of N = 256, and the softmax keeps ahead of it.
//   warps 4-11  softmax: two warpgroups per row set, each taking half of every S tile's
//               columns and half of O's; ancestor mask on tree tiles, running max with
//               lazy O rescaling (only when the max grows by more than 2^8); zeroes V rows
//               of padding tree nodes before their MMA; epilogue O / l to global (or a
//               split-KV partial that k_attn_merge combines).
// Every mbarrier wait is bounded; on a timeout the CTA drains its copies and MMAs,
// frees TMEM, and reports DDT_ERR_TIMEOUT in the request's status word.
#include <cuda.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace ddt {

namespace {

constexpr int kBM = 128;     // query rows per CTA (TMEM lanes)
constexpr int kBN = 64;      // keys per tile
constexpr float kTau = 8.f;  // rescale O only when the row max grows by more than 2^kTau

struct TcParams {
    int L, B, N, Hq, Hkv, G, MT, S, chunk, Pcap, W;
    int MP;  // pair kernel: 256-row tiles per (layer, request, kv head); MT = 2 MP there
    // paged prefix caches: page_rows positions a page, block_table [B][max_pages] of
    // physical pages out of num_pages (paged == 0: one contiguous slab per request)
    int paged, page_rows, num_pages, max_pages;
    const int32_t* block_table;
    const __nv_bfloat16* q;
    const int32_t* prefix_len;
    const int32_t* n_nodes;
    const uint32_t* anc;
    const int32_t* perm;  // requests by prefix length, longest first
    void* o;              // final output (S == 1)
    float* part_o;        // [S][L][B][Hkv][MT*128][D] unnormalised partial O (S > 1)
    float2* part_ml;      // [S][L][B][Hkv][MT*128] (row max in log2 units, row sum)
    int32_t* status;
    float scale_log2;
    // rotary embedding of q by tree-row position (rope_rot == 0: q is already rotated):
    // pairs (i, i + rope_rot / 2) of the first rope_rot channels, cos/sin per row from
    // rope_table [B][N][rope_rot]
    int rope_rot;
    const float* rope_table;
};

constexpr int kThreads = 384;  // 0 TMA, 1 MMA, 2-3 setup, 4-11 softmax

template <int D>
struct TcCfg {
    static constexpr int kBlocks = D / 64;              // 128-byte-swizzle column blocks
    static constexpr int kStageBytes = kBN * D * 2;
    // K/V ring depth (K and V tiles alternate): as deep as shared memory allows, so that
    // about three tiles of keys are in flight per CTA
    static constexpr int kStages = D == 256 ? 6 : 8;
    // TMEM columns: S double buffer [0, 2 kBN), O [kOCol, kOCol + D), Q (bf16, two per
    // column, the A operand of S = Q K^T) [kQCol, kQCol + D/2)
    static constexpr int kOCol = 2 * kBN;
    static constexpr int kQCol = kOCol + D;
    static constexpr int kTmemCols = (kQCol + D / 2) <= 256 ? 256 : 512;
    static constexpr int kBarBytes = 512;
    static constexpr int kXchBytes = 4096;  // softmax halves: tile row max (x2 parity), row sum
    static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes + kXchBytes;
};

struct Tile {
    int tree;  // 0 = prefix tile, 1 = tree tile
    int y;     // first key: prefix position or tree node
    int lo;    // prefix tiles: keys below lo were handled by the previous tile
};

// ragged: the chunk's last prefix tile is partial.  Contiguous caches shift it to end at
// the chunk's end (no row past the prefix is read); paged caches keep it aligned (a
// shifted tile could straddle pages) and mask the rows past the end instead.
__device__ __forceinline__ Tile tile_of(int j, int n_pre, int c0, int c1, bool ragged) {
    Tile t;
    if (j < n_pre) {
        t.tree = 0;
        t.lo = c0 + j * kBN;
        t.y = (j == n_pre - 1 && ragged) ? c1 - kBN : t.lo;
    } else {
        t.tree = 1;
        t.y = (j - n_pre) * kBN;
        t.lo = 0;
    }
    return t;
}

// Bounded wait that ignores the abort flag: used only to drain in-flight work.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!tc::mbar_try(bar, parity))
        if (clock64() - t0 > tc::kWaitCycles) return;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <typename Tout>
__device__ __forceinline__ void store_row32(Tout* dst, const float* v);
template <>
__device__ __forceinline__ void store_row32<float>(float* dst, const float* v) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}
template <>
__device__ __forceinline__ void store_row32<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
        uint4 u;
        u.x = pack_bf16(v[i], v[i + 1]);
        u.y = pack_bf16(v[i + 2], v[i + 3]);
        u.z = pack_bf16(v[i + 4], v[i + 5]);
        u.w = pack_bf16(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4*>(dst + i) = u;
    }
}

}  // namespace

template <int D, typename Tout>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const TcParams p, const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
              const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt) {
    using Cfg = TcCfg<D>;
    extern __shared__ unsigned char smem_raw[];
    // align to 1024 B by pointer arithmetic on the shared array (keeps the address space)
    unsigned char* base = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int kStages = Cfg::kStages;
    unsigned char* sRing = base;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + kStages * Cfg::kStageBytes);
    uint64_t* full = bars;                 // [kStages] TMA landed
    // [kSlots] tile slot free: the P.V MMAs of the slot's last tile are done, so its K and
    // V stages may be refilled and O holds that tile.  One commit per tile instead of one
    // per stage and one more for O: each commit costs the single issuing thread ~100 cycles.
    constexpr int kSlots = kStages / 2;
    uint64_t* tfree = bars + kStages;
    uint64_t* s_full = bars + 2 * kStages; // [2] S_j in TMEM
    uint64_t* p_full = s_full + 2;         // [2] P_j in TMEM (128 arrivals)
    uint64_t* drain = p_full + 2;
    // Single-phase barrier for the epilogue: a tile-slot barrier may be behind by more
    // than one phase when the softmax finishes, which a parity wait cannot tell apart.
    uint64_t* o_final = drain + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_final + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    float* xch = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(bars) + Cfg::kBarBytes);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int x = blockIdx.x;
    const int s = x % p.S;
    x /= p.S;
    const int mt = x % p.MT;
    x /= p.MT;
    const int g = x % p.Hkv;
    const int l = x / p.Hkv;
    const int b = p.perm[blockIdx.y];
    const long lb = (long)l * p.B + b;
    const int P = p.prefix_len[b], nn = p.n_nodes[b];
    bool bad = P < 0 || P > p.Pcap || nn < 1 || nn > p.N;
    int bad_table = 0;
    if (p.paged && !bad) {  // every page the prefix uses must exist
        const int np = (P + p.page_rows - 1) / p.page_rows;
        for (int i = tid; i < np; i += kThreads) {
            const int pg = p.block_table[(long)b * p.max_pages + i];
            bad_table |= (pg < 0 || pg >= p.num_pages);
        }
    }
    bad_table = __syncthreads_or(bad_table);
    bad = bad || bad_table;
    const long prow0 = ((((long)s * p.L + l) * p.B + b) * p.Hkv + g) * (long)(p.MT * kBM) + mt * kBM;

    if (bad) {
        if (tid == 0 && s == 0 && mt == 0 && g == 0 && l == 0)
            p.status[b] = (P < 0 || P > p.Pcap) ? DDT_ERR_CAPACITY : (bad_table ? DDT_ERR_INVALID_ARG : DDT_ERR_TREE);
        if (p.S == 1) {
            for (int e = tid; e < kBM * D; e += kThreads) {
                const int R = mt * kBM + e / D;
                if (R >= p.N * p.G) continue;
                const int node = R / p.G, h = g * p.G + R % p.G;
                static_cast<Tout*>(p.o)[((lb * p.N + node) * p.Hq + h) * D + e % D] = from_f32<Tout>(0.f);
            }
        } else if (tid < kBM) {
            p.part_ml[prow0 + tid] = make_float2(-INFINITY, 0.f);
        }
        return;
    }

    const int c0 = s * p.chunk;
    const int s_last = P > 0 ? (P - 1) / p.chunk : 0;
    int n_pre = 0, c1 = c0;
    if (c0 < P) {
        c1 = min(c0 + p.chunk, P);
        n_pre = (c1 - c0 + kBN - 1) / kBN;
    }
    const int n_tree = (s == s_last) ? (nn + kBN - 1) / kBN : 0;
    const int T = n_pre + n_tree;
    const bool ragged = !p.paged && ((c1 - c0) % kBN) != 0;
    if (T == 0) {  // an empty split (only when S > 1)
        if (tid < kBM) p.part_ml[prow0 + tid] = make_float2(-INFINITY, 0.f);
        return;
    }

    // ---- setup: barriers, TMEM, Q rows into TMEM
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(full + i, 1);
            if (i < kSlots) tc::mbar_init(tfree + i, 1);
        }
        tc::mbar_init(s_full, 1);
        tc::mbar_init(s_full + 1, 1);
        tc::mbar_init(p_full, 256);
        tc::mbar_init(p_full + 1, 256);
        tc::mbar_init(drain, 1);
        tc::mbar_init(o_final, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tc::tmem_relinquish();
    }
    if (tid == 64) {
        tc::prefetch_tmap(&tm_kc);
        tc::prefetch_tmap(&tm_vc);
        tc::prefetch_tmap(&tm_kt);
        tc::prefetch_tmap(&tm_vt);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Q rows into TMEM (lane = query row): the softmax warps, half hf writes columns
    // [hf D/4, (hf+1) D/4) of the packed bf16 row
    if (warp >= 4 && warp < 12) {
        const int hf = (warp - 4) >> 2, ws = (warp - 4) & 3, r = 32 * ws + lane;
        const int R = mt * kBM + r;
        const __nv_bfloat16* qrow = nullptr;
        if (R < p.N * p.G) {
            const int node = R / p.G, h = g * p.G + R % p.G;
            if (node < nn) qrow = p.q + ((lb * p.N + node) * p.Hq + h) * D;
        }
        const uint32_t qaddr = tmem + (static_cast<uint32_t>(32 * ws) << 16) + Cfg::kQCol + hf * (D / 4);
#pragma unroll
        for (int cb = 0; cb < D / 4; cb += 16) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                uint4 v = make_uint4(0, 0, 0, 0);
                if (qrow) v = __ldg(reinterpret_cast<const uint4*>(qrow + hf * (D / 2) + 2 * (cb + i)));
                w[i] = v.x;
                w[i + 1] = v.y;
                w[i + 2] = v.z;
                w[i + 3] = v.w;
            }
            tc::tmem_st16(qaddr + cb, w);
        }
        tc::tmem_wait_st();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();


    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            const int grp = (int)((lb * p.Hkv) + g);
            int issued = 0;
            for (int j = 0; j < T && !*abort_flag; ++j) {
                const Tile t = tile_of(j, n_pre, c0, c1, ragged);
                // both stages of tile j sit in slot j % kSlots (stages 2j and 2j + 1 mod kStages)
                bool ok = tc::mbar_wait(tfree + j % kSlots, ((j / kSlots) & 1) ^ 1, abort_flag);
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int u = 2 * j + kv, st = u % kStages;
                    tc::mbar_expect_tx(full + st, Cfg::kStageBytes);
                    unsigned char* dst = sRing + st * Cfg::kStageBytes;
                    if (!t.tree && p.paged) {
                        // one box per page slice of the tile (pages of fewer than 64 rows);
                        // rows past the prefix come from its last page and are masked
                        const int sub = min(kBN, p.page_rows), last = (P - 1) / p.page_rows;
                        for (int r0 = 0; r0 < kBN; r0 += sub) {
                            const int pos = t.y + r0;
                            const int lp = min(pos / p.page_rows, last);
                            const int phys = p.block_table[(long)b * p.max_pages + lp];
                            const int plane = (int)(((long)l * p.num_pages + phys) * p.Hkv + g);
#pragma unroll
                            for (int blk = 0; blk < Cfg::kBlocks; ++blk)
                                tc::tma_load_3d(dst + blk * (kBN * 128) + r0 * 128, kv ? &tm_vc : &tm_kc, full + st,
                                                blk * 64, pos % p.page_rows, plane);
                        }
                    } else {
#pragma unroll
                        for (int blk = 0; blk < Cfg::kBlocks; ++blk) {
                            if (!t.tree)
                                tc::tma_load_3d(dst + blk * (kBN * 128), kv ? &tm_vc : &tm_kc, full + st, blk * 64, t.y,
                                                grp);
                            else
                                tc::tma_load_4d(dst + blk * (kBN * 128), kv ? &tm_vt : &tm_kt, full + st, blk * 64, g,
                                                t.y, (int)lb);
                        }
                    }
                    issued = u + 1;
                }
                if (!ok) break;
            }
            for (int u = max(0, issued - kStages); u < issued; ++u) drain_wait(full + u % kStages, (u / kStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = tc::idesc_bf16(kBM, kBN, false, false);
            constexpr uint32_t idesc_pv = tc::idesc_bf16(kBM, D, false, true);
            const uint32_t sRa = tc::smem_u32(sRing);
            // Descriptors are built once; a k-step or a ring stage only moves the start
            // address, i.e. adds (byte offset >> 4) to the low 14-bit field, which cannot
            // overflow for addresses inside this CTA's shared memory.  Keeping the per-MMA
            // work to one add matters: the single issuing thread, not the tensor core, was
            // the bound when every MMA rebuilt its 64-bit descriptor.
            const uint64_t kdesc0 = tc::desc_sw128(sRa, 16, 1024);
            const uint64_t vdesc0 = tc::desc_sw128(sRa, kBN * 128, 1024);
            auto pv = [&](int i) -> bool {
                if (!tc::mbar_wait(p_full + (i & 1), (i >> 1) & 1, abort_flag)) return false;
                const int u = 2 * i + 1, st = u % kStages;
                if (!tc::mbar_wait(full + st, (u / kStages) & 1, abort_flag)) return false;
                tc::tc_fence_after();
                const uint64_t vd = vdesc0 + static_cast<uint64_t>((st * Cfg::kStageBytes) >> 4);
                const uint32_t pa = tmem + (i & 1) * kBN;
                // first MMA of the chunk may start the accumulator, the rest accumulate
                tc::mma_f16_ts(tmem + Cfg::kOCol, pa, vd, idesc_pv, i > 0 ? 1u : 0u);
#pragma unroll
                for (int q = 1; q < 2 * (kBN / 16); ++q) {  // P_hi k-steps, then P_lo k-steps
                    const int part = q / (kBN / 16), kk = q % (kBN / 16);
                    // V tile: 16 keys = two 8-row swizzle atoms down the K dimension
                    tc::mma_f16_ts_acc(tmem + Cfg::kOCol, pa + part * (kBN / 2) + kk * 8,
                                       vd + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv);
                }
                tc::mma_commit(tfree + i % kSlots);
                return true;
            };
            bool ok = true;
            for (int j = 0; j < T && ok; ++j) {
                const int u = 2 * j, st = u % kStages;
                if (!tc::mbar_wait(full + st, (u / kStages) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint64_t kd = kdesc0 + static_cast<uint64_t>((st * Cfg::kStageBytes) >> 4);
                const uint32_t sd = tmem + (j & 1) * kBN, qa = tmem + Cfg::kQCol;
                tc::mma_f16_ts(sd, qa, kd, idesc_qk, 0u);
#pragma unroll
                for (int kk = 1; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;
                    tc::mma_f16_ts_acc(sd, qa + kk * 8, kd + static_cast<uint64_t>(koff >> 4), idesc_qk);
                }
                tc::mma_commit(s_full + (j & 1));
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok && pv(T - 1)) tc::mma_commit(o_final);
            tc::mma_commit(drain);
            drain_wait(drain, 0);
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------------ softmax
        // Two warpgroups share each row: half hf takes key columns [32 hf, 32 hf + 32) of
        // every S tile and value columns [hf D/2, (hf+1) D/2) of O.  The tile's row max is
        // exchanged through shared memory, so both halves keep the same reference max.
        const int hf = (warp - 4) >> 2, ws = (warp - 4) & 3, r = 32 * ws + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * ws) << 16;
        const int R = mt * kBM + r;
        const bool in_rows = R < p.N * p.G;
        const int node = in_rows ? R / p.G : 0;
        const int h = g * p.G + (in_rows ? R % p.G : 0);
        const bool live = in_rows && node < nn;
        const uint32_t* anc_row = p.anc + ((long)b * p.N + node) * p.W;
        float m_used = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const Tile t = tile_of(j, n_pre, c0, c1, ragged);
            if (ok) ok = tc::mbar_wait(s_full + (j & 1), (j >> 1) & 1, abort_flag);
            ok = __all_sync(kFull, ok);
            float sv[32];
            float mtile = -INFINITY;
            if (ok) {
                tc::tc_fence_after();
                uint32_t sr[32];
                tc::tmem_ld32(tmem + lane_base + (j & 1) * kBN + 32 * hf, sr);
                tc::tmem_wait_ld();
                uint32_t vis;
                if (!t.tree) {
                    const int skip = t.lo - t.y - 32 * hf;  // keys of this half already seen
                    const int lim = c1 - t.y - 32 * hf;     // keys of this half before the chunk's end
                    vis = skip <= 0 ? ~0u : (skip >= 32 ? 0u : (~0u << skip));
                    vis &= lim >= 32 ? ~0u : (lim <= 0 ? 0u : ((1u << lim) - 1u));
                } else {
                    const int w = (t.y >> 5) + hf;
                    vis = (live && w < p.W) ? anc_row[w] : 0u;
                }
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sv[c] = ((vis >> c) & 1u) ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
                    mtile = fmaxf(mtile, sv[c]);
                }
            }
            // row max of the whole tile: exchange with the other half
            float* xm = xch + (j & 1) * 256;
            xm[hf * 128 + r] = mtile;
            tc::named_bar(1, 256);
            mtile = fmaxf(mtile, xm[(hf ^ 1) * 128 + r]);
            if (!ok) continue;
            // lazy rescale: only when the max grows by more than 2^kTau
            const bool grow = mtile > m_used + kTau;
            const bool need = grow && (m_used != -INFINITY);  // O already holds this row's data
            if (__any_sync(kFull, need)) {
                ok = __all_sync(kFull, tc::mbar_wait(tfree + (j - 1) % kSlots, ((j - 1) / kSlots) & 1, abort_flag));
                if (!ok) continue;
                tc::tc_fence_after();
                const float f = need ? tc::ex2(m_used - mtile) : 1.f;
#pragma unroll 1
                for (int cb = hf * (D / 2); cb < (hf + 1) * (D / 2); cb += 32) {
                    uint32_t ov[32];
                    tc::tmem_ld32(tmem + lane_base + Cfg::kOCol + cb, ov);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
                    tc::tmem_st32(tmem + lane_base + Cfg::kOCol + cb, ov);
                }
                tc::tmem_wait_st();
                if (need) l_run *= f;
            }
            if (grow) m_used = mtile;
            uint32_t phi[16], plo[16];
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
                const float a = (sv[c] == -INFINITY) ? 0.f : tc::ex2(sv[c] - m_used);
                const float bb = (sv[c + 1] == -INFINITY) ? 0.f : tc::ex2(sv[c + 1] - m_used);
                sum += a + bb;
                const __nv_bfloat162 hi = __floats2bfloat162_rn(a, bb);
                phi[c >> 1] = *reinterpret_cast<const uint32_t*>(&hi);
                plo[c >> 1] = pack_bf16(a - __low2float(hi), bb - __high2float(hi));
            }
            l_run += sum;
            if (t.tree || t.y + kBN > c1) {
                // V rows of padding nodes (or, paged, rows past the prefix) may hold anything,
                // even NaN: zero them before the MMA reads them (a zero P does not cancel NaN)
                const int u = 2 * j + 1, st = u % kStages;
                ok = __all_sync(kFull, tc::mbar_wait(full + st, (u / kStages) & 1, abort_flag));
                const int first = t.tree ? max(0, nn - t.y) : c1 - t.y;
                if (ok && first < kBN) {
                    unsigned char* vst = sRing + st * Cfg::kStageBytes;
                    const int per_blk = (kBN - first) * 8;
                    for (int e = hf * 128 + r; e < per_blk * Cfg::kBlocks; e += 256) {
                        const int blk = e / per_blk, rem = e % per_blk;
                        *reinterpret_cast<uint4*>(vst + blk * (kBN * 128) + (first + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    tc::fence_proxy_async();
                }
                if (!ok) continue;
            }
            tc::tmem_st16(tmem + lane_base + (j & 1) * kBN + 16 * hf, phi);
            tc::tmem_st16(tmem + lane_base + (j & 1) * kBN + kBN / 2 + 16 * hf, plo);
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(p_full + (j & 1));
        }
        if (ok) ok = tc::mbar_wait(o_final, 0, abort_flag);
        ok = __all_sync(kFull, ok);
        // row sum of both halves
        xch[512 + hf * 128 + r] = l_run;
        tc::named_bar(1, 256);
        const float l_tot = l_run + xch[512 + (hf ^ 1) * 128 + r];
        if (ok) {
            tc::tc_fence_after();
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll 1
            for (int cb = hf * (D / 2); cb < (hf + 1) * (D / 2); cb += 32) {
                uint32_t ov[32];
                tc::tmem_ld32(tmem + lane_base + Cfg::kOCol + cb, ov);
                tc::tmem_wait_ld();
                float f[32];
                if (p.S == 1) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] = live ? __uint_as_float(ov[i]) * inv : 0.f;
                    if (in_rows)
                        store_row32<Tout>(static_cast<Tout*>(p.o) + ((lb * p.N + node) * p.Hq + h) * D + cb, f);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(ov[i]);
                    store_row32<float>(p.part_o + (prow0 + r) * D + cb, f);
                }
            }
            if (p.S > 1 && hf == 0) p.part_ml[prow0 + r] = make_float2(m_used, l_tot);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, Cfg::kTmemCols);
    }
    if (tid == 0 && *abort_flag) atomicExch(p.status + b, (int)DDT_ERR_TIMEOUT);
}

// ------------------------------------------------------------------------------------
// The CTA-pair kernel (head sizes 128 and 256).  Two CTAs on a pair of SMs (a cluster of
// two) share each MMA (tcgen05 cta_group::2): one 256-row M tile, 128 query rows per
// CTA, and 128 keys per tile, so S = Q K^T runs as N = 128 MMAs at the full tensor rate
// and every MMA does twice the work of a one-SM instruction.  Each CTA keeps its own
// 128 query rows in shared memory (the A operand), loads half of every key tile (64 keys
// x d for Q K^T, all 128 keys x d/2 value columns for P V), and receives its rows of S
// and O in its own tensor memory: S/P double buffer in columns [0, 256), O in
// [256, 256 + d).  Roles:
//   warp 0      TMA producer in each CTA (its own halves).  K halves report to the even
//               CTA's barrier (the MMA waits there for both); V halves to the CTA's own,
//               which its softmax warps wait on.
//   warp 1      MMA issuer, even CTA only.
//   warps 4-11  softmax, as in k_attn_tc but over 64 keys per thread; once P_j is in
//               tensor memory and the CTA's V_j half has landed (padding rows zeroed),
//               each warp arrives on the even CTA's P barrier: that arrival certifies
//               both P and V of the CTA.
// Every wait is bounded; the even CTA drains both CTAs' K loads, each CTA its own V loads,
// and a cluster barrier keeps either CTA from leaving while the pair may still touch it.
namespace {
constexpr int kPN = 128;  // keys per tile of the pair kernel

template <int D>
struct Tc2Cfg {
    static constexpr int kBlocks = D / 64;
    static constexpr int kQBytes = 128 * D * 2;     // this CTA's query rows
    static constexpr int kStageBytes = 64 * D * 2;  // a K half (64 keys x D) or a V half (128 keys x D/2)
    // separate K and V rings: a K stage frees as its tile's Q K^T finishes, about 5000
    // cycles before the tile two ahead needs it; a V stage frees only as its tile's P.V
    // finishes, so V gets the deeper ring
    static constexpr int kKS = D == 256 ? 2 : 4;
    static constexpr int kVS = D == 256 ? 3 : 4;
    static constexpr int kStages = kKS + kVS;
    static constexpr int kOCol = 2 * kPN;
    static constexpr int kBarBytes = 256;
    static constexpr int kXchBytes = 2048;  // row maxima of the two column halves (two parities)
    static constexpr int kUsed = kQBytes + kStages * kStageBytes + kBarBytes + kXchBytes;
    // dynamic shared memory requested: what the layout uses plus room to align it to 1024
    // bytes, capped at the per-block maximum; the kernel checks the slack it gets
    static constexpr int kSmem = kUsed + 1024 <= 232448 ? kUsed + 1024 : 232448;
};

__device__ __forceinline__ Tile tile2_of(int j, int n_pre, int c0, int c1, bool ragged) {
    Tile t;
    if (j < n_pre) {
        t.tree = 0;
        t.lo = c0 + j * kPN;
        t.y = (j == n_pre - 1 && ragged) ? c1 - kPN : t.lo;
    } else {
        t.tree = 1;
        t.y = (j - n_pre) * kPN;
        t.lo = 0;
    }
    return t;
}

// visibility bits of 32 consecutive keys starting at key k0 of a prefix tile
__device__ __forceinline__ uint32_t prefix_vis(int lo, int c1, int k0) {
    const int skip = lo - k0, lim = c1 - k0;
    uint32_t v = skip <= 0 ? ~0u : (skip >= 32 ? 0u : (~0u << skip));
    v &= lim >= 32 ? ~0u : (lim <= 0 ? 0u : ((1u << lim) - 1u));
    return v;
}
}  // namespace

template <int D, typename Tout>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_attn_tc2(const TcParams p, const __grid_constant__ CUtensorMap tm_kc, const __grid_constant__ CUtensorMap tm_vc,
               const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt) {
    using Cfg = Tc2Cfg<D>;
    constexpr int kStages = Cfg::kStages, kKS = Cfg::kKS, kVS = Cfg::kVS;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t slack = (1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u;
    unsigned char* base = smem_raw + slack;
    unsigned char* sQ = base;
    unsigned char* sRing = base + Cfg::kQBytes;  // stages [0, kKS): K ring; [kKS, kStages): V ring
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + kStages * Cfg::kStageBytes);
    uint64_t* full = bars;                 // [kStages] K: both CTAs' halves (even CTA's copy); V: own half
    uint64_t* sfree = bars + kStages;      // [kStages] the MMAs that read the stage are done (both CTAs)
    uint64_t* s_full = bars + 2 * kStages; // [2] S_j in tensor memory (both CTAs)
    // [2] P_j and V_j ready: in the even CTA its 8 softmax warps plus one arrival forwarded
    // from the odd CTA; in the odd CTA its own 8 warps (which a forwarding thread waits on)
    uint64_t* p_full = s_full + 2;
    uint64_t* drain = p_full + 2;
    uint64_t* o_final = drain + 1;         // single phase: O complete (both CTAs)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_final + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    float* xch = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(bars) + Cfg::kBarBytes);

    const uint32_t rank = tc::cluster_ctarank();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int x = blockIdx.x >> 1;
    const int s = x % p.S;
    x /= p.S;
    const int mp = x % p.MP;
    x /= p.MP;
    const int g = x % p.Hkv;
    const int l = x / p.Hkv;
    const int b = p.perm[blockIdx.y];
    const long lb = (long)l * p.B + b;
    const int row0 = mp * 256 + (int)rank * 128;  // this CTA's first query row
    const int P = p.prefix_len[b], nn = p.n_nodes[b];
    bool bad = P < 0 || P > p.Pcap || nn < 1 || nn > p.N;
    int bad_table = 0;
    if (p.paged && !bad) {  // every page the prefix uses must exist
        const int np = (P + p.page_rows - 1) / p.page_rows;
        for (int i = tid; i < np; i += kThreads) {
            const int pg = p.block_table[(long)b * p.max_pages + i];
            bad_table |= (pg < 0 || pg >= p.num_pages);
        }
    }
    bad_table = __syncthreads_or(bad_table);
    bad = bad || bad_table;
    const long prow0 = ((((long)s * p.L + l) * p.B + b) * p.Hkv + g) * (long)(p.MP * 256) + row0;
    if (slack + Cfg::kUsed > (uint32_t)Cfg::kSmem) {  // the layout would not fit: refuse, touch nothing
        if (tid == 0) atomicExch(p.status + b, (int)DDT_ERR_UNSUPPORTED);
        return;
    }
    // (both CTAs of a pair see the same request, so they leave here together)
    if (bad) {
        if (tid == 0 && rank == 0 && s == 0 && mp == 0 && g == 0 && l == 0)
            p.status[b] = (P < 0 || P > p.Pcap) ? DDT_ERR_CAPACITY : (bad_table ? DDT_ERR_INVALID_ARG : DDT_ERR_TREE);
        if (p.S == 1) {
            for (int e = tid; e < 128 * D; e += kThreads) {
                const int R = row0 + e / D;
                if (R >= p.N * p.G) continue;
                const int node = R / p.G, h = g * p.G + R % p.G;
                static_cast<Tout*>(p.o)[((lb * p.N + node) * p.Hq + h) * D + e % D] = from_f32<Tout>(0.f);
            }
        } else if (tid < 128) {
            p.part_ml[prow0 + tid] = make_float2(-INFINITY, 0.f);
        }
        return;
    }
    const int c0 = s * p.chunk;
    const int s_last = P > 0 ? (P - 1) / p.chunk : 0;
    int n_pre = 0, c1 = c0;
    if (c0 < P) {
        c1 = min(c0 + p.chunk, P);
        n_pre = (c1 - c0 + kPN - 1) / kPN;
    }
    const int n_tree = (s == s_last) ? (nn + kPN - 1) / kPN : 0;
    const int T = n_pre + n_tree;
    const bool ragged = !p.paged && ((c1 - c0) % kPN) != 0;
    if (T == 0) {
        if (tid < 128) p.part_ml[prow0 + tid] = make_float2(-INFINITY, 0.f);
        return;
    }

    // ---- setup: barriers, tensor memory (allocated for the pair), Q rows into shared memory
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(full + i, 1);
            tc::mbar_init(sfree + i, 1);
        }
        tc::mbar_init(s_full, 1);
        tc::mbar_init(s_full + 1, 1);
        tc::mbar_init(p_full, rank == 0 ? 9 : 8);
        tc::mbar_init(p_full + 1, rank == 0 ? 9 : 8);
        tc::mbar_init(drain, 1);
        tc::mbar_init(o_final, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc2(tmem_slot, 512);
        tc::tmem_relinquish2();
    }
    if (tid == 64) {
        tc::prefetch_tmap(&tm_kc);
        tc::prefetch_tmap(&tm_vc);
        tc::prefetch_tmap(&tm_kt);
        tc::prefetch_tmap(&tm_vt);
    }
    // Q: 128 rows x D bf16, K-major with the 128-byte swizzle (64-column blocks of 128 rows).
    // With a rotary table, 16-byte chunk c < rot/16 and its partner c + rot/16 are rotated
    // together in fp32 (the arithmetic of ddt_rope_tree) and rounded once to bf16.
    {
        auto qstore = [&](int r, int c, uint4 v) {
            *reinterpret_cast<uint4*>(sQ + (c >> 3) * (128 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
        };
        const int rc = p.rope_rot / 8;  // rotated 16-byte chunks
        for (int e = tid; e < 128 * (D / 8); e += blockDim.x) {
            const int r = e / (D / 8), c = e % (D / 8);
            if (c >= rc / 2 && c < rc) continue;  // second half of a rotary pair: with its partner
            const int R = row0 + r;
            const __nv_bfloat16* qrow = nullptr;
            int node = 0;
            if (R < p.N * p.G) {
                node = R / p.G;
                const int h = g * p.G + R % p.G;
                if (node < nn) qrow = p.q + ((lb * p.N + node) * p.Hq + h) * D;
            }
            if (c >= rc) {
                qstore(r, c, qrow ? __ldg(reinterpret_cast<const uint4*>(qrow) + c) : make_uint4(0, 0, 0, 0));
                continue;
            }
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (qrow) {
                const uint4 a = __ldg(reinterpret_cast<const uint4*>(qrow) + c);
                const uint4 bq = __ldg(reinterpret_cast<const uint4*>(qrow) + c + rc / 2);
                const float* cs = p.rope_table + ((long)b * p.N + node) * p.rope_rot + 8 * c;
                const float* sn = cs + p.rope_rot / 2;
                const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {bq.x, bq.y, bq.z, bq.w};
                uint32_t ow0[4], ow1[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float x0[2], x1[2], y0[2], y1[2];
                    x0[0] = __uint_as_float(aw[u] << 16);
                    x0[1] = __uint_as_float(aw[u] & 0xffff0000u);
                    x1[0] = __uint_as_float(bw[u] << 16);
                    x1[1] = __uint_as_float(bw[u] & 0xffff0000u);
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const float cz = cs[2 * u + z], sz = sn[2 * u + z];
                        y0[z] = __fmaf_rn(x0[z], cz, __fmul_rn(-x1[z], sz));
                        y1[z] = __fmaf_rn(x1[z], cz, __fmul_rn(x0[z], sz));
                    }
                    ow0[u] = pack_bf16(y0[0], y0[1]);
                    ow1[u] = pack_bf16(y1[0], y1[1]);
                }
                lo = make_uint4(ow0[0], ow0[1], ow0[2], ow0[3]);
                hi = make_uint4(ow1[0], ow1[1], ow1[2], ow1[3]);
            }
            qstore(r, c, lo);
            qstore(r, c + rc / 2, hi);
        }
    }
    tc::fence_proxy_async();
    tc::tc_fence_before();
    tc::cluster_sync();  // both CTAs' barriers, tensor memory and Q before the pipeline starts
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            const int grp = (int)((lb * p.Hkv) + g);
            const uint32_t full_c = tc::mapa_shared(tc::smem_u32(full), 0);  // the even CTA's K barriers
            int issued = 0;
            for (int j = 0; j < T && !*abort_flag; ++j) {
                const Tile t = tile2_of(j, n_pre, c0, c1, ragged);
                if (j + 2 < T && !p.paged) {
                    // warm L2 with tile j + 2's halves: their stages free up only as tile j's
                    // MMAs finish, and the load must then land within about one tile's time
                    const Tile t2 = tile2_of(j + 2, n_pre, c0, c1, ragged);
                    const int yk = t2.y + 64 * (int)rank, xv = (int)rank * (D / 2);
#pragma unroll
                    for (int blk = 0; blk < Cfg::kBlocks; ++blk) {
                        if (!t2.tree) tc::tma_prefetch_3d(&tm_kc, blk * 64, yk, grp);
                        else tc::tma_prefetch_4d(&tm_kt, blk * 64, g, yk, (int)lb);
                    }
#pragma unroll
                    for (int blk = 0; blk < Cfg::kBlocks / 2; ++blk) {
                        if (!t2.tree) tc::tma_prefetch_3d(&tm_vc, xv + blk * 64, t2.y, grp);
                        else tc::tma_prefetch_4d(&tm_vt, xv + blk * 64, g, t2.y, (int)lb);
                    }
                }
                bool ok = true;
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int st = kv == 0 ? j % kKS : kKS + j % kVS;
                    const int ph = kv == 0 ? (j / kKS) & 1 : (j / kVS) & 1;
                    ok = tc::mbar_wait(sfree + st, ph ^ 1, abort_flag);
                    if (!ok) break;
                    unsigned char* dst = sRing + st * Cfg::kStageBytes;
                    if (kv == 0) {
                        // K half: keys [y + 64 rank, +64), all D columns
                        if (rank == 0) tc::mbar_expect_tx(full + st, 2 * Cfg::kStageBytes);
                        const uint32_t cb = full_c + st * 8;
                        const int y = t.y + 64 * (int)rank;
                        if (!t.tree && p.paged) {
                            const int sub = min(64, p.page_rows), last = (P - 1) / p.page_rows;
                            for (int r0 = 0; r0 < 64; r0 += sub) {
                                const int pos = y + r0;
                                const int lp = min(pos / p.page_rows, last);
                                const int phys = p.block_table[(long)b * p.max_pages + lp];
                                const int plane = (int)(((long)l * p.num_pages + phys) * p.Hkv + g);
#pragma unroll
                                for (int blk = 0; blk < Cfg::kBlocks; ++blk)
                                    tc::tma_load_3d_pair(dst + blk * (64 * 128) + r0 * 128, &tm_kc, cb, blk * 64,
                                                         pos % p.page_rows, plane);
                            }
                        } else {
#pragma unroll
                            for (int blk = 0; blk < Cfg::kBlocks; ++blk) {
                                if (!t.tree)
                                    tc::tma_load_3d_pair(dst + blk * (64 * 128), &tm_kc, cb, blk * 64, y, grp);
                                else
                                    tc::tma_load_4d_pair(dst + blk * (64 * 128), &tm_kt, cb, blk * 64, g, y, (int)lb);
                            }
                        }
                    } else {
                        // V half: keys [y, +128), value columns [rank D/2, (rank + 1) D/2)
                        tc::mbar_expect_tx(full + st, Cfg::kStageBytes);
                        const int xc = (int)rank * (D / 2);
                        if (!t.tree && p.paged) {
                            const int sub = min(kPN, p.page_rows), last = (P - 1) / p.page_rows;
                            for (int r0 = 0; r0 < kPN; r0 += sub) {
                                const int pos = t.y + r0;
                                const int lp = min(pos / p.page_rows, last);
                                const int phys = p.block_table[(long)b * p.max_pages + lp];
                                const int plane = (int)(((long)l * p.num_pages + phys) * p.Hkv + g);
#pragma unroll
                                for (int blk = 0; blk < Cfg::kBlocks / 2; ++blk)
                                    tc::tma_load_3d(dst + blk * (kPN * 128) + r0 * 128, &tm_vc, full + st,
                                                    xc + blk * 64, pos % p.page_rows, plane);
                            }
                        } else {
#pragma unroll
                            for (int blk = 0; blk < Cfg::kBlocks / 2; ++blk) {
                                if (!t.tree)
                                    tc::tma_load_3d(dst + blk * (kPN * 128), &tm_vc, full + st, xc + blk * 64, t.y,
                                                    grp);
                                else
                                    tc::tma_load_4d(dst + blk * (kPN * 128), &tm_vt, full + st, xc + blk * 64, g, t.y,
                                                    (int)lb);
                            }
                        }
                    }
                    issued = 2 * j + kv + 1;
                }
                if (!ok) break;
            }
            // drain: the even CTA waits for its last K stages (both halves) and its V stages,
            // the odd CTA for its own V stages
            const int nk = (issued + 1) / 2, nv = issued / 2;  // K and V tiles issued
            if (rank == 0)
                for (int i = max(0, nk - kKS); i < nk; ++i) drain_wait(full + i % kKS, (i / kKS) & 1);
            for (int i = max(0, nv - kVS); i < nv; ++i) drain_wait(full + kKS + i % kVS, (i / kVS) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc_qk = tc::idesc_bf16(256, kPN, false, false);
            constexpr uint32_t idesc_pv = tc::idesc_bf16(256, D, false, true);
            const uint32_t sRa = tc::smem_u32(sRing);
            const uint64_t qdesc0 = tc::desc_sw128(tc::smem_u32(sQ), 16, 1024);
            const uint64_t kdesc0 = tc::desc_sw128(sRa, 16, 1024);
            const uint64_t vdesc0 = tc::desc_sw128(sRa, kPN * 128, 1024);
            auto pv = [&](int i) -> bool {
                // P_i and both V_i halves (padding rows zeroed) are ready once all 16
                // softmax warps of the pair have arrived
                if (!tc::mbar_wait_cluster(p_full + (i & 1), (i >> 1) & 1, abort_flag)) return false;
                tc::tc_fence_after();
                const int st = kKS + i % kVS;
                const uint64_t vd = vdesc0 + static_cast<uint64_t>((st * Cfg::kStageBytes) >> 4);
                const uint32_t pa = tmem + (i & 1) * kPN;
#pragma unroll
                for (int q = 0; q < 2 * (kPN / 16); ++q) {  // P_hi k-steps, then P_lo k-steps
                    const int part = q / (kPN / 16), kk = q % (kPN / 16);
                    tc::mma2_f16_ts(tmem + Cfg::kOCol, pa + part * (kPN / 2) + kk * 8,
                                    vd + static_cast<uint64_t>((kk * 2048) >> 4), idesc_pv, (i > 0 || q > 0) ? 1u : 0u);
                }
                tc::mma2_commit_mc(sfree + st, 3);  // V stage free; also: O holds tile i
                return true;
            };
            bool ok = true;
            for (int j = 0; j < T && ok; ++j) {
                const int st = j % kKS;
                if (!tc::mbar_wait_cluster(full + st, (j / kKS) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint64_t kd = kdesc0 + static_cast<uint64_t>((st * Cfg::kStageBytes) >> 4);
                const uint32_t sd = tmem + (j & 1) * kPN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qoff = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
                    const uint32_t koff = (kk >> 2) * (64 * 128) + (kk & 3) * 32;
                    tc::mma2_f16_ss(sd, qdesc0 + static_cast<uint64_t>(qoff >> 4),
                                    kd + static_cast<uint64_t>(koff >> 4), idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc::mma2_commit_mc(sfree + st, 3);       // K stage free in both CTAs
                tc::mma2_commit_mc(s_full + (j & 1), 3); // S_j ready in both CTAs
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok && pv(T - 1)) tc::mma2_commit_mc(o_final, 3);
            tc::mma2_commit_mc(drain, 1);
            drain_wait(drain, 0);
        }
    } else if (warp == 2) {
        // ------------------------------------------------- forwarder (odd CTA)
        // one cluster-scope arrival a tile on the even CTA's P barrier, once this CTA's 8
        // softmax warps have arrived locally (cheaper than 8 remote arrivals on their path)
        if (lane == 0 && rank == 1) {
            const uint32_t pf_remote = tc::mapa_shared(tc::smem_u32(p_full), 0);
            for (int j = 0; j < T; ++j) {
                if (!tc::mbar_wait(p_full + (j & 1), (j >> 1) & 1, abort_flag)) break;
                tc::mbar_arrive_cluster(pf_remote + (j & 1) * 8);
            }
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------------ softmax
        const int hf = (warp - 4) >> 2, ws = (warp - 4) & 3, r = 32 * ws + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * ws) << 16;
        const int R = row0 + r;
        const bool in_rows = R < p.N * p.G;
        const int node = in_rows ? R / p.G : 0;
        const int h = g * p.G + (in_rows ? R % p.G : 0);
        const bool live = in_rows && node < nn;
        const uint32_t* anc_row = p.anc + ((long)b * p.N + node) * p.W;
        float m_used = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            const Tile t = tile2_of(j, n_pre, c0, c1, ragged);
            if (ok) ok = tc::mbar_wait(s_full + (j & 1), (j >> 1) & 1, abort_flag);
            ok = __all_sync(kFull, ok);
            float sv[64];  // raw scores, -inf where the key is not visible
            float mtile = -INFINITY;
            if (ok) {
                tc::tc_fence_after();
                const int k0 = t.y + 64 * hf;  // this half's first key
                uint32_t vis[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    if (!t.tree) {
                        vis[w] = prefix_vis(t.lo, c1, k0 + 32 * w);
                    } else {
                        const int wd = (t.y >> 5) + 2 * hf + w;
                        vis[w] = (live && wd < p.W) ? anc_row[wd] : 0u;
                    }
                }
                const bool all_vis = __all_sync(kFull, (vis[0] & vis[1]) == ~0u);
                uint32_t sr[32];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    tc::tmem_ld32(tmem + lane_base + (j & 1) * kPN + 64 * hf + 32 * w, sr);
                    tc::tmem_wait_ld();
                    if (all_vis) {  // every key of the half visible (nearly every prefix tile)
#pragma unroll
                        for (int c = 0; c < 32; ++c) sv[32 * w + c] = __uint_as_float(sr[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            sv[32 * w + c] = ((vis[w] >> c) & 1u) ? __uint_as_float(sr[c]) : -INFINITY;
                    }
                }
                // tile max as a tree (short dependency chains), then into log2 units
                float mx[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) mx[c] = fmaxf(fmaxf(sv[c], sv[c + 16]), fmaxf(sv[c + 32], sv[c + 48]));
#pragma unroll
                for (int w = 8; w > 0; w >>= 1)
#pragma unroll
                    for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
                mtile = mx[0] * p.scale_log2;
            }
            float* xm = xch + (j & 1) * 256;
            xm[hf * 128 + r] = mtile;
            tc::named_bar(1, 256);
            mtile = fmaxf(mtile, xm[(hf ^ 1) * 128 + r]);
            if (!ok) continue;
            const bool grow = mtile > m_used + kTau;
            const bool need = grow && (m_used != -INFINITY);
            if (__any_sync(kFull, need)) {
                // O must hold tile j - 1 before it is rescaled: wait for that tile's P.V
                ok = __all_sync(kFull,
                                tc::mbar_wait(sfree + kKS + (j - 1) % kVS, ((j - 1) / kVS) & 1, abort_flag));
                if (!ok) continue;
                tc::tc_fence_after();
                const float f = need ? tc::ex2(m_used - mtile) : 1.f;
#pragma unroll 1
                for (int cb = hf * (D / 2); cb < (hf + 1) * (D / 2); cb += 32) {
                    uint32_t ov[32];
                    tc::tmem_ld32(tmem + lane_base + Cfg::kOCol + cb, ov);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
                    tc::tmem_st32(tmem + lane_base + Cfg::kOCol + cb, ov);
                }
                tc::tmem_wait_st();
                if (need) l_run *= f;
            }
            if (grow) m_used = mtile;
            float sum = 0.f;
            // a row that has seen no visible key yet has no reference: its P is all zeros
            const float mref = m_used == -INFINITY ? 0.f : m_used;
            const float sc = p.scale_log2;
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                uint32_t phi[16], plo[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    // ex2(-inf) = 0 for keys that are not visible.  P = P_hi + P_lo with P_hi
                    // the top 16 bits of P (exact as bf16) and P_lo = bf16(P - P_hi): the
                    // pair carries P to ~2^-16 relative
                    const float a = tc::ex2(fmaf(sv[32 * w + c], sc, -mref));
                    const float bb = tc::ex2(fmaf(sv[32 * w + c + 1], sc, -mref));
                    sum += a + bb;
                    const uint32_t ah = __float_as_uint(a) & 0xffff0000u, bh = __float_as_uint(bb) & 0xffff0000u;
                    phi[c >> 1] = (ah >> 16) | bh;
                    plo[c >> 1] = pack_bf16(a - __uint_as_float(ah), bb - __uint_as_float(bh));
                }
                // P_hi in columns [0, 64) of the buffer, P_lo in [64, 128); this half's 64
                // keys are 32 packed columns of each
                tc::tmem_st16(tmem + lane_base + (j & 1) * kPN + 32 * hf + 16 * w, phi);
                tc::tmem_st16(tmem + lane_base + (j & 1) * kPN + kPN / 2 + 32 * hf + 16 * w, plo);
            }
            l_run += sum;
            tc::tmem_wait_st();
            tc::tc_fence_before();
            // this CTA's V half of tile j: wait for it, and zero the rows the MMA must not
            // see (padding tree nodes may hold anything, even NaN, and a zero P does not
            // cancel NaN; paged tiles read rows past the prefix)
            {
                const int st = kKS + j % kVS;
                ok = __all_sync(kFull, tc::mbar_wait(full + st, (j / kVS) & 1, abort_flag));
                const int first = t.tree ? max(0, nn - t.y) : (t.y + kPN > c1 ? c1 - t.y : kPN);
                if (ok && first < kPN) {
                    unsigned char* vst = sRing + st * Cfg::kStageBytes;
                    const int per_blk = (kPN - first) * 8;  // 16-byte chunks of the zeroed rows of a block
                    for (int e = hf * 128 + r; e < per_blk * (Cfg::kBlocks / 2); e += 256) {
                        const int blk = e / per_blk, rem = e % per_blk;
                        *reinterpret_cast<uint4*>(vst + blk * (kPN * 128) + (first + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    tc::fence_proxy_async();
                }
            }
            __syncwarp();
            if (!ok) continue;
            if (lane == 0) tc::mbar_arrive(p_full + (j & 1));
        }
        if (ok) ok = tc::mbar_wait(o_final, 0, abort_flag);
        ok = __all_sync(kFull, ok);
        // row sums of both halves, through the max buffer of the parity tile T - 1 did not use
        float* xs = xch + (T & 1) * 256;
        xs[hf * 128 + r] = l_run;
        tc::named_bar(1, 256);
        const float l_tot = l_run + xs[(hf ^ 1) * 128 + r];
        if (ok) {
            tc::tc_fence_after();
            const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll 1
            for (int cb = hf * (D / 2); cb < (hf + 1) * (D / 2); cb += 32) {
                uint32_t ov[32];
                tc::tmem_ld32(tmem + lane_base + Cfg::kOCol + cb, ov);
                tc::tmem_wait_ld();
                float f[32];
                if (p.S == 1) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] = live ? __uint_as_float(ov[i]) * inv : 0.f;
                    if (in_rows)
                        store_row32<Tout>(static_cast<Tout*>(p.o) + ((lb * p.N + node) * p.Hq + h) * D + cb, f);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(ov[i]);
                    store_row32<float>(p.part_o + (prow0 + r) * D + cb, f);
                }
            }
            if (p.S > 1 && hf == 0) p.part_ml[prow0 + r] = make_float2(m_used, l_tot);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();  // neither CTA frees tensor memory or leaves while the pair may touch it
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc2(tmem, 512);
    }
    if (tid == 0 && *abort_flag) atomicExch(p.status + b, (int)DDT_ERR_TIMEOUT);
}

// Combines split-KV partials: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s.
template <int D, typename Tout>
__global__ void __launch_bounds__(D) k_attn_merge(const TcParams p) {
    const int row = blockIdx.x;  // node * Hq + head
    const int lbi = blockIdx.y;
    const int l = lbi / p.B, b = lbi % p.B;
    const int node = row / p.Hq, hq = row % p.Hq;
    const int g = hq / p.G, R = node * p.G + hq % p.G;
    const int c = threadIdx.x;
    const int P = p.prefix_len[b], nn = p.n_nodes[b];
    Tout* out = static_cast<Tout*>(p.o) + (((long)l * p.B + b) * p.N * p.Hq + row) * D + c;
    if (P < 0 || P > p.Pcap || nn < 1 || nn > p.N || node >= nn) {
        *out = from_f32<Tout>(0.f);
        return;
    }
    const long stride_s = (long)p.L * p.B * p.Hkv * p.MT * kBM;
    const long r0 = ((((long)l * p.B + b) * p.Hkv + g) * (long)(p.MT * kBM)) + R;
    float M = -INFINITY;
    for (int s = 0; s < p.S; ++s) {
        const float2 ml = p.part_ml[s * stride_s + r0];
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    float acc = 0.f, lsum = 0.f;
    for (int s = 0; s < p.S; ++s) {
        const float2 ml = p.part_ml[s * stride_s + r0];
        if (!(ml.y > 0.f)) continue;
        const float w = tc::ex2(ml.x - M);
        lsum += w * ml.y;
        acc += w * p.part_o[(s * stride_s + r0) * D + c];
    }
    *out = from_f32<Tout>(lsum > 0.f ? acc / lsum : 0.f);
}

// Requests ordered by prefix length, longest first (ties by index): long units start
// first.  Also clears the status words, which the attention CTAs only ever set to errors.
__global__ void k_attn_order(int B, const int32_t* __restrict__ prefix_len, int32_t* __restrict__ perm,
                             int32_t* __restrict__ status) {
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        status[b] = DDT_OK;
        const int pb = prefix_len[b];
        int rank = 0;
        for (int o = 0; o < B; ++o) {
            const int po = prefix_len[o];
            rank += (po > pb) || (po == pb && o < b);
        }
        perm[rank] = b;
    }
}

// ------------------------------------------------------------------------------ host
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

int sm_count() {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}

// Split of the prefix into `S` chunks so that very small grids still use the GPU.  A
// split CTA writes a 128 x D fp32 partial that k_attn_merge reads back, and every CTA
// pays its setup, so a split pays only while all splits still run in one wave: S is the
// number of copies of the grid that fit on the SMs, and each chunk keeps >= 1024 keys.
// (One request, 16 layers, P = 4096, 256 CTAs: 0.18 ms unsplit against 0.28-0.52 ms
// for 2 to 8 splits.)
void choose_split(int L, int B, int Hkv, int MT, int Pcap, int n_sms, int* S, int* chunk) {
    const long base = (long)L * B * Hkv * MT;
    int s = 1;
    if (base < n_sms && Pcap > 0) {
        s = (int)(n_sms / base);
        s = max(1, min(s, Pcap / 1024));
    }
    int c = Pcap > 0 ? (Pcap + s - 1) / s : kBN;
    c = ((c + kBN - 1) / kBN) * kBN;
    *chunk = c;
    *S = Pcap > 0 ? (Pcap + c - 1) / c : 1;
}

}  // namespace

// head sizes the CTA-pair kernel takes (the others use k_attn_tc)
static bool pair_kernel(int d) { return d == 128 || d == 256; }

size_t attn_tc_ws_bytes(int L, int B, int N, int Hq, int Hkv, int d, int Pcap) {
    const int G = Hq / Hkv;
    // rows of the split-KV partials: 128-row tiles, or 256-row pair tiles (the pair kernel
    // splits by SM pairs); the workspace covers both
    const int MT = (N * G + kBM - 1) / kBM, MP = (N * G + 255) / 256;
    int S1, S2, chunk;
    choose_split(L, B, Hkv, MT, Pcap, 256, &S1, &chunk);  // 256 bounds the SM count from above
    choose_split(L, B, Hkv, MP, Pcap, 128, &S2, &chunk);
    size_t bytes = ((size_t)B * sizeof(int32_t) + 255) & ~(size_t)255;
    const size_t rows1 = S1 > 1 ? (size_t)S1 * L * B * Hkv * MT * kBM : 0;
    const size_t rows2 = S2 > 1 ? (size_t)S2 * L * B * Hkv * MP * 256 : 0;
    const size_t rows = rows1 > rows2 ? rows1 : rows2;
    bytes += rows * d * sizeof(float) + rows * sizeof(float2);
    return bytes + 256;
}

bool attn_tc_supported(int d, ddt_dtype in) { return in == DDT_BF16 && (d == 64 || d == 128 || d == 256); }

template <int D, typename Tout>
static cudaError_t attn_tc_go(const TcParams& prm, const CUtensorMap* maps, cudaStream_t st) {
    using Cfg = TcCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(k_attn_tc<D, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(prm.S * prm.MT * prm.Hkv * prm.L, prm.B);
    k_attn_tc<D, Tout><<<counted(grid), kThreads, Cfg::kSmem, st>>>(prm, maps[0], maps[1], maps[2], maps[3]);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (prm.S > 1) {
        k_attn_merge<D, Tout><<<counted(dim3(prm.N * prm.Hq, prm.L * prm.B)), D, 0, st>>>(prm);
        e = cudaGetLastError();
    }
    return e;
}

template <int D, typename Tout>
static cudaError_t attn_tc2_go(const TcParams& prm, const CUtensorMap* maps, cudaStream_t st) {
    using Cfg = Tc2Cfg<D>;
    cudaError_t e = cudaFuncSetAttribute(k_attn_tc2<D, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(2 * prm.S * prm.MP * prm.Hkv * prm.L, prm.B);
    k_attn_tc2<D, Tout><<<counted(grid), kThreads, Cfg::kSmem, st>>>(prm, maps[0], maps[1], maps[2], maps[3]);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (prm.S > 1) {
        k_attn_merge<D, Tout><<<counted(dim3(prm.N * prm.Hq, prm.L * prm.B)), D, 0, st>>>(prm);
        e = cudaGetLastError();
    }
    return e;
}

// pg == nullptr: contiguous caches [L][B][Hkv][Pcap][d]; else paged caches
// [L][num_pages][Hkv][page_rows][d] with Pcap = max_pages * page_rows.
static cudaError_t attn_tc_launch(int L, int B, int N, int Hq, int Hkv, int d, int Pcap, ddt_dtype out,
                                  const void* q, const void* k_tree, const void* v_tree, const void* k_cache,
                                  const void* v_cache, const AttnPaging* pg, const int32_t* prefix_len,
                                  const int32_t* n_nodes, const uint32_t* anc, float scale, void* o, int32_t* status,
                                  void* ws, size_t ws_bytes, cudaStream_t st, const AttnRope* rope) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    TcParams prm;
    prm.L = L;
    prm.B = B;
    prm.N = N;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.G = Hq / Hkv;
    prm.MT = (N * prm.G + kBM - 1) / kBM;
    prm.Pcap = Pcap;
    prm.W = (N + 31) / 32;
    const bool pair = pair_kernel(d);
    prm.MP = (N * prm.G + 255) / 256;
    if (pair) {
        // the pair kernel's units are SM pairs of 256 query rows; its partial rows are laid
        // out as 2 MP tiles of 128 for the merge
        choose_split(L, B, Hkv, prm.MP, Pcap, sm_count() / 2, &prm.S, &prm.chunk);
        prm.chunk = ((prm.chunk + kPN - 1) / kPN) * kPN;
        prm.S = Pcap > 0 ? (Pcap + prm.chunk - 1) / prm.chunk : 1;
        prm.MT = 2 * prm.MP;
    } else {
        choose_split(L, B, Hkv, prm.MT, Pcap, sm_count(), &prm.S, &prm.chunk);
    }
    if (ws_bytes < attn_tc_ws_bytes(L, B, N, Hq, Hkv, d, Pcap)) return cudaErrorInvalidValue;
    unsigned char* w = static_cast<unsigned char*>(ws);
    int32_t* perm = reinterpret_cast<int32_t*>(w);
    prm.perm = perm;
    const size_t perm_bytes = ((size_t)B * sizeof(int32_t) + 255) & ~(size_t)255;
    const size_t rows = (size_t)prm.S * L * B * Hkv * prm.MT * kBM;
    prm.part_o = reinterpret_cast<float*>(w + perm_bytes);
    prm.part_ml = reinterpret_cast<float2*>(w + perm_bytes + (prm.S > 1 ? rows * d * sizeof(float) : 0));
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.prefix_len = prefix_len;
    prm.n_nodes = n_nodes;
    prm.anc = anc;
    prm.o = o;
    prm.status = status;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.paged = pg != nullptr;
    prm.page_rows = pg ? pg->page_rows : 0;
    prm.num_pages = pg ? pg->num_pages : 0;
    prm.max_pages = pg ? pg->max_pages : 0;
    prm.block_table = pg ? pg->block_table : nullptr;
    prm.rope_rot = rope ? rope->rot : 0;
    prm.rope_table = rope ? rope->table : nullptr;
    if (rope && !pair) return cudaErrorInvalidValue;  // q rotation is staged by the pair kernel only

    // tensor maps: caches (d, position, layer*B*Hkv), tree rows (d, kv head, node, layer*B)
    CUtensorMap maps[4];
    // (paged: the plane is (layer, physical page, kv head) and a box spans at most a page)
    // box rows: the one-SM kernel loads 64 keys of K and of V; the pair kernel 64 keys of
    // K and 128 of V per CTA (a box spans at most one page)
    const int kbox = kBN, vbox = pair ? kPN : kBN;
    const int rows3 = pg ? pg->page_rows : (Pcap > 0 ? Pcap : 1);
    const cuuint32_t box3k[3] = {64, (cuuint32_t)(pg ? (pg->page_rows < kbox ? pg->page_rows : kbox) : kbox), 1};
    const cuuint32_t box3v[3] = {64, (cuuint32_t)(pg ? (pg->page_rows < vbox ? pg->page_rows : vbox) : vbox), 1};
    const cuuint32_t es3[3] = {1, 1, 1};
    const cuuint64_t dims3[3] = {(cuuint64_t)d, (cuuint64_t)rows3,
                                 (cuuint64_t)L * (pg ? (long)pg->num_pages : (long)B) * Hkv};
    const cuuint64_t str3[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows3 * d * 2};
    const cuuint32_t box4k[4] = {64, 1, (cuuint32_t)kbox, 1};
    const cuuint32_t box4v[4] = {64, 1, (cuuint32_t)vbox, 1};
    const cuuint32_t es4[4] = {1, 1, 1, 1};
    const cuuint64_t dims4[4] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)N, (cuuint64_t)L * B};
    const cuuint64_t str4[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hkv * d * 2, (cuuint64_t)N * Hkv * d * 2};
    const void* kc = Pcap > 0 ? k_cache : k_tree;  // with no prefix the cache maps are never used
    const void* vc = Pcap > 0 ? v_cache : v_tree;
    CUresult r = CUDA_SUCCESS;
    r = r != CUDA_SUCCESS ? r
                          : enc(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kc), dims3, str3, box3k,
                                es3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    r = r != CUDA_SUCCESS ? r
                          : enc(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(vc), dims3, str3, box3v,
                                es3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    r = r != CUDA_SUCCESS ? r
                          : enc(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(k_tree), dims4, str4,
                                box4k, es4, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    r = r != CUDA_SUCCESS ? r
                          : enc(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v_tree), dims4, str4,
                                box4v, es4, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

    k_attn_order<<<counted(1), 256, 0, st>>>(B, prefix_len, perm, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const bool bf = out == DDT_BF16;
    switch (d) {
        case 64: return bf ? attn_tc_go<64, __nv_bfloat16>(prm, maps, st) : attn_tc_go<64, float>(prm, maps, st);
        case 128: return bf ? attn_tc2_go<128, __nv_bfloat16>(prm, maps, st) : attn_tc2_go<128, float>(prm, maps, st);
        case 256: return bf ? attn_tc2_go<256, __nv_bfloat16>(prm, maps, st) : attn_tc2_go<256, float>(prm, maps, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_tc(int L, int B, int N, int Hq, int Hkv, int d, int Pcap, ddt_dtype out, const void* q,
                           const void* k_tree, const void* v_tree, const void* k_cache, const void* v_cache,
                           const int32_t* prefix_len, const int32_t* n_nodes, const uint32_t* anc, float scale,
                           void* o, int32_t* status, void* ws, size_t ws_bytes, cudaStream_t st,
                           const AttnRope* rope) {
    return attn_tc_launch(L, B, N, Hq, Hkv, d, Pcap, out, q, k_tree, v_tree, k_cache, v_cache, nullptr, prefix_len,
                          n_nodes, anc, scale, o, status, ws, ws_bytes, st, rope);
}

cudaError_t launch_attn_tc_paged(int L, int B, int N, int Hq, int Hkv, int d, const AttnPaging& pg, ddt_dtype out,
                                 const void* q, const void* k_tree, const void* v_tree, const void* k_pages,
                                 const void* v_pages, const int32_t* prefix_len, const int32_t* n_nodes,
                                 const uint32_t* anc, float scale, void* o, int32_t* status, void* ws,
                                 size_t ws_bytes, cudaStream_t st, const AttnRope* rope) {
    return attn_tc_launch(L, B, N, Hq, Hkv, d, pg.max_pages * pg.page_rows, out, q, k_tree, v_tree, k_pages, v_pages,
                          &pg, prefix_len, n_nodes, anc, scale, o, status, ws, ws_bytes, st, rope);
}

}  // namespace ddt
