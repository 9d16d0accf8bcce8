// Decode-time expert FFN: permute (P1), gate/up dequantising GEMV with SwiGLU (G1), down
// GEMV with the router-weighted scatter (G2), combine (C1).
//
// What is computed (pages 1-5, see moe.h): for every route (t, j) of a token t to its
// j-th selected expert e, h = silu(Wg_e x_t) * (Wu_e x_t) and
// partial[t][j] = w[t][j] * (Wd_e h); the combine sums partial over j.  Weights stay in
// their quantised blocks (page 5, section 1.2) and are dequantised in registers.
//
// GB300 mapping (the decode GEMVs stream the selected experts' bytes from HBM once):
//  * work unit = two 32-row tiles over a K range whose bytes are one contiguous run per
//    tile and region in the slot image: the gate and the up tile of the same rows (G1), or
//    two neighbouring down tiles (G2);
//  * persistent CTAs of 16 warps, one per SM: each walks a contiguous, work-balanced range
//    of units (precomputed by the permute kernel) through a ring of shared-memory stages;
//    thread 0 keeps the next units' bulk copies (TMA engine, cp.async.bulk) in flight
//    while the current one is computed;
//  * lane l of every warp owns row l of both tiles and keeps its dot products in registers
//    (no cross-lane reduction); each activation value read from shared memory (a warp
//    broadcast) feeds both rows; the 16 warps split the K range and are reduced in shared
//    memory in a fixed order;
//  * codes become fp32 with exponent tricks (no int->float conversions), accumulate with
//    packed fp32x2 FMAs, and block scales are applied once per 32 weights;
//  * the warp that reduces a token's gate and up rows applies SwiGLU and writes h; when the
//    K range is split (large H), the partial sums go to the workspace and the down kernel
//    sums them in a fixed order while it stages its activations;
//  * an expert that missed in a device-managed pool is read from its pinned host image and
//    written through to its slot by the unit that uses the bytes ("fill" units).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <algorithm>
#include <mutex>

#include "moe_ptx.cuh"

#define GV_WARPS 16
#define GV_THREADS (GV_WARPS * 32)
#define GV_TOK 8                  // tokens per pass (one per reducing warp)
#define GV_SMEM_MAX (220 * 1024)  // dynamic shared memory a ring kernel may take
#define GV_FILL_BATCH 4           // 16-byte pieces per thread loaded together by a fill unit
#define GV_ICACHE 64              // active experts of a CTA's range kept in shared memory
#define GV_RCACHE 512             // routes (and router weights) of a CTA's range in shared memory
#define GV_MAX_GRID 1024          // CTAs per launch (bounds the precomputed range tables)

namespace {

// Work of one unit of an expert with n_e tokens, in units of a token's dot products: the
// unit's bytes and dequantisation cost about as much as GV_COST_MEM tokens.
#define GV_COST_MEM 4
__host__ __device__ inline int unit_cost(int n_e) { return n_e > 0 ? GV_COST_MEM + n_e : 1; }

// ------------------------------------------------------------------ shared-memory layout

struct RingSmem {
    size_t bars, stages, stage_bytes, tile_bytes, scale_off, act, asum, red, info, rts, wts, total;
};

// nbr blocks of 32 columns per tile, `tiles` tiles per unit, ntok staged token rows, S stages.
__host__ __device__ inline RingSmem ring_smem(int qtype, int nbr, int tiles, int ntok, int S) {
    RingSmem L;
    const int QB = qtype == MOE_Q8_0 ? 1024 : 512;       // code bytes per block of a 32-row tile
    const int SB = 32 * moe_scale_entry_bytes(qtype);    // scale bytes per block of a tile
    L.scale_off = (size_t)nbr * QB;
    L.tile_bytes = L.scale_off + ((size_t)nbr * SB + 127) / 128 * 128;
    L.stage_bytes = (size_t)tiles * L.tile_bytes;
    size_t off = 0;
    L.bars = off;   off += 128;
    L.stages = off; off += (size_t)S * L.stage_bytes;
    L.act = off;    off += (size_t)ntok * nbr * 32 * 4;
    L.asum = off;   off += ((size_t)ntok * nbr * 4 + 15) / 16 * 16;
    L.red = off;    off += (size_t)GV_WARPS * ntok * 2 * 32 * 4;
    L.info = off;   off += (size_t)GV_ICACHE * 32;
    L.rts = off;    off += (size_t)GV_RCACHE * 4;
    L.wts = off;    off += (size_t)GV_RCACHE * 4;
    L.total = off;
    return L;
}

// Launch plan of one decode FFN: the gate/up K split and ring depth, the down tiles per unit
// and ring depth, chosen so that each kernel's shared memory fits.
struct GvPlan {
    int KS, S1, TPU, S2;
};

// Units are made small enough that a launch has about GV_UNITS_TARGET of them (a CTA's share
// is then several units and the work-balanced split is fine-grained), but no smaller than one
// 32-column block per warp.
#define GV_UNITS_TARGET 1024

inline bool gv_plan(int T, int H, int F, int qtype, int n_act_max, GvPlan *pl) {
    const int ntok = T < GV_TOK ? T : GV_TOK;
    const int NB = H / 32, RTF = F / 32, RTH = H / 32;
    pl->KS = 0;
    for (int ks = 1; ks <= NB && !pl->KS; ks *= 2) {
        if (NB % ks) break;
        const bool more = (long)n_act_max * ks * RTF < GV_UNITS_TARGET && NB % (2 * ks) == 0 &&
                          NB / (2 * ks) >= GV_WARPS;
        for (int S = 3; S >= 2 && !pl->KS; --S)
            if (!more && ring_smem(qtype, NB / ks, 2, ntok, S).total <= GV_SMEM_MAX) {
                pl->KS = ks;
                pl->S1 = S;
            }
    }
    if (!pl->KS) {  // a single stage of the smallest split
        int ks = 1;
        while (NB % (2 * ks) == 0 && ring_smem(qtype, NB / ks, 2, ntok, 1).total > GV_SMEM_MAX) ks *= 2;
        if (ring_smem(qtype, NB / ks, 2, ntok, 1).total > GV_SMEM_MAX) return false;
        pl->KS = ks;
        pl->S1 = 1;
    }
    pl->TPU = 0;
    const bool pairs = RTH % 2 == 0 && (long)n_act_max * (RTH / 2) >= GV_UNITS_TARGET;
    const int cand[7][2] = {{2, 4}, {2, 3}, {2, 2}, {1, 4}, {1, 3}, {1, 2}, {1, 1}};
    for (int i = 0; i < 7 && !pl->TPU; ++i) {
        if (cand[i][0] == 2 && !pairs) continue;
        if (ring_smem(qtype, F / 32, cand[i][0], ntok, cand[i][1]).total <= GV_SMEM_MAX) {
            pl->TPU = cand[i][0];
            pl->S2 = cand[i][1];
        }
    }
    return pl->TPU != 0;
}

inline int gv_n_act_max(int T, int E, int k) { return T * k < E ? T * k : E; }

// ------------------------------------------------------------------ workspace layout

// Per active expert, written by the permute kernel.
struct ActInfo {
    unsigned long long src;  // image base the weights are read from (slot, or pinned host image)
    unsigned long long dst;  // slot base (written through when fill != 0)
    int e, pos0, n_e, fill;  // n_e == 0: skip (invalid slot)
};

// int32 region: [0] n_active | active [E] | a_off [E+1] | routes [R] | ranges1 | ranges2
__host__ __device__ inline int ws_active_off() { return 16; }
__host__ __device__ inline int ws_aoff_off(int E) { return 16 + E; }
__host__ __device__ inline int ws_routes_off(int E) { return 16 + 2 * E + 1; }
__host__ __device__ inline int ws_ranges_off(int E, int R, int which) {
    return 16 + 2 * E + 1 + R + which * (GV_MAX_GRID + 1);
}

struct WsLayout {
    size_t ints_off, info_off;
    size_t gu_off;     // float [KS][2][R][F] gate/up partial sums (KS > 1)
    size_t h_off;      // float [R][F] silu(gate) * up (KS == 1)
    size_t total;
};

inline WsLayout ws_layout(int T, int H, int F, int qtype, int E, int k) {
    WsLayout L;
    const size_t R = (size_t)T * k;
    GvPlan pl;
    if (!gv_plan(T, H, F, qtype, gv_n_act_max(T, E, k), &pl)) pl.KS = 1;
    const size_t ints = 16 + 2 * (size_t)E + 1 + R + 2 * (GV_MAX_GRID + 1);
    L.ints_off = 0;
    L.info_off = (ints * 4 + 255) / 256 * 256;
    L.gu_off = L.info_off + ((size_t)E * sizeof(ActInfo) + 255) / 256 * 256;
    const size_t gu = pl.KS > 1 ? (size_t)pl.KS * 2 * R * F * 4 : 0;
    L.h_off = L.gu_off + (gu + 255) / 256 * 256;
    const size_t hb = pl.KS > 1 ? 0 : R * F * 4;
    L.total = L.h_off + (hb + 255) / 256 * 256;
    return L;
}

__device__ __forceinline__ void warp_blocks(int nbr, int w, int &b0, int &b1) {
    b0 = (w * nbr) / GV_WARPS;
    b1 = ((w + 1) * nbr) / GV_WARPS;
}

// Bulk copies of one 32-row tile into a stage: rows [32g, 32g+32) of matrix `mat` [R][K],
// blocks [kb0, kb0+nbr) — the codes and the scales are one contiguous run each.
template <int QT>
__device__ __forceinline__ void issue_tile(const uint8_t *mat, int R, int K, int g, int kb0, int nbr,
                                           unsigned char *tile, size_t scale_off, uint64_t *bar) {
    const int QB = QT == MOE_Q8_0 ? 1024 : 512;
    const int SB = 32 * moe_scale_entry_bytes(QT);
    const int PPB = QT == MOE_Q8_0 ? 2 : 1;  // 16-byte pieces per block
    bulk_g2s(tile, mat + moe_piece_offset(QT, K, g, kb0 * PPB), (uint32_t)nbr * QB, bar);
    bulk_g2s(tile + scale_off, mat + moe_quant_bytes(QT, R, K) + moe_scale_offset(QT, K, g, kb0),
             (uint32_t)nbr * SB, bar);
}

// Fill path of a tile whose expert missed: its bytes come from the expert's pinned host
// image over the CPU-GPU link (16-byte loads by every thread, GV_FILL_BATCH in flight per
// thread) and are written both to the stage and through to the expert's slot, so the slot
// is filled by the kernels that use it.  Same byte ranges as issue_tile.
template <int QT>
__device__ void fill_tile(const uint8_t *src_mat, uint8_t *dst_mat, int R, int K, int g, int kb0, int nbr,
                          unsigned char *tile, size_t scale_off) {
    const int QB = QT == MOE_Q8_0 ? 1024 : 512;
    const int SB = 32 * moe_scale_entry_bytes(QT);
    const int PPB = QT == MOE_Q8_0 ? 2 : 1;
    const size_t qoff = moe_piece_offset(QT, K, g, kb0 * PPB);
    const size_t soff = moe_quant_bytes(QT, R, K) + moe_scale_offset(QT, K, g, kb0);
    const int nq = nbr * QB / 16, ns = nbr * SB / 16;
    constexpr int NB = GV_FILL_BATCH;
    for (int i0 = 0; i0 < nq + ns; i0 += NB * GV_THREADS) {
        uint4 v[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int i = i0 + b * GV_THREADS + threadIdx.x;
            if (i < nq + ns) {
                const size_t off = i < nq ? qoff + (size_t)i * 16 : soff + (size_t)(i - nq) * 16;
                v[b] = __ldcs((const uint4 *)(src_mat + off));
            }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int i = i0 + b * GV_THREADS + threadIdx.x;
            if (i < nq + ns) {
                const bool q = i < nq;
                const size_t off = q ? qoff + (size_t)i * 16 : soff + (size_t)(i - nq) * 16;
                *(uint4 *)(tile + (q ? (size_t)i * 16 : scale_off + (size_t)(i - nq) * 16)) = v[b];
                __stcs((uint4 *)(dst_mat + off), v[b]);
            }
        }
    }
}

// fp32 scale of column c of a 4-bit block in the activation copy: code j = c % 8 of a
// word decodes to q * 16^j (j <= 4) or q * 16^(j-5) (j >= 5), so the activation is
// pre-multiplied by the inverse power of two (exact).
__device__ __forceinline__ float q4_act_scale(int c) {
    const int j = c & 7;
    const int e = j <= 4 ? j : j - 5;
    return __int_as_float((127 - 4 * e) << 23);
}

__device__ __forceinline__ float q4_act_unscale(int c) {
    const int j = c & 7;
    const int e = j <= 4 ? j : j - 5;
    return __int_as_float((127 + 4 * e) << 23);
}

// Decoded fp32 pairs of one 32-bit word of codes (q8_0: 4 codes -> 2 pairs; 4-bit: 8 codes
// -> 4 pairs, code j scaled by 16^j or 16^(j-5)).
template <int QT>
__device__ __forceinline__ void decode_word(uint32_t w, unsigned long long (&p)[QT == MOE_Q8_0 ? 2 : 4]) {
    if constexpr (QT == MOE_Q8_0) {
        const unsigned long long MAG8 = f2_pack(-8388736.0f, -8388736.0f);  // 2^23 + 128
        const uint32_t wx = w ^ 0x80808080u;  // int8 -> offset-128 bytes
        const float v0 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7440));
        const float v1 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7441));
        const float v2 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7442));
        const float v3 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7443));
        p[0] = f2_add(f2_pack(v0, v1), MAG8);
        p[1] = f2_add(f2_pack(v2, v3), MAG8);
    } else {
        const unsigned long long MAG4 = f2_pack(-8388608.0f, -8388608.0f);  // 2^23
        const uint32_t w5 = w >> 20;
        const float v0 = __int_as_float((w & 0xFu) | 0x4B000000u);
        const float v1 = __int_as_float((w & 0xF0u) | 0x4B000000u);
        const float v2 = __int_as_float((w & 0xF00u) | 0x4B000000u);
        const float v3 = __int_as_float((w & 0xF000u) | 0x4B000000u);
        const float v4 = __int_as_float((w & 0xF0000u) | 0x4B000000u);
        const float v5 = __int_as_float((w5 & 0xFu) | 0x4B000000u);
        const float v6 = __int_as_float((w5 & 0xF0u) | 0x4B000000u);
        const float v7 = __int_as_float((w5 & 0xF00u) | 0x4B000000u);
        p[0] = f2_add(f2_pack(v0, v1), MAG4);
        p[1] = f2_add(f2_pack(v2, v3), MAG4);
        p[2] = f2_add(f2_pack(v4, v5), MAG4);
        p[3] = f2_add(f2_pack(v6, v7), MAG4);
    }
}

// One block b of the lane's row in NTL tiles against NT staged activation rows:
// acc[i][t] += d_i * sum (+ m_i * asum for 4-bit).  Each activation vector read from
// shared memory serves every tile.  act: [NT][Kr] fp32, asum: [NT][nbr].
template <int QT, int NT, int NTL>
__device__ __forceinline__ void block_dot(const unsigned char *tile0, const unsigned char *tile1, size_t scale_off,
                                          const float *act, const float *asum, int Kr, int nbr, int b, int lane,
                                          float (&acc)[2][GV_TOK]) {
    constexpr int WPB = QT == MOE_Q8_0 ? 8 : 4;  // 32-bit code words per lane and block
    constexpr int PPW = QT == MOE_Q8_0 ? 2 : 4;  // fp32 pairs per word
    const unsigned char *tl[2] = {tile0, tile1};
    uint32_t wd[NTL][WPB];
    uint32_t sc[NTL];
#pragma unroll
    for (int i = 0; i < NTL; ++i) {
        if constexpr (QT == MOE_Q8_0) {
            const uint4 qa = *(const uint4 *)(tl[i] + ((size_t)(2 * b) * 32 + lane) * 16);
            const uint4 qb = *(const uint4 *)(tl[i] + ((size_t)(2 * b + 1) * 32 + lane) * 16);
            wd[i][0] = qa.x; wd[i][1] = qa.y; wd[i][2] = qa.z; wd[i][3] = qa.w;
            wd[i][4] = qb.x; wd[i][5] = qb.y; wd[i][6] = qb.z; wd[i][7] = qb.w;
            sc[i] = *(const unsigned short *)(tl[i] + scale_off + ((size_t)b * 32 + lane) * 2);
        } else {
            const uint4 q = *(const uint4 *)(tl[i] + ((size_t)b * 32 + lane) * 16);
            wd[i][0] = q.x; wd[i][1] = q.y; wd[i][2] = q.z; wd[i][3] = q.w;
            sc[i] = *(const uint32_t *)(tl[i] + scale_off + ((size_t)b * 32 + lane) * 4);
        }
    }
    unsigned long long inner[NTL][NT];
#pragma unroll
    for (int i = 0; i < NTL; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t) inner[i][t] = 0ull;
#pragma unroll
    for (int wi = 0; wi < WPB; ++wi) {
        unsigned long long pr[NTL][PPW];
#pragma unroll
        for (int i = 0; i < NTL; ++i) decode_word<QT>(wd[i][wi], pr[i]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float *ap = act + (size_t)t * Kr + b * 32 + 2 * PPW * wi;
            const float4 xa = *(const float4 *)ap;
            const unsigned long long x01 = f2_pack(xa.x, xa.y), x23 = f2_pack(xa.z, xa.w);
            unsigned long long x45 = 0ull, x67 = 0ull;
            if constexpr (PPW == 4) {
                const float4 xb = *(const float4 *)(ap + 4);
                x45 = f2_pack(xb.x, xb.y);
                x67 = f2_pack(xb.z, xb.w);
            }
#pragma unroll
            for (int i = 0; i < NTL; ++i) {
                inner[i][t] = f2_fma(pr[i][0], x01, inner[i][t]);
                inner[i][t] = f2_fma(pr[i][1], x23, inner[i][t]);
                if constexpr (PPW == 4) {
                    inner[i][t] = f2_fma(pr[i][2], x45, inner[i][t]);
                    inner[i][t] = f2_fma(pr[i][3], x67, inner[i][t]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NTL; ++i) {
        const float d = __half2float(__ushort_as_half((unsigned short)(sc[i] & 0xFFFFu)));
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            float lo, hi;
            f2_unpack(inner[i][t], lo, hi);
            if constexpr (QT == MOE_Q8_0) {
                acc[i][t] = fmaf(d, lo + hi, acc[i][t]);
            } else {
                const float m = __half2float(__ushort_as_half((unsigned short)(sc[i] >> 16)));
                acc[i][t] = fmaf(d, lo + hi, fmaf(m, asum[(size_t)t * nbr + b], acc[i][t]));
            }
        }
    }
}

template <int QT, int NTL>
__device__ __forceinline__ void tile_dot_dispatch(int nt, const unsigned char *tile0, const unsigned char *tile1,
                                                  size_t scale_off, const float *act, const float *asum, int Kr,
                                                  int nbr, int b0, int b1, int lane, float (&acc)[2][GV_TOK]) {
#define GV_DOT(N)                                                                                    \
    for (int b = b0; b < b1; ++b)                                                                    \
        block_dot<QT, N, NTL>(tile0, tile1, scale_off, act, asum, Kr, nbr, b, lane, acc);           \
    break;
    switch (nt) {
        case 1: GV_DOT(1)
        case 2: GV_DOT(2)
        case 3: GV_DOT(3)
        case 4: GV_DOT(4)
        case 5: GV_DOT(5)
        case 6: GV_DOT(6)
        case 7: GV_DOT(7)
        default: GV_DOT(8)
    }
#undef GV_DOT
}

// Block sums of the (unscaled) activations for the 4-bit min term.
template <int QT>
__device__ __forceinline__ void compute_asum(const float *act, float *asum, int nt, int nbr, int Kr) {
    if constexpr (QT == MOE_Q4_SM) {
        for (int i = threadIdx.x; i < nt * nbr; i += GV_THREADS) {
            const int t = i / nbr, b = i % nbr;
            float s = 0.f;
            for (int c = 0; c < 32; ++c) s += act[(size_t)t * Kr + b * 32 + c] * q4_act_unscale(c);
            asum[i] = s;
        }
    }
}

struct FfnParams {
    const void *x;
    int T, H, F, k, E, KS, RT, TPU;
    const float *weights;
    const int32_t *ws_ints;
    const int32_t *ranges;  // this launch's CTA boundaries: CTA c takes units [ranges[c], ranges[c+1])
    const ActInfo *info;
    float *gu;
    float *h;
    float *partial;
    int *status;
    int stages;        // ring stages of this launch
    int x_vec;         // x is 16-byte aligned: vector loads
};

__device__ __forceinline__ void mbar_arrive_plain(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Stage the activations of route positions [pos, pos+nt) for columns [c0, c0+Kr): gate/up
// reads x (fp32 or bf16) of the routes' tokens (route of position pos+t at rbase[rpos+t]);
// down reads h, or forms silu(sum gate) * (sum up) from the K-split partial sums.
template <int QT, int XT, bool DOWN>
__device__ __forceinline__ void load_act(const FfnParams &p, const int *rbase, int rpos, int pos, int nt, int c0,
                                         int Kr, float *act) {
    const int nq = Kr / 4;
    for (int idx = threadIdx.x; idx < nt * nq; idx += GV_THREADS) {
        const int t = idx / nq, c = 4 * (idx - t * nq);
        float4 v;
        if (DOWN) {
            const size_t q = (size_t)(pos + t) * p.F + c;
            if (p.KS == 1) {
                v = *(const float4 *)(p.h + q);
            } else {
                float4 gs = make_float4(0.f, 0.f, 0.f, 0.f), us = gs;
                for (int ks = 0; ks < p.KS; ++ks) {  // fixed order over the K ranges
                    const float4 gv = *(const float4 *)(p.gu + ((size_t)ks * 2 + 0) * p.RT * p.F + q);
                    const float4 uv = *(const float4 *)(p.gu + ((size_t)ks * 2 + 1) * p.RT * p.F + q);
                    gs.x += gv.x; gs.y += gv.y; gs.z += gv.z; gs.w += gv.w;
                    us.x += uv.x; us.y += uv.y; us.z += uv.z; us.w += uv.w;
                }
                v = make_float4(silu_mul(gs.x, us.x), silu_mul(gs.y, us.y), silu_mul(gs.z, us.z),
                                silu_mul(gs.w, us.w));
            }
        } else {
            const size_t off = (size_t)(rbase[rpos + t] / p.k) * p.H + c0 + c;
            if (XT == MOE_BF16) {
                const __nv_bfloat16 *xb = (const __nv_bfloat16 *)p.x + off;
                if (p.x_vec) {
                    const uint2 r = *(const uint2 *)xb;
                    const float2 lo = __bfloat1622float2(*(const __nv_bfloat162 *)&r.x);
                    const float2 hi = __bfloat1622float2(*(const __nv_bfloat162 *)&r.y);
                    v = make_float4(lo.x, lo.y, hi.x, hi.y);
                } else {
                    v = make_float4(__bfloat162float(xb[0]), __bfloat162float(xb[1]), __bfloat162float(xb[2]),
                                    __bfloat162float(xb[3]));
                }
            } else {
                const float *xf = (const float *)p.x + off;
                v = p.x_vec ? *(const float4 *)xf : make_float4(xf[0], xf[1], xf[2], xf[3]);
            }
        }
        if (QT == MOE_Q4_SM) {
            v.x *= q4_act_scale(c);
            v.y *= q4_act_scale(c + 1);
            v.z *= q4_act_scale(c + 2);
            v.w *= q4_act_scale(c + 3);
        }
        *(float4 *)(act + (size_t)t * Kr + c) = v;
    }
}

// ------------------------------------------------------------------ G1 / G2: the ring kernel
//
// G1 (gate/up): units per active expert are KS K ranges x F/32 row tiles, ordered (ks, g);
// unit (ks, g) holds the gate tile g and the up tile g over K range ks, so consecutive units
// of a CTA share the expert's activations.  The reducing warp of token t forms
// h = silu(gate) * up (KS = 1) or stores both partial sums (KS > 1).
// G2 (down): units per active expert are H/(32 TPU) groups of TPU row tiles over the whole
// of F with h as activations; each unit writes w[r] * (Wd h) for its routes r.
//
// Ring protocol: stage s = i % S holds the CTA's i-th unit.  Thread 0 issues unit i+S-1
// at the top of iteration i, into the stage that unit i-1 used; every thread has finished
// reading that stage before the barrier that ends unit i-1's dot products.  A fill unit or
// a skipped expert arrives on its stage's mbarrier without bytes, so each stage completes
// exactly one phase per use and the waits use parity (i / S) & 1.

template <int QT, int XT, bool DOWN>
__global__ void __launch_bounds__(GV_THREADS, 1) ffn_ring_kernel(FfnParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = p.stages;
    const int RTF = p.F / 32, RTH = p.H / 32;
    const int NTL = DOWN ? p.TPU : 2;
    const int nbr = DOWN ? p.F / 32 : (p.H / 32) / p.KS, Kr = nbr * 32;
    const int R = DOWN ? p.H : p.F, K = DOWN ? p.F : p.H;
    const int per_a = DOWN ? RTH / p.TPU : p.KS * RTF;
    const int u0 = p.ranges[blockIdx.x], u1 = p.ranges[blockIdx.x + 1];
    if (u0 >= u1) return;
    const int ntok = min(p.T, GV_TOK);
    const RingSmem L = ring_smem(QT, nbr, NTL, ntok, S);
    uint64_t *bars = (uint64_t *)(smem + L.bars);
    unsigned char *stages = smem + L.stages;
    float *act = (float *)(smem + L.act);
    float *asum = (float *)(smem + L.asum);
    float *red = (float *)(smem + L.red);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int *routes = p.ws_ints + ws_routes_off(p.E);

    // the experts and routes of this CTA's range, in shared memory when they fit
    const int a_lo = u0 / per_a, a_hi = (u1 - 1) / per_a;
    const bool icache = a_hi - a_lo < GV_ICACHE;
    ActInfo *info_s = (ActInfo *)(smem + L.info);
    const int pos_lo = p.info[a_lo].pos0, pos_hi = p.info[a_hi].pos0 + p.info[a_hi].n_e;
    const bool rcache = pos_hi - pos_lo <= GV_RCACHE;
    int *rts_s = (int *)(smem + L.rts);
    float *wts_s = (float *)(smem + L.wts);
    if (icache)
        for (int a = a_lo + threadIdx.x; a <= a_hi; a += GV_THREADS) info_s[a - a_lo] = p.info[a];
    if (rcache)
        for (int q = pos_lo + threadIdx.x; q < pos_hi; q += GV_THREADS) {
            const int r = routes[q];
            rts_s[q - pos_lo] = r;
            if (DOWN) wts_s[q - pos_lo] = p.weights[r];
        }
    auto info_at = [&](int a) { return icache ? info_s[a - a_lo] : p.info[a]; };
    const int *rbase = rcache ? rts_s : routes;
    const int rpos0 = rcache ? pos_lo : 0;  // route position q is at rbase[q - rpos0]

    // unit u -> active expert a, K range ks, first row tile g (tile i: matrix mats[i], row tile g + i*DOWN)
    auto decode = [&](int u, int &a, int &ks, int &g) {
        a = u / per_a;
        const int r = u - a * per_a;
        if (DOWN) {
            ks = 0;
            g = r * p.TPU;
        } else {
            ks = r / RTF;
            g = r - ks * RTF;
        }
    };
    auto tile_mat = [&](int i) { return DOWN ? 2 : i; };
    auto tile_row = [&](int g, int i) { return DOWN ? g + i : g; };
    auto issue = [&](int u, int s, bool cached) {  // thread 0 only
        int a, ks, g;
        decode(u, a, ks, g);
        const ActInfo in = cached ? info_at(a) : p.info[a];
        if (in.n_e == 0 || in.fill) {
            mbar_arrive_plain(&bars[s]);
            return;
        }
        const int QB = QT == MOE_Q8_0 ? 1024 : 512, SB = 32 * moe_scale_entry_bytes(QT);
        mbar_arrive_expect_tx(&bars[s], (uint32_t)(NTL * nbr * (QB + SB)));
        for (int i = 0; i < NTL; ++i)
            issue_tile<QT>((const uint8_t *)in.src + moe_expert_matrix_offset(QT, p.H, p.F, tile_mat(i)), R, K,
                           tile_row(g, i), ks * nbr, nbr, stages + (size_t)s * L.stage_bytes + i * L.tile_bytes,
                           L.scale_off, &bars[s]);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
        for (int j = 0; j < S - 1 && u0 + j < u1; ++j) issue(u0 + j, j, false);
    }
    __syncthreads();

    int b0, b1;
    warp_blocks(nbr, warp, b0, b1);
    int cur_a = -1, cur_ks = -1, cur_tg = -1;
    int i = 0;
    bool failed = false;
    for (; u0 + i < u1; ++i) {
        const int u = u0 + i, s = i % S;
        if (threadIdx.x == 0 && u + S - 1 < u1) issue(u + S - 1, (i + S - 1) % S, true);
        int a, ks, g;
        decode(u, a, ks, g);
        const ActInfo in = info_at(a);
        unsigned char *stage = stages + (size_t)s * L.stage_bytes;
        // activations of the first token pass, loaded while the unit's bytes arrive
        const bool fresh = in.n_e > 0 && (a != cur_a || ks != cur_ks || cur_tg != 0);
        if (fresh)
            load_act<QT, XT, DOWN>(p, rbase, in.pos0 - rpos0, in.pos0, min(GV_TOK, in.n_e), ks * Kr, Kr, act);
        // warp 0 waits for the stage; the barrier below publishes it to the other warps
        const bool ok = warp == 0 ? mbar_wait_bounded(&bars[s], (i / S) & 1, p.status) : true;
        if (in.fill && in.n_e > 0) {
            for (int t = 0; t < NTL; ++t) {
                const size_t mo = moe_expert_matrix_offset(QT, p.H, p.F, tile_mat(t));
                fill_tile<QT>((const uint8_t *)in.src + mo, (uint8_t *)in.dst + mo, R, K, tile_row(g, t), ks * nbr,
                              nbr, stage + t * L.tile_bytes, L.scale_off);
            }
            fence_proxy_async_smem();  // a later bulk copy overwrites this stage
        }
        // uniform: every thread saw its stage complete; the activations and a filled stage
        // are visible; this unit's writes of red follow the previous unit's reads
        if (!__syncthreads_and(ok)) {
            failed = true;
            break;
        }
        if (fresh) {
            cur_a = a;
            cur_ks = ks;
            cur_tg = 0;
            if (QT == MOE_Q4_SM) {
                compute_asum<QT>(act, asum, min(GV_TOK, in.n_e), nbr, Kr);
                __syncthreads();
            }
        }
        for (int tg = 0; tg < in.n_e; tg += GV_TOK) {
            const int nt = min(GV_TOK, in.n_e - tg);
            if (tg != cur_tg) {  // further passes of an expert with more than 8 tokens
                load_act<QT, XT, DOWN>(p, rbase, in.pos0 + tg - rpos0, in.pos0 + tg, nt, ks * Kr, Kr, act);
                __syncthreads();
                if (QT == MOE_Q4_SM) {
                    compute_asum<QT>(act, asum, nt, nbr, Kr);
                    __syncthreads();
                }
                cur_tg = tg;
            }
            float acc[2][GV_TOK];
#pragma unroll
            for (int t = 0; t < GV_TOK; ++t) acc[0][t] = acc[1][t] = 0.f;
            if (NTL == 2)
                tile_dot_dispatch<QT, 2>(nt, stage, stage + L.tile_bytes, L.scale_off, act, asum, Kr, nbr, b0, b1,
                                         lane, acc);
            else
                tile_dot_dispatch<QT, 1>(nt, stage, stage, L.scale_off, act, asum, Kr, nbr, b0, b1, lane, acc);
#pragma unroll
            for (int t = 0; t < GV_TOK; ++t)
                if (t < nt) {
                    red[(((size_t)warp * ntok + t) * 2 + 0) * 32 + lane] = acc[0][t];
                    red[(((size_t)warp * ntok + t) * 2 + 1) * 32 + lane] = acc[1][t];
                }
            __syncthreads();  // red complete; every thread is done reading this stage and act
            if (warp < nt) {
                float v0 = 0.f, v1 = 0.f;
#pragma unroll
                for (int w = 0; w < GV_WARPS; ++w) {
                    v0 += red[(((size_t)w * ntok + warp) * 2 + 0) * 32 + lane];
                    v1 += red[(((size_t)w * ntok + warp) * 2 + 1) * 32 + lane];
                }
                const int pos = in.pos0 + tg + warp;
                if (DOWN) {
                    const int r = rbase[pos - rpos0];
                    const float wr = rcache ? wts_s[pos - rpos0] : p.weights[r];
                    p.partial[(size_t)r * p.H + 32 * g + lane] = wr * v0;
                    if (NTL == 2) p.partial[(size_t)r * p.H + 32 * (g + 1) + lane] = wr * v1;
                } else if (p.KS == 1) {
                    p.h[(size_t)pos * p.F + 32 * g + lane] = silu_mul(v0, v1);
                } else {
                    p.gu[(((size_t)ks * 2 + 0) * p.RT + pos) * p.F + 32 * g + lane] = v0;
                    p.gu[(((size_t)ks * 2 + 1) * p.RT + pos) * p.F + 32 * g + lane] = v1;
                }
            }
            if (tg + GV_TOK < in.n_e) __syncthreads();  // red and act are rewritten by the next pass
        }
    }
    // A wait ran out: never leave with copies in flight.  Units i .. last issued are
    // unconsumed; give each a second bounded wait.
    if (failed && threadIdx.x == 0) {
        const int last = min(u1 - 1, u0 + i + S - 1);
        for (int j = i; u0 + j <= last; ++j) mbar_wait_bounded(&bars[j % S], (j / S) & 1, p.status);
    }
}

// ------------------------------------------------------------------ P1: permute

// First unit whose start cost is >= x: unit u of active expert a starts at cost
// per_a * P[a] + (u - a * per_a) * cost[a].
__device__ __forceinline__ int unit_at_cost(long long x, int n_act, int per_a, const int *P, const int *cost) {
    const long long C = (long long)per_a * P[n_act];
    if (x >= C) return n_act * per_a;
    int lo = 0, hi = n_act - 1;  // largest a with per_a * P[a] <= x
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if ((long long)per_a * P[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    const long long rem = x - (long long)per_a * P[lo];
    return lo * per_a + (int)((rem + cost[lo] - 1) / cost[lo]);
}

// Stable counting sort of the routes r = t*k + j by expert (restricted to a subset), the
// ascending list of active experts, their route ranges, per active expert where its weights
// are read from (slot in the pool, or its pinned host image for a fill), and the unit
// ranges of the CTAs of both GEMV launches, balanced by work (unit_cost).
__global__ void __launch_bounds__(256) permute_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                      const int32_t *__restrict__ subset, int n_subset,
                                                      int32_t *__restrict__ ints, ActInfo *__restrict__ info,
                                                      const int32_t *__restrict__ slot_table, int n_slots,
                                                      const uint8_t *pool, size_t slot_bytes,
                                                      const unsigned long long *__restrict__ fill_src,
                                                      int G1, int per_a1, int G2, int per_a2, int *status) {
    __shared__ int cnt[MOE_MAX_E], off[MOE_MAX_E + 1], run[MOE_MAX_E];
    __shared__ int P[MOE_MAX_E + 1], cost[MOE_MAX_E];
    __shared__ unsigned char insub[MOE_MAX_E];
    __shared__ int chunk_e[256];
    __shared__ int n_act;
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += 256) {
        cnt[e] = 0;
        run[e] = 0;
        insub[e] = subset ? 0 : 1;
    }
    __syncthreads();
    if (subset) {
        for (int i = tid; i < n_subset; i += 256) {
            const int e = subset[i];
            if (e >= 0 && e < E) insub[e] = 1;
            else moe_set_status(status, MOE_ERR_INVALID);
        }
    }
    __syncthreads();
    for (int r = tid; r < R; r += 256) {
        const int e = ids[r];
        if (e < 0 || e >= E) { moe_set_status(status, MOE_ERR_INVALID); continue; }
        if (insub[e]) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    int *active = ints + ws_active_off();
    int *aoff = ints + ws_aoff_off(E);
    if (tid == 0) {
        int s = 0, na = 0;
        for (int e = 0; e < E; ++e) {
            off[e] = s;
            if (cnt[e] > 0) {
                active[na] = e;
                aoff[na] = s;
                ++na;
            }
            s += cnt[e];
        }
        aoff[na] = s;
        ints[0] = na;
        n_act = na;
    }
    __syncthreads();
    for (int a = tid; a < n_act; a += 256) {
        const int e = active[a];
        const int slot = slot_table ? slot_table[e] : e;
        ActInfo in;
        in.e = e;
        in.pos0 = aoff[a];
        in.n_e = aoff[a + 1] - aoff[a];
        in.fill = 0;
        in.src = in.dst = 0ull;
        if (slot < 0 || slot >= n_slots) {
            moe_set_status(status, MOE_ERR_INVALID);
            in.n_e = 0;  // nothing of this expert is read
        } else {
            in.dst = (unsigned long long)(pool + (size_t)slot * slot_bytes);
            const unsigned long long f = fill_src ? fill_src[e] : 0ull;
            in.fill = f != 0ull;
            in.src = f ? f : in.dst;
        }
        info[a] = in;
        cost[a] = unit_cost(in.n_e);
    }
    __syncthreads();
    if (tid == 0) {  // work prefix over the active experts (skipped experts cost 1 per unit)
        int c = 0;
        for (int a = 0; a < n_act; ++a) {
            P[a] = c;
            c += cost[a];
        }
        P[n_act] = c;
    }
    __syncthreads();
    {
        int *r1 = ints + ws_ranges_off(E, R, 0), *r2 = ints + ws_ranges_off(E, R, 1);
        const long long C1 = (long long)per_a1 * P[n_act], C2 = (long long)per_a2 * P[n_act];
        for (int c = tid; c <= G1; c += 256) r1[c] = unit_at_cost(C1 * c / G1, n_act, per_a1, P, cost);
        for (int c = tid; c <= G2; c += 256) r2[c] = unit_at_cost(C2 * c / G2, n_act, per_a2, P, cost);
    }
    int *routes = ints + ws_routes_off(E);
    for (int c0 = 0; c0 < R; c0 += 256) {
        const int r = c0 + tid;
        int e = -1;
        if (r < R) {
            e = ids[r];
            if (e < 0 || e >= E || !insub[e]) e = -1;
        }
        chunk_e[tid] = e;
        __syncthreads();
        if (e >= 0) {
            int rank = 0;
            for (int i = 0; i < tid; ++i) rank += (chunk_e[i] == e);
            routes[off[e] + run[e] + rank] = r;
        }
        __syncthreads();
        if (e >= 0) atomicAdd(&run[e], 1);
        __syncthreads();
    }
}

// ------------------------------------------------------------------ C1: combine

__global__ void combine_kernel(const float4 *__restrict__ partial, int T, int k, int H4,
                               const float4 *extra, float4 *y) {
    const size_t n = (size_t)T * H4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t t = i / H4, h = i % H4;
        float4 s = extra ? extra[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float4 v = partial[(t * k + j) * H4 + h];
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
        y[i] = s;
    }
}

// Combine + RMSNorm for the stack: one CTA per token.  y = extra + sum_j partial[j] (fixed
// order), then xn = y / sqrt(mean(y^2) + eps) with a fixed-order block reduction.
__global__ void __launch_bounds__(256) combine_norm_kernel(const float4 *__restrict__ partial, int k, int H4,
                                                           const float4 *extra, float4 *y, float4 *xn,
                                                           float eps) {
    __shared__ float red[8];
    const int t = blockIdx.x;
    float ss = 0.f;
    for (int h = threadIdx.x; h < H4; h += blockDim.x) {
        float4 s = extra ? extra[(size_t)t * H4 + h] : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float4 v = partial[((size_t)t * k + j) * H4 + h];
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
        if (y) y[(size_t)t * H4 + h] = s;
        ss += s.x * s.x + s.y * s.y + s.z * s.z + s.w * s.w;
        if (xn) xn[(size_t)t * H4 + h] = s;  // scaled below
    }
    if (!xn) return;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)(4 * H4) + eps);
    for (int h = threadIdx.x; h < H4; h += blockDim.x) {
        float4 v = xn[(size_t)t * H4 + h];
        v.x *= inv; v.y *= inv; v.z *= inv; v.w *= inv;
        xn[(size_t)t * H4 + h] = v;
    }
}

// Resident CTAs of a ring kernel on the whole device at a dynamic shared-memory size,
// cached per (device, kernel, size).  The kernel's shared-memory limit is only ever raised,
// so every cached size stays launchable.
struct OccEntry {
    int dev;
    const void *fn;
    size_t smem;
    int ctas;
};

int ring_grid_capacity(const void *fn, size_t smem, int *ctas) {
    static std::mutex mu;
    static OccEntry tab[64];
    static int n_tab = 0;
    static struct { int dev; const void *fn; size_t max; } lim[32];
    static int n_lim = 0;
    int dev = 0;
    MOE_TRY_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> g(mu);
    for (int i = 0; i < n_tab; ++i)
        if (tab[i].dev == dev && tab[i].fn == fn && tab[i].smem == smem) {
            *ctas = tab[i].ctas;
            return MOE_OK;
        }
    int li = -1;
    for (int i = 0; i < n_lim; ++i)
        if (lim[i].dev == dev && lim[i].fn == fn) li = i;
    if (li < 0 || lim[li].max < smem) {
        MOE_TRY_CUDA(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        if (li < 0 && n_lim < 32) li = n_lim++;
        if (li >= 0) lim[li] = {dev, fn, smem};
    }
    int occ = 0, sms = 0;
    MOE_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, GV_THREADS, smem));
    MOE_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (occ < 1 || sms < 1) return MOE_ERR_UNSUPPORTED;
    *ctas = std::min(occ * sms, GV_MAX_GRID);
    if (n_tab < 64) tab[n_tab++] = {dev, fn, smem, *ctas};
    return MOE_OK;
}

template <int QT, int XT, bool DOWN>
const void *ring_fn() {
    return (const void *)ffn_ring_kernel<QT, XT, DOWN>;
}

const void *ring_kernel_for(int qtype, int xtype, bool down) {
    if (qtype == MOE_Q8_0) {
        if (down) return ring_fn<MOE_Q8_0, MOE_F32, true>();
        return xtype == MOE_F32 ? ring_fn<MOE_Q8_0, MOE_F32, false>() : ring_fn<MOE_Q8_0, MOE_BF16, false>();
    }
    if (down) return ring_fn<MOE_Q4_SM, MOE_F32, true>();
    return xtype == MOE_F32 ? ring_fn<MOE_Q4_SM, MOE_F32, false>() : ring_fn<MOE_Q4_SM, MOE_BF16, false>();
}

}  // namespace

size_t moe_decode_workspace_bytes(int T, int H, int F, int qtype, int E, int k) {
    return ws_layout(T, H, F, qtype, E, k).total;
}

size_t moe_ffn_workspace_bytes(int T, int H, int F, int qtype, int xtype, int E, int k) {
    if (moe_prefill_eligible(T, H, F, qtype, xtype)) return moe_prefill_workspace_bytes(T, H, F, E, k);
    return moe_decode_workspace_bytes(T, H, F, qtype, E, k);
}

int moe_expert_ffn_impl(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                        const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                        int n_slots, const void *pool, size_t slot_bytes,
                        const int32_t *expert_subset, int n_subset, float *partial,
                        void *workspace, size_t ws_bytes, cudaStream_t s,
                        const moe_ffn_timing *timing) {
    return moe_expert_ffn_core(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots, pool,
                               slot_bytes, expert_subset, n_subset, nullptr, partial, workspace, ws_bytes, s,
                               timing);
}

int moe_expert_ffn_core(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                        const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                        int n_slots, const void *pool, size_t slot_bytes,
                        const int32_t *expert_subset, int n_subset, const uint64_t *d_fill_src,
                        float *partial, void *workspace, size_t ws_bytes, cudaStream_t s,
                        const moe_ffn_timing *timing) {
    MOE_CHECK(T >= 0);
    MOE_CHECK(qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
    MOE_CHECK(xtype == MOE_F32 || xtype == MOE_BF16);
    MOE_CHECK(H > 0 && F > 0 && H % 32 == 0 && F % 32 == 0);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K && k <= E);
    MOE_CHECK(n_subset >= 0 && n_subset <= E);
    if (T == 0 || (expert_subset && n_subset == 0)) return MOE_OK;
    MOE_CHECK(x && ids && weights && pool && partial && workspace);
    MOE_CHECK(n_slots >= 1);
    MOE_CHECK(((uintptr_t)pool & 15) == 0 && (slot_bytes & 15) == 0);
    MOE_CHECK(slot_bytes >= moe_expert_image_bytes(qtype, H, F));
    MOE_CHECK(((uintptr_t)workspace & 255) == 0);
    if (moe_prefill_eligible(T, H, F, qtype, xtype)) {
        if (d_fill_src) return MOE_ERR_UNSUPPORTED;  // slot filling is a decode-path feature
        MOE_CHECK(ws_bytes >= moe_prefill_workspace_bytes(T, H, F, E, k));
        return moe_prefill_ffn(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots, pool,
                               slot_bytes, expert_subset, n_subset, partial, workspace, ws_bytes, s, timing);
    }
    const WsLayout W = ws_layout(T, H, F, qtype, E, k);
    MOE_CHECK(ws_bytes >= W.total);
    if ((size_t)T * k > (1u << 20)) return MOE_ERR_UNSUPPORTED;
    GvPlan pl;  // planned for every expert routable (the workspace does not depend on a subset)
    if (!gv_plan(T, H, F, qtype, gv_n_act_max(T, E, k), &pl)) return MOE_ERR_UNSUPPORTED;
    const int ntok = T < GV_TOK ? T : GV_TOK;
    const int RTF = F / 32, RTH = H / 32;
    const int nb1 = (H / 32) / pl.KS, nb2 = F / 32;
    const size_t smem1 = ring_smem(qtype, nb1, 2, ntok, pl.S1).total;
    const size_t smem2 = ring_smem(qtype, nb2, pl.TPU, ntok, pl.S2).total;
    const void *k1 = ring_kernel_for(qtype, xtype, false), *k2 = ring_kernel_for(qtype, xtype, true);
    int cap1 = 0, cap2 = 0, rc;
    if ((rc = ring_grid_capacity(k1, smem1, &cap1)) != MOE_OK) return rc;
    if ((rc = ring_grid_capacity(k2, smem2, &cap2)) != MOE_OK) return rc;
    const int n_act_max = expert_subset ? n_subset : (T * k < E ? T * k : E);
    const int per_a1 = pl.KS * RTF, per_a2 = RTH / pl.TPU;
    const int G1 = std::max(1, std::min(cap1, n_act_max * per_a1));
    const int G2 = std::max(1, std::min(cap2, n_act_max * per_a2));

    FfnParams p;
    p.x = x;
    p.T = T; p.H = H; p.F = F; p.k = k; p.E = E;
    p.KS = pl.KS;
    p.TPU = pl.TPU;
    p.RT = T * k;
    p.weights = weights;
    p.ws_ints = (const int32_t *)((char *)workspace + W.ints_off);
    p.info = (const ActInfo *)((char *)workspace + W.info_off);
    p.gu = (float *)((char *)workspace + W.gu_off);
    p.h = (float *)((char *)workspace + W.h_off);
    p.partial = partial;
    p.status = moe_status_word_device_ptr();
    p.x_vec = ((uintptr_t)x % (xtype == MOE_F32 ? 16 : 8)) == 0;

    if (timing && timing->permute0) MOE_TRY_CUDA(cudaEventRecord(timing->permute0, s));
    permute_kernel<<<1, 256, 0, s>>>(ids, T * k, E, expert_subset, n_subset,
                                     (int32_t *)((char *)workspace + W.ints_off),
                                     (ActInfo *)((char *)workspace + W.info_off), d_slot_table, n_slots,
                                     (const uint8_t *)pool, slot_bytes, (const unsigned long long *)d_fill_src,
                                     G1, per_a1, G2, per_a2, p.status);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->permute1) MOE_TRY_CUDA(cudaEventRecord(timing->permute1, s));
    if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
    p.stages = pl.S1;
    p.ranges = p.ws_ints + ws_ranges_off(E, T * k, 0);
    if (qtype == MOE_Q8_0) {
        if (xtype == MOE_F32) ffn_ring_kernel<MOE_Q8_0, MOE_F32, false><<<G1, GV_THREADS, smem1, s>>>(p);
        else ffn_ring_kernel<MOE_Q8_0, MOE_BF16, false><<<G1, GV_THREADS, smem1, s>>>(p);
    } else {
        if (xtype == MOE_F32) ffn_ring_kernel<MOE_Q4_SM, MOE_F32, false><<<G1, GV_THREADS, smem1, s>>>(p);
        else ffn_ring_kernel<MOE_Q4_SM, MOE_BF16, false><<<G1, GV_THREADS, smem1, s>>>(p);
    }
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->gateup1) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
    p.stages = pl.S2;
    p.ranges = p.ws_ints + ws_ranges_off(E, T * k, 1);
    if (qtype == MOE_Q8_0) ffn_ring_kernel<MOE_Q8_0, MOE_F32, true><<<G2, GV_THREADS, smem2, s>>>(p);
    else ffn_ring_kernel<MOE_Q4_SM, MOE_F32, true><<<G2, GV_THREADS, smem2, s>>>(p);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->down1) MOE_TRY_CUDA(cudaEventRecord(timing->down1, s));
    return MOE_OK;
}

extern "C" int moe_expert_ffn(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                              const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                              int n_slots, const void *pool, size_t slot_bytes,
                              const int32_t *expert_subset, int n_subset, float *partial,
                              void *workspace, size_t ws_bytes, moe_stream_t s) {
    return moe_expert_ffn_impl(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots,
                               pool, slot_bytes, expert_subset, n_subset, partial, workspace,
                               ws_bytes, moe_cuda_stream(s), nullptr);
}

extern "C" int moe_expert_ffn_fill(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k,
                                   const int32_t *ids, const float *weights, const int32_t *d_slot_table,
                                   int n_slots, void *pool, size_t slot_bytes, const uint64_t *d_fill_src,
                                   float *partial, void *workspace, size_t ws_bytes, moe_stream_t s) {
    MOE_CHECK(d_slot_table && d_fill_src);
    return moe_expert_ffn_core(x, xtype, T, H, F, qtype, E, k, ids, weights, d_slot_table, n_slots, pool,
                               slot_bytes, nullptr, 0, d_fill_src, partial, workspace, ws_bytes,
                               moe_cuda_stream(s), nullptr);
}

extern "C" int moe_expert_ffn_workspace(int T, int H, int F, int qtype, int xtype, int E, int k,
                                        size_t *bytes) {
    MOE_CHECK(bytes);
    MOE_CHECK(T >= 0 && H > 0 && F > 0 && H % 32 == 0 && F % 32 == 0);
    MOE_CHECK(qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
    MOE_CHECK(xtype == MOE_F32 || xtype == MOE_BF16);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K);
    *bytes = moe_ffn_workspace_bytes(T, H, F, qtype, xtype, E, k);
    return MOE_OK;
}

extern "C" int moe_combine_rmsnorm(const float *partial, int T, int k, int H, const float *extra, float *y,
                                   float *xn, float eps, moe_stream_t s) {
    MOE_CHECK(T >= 0 && k >= 0 && k <= 64 && H > 0 && H % 4 == 0 && eps >= 0.f);
    if (T == 0) return MOE_OK;
    MOE_CHECK(k == 0 || partial);
    MOE_CHECK(y || xn);
    MOE_CHECK(((uintptr_t)partial & 15) == 0 && ((uintptr_t)y & 15) == 0 && ((uintptr_t)extra & 15) == 0 &&
              ((uintptr_t)xn & 15) == 0);
    MOE_CHECK(!(xn && (xn == extra || xn == y)));
    combine_norm_kernel<<<T, 256, 0, moe_cuda_stream(s)>>>((const float4 *)partial, k, H / 4,
                                                           (const float4 *)extra, (float4 *)y, (float4 *)xn, eps);
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
}

extern "C" int moe_combine(const float *partial, int T, int k, int H, const float *extra, float *y,
                           moe_stream_t s) {
    MOE_CHECK(T >= 0 && k >= 1 && k <= 64 && H > 0 && H % 4 == 0);
    if (T == 0) return MOE_OK;
    MOE_CHECK(partial && y);
    MOE_CHECK(((uintptr_t)partial & 15) == 0 && ((uintptr_t)y & 15) == 0 &&
              ((uintptr_t)extra & 15) == 0);
    const int H4 = H / 4;
    const size_t n = (size_t)T * H4;
    int grid = (int)((n + 255) / 256);
    if (grid > 152 * 8) grid = 152 * 8;
    combine_kernel<<<grid, 256, 0, moe_cuda_stream(s)>>>((const float4 *)partial, T, k, H4,
                                                          (const float4 *)extra, (float4 *)y);
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
}
