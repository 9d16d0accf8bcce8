// Prefill (batches above the decode limit): grouped GEMM on tcgen05 tensor cores.
//
// Page 4 ("llama.cpp MoE缓存实测", section "MoE缓存到底缓存了什么"): batches of more than
// 32 tokens (prompt processing) do not use the decode slots.  Here every routed token
// row is permuted into per-expert token tiles and each expert's FFN becomes two small
// GEMMs: [gate;up] (F x H) times the expert's tokens, SwiGLU, then down (H x F).
//
// GB300 mapping:
//  * route kernel: per-expert counts, token tiles of 128 routes, route of every tile row;
//  * gather kernel: activations -> fp16 tiles already in the UMMA 128-byte-swizzled
//    K-major layout, one contiguous block per (tile, 64-column chunk), so one bulk copy
//    (TMA engine) brings an A operand stage;
//  * GEMM kernels: persistent, one CTA per SM, each walking a strided list of work items
//    (token tile, 256-row weight slab) with warp-specialised roles and mbarrier rings
//    that run on across items.  The MMA is D[128 tokens][256 rows] += A[tokens][K] .
//    B[rows][K]^T (tcgen05.mma kind::f16, M=128, N=256, K=16 per instruction):
//      warp 0      bulk copies of the quantised weight pieces and the token tile of each
//                  64-column K stage into a raw ring;
//      warps 2-17  dequantise the codes to fp16 into a B ring in the swizzled layout
//                  (integer codes become fp16 by exponent tricks, then one fp16 FMA
//                  d*q [+ m] — a single rounding), one (row, 32-column block) per thread;
//      warp 1      issues the MMAs into one of two 256-column TMEM accumulators;
//      warps 18-21 the epilogue of the previous item from the other accumulator, one
//                  token per thread: GEMM 1 holds gate rows in columns 0-127 and up rows
//                  in 128-255, applies SwiGLU and writes the fp16 h row segment (the A
//                  operand of GEMM 2) with 16-byte stores; GEMM 2 scales by the router
//                  weight and writes 256 consecutive outputs of partial[t][j].
//  * Operands are fp16 (activations arrive as bf16 or fp32 and are rounded to fp16; bf16
//    operands would exceed the 2e-3 output tolerance on the Qwen-shaped layer).
//  * 4-bit operands: one 32-bit word of codes decodes into the fp16 pairs (q0,q4), (q1,q5),
//    (q2,q6), (q3,q7), so inside every 8-element group of K both operands of a 4-bit GEMM
//    are stored in the order 0,4,1,5,2,6,3,7 (the same permutation of K on both sides
//    leaves the products unchanged).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_tc.cuh"

#define PF_TM 128          // token rows per tile (MMA M)
#define PF_WN 256          // weight rows per item (MMA N)
#define PF_BK 64           // K columns per stage
#define PF_DQ_WARPS 16
#define PF_EPI_WARPS 4
#define PF_THREADS ((2 + PF_DQ_WARPS + PF_EPI_WARPS) * 32)
#define PF_AS 3            // dequantised (B operand) ring stages

namespace {

// ------------------------------------------------------------------ workspace layout

struct PfLayout {
    int max_tiles;
    size_t o_cnt, o_cursor, o_tbase, o_texp, o_trows, o_troute;  // int offsets (in ints)
    size_t ints_bytes, xp, hp, total;
};

inline PfLayout pf_layout(int T, int H, int F, int E, int k) {
    PfLayout L;
    const long R = (long)T * k;
    L.max_tiles = (int)(E + (R + PF_TM - 1) / PF_TM);
    size_t o = 16;
    L.o_cnt = o;    o += E;
    L.o_cursor = o; o += E;
    L.o_tbase = o;  o += E + 1;
    L.o_texp = o;   o += L.max_tiles;
    L.o_trows = o;  o += L.max_tiles;
    L.o_troute = o; o += (size_t)L.max_tiles * PF_TM;
    L.ints_bytes = (o * 4 + 1023) / 1024 * 1024;
    L.xp = L.ints_bytes;
    L.hp = L.xp + (size_t)L.max_tiles * H * PF_TM * 2;
    L.total = L.hp + (size_t)L.max_tiles * F * PF_TM * 2;
    L.total = (L.total + 255) / 256 * 256;
    return L;
}

// TMA tensor maps over the pool, one per matrix: 64-bit words of a tile block (codes and
// scales of 32 rows x 32 columns) x blocks x 32-row tiles x slots, so one copy brings a
// stage's box of 2 blocks of several row tiles of one matrix.
struct PfMaps {
    CUtensorMap blk[3];  // gate, up, down
};

struct PfParams {
    PfMaps maps;
    const void *x;
    int T, H, F, k, E;
    const float *weights;
    const int32_t *slot_table;
    int n_slots;
    const uint8_t *pool;
    size_t slot_bytes;
    int32_t *ints;
    uint8_t *xp, *hp;
    float *partial;
    int *status;
    size_t o_texp, o_trows, o_troute;
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 4-D TMA tile load global -> shared completing on `bar`; coordinates (x, y, z, w) in elements
// of the map (x is always 0 here, so the 16-byte alignment of the innermost coordinate holds).
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
        "[%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------------ route + gather

// Per-expert token tiles: tile i of expert e holds routes [i*128, (i+1)*128) of e in
// troute (-1 beyond the expert's count).  An expert whose slot is out of range is
// reported and its tiles get expert -1 (skipped by the GEMMs).
__global__ void __launch_bounds__(1024) pf_route_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                        const int32_t *__restrict__ subset, int n_subset,
                                                        const int32_t *__restrict__ slot_table, int n_slots,
                                                        int32_t *__restrict__ ints, size_t o_cnt,
                                                        size_t o_cursor, size_t o_tbase, size_t o_texp,
                                                        size_t o_trows, size_t o_troute, int *status) {
    __shared__ int cnt[MOE_MAX_E], cur[MOE_MAX_E], tb[MOE_MAX_E + 1];
    __shared__ unsigned char insub[MOE_MAX_E];
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) {
        cnt[e] = 0;
        cur[e] = 0;
        insub[e] = subset ? 0 : 1;
    }
    __syncthreads();
    if (subset)
        for (int i = tid; i < n_subset; i += blockDim.x) {
            const int e = subset[i];
            if (e >= 0 && e < E) insub[e] = 1;
            else moe_set_status(status, MOE_ERR_INVALID);
        }
    __syncthreads();
    // ids are read RB per thread at a time so that the loads overlap
    constexpr int RB = 8;
    for (int r0 = 0; r0 < R; r0 += RB * (int)blockDim.x) {
        int e8[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const int r = r0 + i * blockDim.x + tid;
            e8[i] = r < R ? ids[r] : 0;
        }
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            if (r0 + i * (int)blockDim.x + tid >= R) continue;
            const int e = e8[i];
            if (e < 0 || e >= E) { moe_set_status(status, MOE_ERR_INVALID); continue; }
            if (insub[e]) atomicAdd(&cnt[e], 1);
        }
    }
    __syncthreads();
    if (tid == 0) {
        int t = 0;
        for (int e = 0; e < E; ++e) {
            tb[e] = t;
            const int nt = (cnt[e] + PF_TM - 1) / PF_TM;
            const int slot = slot_table ? slot_table[e] : e;
            const bool valid = slot >= 0 && slot < n_slots;
            if (nt > 0 && !valid) moe_set_status(status, MOE_ERR_INVALID);
            for (int i = 0; i < nt; ++i) {
                ints[o_texp + t + i] = valid ? e : -1;
                ints[o_trows + t + i] = min(PF_TM, cnt[e] - i * PF_TM);
            }
            t += nt;
        }
        tb[E] = t;
        ints[0] = t;
    }
    __syncthreads();
    const int n_tiles = tb[E];
    for (int i = tid; i < n_tiles * PF_TM; i += blockDim.x) ints[o_troute + i] = -1;
    for (int e = tid; e < E; e += blockDim.x) {
        ints[o_cnt + e] = cnt[e];
        ints[o_tbase + e] = tb[e];
    }
    __syncthreads();
    for (int r0 = 0; r0 < R; r0 += RB * (int)blockDim.x) {
        int e8[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const int r = r0 + i * blockDim.x + tid;
            e8[i] = r < R ? ids[r] : -1;
        }
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const int e = e8[i];  // -1 beyond R
            if (e < 0 || e >= E || !insub[e]) continue;
            const int j = atomicAdd(&cur[e], 1);
            ints[o_troute + (size_t)(tb[e] + j / PF_TM) * PF_TM + (j % PF_TM)] = r0 + i * blockDim.x + tid;
        }
    }
}

// Activation rows of every tile -> fp16, 128-byte-swizzled K-major blocks (K in the
// 4-bit order when Q4).
template <int XT, bool Q4>
__global__ void __launch_bounds__(256) pf_gather_kernel(const void *__restrict__ x, int H, int k,
                                                        const int32_t *__restrict__ ints, size_t o_troute,
                                                        uint8_t *__restrict__ xp) {
    __shared__ int rt[PF_TM];
    const int tile = blockIdx.x;
    if (tile >= ints[0]) return;
    for (int i = threadIdx.x; i < PF_TM; i += blockDim.x) rt[i] = ints[o_troute + (size_t)tile * PF_TM + i];
    __syncthreads();
    const int NKC = H / PF_BK, C8 = H / 8;
#pragma unroll 4
    for (int idx = threadIdx.x; idx < PF_TM * C8; idx += blockDim.x) {
        const int row = idx / C8, c8 = idx % C8;
        const int r = rt[row];
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r >= 0) {
            const size_t base = (size_t)(r / k) * H + (size_t)c8 * 8;
            __half2 h[4];
            if (XT == MOE_BF16) {
                const uint4 raw = *(const uint4 *)((const __nv_bfloat16 *)x + base);
                const __nv_bfloat162 *b2 = (const __nv_bfloat162 *)&raw;
#pragma unroll
                for (int i = 0; i < 4; ++i) h[i] = __float22half2_rn(__bfloat1622float2(b2[i]));
            } else {
                const float4 a = *(const float4 *)((const float *)x + base);
                const float4 b = *(const float4 *)((const float *)x + base + 4);
                h[0] = __floats2half2_rn(a.x, a.y);
                h[1] = __floats2half2_rn(a.z, a.w);
                h[2] = __floats2half2_rn(b.x, b.y);
                h[3] = __floats2half2_rn(b.z, b.w);
            }
            const uint32_t *w = (const uint32_t *)h;
            if (Q4)  // (e0,e1)(e2,e3)(e4,e5)(e6,e7) -> (e0,e4)(e1,e5)(e2,e6)(e3,e7)
                v = make_uint4(__byte_perm(w[0], w[2], 0x5410), __byte_perm(w[0], w[2], 0x7632),
                               __byte_perm(w[1], w[3], 0x5410), __byte_perm(w[1], w[3], 0x7632));
            else
                v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        const int kc = c8 / 8;
        uint8_t *blk = xp + ((size_t)tile * NKC + kc) * PF_TM * 128;
        *(uint4 *)(blk + sw128_offset(row, (c8 % 8) * 8)) = v;
    }
}

// ------------------------------------------------------------------ dequant of one piece

// Raw stage layout (both GEMMs): 8 row tiles of 32 weight rows x 2 tile blocks (each the
// codes of 32 rows x 32 columns, then their 32 scale entries; slot image layout).  GEMM 1:
// row tiles 0-3 gate, 4-7 up; GEMM 2: down.
template <int QT> struct RawGeom {
    static constexpr int TBB = QT == MOE_Q8_0 ? 1088 : 640;   // bytes of a tile block
    static constexpr int SC = QT == MOE_Q8_0 ? 1024 : 512;    // its scale entries' offset
    static constexpr int BYTES = 8 * 2 * TBB;
};

__device__ __forceinline__ __half2 u32_as_half2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ uint32_t half2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Dequantise (row, block) of the raw stage into the swizzled fp16 B tile (256 rows).
//  q8_0: the offset-binary bytes q + 128 placed under the fp16 exponent of 1024 give
//        1152 + q exactly; subtracting 1152 leaves q, and one fp16 multiply by d rounds d*q
//        once.
//  4-bit: nibble pairs (n, n+4) masked under the exponent of 1024 give 1024 + q; then
//        q*d + m in one fp16 FMA (one rounding).
template <int QT>
__device__ __forceinline__ void dequant_piece(const uint8_t *raw, int row, int blk, uint8_t *b_tile) {
    using G = RawGeom<QT>;
    const int rt = row >> 5, lr = row & 31;
    if constexpr (QT == MOE_Q8_0) {
        const uint8_t *tb = raw + (size_t)(rt * 2 + blk) * G::TBB;
        const __half dh = __ushort_as_half(*(const unsigned short *)(tb + G::SC + moe_scale_pos(lr) * 2));
        const __half2 d2 = __halves2half2(dh, dh);
        const __half2 off = __float2half2_rn(1152.0f);
        uint4 q[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) q[h] = *(const uint4 *)(tb + moe_piece_in_block(h, lr));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t wd[4] = {q[h].x, q[h].y, q[h].z, q[h].w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 lo = __hsub2(u32_as_half2(__byte_perm(wd[i], 0x64646464u, 0x4140)), off);
                const __half2 hi = __hsub2(u32_as_half2(__byte_perm(wd[i], 0x64646464u, 0x4342)), off);
                o[2 * i] = half2_as_u32(__hmul2(lo, d2));
                o[2 * i + 1] = half2_as_u32(__hmul2(hi, d2));
            }
            *(uint4 *)(b_tile + sw128_offset(row, blk * 32 + 16 * h)) = make_uint4(o[0], o[1], o[2], o[3]);
            *(uint4 *)(b_tile + sw128_offset(row, blk * 32 + 16 * h + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
    } else {
        const uint8_t *tb = raw + (size_t)(rt * 2 + blk) * G::TBB;
        const uint32_t dm = *(const uint32_t *)(tb + G::SC + moe_scale_pos(lr) * 4);
        const uint4 q = *(const uint4 *)(tb + moe_piece_in_block(0, lr));
        const __half dh = __ushort_as_half((unsigned short)(dm & 0xFFFFu));
        const __half mh = __ushort_as_half((unsigned short)(dm >> 16));
        const __half2 d2 = __halves2half2(dh, dh), m2 = __halves2half2(mh, mh);
        const __half2 off = __float2half2_rn(1024.0f);
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t o[4];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const uint32_t u = ((wd[i] >> (4 * n)) & 0x000F000Fu) | 0x64006400u;
                o[n] = half2_as_u32(__hfma2(__hsub2(u32_as_half2(u), off), d2, m2));
            }
            *(uint4 *)(b_tile + sw128_offset(row, blk * 32 + 8 * i)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    const uint32_t a = smem_u32(p);
    return p + ((1024 - (a & 1023)) & 1023);
}

// Wait for an mbarrier phase; gives up (returns false) when another role has aborted or,
// after the spin limit, records MOE_ERR_TIMEOUT and aborts the CTA.
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, int *status, volatile int *abort_flag) {
    for (uint32_t i = 0; i < MOE_SPIN_LIMIT; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    moe_set_status(status, MOE_ERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

// ------------------------------------------------------------------ the persistent GEMM

template <int QT>
struct PfGeom {
    static constexpr int RS = QT == MOE_Q8_0 ? 3 : 4;         // raw + token tile ring stages
    static constexpr int RSTAGE = ((PF_TM * 128 + RawGeom<QT>::BYTES) + 1023) / 1024 * 1024;
    static constexpr int BSTAGE = PF_WN * 128;                // dequantised weights, fp16
    static constexpr uint32_t NCOLS = 2 * PF_WN;              // two fp32 accumulators of 256 columns
    static constexpr size_t SMEM = 2048 + (size_t)RS * RSTAGE + (size_t)PF_AS * BSTAGE;
};

// Work item j = (token tile j / MT, weight slab j % MT); CTA c takes j = c, c+G, ...
// GEMM 1 (DOWN = false): slab m = gate rows 128m.. and up rows 128m.. of F x H against the
// tile's x; epilogue h = silu(g) * u -> fp16 rows of GEMM 2's A operand.  GEMM 2: slab m =
// down rows 256m.. of H x F against h; epilogue w[r] * (.) -> partial[r][256m ..].
template <int QT, bool DOWN>
__global__ void __launch_bounds__(PF_THREADS, 1) pf_gemm_kernel(const __grid_constant__ PfParams p) {
    extern __shared__ uint8_t smem_raw[];
    using G = RawGeom<QT>;
    using PG = PfGeom<QT>;
    constexpr int RS = PG::RS, AS = PF_AS;
    const int MT = DOWN ? p.H / PF_WN : p.F / 128;
    const int NK = (DOWN ? p.F : p.H) / PF_BK;
    const int32_t *ints = p.ints;
    const int n_items = ints[0] * MT;
    if ((int)blockIdx.x >= n_items) return;

    uint8_t *smem = align1024(smem_raw);
    uint64_t *r_full = (uint64_t *)smem;
    uint64_t *r_empty = r_full + RS;
    uint64_t *b_full = r_empty + RS;
    uint64_t *b_empty = b_full + AS;
    uint64_t *acc_full = b_empty + AS;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    uint8_t *rring = smem + 1024;
    uint8_t *bring = rring + (size_t)RS * PG::RSTAGE;
    auto At = [&](int s) { return rring + (size_t)s * PG::RSTAGE; };
    auto RAW = [&](int s) { return rring + (size_t)s * PG::RSTAGE + PF_TM * 128; };
    auto Bt = [&](int s) { return bring + (size_t)s * PG::BSTAGE; };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&r_full[s], 1);
            mbar_init(&r_empty[s], 1);
        }
        for (int s = 0; s < AS; ++s) {
            mbar_init(&b_full[s], PF_DQ_WARPS);
            mbar_init(&b_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], PF_EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, PG::NCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto item_expert = [&](int j) { return ints[p.o_texp + j / MT]; };

    if (warp == 0) {
        // ---------------- producer (lane 0): per K stage the token tile (one bulk copy) and, per
        // weight matrix of the item, one TMA box of tile blocks
        if (lane == 0) {
            using Gq = RawGeom<QT>;
            int g = 0;
            bool ok = true;
            for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
                const int e = item_expert(j);
                if (e < 0) continue;
                const int tile = j / MT, m = j % MT;
                const int slot = p.slot_table ? p.slot_table[e] : e;
                const uint8_t *asrc = (DOWN ? p.hp : p.xp) + (size_t)tile * NK * PF_TM * 128;
                for (int kc = 0; kc < NK; ++kc, ++g) {
                    const int s = g % RS;
                    if (g >= RS && !(ok = pf_wait(&r_empty[s], ((g / RS) - 1) & 1, p.status, abort_flag))) break;
                    mbar_arrive_expect_tx(&r_full[s], Gq::BYTES + PF_TM * 128);
                    bulk_g2s(At(s), asrc + (size_t)kc * PF_TM * 128, PF_TM * 128, &r_full[s]);
                    if (DOWN) {
                        tma_load_4d(RAW(s), &p.maps.blk[2], 0, 2 * kc, 8 * m, slot, &r_full[s]);
                    } else {
                        for (int mt = 0; mt < 2; ++mt)
                            tma_load_4d(RAW(s) + 4 * mt * 2 * Gq::TBB, &p.maps.blk[mt], 0, 2 * kc, 4 * m, slot,
                                        &r_full[s]);
                    }
                }
            }
            // never leave with copies in flight: wait for the last phase issued on each stage
            for (int s = 0; s < RS && s < g; ++s) {
                const int last = s + ((g - 1 - s) / RS) * RS;
                mbar_wait_bounded(&r_full[s], (last / RS) & 1, p.status);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(PF_TM, PF_WN);
            int g = 0, jl = 0;
            bool ok = true;
            for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
                if (item_expert(j) < 0) continue;
                const int buf = jl & 1;
                if (jl >= 2 && !(ok = pf_wait(&acc_empty[buf], ((jl / 2) - 1) & 1, p.status, abort_flag))) break;
                tc_fence_after();
                const uint32_t d = tmem + buf * PF_WN;
                for (int kc = 0; kc < NK; ++kc, ++g) {
                    const int s = g % RS, sb = g % AS;
                    if (!(ok = pf_wait(&b_full[sb], (g / AS) & 1, p.status, abort_flag))) break;
                    if (!(ok = pf_wait(&r_full[s], (g / RS) & 1, p.status, abort_flag))) break;
                    tc_fence_after();
                    const uint64_t a = umma_desc_sw128(smem_u32(At(s)));
                    const uint64_t b = umma_desc_sw128(smem_u32(Bt(sb)));
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk)
                        umma_f16(d, a + 2 * kk, b + 2 * kk, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&b_empty[sb]);
                    umma_commit(&r_empty[s]);
                }
                if (ok) umma_commit(&acc_full[buf]);
                ++jl;
            }
            // every MMA of this CTA has completed before TMEM is released
            umma_commit(mma_done);
            mbar_wait_bounded(mma_done, 0, p.status);
        }
    } else if (warp < 2 + PF_DQ_WARPS) {
        // ---------------- dequant: thread -> (weight row 0..255, 32-column block) of the stage
        const int it = (warp - 2) * 32 + lane;
        const int blk = it >> 8, row = it & 255;
        int g = 0;
        bool ok = true;
        for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
            if (item_expert(j) < 0) continue;
            for (int kc = 0; kc < NK; ++kc, ++g) {
                const int s = g % RS, sb = g % AS;
                bool w = pf_wait(&r_full[s], (g / RS) & 1, p.status, abort_flag);
                if (w && g >= AS) w = pf_wait(&b_empty[sb], ((g / AS) - 1) & 1, p.status, abort_flag);
                if (!(ok = __all_sync(0xffffffffu, w))) break;  // the warp leaves together
                dequant_piece<QT>(RAW(s), row, blk, Bt(sb));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&b_full[sb]);
            }
        }
    } else {
        // ---------------- epilogue: TMEM lane = token row t = 32q + lane (q = warp % 4)
        const int q = warp & 3;
        const int t = 32 * q + lane;
        int jl = 0;
        bool ok = true;
        for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
            if (item_expert(j) < 0) continue;
            const int tile = j / MT, m = j % MT;
            // this token's route and router weight (GEMM 2), read before the accumulator is ready
            int route = -1;
            float wr = 0.f;
            if (DOWN) {
                if (t < ints[p.o_trows + tile]) {
                    route = ints[p.o_troute + (size_t)tile * PF_TM + t];
                    wr = p.weights[route];
                }
            }
            const int buf = jl & 1;
            ok = pf_wait(&acc_full[buf], (jl / 2) & 1, p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + buf * PF_WN;
            if (!DOWN) {
                // columns c (gate row 128m + c) and 128 + c (up row 128m + c) -> h[t][128m + c]
                uint8_t *hrow = p.hp + (size_t)tile * (p.F / PF_BK) * PF_TM * 128;
                for (int c0 = 0; c0 < 128; c0 += 16) {
                    uint32_t g16[16], u16[16];
                    tmem_ld16(tb + c0, g16);
                    tmem_ld16(tb + 128 + c0, u16);
                    tmem_ld_wait();
                    float h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float gv = __uint_as_float(g16[i]), uv = __uint_as_float(u16[i]);
                        h[i] = gv / (1.0f + __expf(-gv)) * uv;
                    }
                    const int f0 = 128 * m + c0;  // 16 consecutive F columns, two 8-column chunks
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t wds[4];
#pragma unroll
                        for (int pq = 0; pq < 4; ++pq) {
                            // physical slots 2pq, 2pq+1 hold logical (pq, pq+4) for 4-bit, (2pq, 2pq+1) otherwise
                            const float lo = QT == MOE_Q4_SM ? h[8 * ch + pq] : h[8 * ch + 2 * pq];
                            const float hi = QT == MOE_Q4_SM ? h[8 * ch + pq + 4] : h[8 * ch + 2 * pq + 1];
                            wds[pq] = half2_as_u32(__floats2half2_rn(lo, hi));
                        }
                        const int f = f0 + 8 * ch;
                        uint8_t *blkp = hrow + (size_t)(f / PF_BK) * PF_TM * 128;
                        *(uint4 *)(blkp + sw128_offset(t, f % PF_BK)) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
                    }
                }
            } else {
                // columns c -> output rows 256m + c of this token's route
                float *dst = route >= 0 ? p.partial + (size_t)route * p.H + PF_WN * m : nullptr;
                for (int c0 = 0; c0 < PF_WN; c0 += 16) {
                    uint32_t d16[16];
                    tmem_ld16(tb + c0, d16);
                    tmem_ld_wait();
                    if (dst) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *(float4 *)(dst + c0 + i) =
                                make_float4(wr * __uint_as_float(d16[i]), wr * __uint_as_float(d16[i + 1]),
                                            wr * __uint_as_float(d16[i + 2]), wr * __uint_as_float(d16[i + 3]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            ++jl;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, PG::NCOLS);
    }
}

// cuTensorMapEncodeTiled from the driver (looked up once through the runtime).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
    });
    return fn;
}

// Map of one matrix (mat: 0 gate, 1 up, 2 down) of every slot: tile blocks as [slot][row
// tile][block][TBB / 8 x uint64]; boxes of 2 K blocks x `tiles` row tiles.
template <int QT>
int encode_matrix_map(const uint8_t *pool, int n_slots, size_t slot_bytes, int H, int F, int mat, int tiles,
                      CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return MOE_ERR_UNSUPPORTED;
    using G = RawGeom<QT>;
    const int R = mat == 2 ? H : F, K = mat == 2 ? F : H;
    const int NB = K / 32;
    const uint8_t *base = pool + moe_expert_matrix_offset(QT, H, F, mat);
    const cuuint64_t dims[4] = {(cuuint64_t)(G::TBB / 8), (cuuint64_t)NB, (cuuint64_t)(R / 32), (cuuint64_t)n_slots};
    const cuuint64_t strides[3] = {(cuuint64_t)G::TBB, (cuuint64_t)NB * G::TBB, (cuuint64_t)slot_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)(G::TBB / 8), 2, (cuuint32_t)tiles, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, (void *)base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int sm_count_cached() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
    }
    return n;
}

template <int QT>
int launch_gemms(PfParams &p, int max_tiles, cudaStream_t s, const moe_ffn_timing *timing) {
    using PG = PfGeom<QT>;
    if (PG::SMEM > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    for (int mat = 0; mat < 3; ++mat) {
        const int rc = encode_matrix_map<QT>(p.pool, p.n_slots, p.slot_bytes, p.H, p.F, mat, mat == 2 ? 8 : 4,
                                             &p.maps.blk[mat]);
        if (rc != MOE_OK) return rc;
    }
    MOE_TRY_CUDA(cudaFuncSetAttribute(pf_gemm_kernel<QT, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)PG::SMEM));
    MOE_TRY_CUDA(cudaFuncSetAttribute(pf_gemm_kernel<QT, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)PG::SMEM));
    const int sms = sm_count_cached();
    const int items1 = max_tiles * (p.F / 128), items2 = max_tiles * (p.H / PF_WN);
    if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
    pf_gemm_kernel<QT, false><<<std::min(items1, sms), PF_THREADS, PG::SMEM, s>>>(p);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->gateup1) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
    pf_gemm_kernel<QT, true><<<std::min(items2, sms), PF_THREADS, PG::SMEM, s>>>(p);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->down1) MOE_TRY_CUDA(cudaEventRecord(timing->down1, s));
    return MOE_OK;
}

}  // namespace

bool moe_prefill_eligible(int T, int H, int F, int qtype, int xtype) {
    return T > MOE_DECODE_MAX_T && xtype == MOE_BF16 && H % PF_WN == 0 && F % 128 == 0 &&
           (qtype == MOE_Q8_0 || qtype == MOE_Q4_SM);
}

size_t moe_prefill_workspace_bytes(int T, int H, int F, int E, int k) { return pf_layout(T, H, F, E, k).total; }

int moe_prefill_ffn(const void *x, int xtype, int T, int H, int F, int qtype, int E, int k, const int32_t *ids,
                    const float *weights, const int32_t *d_slot_table, int n_slots, const void *pool,
                    size_t slot_bytes, const int32_t *expert_subset, int n_subset, float *partial,
                    void *workspace, size_t ws_bytes, cudaStream_t s, const moe_ffn_timing *timing) {
    const PfLayout L = pf_layout(T, H, F, E, k);
    MOE_CHECK(ws_bytes >= L.total);
    PfParams p;
    p.x = x;
    p.T = T; p.H = H; p.F = F; p.k = k; p.E = E;
    p.weights = weights;
    p.slot_table = d_slot_table;
    p.n_slots = n_slots;
    p.pool = (const uint8_t *)pool;
    p.slot_bytes = slot_bytes;
    p.ints = (int32_t *)workspace;
    p.xp = (uint8_t *)workspace + L.xp;
    p.hp = (uint8_t *)workspace + L.hp;
    p.partial = partial;
    p.status = moe_status_word_device_ptr();
    p.o_texp = L.o_texp;
    p.o_trows = L.o_trows;
    p.o_troute = L.o_troute;
    if (timing && timing->permute0) MOE_TRY_CUDA(cudaEventRecord(timing->permute0, s));
    pf_route_kernel<<<1, 1024, 0, s>>>(ids, T * k, E, expert_subset, n_subset, d_slot_table, n_slots, p.ints,
                                       L.o_cnt, L.o_cursor, L.o_tbase, L.o_texp, L.o_trows, L.o_troute, p.status);
    MOE_TRY_CUDA(cudaGetLastError());
    const bool q4 = qtype == MOE_Q4_SM;
    if (xtype == MOE_BF16) {
        if (q4) pf_gather_kernel<MOE_BF16, true><<<L.max_tiles, 256, 0, s>>>(x, H, k, p.ints, L.o_troute, p.xp);
        else pf_gather_kernel<MOE_BF16, false><<<L.max_tiles, 256, 0, s>>>(x, H, k, p.ints, L.o_troute, p.xp);
    } else {
        if (q4) pf_gather_kernel<MOE_F32, true><<<L.max_tiles, 256, 0, s>>>(x, H, k, p.ints, L.o_troute, p.xp);
        else pf_gather_kernel<MOE_F32, false><<<L.max_tiles, 256, 0, s>>>(x, H, k, p.ints, L.o_troute, p.xp);
    }
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->permute1) MOE_TRY_CUDA(cudaEventRecord(timing->permute1, s));
    return qtype == MOE_Q8_0 ? launch_gemms<MOE_Q8_0>(p, L.max_tiles, s, timing)
                             : launch_gemms<MOE_Q4_SM>(p, L.max_tiles, s, timing);
}
