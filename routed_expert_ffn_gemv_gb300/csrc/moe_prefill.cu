// Prefill (batches above the decode limit): grouped GEMM on tcgen05 tensor cores.
//
// Page 4 ("llama.cpp MoE缓存实测", section "MoE缓存到底缓存了什么"): batches of more than
// 32 tokens (prompt processing) do not use the decode slots.  Here every routed token
// row is permuted into per-expert token tiles and each expert's FFN becomes two small
// GEMMs: [gate;up] (F x H) times the expert's tokens, SwiGLU, then down (H x F).
//
// GB300 mapping:
//  * route kernel: per-expert counts, token tiles of BN rows, route of every tile row;
//  * gather kernel: activations -> fp16 tiles already in the UMMA 128-byte-swizzled
//    K-major layout, one contiguous block per (tile, 64-column chunk), so one bulk copy
//    (TMA engine) brings a B operand stage;
//  * GEMM kernels: persistent, one CTA per SM, each walking a strided list of work items
//    (token tile, 128-row weight tile) with warp-specialised roles and mbarrier rings
//    that run on across items:
//      warp 0     bulk copies of the quantised weight pieces and the B tile of each
//                 64-column K stage into a raw ring;
//      warps 2-9  dequantise the codes to fp16 into an A ring in the swizzled layout
//                 (integer codes become fp16 by exponent tricks, then one fp16 FMA
//                 d*q [+ m] — a single rounding);
//      warp 1     issues tcgen05.mma (M=128, N=BN, K=16 steps) into one of two TMEM
//                 accumulator buffers and commits stage releases;
//      warps 10-13 the epilogue of the previous item from the other TMEM buffer: GEMM 1
//                 applies SwiGLU and writes fp16 h tiles in the B layout of GEMM 2;
//                 GEMM 2 applies the router weight and scatters rows to partial[t][j].
//  * Operands are fp16 (activations arrive as bf16 or fp32 and are rounded to fp16; bf16
//    operands would exceed the 2e-3 output tolerance on the Qwen-shaped layer).
//  * 4-bit operands: one 32-bit word of codes decodes into the fp16 pairs (q0,q4), (q1,q5),
//    (q2,q6), (q3,q7), so inside every 8-element group of K both operands of a 4-bit GEMM
//    are stored in the order 0,4,1,5,2,6,3,7 (the same permutation of K on both sides
//    leaves the products unchanged).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "moe_tc.cuh"

#define PF_DQ_WARPS 8
#define PF_EPI_WARPS 4
#define PF_THREADS ((2 + PF_DQ_WARPS + PF_EPI_WARPS) * 32)
#define PF_BM 128
#define PF_BK 64
#define PF_R1 4   // raw/B ring stages, gate/up GEMM
#define PF_A1 2   // A ring stages, gate/up GEMM
#define PF_R2 6   // raw/B ring stages, down GEMM
#define PF_A2 3   // A ring stages, down GEMM

namespace {

// ------------------------------------------------------------------ workspace layout

// ------------------------------------------------------------------ workspace layout

struct PfLayout {
    int BN, max_tiles;
    size_t o_cnt, o_cursor, o_tbase, o_texp, o_trows, o_troute;  // int offsets (in ints)
    size_t ints_bytes, xp, hp, total;
};

inline int pf_block_n(int T, int k, int E) { return ((long)T * k / E > 96) ? 128 : 64; }

inline PfLayout pf_layout(int T, int H, int F, int E, int k) {
    PfLayout L;
    L.BN = pf_block_n(T, k, E);
    const long R = (long)T * k;
    L.max_tiles = (int)(E + (R + L.BN - 1) / L.BN);
    size_t o = 16;
    L.o_cnt = o;    o += E;
    L.o_cursor = o; o += E;
    L.o_tbase = o;  o += E + 1;
    L.o_texp = o;   o += L.max_tiles;
    L.o_trows = o;  o += L.max_tiles;
    L.o_troute = o; o += (size_t)L.max_tiles * L.BN;
    L.ints_bytes = (o * 4 + 1023) / 1024 * 1024;
    L.xp = L.ints_bytes;
    L.hp = L.xp + (size_t)L.max_tiles * H * L.BN * 2;
    L.total = L.hp + (size_t)L.max_tiles * F * L.BN * 2;
    L.total = (L.total + 255) / 256 * 256;
    return L;
}

struct PfParams {
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


// Physical position, inside an 8-element group of K, of logical element j of a 4-bit GEMM
// operand (order 0,4,1,5,2,6,3,7).
__host__ __device__ __forceinline__ int q4_kpos(int j) { return j < 4 ? 2 * j : 2 * (j - 4) + 1; }

// ------------------------------------------------------------------ route + gather

// Per-expert token tiles: tile i of expert e holds routes [i*BN, (i+1)*BN) of e in
// troute (-1 beyond the expert's count).  An expert whose slot is out of range is
// reported and its tiles get expert -1 (skipped by the GEMMs).
__global__ void __launch_bounds__(1024) pf_route_kernel(const int32_t *__restrict__ ids, int R, int E, int BN,
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
    for (int r = tid; r < R; r += blockDim.x) {
        const int e = ids[r];
        if (e < 0 || e >= E) { moe_set_status(status, MOE_ERR_INVALID); continue; }
        if (insub[e]) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int t = 0;
        for (int e = 0; e < E; ++e) {
            tb[e] = t;
            const int nt = (cnt[e] + BN - 1) / BN;
            const int slot = slot_table ? slot_table[e] : e;
            const bool valid = slot >= 0 && slot < n_slots;
            if (nt > 0 && !valid) moe_set_status(status, MOE_ERR_INVALID);
            for (int i = 0; i < nt; ++i) {
                ints[o_texp + t + i] = valid ? e : -1;
                ints[o_trows + t + i] = min(BN, cnt[e] - i * BN);
            }
            t += nt;
        }
        tb[E] = t;
        ints[0] = t;
    }
    __syncthreads();
    const int n_tiles = tb[E];
    for (int i = tid; i < n_tiles * BN; i += blockDim.x) ints[o_troute + i] = -1;
    for (int e = tid; e < E; e += blockDim.x) {
        ints[o_cnt + e] = cnt[e];
        ints[o_tbase + e] = tb[e];
    }
    __syncthreads();
    for (int r = tid; r < R; r += blockDim.x) {
        const int e = ids[r];
        if (e < 0 || e >= E || !insub[e]) continue;
        const int i = atomicAdd(&cur[e], 1);
        ints[o_troute + (size_t)(tb[e] + i / BN) * BN + (i % BN)] = r;
    }
}

// Activation rows of every tile -> fp16, 128-byte-swizzled K-major blocks (K in the
// 4-bit order when Q4).
template <int XT, bool Q4>
__global__ void __launch_bounds__(256) pf_gather_kernel(const void *__restrict__ x, int H, int k, int BN,
                                                        const int32_t *__restrict__ ints, size_t o_troute,
                                                        uint8_t *__restrict__ xp) {
    const int tile = blockIdx.x;
    if (tile >= ints[0]) return;
    const int NKC = H / PF_BK, C8 = H / 8;
    for (int idx = threadIdx.x; idx < BN * C8; idx += blockDim.x) {
        const int row = idx / C8, c8 = idx % C8;
        const int r = ints[o_troute + (size_t)tile * BN + row];
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
        uint8_t *blk = xp + ((size_t)tile * NKC + kc) * BN * 128;
        *(uint4 *)(blk + sw128_offset(row, (c8 % 8) * 8)) = v;
    }
}

// ------------------------------------------------------------------ dequant of one piece

// Raw stage layout per matrix: 4 row tiles x [codes of 2 blocks] then 4 row tiles x
// [scales of 2 blocks].
template <int QT> struct RawGeom {
    static constexpr int QPB = QT == MOE_Q8_0 ? 2048 : 1024;  // code bytes per row tile (2 blocks)
    static constexpr int SPB = 2 * 32 * (QT == MOE_Q8_0 ? 2 : 4);
    static constexpr int BYTES = 4 * (QPB + SPB);
    static constexpr int PPB = QT == MOE_Q8_0 ? 2 : 1;         // 16-byte pieces per block
};

__device__ __forceinline__ __half2 u32_as_half2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ uint32_t half2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Dequantise (row, block) of the raw stage into the swizzled fp16 A tile.
//  q8_0: bytes x ^ 0x80 placed under the fp16 exponent of 1024 give 1152 + q exactly;
//        subtracting 1152 leaves q, and one fp16 multiply by d rounds d*q once.
//  4-bit: nibble pairs (n, n+4) masked under the exponent of 1024 give 1024 + q; then
//        q*d + m in one fp16 FMA (one rounding).
template <int QT>
__device__ __forceinline__ void dequant_piece(const uint8_t *raw, int row, int blk, uint8_t *a_tile) {
    using G = RawGeom<QT>;
    const int rt = row >> 5, lr = row & 31;
    if constexpr (QT == MOE_Q8_0) {
        const __half dh = __ushort_as_half(
            *(const unsigned short *)(raw + 4 * G::QPB + rt * G::SPB + (blk * 32 + lr) * 2));
        const __half2 d2 = __halves2half2(dh, dh);
        const __half2 off = __float2half2_rn(1152.0f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 q = *(const uint4 *)(raw + rt * G::QPB + ((2 * blk + h) * 32 + lr) * 16);
            const uint32_t wd[4] = {q.x ^ 0x80808080u, q.y ^ 0x80808080u, q.z ^ 0x80808080u, q.w ^ 0x80808080u};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 lo = __hsub2(u32_as_half2(__byte_perm(wd[i], 0x64646464u, 0x4140)), off);
                const __half2 hi = __hsub2(u32_as_half2(__byte_perm(wd[i], 0x64646464u, 0x4342)), off);
                o[2 * i] = half2_as_u32(__hmul2(lo, d2));
                o[2 * i + 1] = half2_as_u32(__hmul2(hi, d2));
            }
            *(uint4 *)(a_tile + sw128_offset(row, blk * 32 + 16 * h)) = make_uint4(o[0], o[1], o[2], o[3]);
            *(uint4 *)(a_tile + sw128_offset(row, blk * 32 + 16 * h + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
    } else {
        const uint32_t dm = *(const uint32_t *)(raw + 4 * G::QPB + rt * G::SPB + (blk * 32 + lr) * 4);
        const __half dh = __ushort_as_half((unsigned short)(dm & 0xFFFFu));
        const __half mh = __ushort_as_half((unsigned short)(dm >> 16));
        const __half2 d2 = __halves2half2(dh, dh), m2 = __halves2half2(mh, mh);
        const __half2 off = __float2half2_rn(1024.0f);
        const uint4 q = *(const uint4 *)(raw + rt * G::QPB + (blk * 32 + lr) * 16);
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t o[4];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const uint32_t u = ((wd[i] >> (4 * n)) & 0x000F000Fu) | 0x64006400u;
                o[n] = half2_as_u32(__hfma2(__hsub2(u32_as_half2(u), off), d2, m2));
            }
            *(uint4 *)(a_tile + sw128_offset(row, blk * 32 + 8 * i)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// Issue the copies of one 64-column stage of a 128-row weight tile (4 row tiles of 32).
template <int QT>
__device__ __forceinline__ void issue_weight_stage(const uint8_t *mat, int R, int K, int m, int kc, uint8_t *raw,
                                                   uint64_t *bar) {
    using G = RawGeom<QT>;
    const uint8_t *scales = mat + moe_quant_bytes(QT, R, K);
    for (int rt = 0; rt < 4; ++rt) {
        const int g = 4 * m + rt;
        bulk_g2s(raw + rt * G::QPB, mat + moe_piece_offset(QT, K, g, 2 * kc * G::PPB), G::QPB, bar);
        bulk_g2s(raw + 4 * G::QPB + rt * G::SPB, scales + moe_scale_offset(QT, K, g, 2 * kc), G::SPB, bar);
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

template <int QT, int BN, bool DOWN>
struct PfGeom {
    static constexpr int NMAT = DOWN ? 1 : 2;                 // weight matrices per item
    static constexpr int RS = DOWN ? PF_R2 : PF_R1;
    static constexpr int AS = DOWN ? PF_A2 : PF_A1;
    static constexpr int RSTAGE = ((BN * 128 + NMAT * RawGeom<QT>::BYTES) + 1023) / 1024 * 1024;
    static constexpr int ASTAGE = NMAT * 16384;
    static constexpr uint32_t ACC = NMAT * BN;                // TMEM columns per accumulator buffer
    static constexpr uint32_t NCOLS = 2 * ACC < 32 ? 32 : 2 * ACC;  // a power of two here
    static constexpr size_t SMEM = 2048 + (size_t)RS * RSTAGE + (size_t)AS * ASTAGE;
};

// Work item j = (token tile j / MT, weight row tile j % MT), CTA c takes j = c, c+G, ...
// GEMM 1 (DOWN = false): [gate; up] rows 128m.. of F x H against the tile's x; epilogue
// h = silu(g) * u -> fp16 B tiles of GEMM 2.  GEMM 2: down rows 128m.. of H x F against
// h; epilogue w[r] * (.) -> partial[r][128m + row].
template <int QT, int BN, bool DOWN>
__global__ void __launch_bounds__(PF_THREADS, 1) pf_gemm_kernel(PfParams p) {
    extern __shared__ uint8_t smem_raw[];
    using G = RawGeom<QT>;
    using PG = PfGeom<QT, BN, DOWN>;
    constexpr int NMAT = PG::NMAT, RS = PG::RS, AS = PG::AS;
    const int MT = (DOWN ? p.H : p.F) / PF_BM;
    const int NK = (DOWN ? p.F : p.H) / PF_BK;
    const int32_t *ints = p.ints;
    const int n_items = ints[0] * MT;
    if ((int)blockIdx.x >= n_items) return;

    uint8_t *smem = align1024(smem_raw);
    uint64_t *r_full = (uint64_t *)smem;
    uint64_t *r_empty = r_full + RS;
    uint64_t *a_full = r_empty + RS;
    uint64_t *a_empty = a_full + AS;
    uint64_t *acc_full = a_empty + AS;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
    volatile int *abort_flag = (volatile int *)(tmem_slot + 1);
    uint8_t *rring = smem + 1024;
    uint8_t *aring = rring + (size_t)RS * PG::RSTAGE;
    auto Bt = [&](int s) { return rring + (size_t)s * PG::RSTAGE; };
    auto RAW = [&](int s) { return rring + (size_t)s * PG::RSTAGE + BN * 128; };
    auto At = [&](int s) { return aring + (size_t)s * PG::ASTAGE; };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&r_full[s], 1);
            mbar_init(&r_empty[s], 1);
        }
        for (int s = 0; s < AS; ++s) {
            mbar_init(&a_full[s], PF_DQ_WARPS);
            mbar_init(&a_empty[s], 1);
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
    auto mat_ptr = [&](int e, int mat) {
        const int slot = p.slot_table ? p.slot_table[e] : e;
        return p.pool + (size_t)slot * p.slot_bytes + moe_expert_matrix_offset(QT, p.H, p.F, DOWN ? 2 : mat);
    };

    if (warp == 0) {
        // ---------------- producer: raw weight pieces + B tile per K stage
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
                const int e = item_expert(j);
                if (e < 0) continue;
                const int tile = j / MT, m = j % MT;
                const uint8_t *mats[2] = {mat_ptr(e, 0), NMAT > 1 ? mat_ptr(e, 1) : nullptr};
                const uint8_t *bsrc = (DOWN ? p.hp : p.xp) + (size_t)tile * NK * BN * 128;
                for (int kc = 0; kc < NK; ++kc, ++g) {
                    const int s = g % RS;
                    if (g >= RS && !(ok = pf_wait(&r_empty[s], ((g / RS) - 1) & 1, p.status, abort_flag))) break;
                    mbar_arrive_expect_tx(&r_full[s], NMAT * G::BYTES + BN * 128);
                    for (int mt = 0; mt < NMAT; ++mt)
                        issue_weight_stage<QT>(mats[mt], DOWN ? p.H : p.F, DOWN ? p.F : p.H, m, kc,
                                               RAW(s) + mt * G::BYTES, &r_full[s]);
                    bulk_g2s(Bt(s), bsrc + (size_t)kc * BN * 128, BN * 128, &r_full[s]);
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
            constexpr uint32_t idesc = umma_idesc_f16_f32(PF_BM, BN);
            int g = 0, jl = 0;
            bool ok = true;
            for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
                if (item_expert(j) < 0) continue;
                const int buf = jl & 1;
                if (jl >= 2 && !(ok = pf_wait(&acc_empty[buf], ((jl / 2) - 1) & 1, p.status, abort_flag))) break;
                tc_fence_after();
                const uint32_t d0 = tmem + buf * PG::ACC;
                for (int kc = 0; kc < NK; ++kc, ++g) {
                    const int s = g % RS, sa = g % AS;
                    if (!(ok = pf_wait(&a_full[sa], (g / AS) & 1, p.status, abort_flag))) break;
                    if (!(ok = pf_wait(&r_full[s], (g / RS) & 1, p.status, abort_flag))) break;
                    tc_fence_after();
                    const uint64_t b = umma_desc_sw128(smem_u32(Bt(s)));
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk) {
                        const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
#pragma unroll
                        for (int mt = 0; mt < NMAT; ++mt)
                            umma_f16(d0 + mt * BN, umma_desc_sw128(smem_u32(At(sa) + mt * 16384)) + 2 * kk,
                                     b + 2 * kk, idesc, acc);
                    }
                    umma_commit(&a_empty[sa]);
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
        // ---------------- dequant: thread -> (row, 32-column block) of the 128 x 64 stage
        const int it = (warp - 2) * 32 + lane;
        const int blk = it >> 7, row = it & 127;
        int g = 0;
        bool ok = true;
        for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
            if (item_expert(j) < 0) continue;
            for (int kc = 0; kc < NK; ++kc, ++g) {
                const int s = g % RS, sa = g % AS;
                bool w = pf_wait(&r_full[s], (g / RS) & 1, p.status, abort_flag);
                if (w && g >= AS) w = pf_wait(&a_empty[sa], ((g / AS) - 1) & 1, p.status, abort_flag);
                if (!(ok = __all_sync(0xffffffffu, w))) break;  // the warp leaves together
#pragma unroll
                for (int mt = 0; mt < NMAT; ++mt) dequant_piece<QT>(RAW(s) + mt * G::BYTES, row, blk, At(sa) + mt * 16384);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[sa]);
            }
        }
    } else {
        // ---------------- epilogue: TMEM lanes 32q.. (q = warp % 4) = weight rows of the item
        const int q = warp & 3;
        const int r = 32 * q + lane;
        int jl = 0;
        bool ok = true;
        for (int j = blockIdx.x; j < n_items && ok; j += gridDim.x) {
            if (item_expert(j) < 0) continue;
            const int tile = j / MT, m = j % MT;
            const int buf = jl & 1;
            ok = pf_wait(&acc_full[buf], (jl / 2) & 1, p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + buf * PG::ACC;
            if (!DOWN) {
                const int f = PF_BM * m + r;
                const int fk = f % PF_BK;
                const int fpos = QT == MOE_Q4_SM ? (fk & ~7) + q4_kpos(fk & 7) : fk;
                uint8_t *hblk = p.hp + ((size_t)tile * (p.F / PF_BK) + f / PF_BK) * BN * 128;
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    uint32_t g16[16], u16[16];
                    tmem_ld16(tb + c0, g16);
                    tmem_ld16(tb + BN + c0, u16);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float gv = __uint_as_float(g16[i]), uv = __uint_as_float(u16[i]);
                        const float h = gv / (1.0f + expf(-gv)) * uv;
                        *(__half *)(hblk + sw128_offset(c0 + i, fpos)) = __float2half_rn(h);
                    }
                }
            } else {
                const int rows = ints[p.o_trows + tile];
                const int hrow = PF_BM * m + r;
                const int32_t *troute = ints + p.o_troute + (size_t)tile * BN;
                for (int c0 = 0; c0 < BN; c0 += 16) {
                    if (c0 >= rows) break;  // warp-uniform
                    uint32_t d16[16];
                    tmem_ld16(tb + c0, d16);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = c0 + i;
                        if (t < rows) {
                            const int route = troute[t];
                            p.partial[(size_t)route * p.H + hrow] = p.weights[route] * __uint_as_float(d16[i]);
                        }
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

template <int QT, int BN>
int launch_gemms(const PfParams &p, int max_tiles, cudaStream_t s, const moe_ffn_timing *timing) {
    using G1 = PfGeom<QT, BN, false>;
    using G2 = PfGeom<QT, BN, true>;
    if (G1::SMEM > 227 * 1024 || G2::SMEM > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    MOE_TRY_CUDA(cudaFuncSetAttribute(pf_gemm_kernel<QT, BN, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)G1::SMEM));
    MOE_TRY_CUDA(cudaFuncSetAttribute(pf_gemm_kernel<QT, BN, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)G2::SMEM));
    const int sms = sm_count_cached();
    const int items1 = max_tiles * (p.F / PF_BM), items2 = max_tiles * (p.H / PF_BM);
    if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
    pf_gemm_kernel<QT, BN, false><<<std::min(items1, sms), PF_THREADS, G1::SMEM, s>>>(p);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->gateup1) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
    pf_gemm_kernel<QT, BN, true><<<std::min(items2, sms), PF_THREADS, G2::SMEM, s>>>(p);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->down1) MOE_TRY_CUDA(cudaEventRecord(timing->down1, s));
    return MOE_OK;
}

}  // namespace
bool moe_prefill_eligible(int T, int H, int F, int qtype, int xtype) {
    return T > MOE_DECODE_MAX_T && xtype == MOE_BF16 && H % PF_BM == 0 && F % PF_BM == 0 &&
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
    pf_route_kernel<<<1, 1024, 0, s>>>(ids, T * k, E, L.BN, expert_subset, n_subset, d_slot_table, n_slots,
                                       p.ints, L.o_cnt, L.o_cursor,
                                       L.o_tbase, L.o_texp, L.o_trows, L.o_troute, p.status);
    MOE_TRY_CUDA(cudaGetLastError());
    const bool q4 = qtype == MOE_Q4_SM;
    if (xtype == MOE_BF16) {
        if (q4) pf_gather_kernel<MOE_BF16, true><<<L.max_tiles, 256, 0, s>>>(x, H, k, L.BN, p.ints, L.o_troute, p.xp);
        else pf_gather_kernel<MOE_BF16, false><<<L.max_tiles, 256, 0, s>>>(x, H, k, L.BN, p.ints, L.o_troute, p.xp);
    } else {
        if (q4) pf_gather_kernel<MOE_F32, true><<<L.max_tiles, 256, 0, s>>>(x, H, k, L.BN, p.ints, L.o_troute, p.xp);
        else pf_gather_kernel<MOE_F32, false><<<L.max_tiles, 256, 0, s>>>(x, H, k, L.BN, p.ints, L.o_troute, p.xp);
    }
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->permute1) MOE_TRY_CUDA(cudaEventRecord(timing->permute1, s));
    if (qtype == MOE_Q8_0)
        return L.BN == 128 ? launch_gemms<MOE_Q8_0, 128>(p, L.max_tiles, s, timing)
                           : launch_gemms<MOE_Q8_0, 64>(p, L.max_tiles, s, timing);
    return L.BN == 128 ? launch_gemms<MOE_Q4_SM, 128>(p, L.max_tiles, s, timing)
                       : launch_gemms<MOE_Q4_SM, 64>(p, L.max_tiles, s, timing);
}
