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
//  * GEMM kernels (one CTA per (token tile, 128-row weight tile)): warp 0 issues bulk
//    copies of the quantised weight pieces and the activation tile, eight warps
//    dequantise the codes to fp16 in the swizzled A layout (w = d*q [+ m], fp32, rounded
//    once), warp 1 owns the TMEM accumulator and issues tcgen05.mma (M=128, N=BN, K=16
//    steps) per 64-column stage; a 3-4 stage mbarrier ring overlaps copies, dequant and
//    MMA.  GEMM 1 keeps gate and up in two TMEM accumulators and its epilogue applies
//    SwiGLU and writes fp16 h tiles in the B layout of GEMM 2; GEMM 2's epilogue applies
//    the router weight and scatters each token row to partial[t][j].
//  * Operands are fp16 (activations arrive as bf16 or fp32 and are rounded to fp16; bf16
//    operands would exceed the 2e-3 output tolerance on the Qwen-shaped layer).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "moe_tc.cuh"

#define PF_DQ_WARPS 8
#define PF_THREADS ((2 + PF_DQ_WARPS) * 32)
#define PF_BM 128
#define PF_BK 64
#define PF_S1 3   // pipeline stages, gate/up GEMM
#define PF_S2 4   // pipeline stages, down GEMM

namespace {

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

// ------------------------------------------------------------------ route + gather

__global__ void __launch_bounds__(1024) pf_route_kernel(const int32_t *__restrict__ ids, int R, int E, int BN,
                                                        const int32_t *__restrict__ subset, int n_subset,
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
            for (int i = 0; i < nt; ++i) {
                ints[o_texp + t + i] = e;
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

// Activation rows of every tile -> fp16, 128-byte-swizzled K-major blocks.
template <int XT>
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
            v = *(const uint4 *)h;
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

// Dequantise (row, block) of the raw stage into the swizzled fp16 A tile.
template <int QT>
__device__ __forceinline__ void dequant_piece(const uint8_t *raw, int row, int blk, uint8_t *a_tile) {
    using G = RawGeom<QT>;
    const int rt = row >> 5, lr = row & 31;
    float w[32];
    if constexpr (QT == MOE_Q8_0) {
        const float d = __half2float(__ushort_as_half(
            *(const unsigned short *)(raw + 4 * G::QPB + rt * G::SPB + (blk * 32 + lr) * 2)));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 q = *(const uint4 *)(raw + rt * G::QPB + ((2 * blk + h) * 32 + lr) * 16);
            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int b = 0; b < 4; ++b) w[16 * h + 4 * i + b] = d * (float)(int8_t)(wd[i] >> (8 * b));
        }
    } else {
        const uint32_t dm = *(const uint32_t *)(raw + 4 * G::QPB + rt * G::SPB + (blk * 32 + lr) * 4);
        const float d = __half2float(__ushort_as_half((unsigned short)(dm & 0xFFFF)));
        const float m = __half2float(__ushort_as_half((unsigned short)(dm >> 16)));
        const uint4 q = *(const uint4 *)(raw + rt * G::QPB + (blk * 32 + lr) * 16);
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) w[8 * i + j] = fmaf(d, (float)((wd[i] >> (4 * j)) & 0xF), m);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        __half2 h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(w[8 * c + 2 * i], w[8 * c + 2 * i + 1]);
        *(uint4 *)(a_tile + sw128_offset(row, blk * 32 + 8 * c)) = *(const uint4 *)h;
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

template <int BN>
__device__ __forceinline__ size_t stage1_bytes(int rawb) {
    return 2 * 16384 + (size_t)BN * 128 + ((rawb * 2 + 1023) / 1024) * 1024;
}

// ------------------------------------------------------------------ GEMM 1: gate/up + SwiGLU

template <int QT, int BN>
__global__ void __launch_bounds__(PF_THREADS, 1) pf_gateup_kernel(PfParams p) {
    extern __shared__ uint8_t smem_raw[];
    using G = RawGeom<QT>;
    constexpr int S = PF_S1;
    constexpr uint32_t NCOLS = 2 * BN;
    const int MT = p.F / PF_BM;
    const int tile = blockIdx.x / MT, m = blockIdx.x % MT;
    const int32_t *ints = p.ints;
    if (tile >= ints[0]) return;
    const int e = ints[p.o_texp + tile];
    const int slot = p.slot_table ? p.slot_table[e] : e;
    if (slot < 0 || slot >= p.n_slots) {
        if (threadIdx.x == 0) moe_set_status(p.status, MOE_ERR_INVALID);
        return;
    }
    const uint8_t *mat_g = p.pool + (size_t)slot * p.slot_bytes + moe_expert_matrix_offset(QT, p.H, p.F, 0);
    const uint8_t *mat_u = p.pool + (size_t)slot * p.slot_bytes + moe_expert_matrix_offset(QT, p.H, p.F, 1);

    uint8_t *smem = align1024(smem_raw);
    uint64_t *full_raw = (uint64_t *)smem;
    uint64_t *full_a = full_raw + S;
    uint64_t *empty = full_a + S;
    uint64_t *acc_full = empty + S;
    uint32_t *tmem_slot = (uint32_t *)(acc_full + 1);
    uint8_t *stages = smem + 1024;
    const size_t SB = stage1_bytes<BN>(G::BYTES);
    auto A_g = [&](int s) { return stages + s * SB; };
    auto A_u = [&](int s) { return stages + s * SB + 16384; };
    auto Bt = [&](int s) { return stages + s * SB + 32768; };
    auto RAW = [&](int s) { return stages + s * SB + 32768 + (size_t)BN * 128; };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_raw[s], 1);
            mbar_init(&full_a[s], PF_DQ_WARPS);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, NCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int NK = p.H / PF_BK, NKF = p.F / PF_BK;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            for (int kc = 0; kc < NK && ok; ++kc) {
                const int s = kc % S;
                if (kc >= S) ok = mbar_wait_bounded(&empty[s], ((kc / S) - 1) & 1, p.status);
                if (!ok) break;
                mbar_arrive_expect_tx(&full_raw[s], 2 * G::BYTES + BN * 128);
                issue_weight_stage<QT>(mat_g, p.F, p.H, m, kc, RAW(s), &full_raw[s]);
                issue_weight_stage<QT>(mat_u, p.F, p.H, m, kc, RAW(s) + G::BYTES, &full_raw[s]);
                bulk_g2s(Bt(s), p.xp + ((size_t)tile * NK + kc) * BN * 128, BN * 128, &full_raw[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(PF_BM, BN);
            for (int kc = 0; kc < NK && ok; ++kc) {
                const int s = kc % S;
                ok = mbar_wait_bounded(&full_a[s], (kc / S) & 1, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ag = umma_desc_sw128(smem_u32(A_g(s)));
                const uint64_t au = umma_desc_sw128(smem_u32(A_u(s)));
                const uint64_t b = umma_desc_sw128(smem_u32(Bt(s)));
#pragma unroll
                for (int kk = 0; kk < PF_BK / 16; ++kk) {
                    const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
                    umma_f16(tmem, ag + 2 * kk, b + 2 * kk, idesc, acc);
                    umma_f16(tmem + BN, au + 2 * kk, b + 2 * kk, idesc, acc);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(acc_full);
        }
    } else {
        const int dw = warp - 2;
        const int it = dw * 32 + lane;
        const int blk = it >> 7, row = it & 127;
        for (int kc = 0; kc < NK; ++kc) {
            const int s = kc % S;
            if (!mbar_wait_bounded(&full_raw[s], (kc / S) & 1, p.status)) { ok = false; break; }
            dequant_piece<QT>(RAW(s), row, blk, A_g(s));
            dequant_piece<QT>(RAW(s) + G::BYTES, row, blk, A_u(s));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_a[s]);
        }
        // epilogue: h = silu(g) * u -> fp16 B tiles of the down GEMM
        if (ok) ok = mbar_wait_bounded(acc_full, 0, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            const int q = warp & 3, half = dw >> 2;
            const int r = 32 * q + lane;             // weight row within the 128-row tile
            const int f = PF_BM * m + r;
            uint8_t *hblk = p.hp + ((size_t)tile * NKF + f / PF_BK) * BN * 128;
            for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 16) {
                uint32_t g16[16], u16[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + c0, g16);
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + BN + c0, u16);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float g = __uint_as_float(g16[i]), u = __uint_as_float(u16[i]);
                    const float h = g / (1.0f + expf(-g)) * u;
                    *(__half *)(hblk + sw128_offset(c0 + i, f % PF_BK)) = __float2half_rn(h);
                }
            }
        }
    }
    // never leave with copies in flight: the producer drains the last phase of each stage
    if (threadIdx.x == 0) {
        for (int s = 0; s < S && s < NK; ++s) {
            const int last = (NK - 1 - s) / S;
            mbar_wait_bounded(&full_raw[s], last & 1, p.status);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, NCOLS);
    }
}

// ------------------------------------------------------------------ GEMM 2: down + weighted scatter

template <int BN>
__device__ __forceinline__ size_t stage2_bytes(int rawb) {
    return 16384 + (size_t)BN * 128 + ((rawb + 1023) / 1024) * 1024;
}

template <int QT, int BN>
__global__ void __launch_bounds__(PF_THREADS, 1) pf_down_kernel(PfParams p) {
    extern __shared__ uint8_t smem_raw[];
    using G = RawGeom<QT>;
    constexpr int S = PF_S2;
    constexpr uint32_t NCOLS = BN < 32 ? 32 : BN;
    const int MT = p.H / PF_BM;
    const int tile = blockIdx.x / MT, m = blockIdx.x % MT;
    const int32_t *ints = p.ints;
    if (tile >= ints[0]) return;
    const int e = ints[p.o_texp + tile];
    const int rows = ints[p.o_trows + tile];
    const int slot = p.slot_table ? p.slot_table[e] : e;
    if (slot < 0 || slot >= p.n_slots) {
        if (threadIdx.x == 0) moe_set_status(p.status, MOE_ERR_INVALID);
        return;
    }
    const uint8_t *mat = p.pool + (size_t)slot * p.slot_bytes + moe_expert_matrix_offset(QT, p.H, p.F, 2);

    uint8_t *smem = align1024(smem_raw);
    uint64_t *full_raw = (uint64_t *)smem;
    uint64_t *full_a = full_raw + S;
    uint64_t *empty = full_a + S;
    uint64_t *acc_full = empty + S;
    uint32_t *tmem_slot = (uint32_t *)(acc_full + 1);
    uint8_t *stages = smem + 1024;
    const size_t SB = stage2_bytes<BN>(G::BYTES);
    auto At = [&](int s) { return stages + s * SB; };
    auto Bt = [&](int s) { return stages + s * SB + 16384; };
    auto RAW = [&](int s) { return stages + s * SB + 16384 + (size_t)BN * 128; };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_raw[s], 1);
            mbar_init(&full_a[s], PF_DQ_WARPS);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, NCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int NK = p.F / PF_BK;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            for (int kc = 0; kc < NK && ok; ++kc) {
                const int s = kc % S;
                if (kc >= S) ok = mbar_wait_bounded(&empty[s], ((kc / S) - 1) & 1, p.status);
                if (!ok) break;
                mbar_arrive_expect_tx(&full_raw[s], G::BYTES + BN * 128);
                issue_weight_stage<QT>(mat, p.H, p.F, m, kc, RAW(s), &full_raw[s]);
                bulk_g2s(Bt(s), p.hp + ((size_t)tile * NK + kc) * BN * 128, BN * 128, &full_raw[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16_f32(PF_BM, BN);
            for (int kc = 0; kc < NK && ok; ++kc) {
                const int s = kc % S;
                ok = mbar_wait_bounded(&full_a[s], (kc / S) & 1, p.status);
                if (!ok) break;
                tc_fence_after();
                const uint64_t a = umma_desc_sw128(smem_u32(At(s)));
                const uint64_t b = umma_desc_sw128(smem_u32(Bt(s)));
#pragma unroll
                for (int kk = 0; kk < PF_BK / 16; ++kk)
                    umma_f16(tmem, a + 2 * kk, b + 2 * kk, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&empty[s]);
            }
            umma_commit(acc_full);
        }
    } else {
        const int dw = warp - 2;
        const int it = dw * 32 + lane;
        const int blk = it >> 7, row = it & 127;
        for (int kc = 0; kc < NK; ++kc) {
            const int s = kc % S;
            if (!mbar_wait_bounded(&full_raw[s], (kc / S) & 1, p.status)) { ok = false; break; }
            dequant_piece<QT>(RAW(s), row, blk, At(s));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_a[s]);
        }
        if (ok) ok = mbar_wait_bounded(acc_full, 0, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            const int q = warp & 3, half = dw >> 2;
            const int r = 32 * q + lane;
            const int hrow = PF_BM * m + r;
            const int32_t *troute = ints + p.o_troute + (size_t)tile * BN;
            for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 16) {
                uint32_t d16[16];
                tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + c0, d16);
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
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < S && s < NK; ++s) {
            const int last = (NK - 1 - s) / S;
            mbar_wait_bounded(&full_raw[s], last & 1, p.status);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, NCOLS);
    }
}

template <int QT, int BN>
size_t gateup_smem() { return 2048 + PF_S1 * (2 * 16384 + (size_t)BN * 128 + ((RawGeom<QT>::BYTES * 2 + 1023) / 1024) * 1024); }
template <int QT, int BN>
size_t down_smem() { return 2048 + PF_S2 * (16384 + (size_t)BN * 128 + ((RawGeom<QT>::BYTES + 1023) / 1024) * 1024); }

template <int QT, int BN>
int launch_gemms(const PfParams &p, int max_tiles, cudaStream_t s, const moe_ffn_timing *timing) {
    const size_t s1 = gateup_smem<QT, BN>(), s2 = down_smem<QT, BN>();
    if (s1 > 227 * 1024 || s2 > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    MOE_TRY_CUDA(cudaFuncSetAttribute(pf_gateup_kernel<QT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1));
    MOE_TRY_CUDA(cudaFuncSetAttribute(pf_down_kernel<QT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2));
    if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
    pf_gateup_kernel<QT, BN><<<max_tiles * (p.F / PF_BM), PF_THREADS, s1, s>>>(p);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->gateup1) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
    pf_down_kernel<QT, BN><<<max_tiles * (p.H / PF_BM), PF_THREADS, s2, s>>>(p);
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
    pf_route_kernel<<<1, 1024, 0, s>>>(ids, T * k, E, L.BN, expert_subset, n_subset, p.ints, L.o_cnt, L.o_cursor,
                                       L.o_tbase, L.o_texp, L.o_trows, L.o_troute, p.status);
    MOE_TRY_CUDA(cudaGetLastError());
    if (xtype == MOE_BF16)
        pf_gather_kernel<MOE_BF16><<<L.max_tiles, 256, 0, s>>>(x, H, k, L.BN, p.ints, L.o_troute, p.xp);
    else
        pf_gather_kernel<MOE_F32><<<L.max_tiles, 256, 0, s>>>(x, H, k, L.BN, p.ints, L.o_troute, p.xp);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->permute1) MOE_TRY_CUDA(cudaEventRecord(timing->permute1, s));
    if (qtype == MOE_Q8_0)
        return L.BN == 128 ? launch_gemms<MOE_Q8_0, 128>(p, L.max_tiles, s, timing)
                           : launch_gemms<MOE_Q8_0, 64>(p, L.max_tiles, s, timing);
    return L.BN == 128 ? launch_gemms<MOE_Q4_SM, 128>(p, L.max_tiles, s, timing)
                       : launch_gemms<MOE_Q4_SM, 64>(p, L.max_tiles, s, timing);
}
