// Decode-time expert FFN: permute (P1), gate/up dequantising GEMV (G1), down GEMV with
// the router-weighted scatter (G2), combine (C1).
//
// What is computed (pages 1-5, see moe.h): for every route (t, j) of a token t to its
// j-th selected expert e, h = silu(Wg_e x_t) * (Wu_e x_t) and
// partial[t][j] = w[t][j] * (Wd_e h); the combine sums partial over j.  Weights stay in
// their quantised blocks (page 5, section 1.2) and are dequantised in registers.
//
// GB300 mapping (the decode GEMVs are HBM-bound):
//  * a CTA owns one unit = (active expert, matrix, 32-row tile, K range); its 4 warps
//    split the K range; lane l owns row l of the tile, so each lane keeps the whole
//    dot product in registers and no cross-lane reduction is needed;
//  * at CTA start one thread issues bulk copies (TMA engine, cp.async.bulk) of every
//    warp's weight bytes into shared memory, so all of a unit's bytes are in flight at
//    once; the slot image layout makes each warp's bytes one contiguous run;
//  * activations of the expert's tokens are staged once in shared memory and read as
//    warp-wide broadcasts; codes become fp32 with exponent tricks (no int->float
//    conversion instructions) and accumulate with packed fp32x2 FMAs; block scales are
//    applied once per 32-weight block;
//  * tokens beyond 8 per expert are processed in further passes over the same
//    shared-memory weights.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "moe_ptx.cuh"

#define GV_WARPS 4
#define GV_THREADS (GV_WARPS * 32)
#define GV_TOK 8            // tokens per pass
#define GV_UNIT_QUANT 16384 // target code bytes per gate/up unit

namespace {

// ------------------------------------------------------------------ workspace layout

struct WsLayout {
    size_t ints_off;   // int32 region: [0] n_active, [16..16+E) active, a_off [E+1], routes [R]
    size_t gu_off;     // float [KS][2][R][F]
    size_t total;
};

__host__ __device__ inline int ws_active_off() { return 16; }
__host__ __device__ inline int ws_aoff_off(int E) { return 16 + E; }
__host__ __device__ inline int ws_routes_off(int E) { return 16 + 2 * E + 1; }

inline WsLayout ws_layout(int T, int H, int F, int qtype, int E, int k) {
    WsLayout L;
    const size_t R = (size_t)T * k;
    const size_t ints = 16 + 2 * (size_t)E + 1 + R;
    L.ints_off = 0;
    L.gu_off = (ints * 4 + 255) / 256 * 256;
    const int KS = moe_gateup_ksplit(qtype, H);
    L.total = L.gu_off + (size_t)KS * 2 * R * F * 4;
    L.total = (L.total + 255) / 256 * 256;
    return L;
}

// ------------------------------------------------------------------ shared-memory layout

struct UnitSmem {
    size_t bars, quant, scale, act, asum, red, total;
};

__host__ __device__ inline UnitSmem unit_smem(int qtype, int nbr, int ntok) {
    UnitSmem L;
    const int QB = qtype == MOE_Q8_0 ? 1024 : 512;           // code bytes per block of a 32-row tile
    const int SB = 32 * moe_scale_entry_bytes(qtype);        // scale bytes per block of a tile
    size_t off = 0;
    L.bars = off;  off += 128;
    L.quant = off; off += (size_t)nbr * QB;
    L.scale = off; off += ((size_t)nbr * SB + 127) / 128 * 128;
    L.act = off;   off += (size_t)ntok * nbr * 32 * 4;
    L.asum = off;  off += ((size_t)ntok * nbr * 4 + 15) / 16 * 16;
    L.red = off;   off += (size_t)GV_WARPS * GV_TOK * 32 * 4;
    L.total = off;
    return L;
}

__device__ __forceinline__ void warp_blocks(int nbr, int w, int &b0, int &b1) {
    b0 = (w * nbr) / GV_WARPS;
    b1 = ((w + 1) * nbr) / GV_WARPS;
}

// Issue the bulk copies of one unit: rows [32g, 32g+32) of matrix `mat` [R][K], blocks
// [kb0, kb0+nbr), warp w's share completing on bars[w].
template <int QT>
__device__ void issue_unit_copies(const uint8_t *mat, int R, int K, int g, int kb0, int nbr,
                                  unsigned char *smem, const UnitSmem &L) {
    uint64_t *bars = (uint64_t *)(smem + L.bars);
    const int QB = QT == MOE_Q8_0 ? 1024 : 512;
    const int SB = 32 * moe_scale_entry_bytes(QT);
    const int PPB = QT == MOE_Q8_0 ? 2 : 1;  // pieces per block
    for (int w = 0; w < GV_WARPS; ++w) mbar_init(&bars[w], 1);
    fence_mbar_init();
    const uint8_t *scales = mat + moe_quant_bytes(QT, R, K);
    for (int w = 0; w < GV_WARPS; ++w) {
        int b0, b1;
        warp_blocks(nbr, w, b0, b1);
        if (b1 <= b0) continue;
        const uint32_t qbytes = (uint32_t)(b1 - b0) * QB, sbytes = (uint32_t)(b1 - b0) * SB;
        mbar_arrive_expect_tx(&bars[w], qbytes + sbytes);
        bulk_g2s(smem + L.quant + (size_t)b0 * QB,
                 mat + moe_piece_offset(QT, K, g, (kb0 + b0) * PPB), qbytes, &bars[w]);
        bulk_g2s(smem + L.scale + (size_t)b0 * SB,
                 scales + moe_scale_offset(QT, K, g, kb0 + b0), sbytes, &bars[w]);
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

// Dot products of one lane's row with NT staged activation rows over warp blocks [b0,b1).
// act: [NT][Kr] (zero rows beyond the real token count), asum: [NT][nbr].
template <int QT, int NT>
__device__ __forceinline__ void tile_dot(const unsigned char *quant_s, const unsigned char *scale_s,
                                         const float *act, const float *asum, int Kr, int nbr,
                                         int b0, int b1, int lane, float *acc) {
    const unsigned long long MAG8 = f2_pack(-8388736.0f, -8388736.0f);  // 2^23 + 128
    const unsigned long long MAG4 = f2_pack(-8388608.0f, -8388608.0f);  // 2^23
    for (int b = b0; b < b1; ++b) {
        unsigned long long inner[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) inner[t] = 0ull;
        if constexpr (QT == MOE_Q8_0) {
            const uint4 qa = *(const uint4 *)(quant_s + ((size_t)(2 * b) * 32 + lane) * 16);
            const uint4 qb = *(const uint4 *)(quant_s + ((size_t)(2 * b + 1) * 32 + lane) * 16);
            const uint32_t wd[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t wx = wd[i] ^ 0x80808080u;  // int8 -> offset-128 bytes
                const float v0 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7440));
                const float v1 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7441));
                const float v2 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7442));
                const float v3 = __int_as_float(__byte_perm(wx, 0x4B000000u, 0x7443));
                const unsigned long long p01 = f2_add(f2_pack(v0, v1), MAG8);
                const unsigned long long p23 = f2_add(f2_pack(v2, v3), MAG8);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4 xv = *(const float4 *)(act + (size_t)t * Kr + b * 32 + 4 * i);
                    inner[t] = f2_fma(p01, f2_pack(xv.x, xv.y), inner[t]);
                    inner[t] = f2_fma(p23, f2_pack(xv.z, xv.w), inner[t]);
                }
            }
            const float d = __half2float(
                __ushort_as_half(*(const unsigned short *)(scale_s + ((size_t)b * 32 + lane) * 2)));
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float lo, hi;
                f2_unpack(inner[t], lo, hi);
                acc[t] = fmaf(d, lo + hi, acc[t]);
            }
        } else {
            const uint4 q = *(const uint4 *)(quant_s + ((size_t)b * 32 + lane) * 16);
            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = wd[i], w5 = wd[i] >> 20;
                const float v0 = __int_as_float((w & 0xFu) | 0x4B000000u);
                const float v1 = __int_as_float((w & 0xF0u) | 0x4B000000u);
                const float v2 = __int_as_float((w & 0xF00u) | 0x4B000000u);
                const float v3 = __int_as_float((w & 0xF000u) | 0x4B000000u);
                const float v4 = __int_as_float((w & 0xF0000u) | 0x4B000000u);
                const float v5 = __int_as_float((w5 & 0xFu) | 0x4B000000u);
                const float v6 = __int_as_float((w5 & 0xF0u) | 0x4B000000u);
                const float v7 = __int_as_float((w5 & 0xF00u) | 0x4B000000u);
                const unsigned long long p01 = f2_add(f2_pack(v0, v1), MAG4);
                const unsigned long long p23 = f2_add(f2_pack(v2, v3), MAG4);
                const unsigned long long p45 = f2_add(f2_pack(v4, v5), MAG4);
                const unsigned long long p67 = f2_add(f2_pack(v6, v7), MAG4);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4 xa = *(const float4 *)(act + (size_t)t * Kr + b * 32 + 8 * i);
                    const float4 xb = *(const float4 *)(act + (size_t)t * Kr + b * 32 + 8 * i + 4);
                    inner[t] = f2_fma(p01, f2_pack(xa.x, xa.y), inner[t]);
                    inner[t] = f2_fma(p23, f2_pack(xa.z, xa.w), inner[t]);
                    inner[t] = f2_fma(p45, f2_pack(xb.x, xb.y), inner[t]);
                    inner[t] = f2_fma(p67, f2_pack(xb.z, xb.w), inner[t]);
                }
            }
            const uint32_t dm = *(const uint32_t *)(scale_s + ((size_t)b * 32 + lane) * 4);
            const float d = __half2float(__ushort_as_half((unsigned short)(dm & 0xFFFFu)));
            const float m = __half2float(__ushort_as_half((unsigned short)(dm >> 16)));
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                float lo, hi;
                f2_unpack(inner[t], lo, hi);
                acc[t] = fmaf(d, lo + hi, fmaf(m, asum[(size_t)t * nbr + b], acc[t]));
            }
        }
    }
}

template <int QT>
__device__ __forceinline__ void tile_dot_dispatch(int ntp, const unsigned char *quant_s,
                                                  const unsigned char *scale_s, const float *act,
                                                  const float *asum, int Kr, int nbr, int b0, int b1,
                                                  int lane, float *acc) {
    switch (ntp) {
        case 1: tile_dot<QT, 1>(quant_s, scale_s, act, asum, Kr, nbr, b0, b1, lane, acc); break;
        case 2: tile_dot<QT, 2>(quant_s, scale_s, act, asum, Kr, nbr, b0, b1, lane, acc); break;
        case 4: tile_dot<QT, 4>(quant_s, scale_s, act, asum, Kr, nbr, b0, b1, lane, acc); break;
        default: tile_dot<QT, 8>(quant_s, scale_s, act, asum, Kr, nbr, b0, b1, lane, acc); break;
    }
}

__host__ __device__ __forceinline__ int pow2_tokens(int nt) { return nt <= 1 ? 1 : nt <= 2 ? 2 : nt <= 4 ? 4 : 8; }

// Block sums of the (unscaled) activations for the 4-bit min term.
template <int QT>
__device__ __forceinline__ void compute_asum(const float *act, float *asum, int ntp, int nbr, int Kr) {
    if constexpr (QT == MOE_Q4_SM) {
    for (int i = threadIdx.x; i < ntp * nbr; i += GV_THREADS) {
        const int t = i / nbr, b = i % nbr;
        float s = 0.f;
        for (int c = 0; c < 32; ++c) s += act[(size_t)t * Kr + b * 32 + c] * q4_act_unscale(c);
        asum[i] = s;
    }
    }
}

// Reduce the 4 warps' accumulators (fixed order) for token t of this pass.
__device__ __forceinline__ float reduce_warps(const float *red, int t, int lane) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < GV_WARPS; ++w) s += red[((size_t)w * GV_TOK + t) * 32 + lane];
    return s;
}

struct FfnParams {
    const void *x;
    int T, H, F, k, E, KS, RT;
    const int32_t *ids;
    const float *weights;
    const int32_t *ws_ints;
    float *gu;
    const int32_t *slot_table;
    int n_slots;
    const uint8_t *pool;
    size_t slot_bytes;
    float *partial;
    int *status;
    int ntok;          // activation rows staged per pass (<= GV_TOK)
    const unsigned long long *fill_src;  // [E]: pinned host image of an expert to fill, or 0
};

// Fill path of a unit whose expert missed: its bytes come from the expert's pinned host
// image over the CPU-GPU link (16-byte loads by every thread) and are written both to the
// unit's shared-memory stage and through to the expert's slot, so the slot is filled by
// the kernels that use it.  Same byte ranges as issue_unit_copies.
template <int QT>
__device__ void fill_unit(const uint8_t *src_mat, uint8_t *dst_mat, int R, int K, int g, int kb0, int nbr,
                          unsigned char *smem, const UnitSmem &L) {
    const int QB = QT == MOE_Q8_0 ? 1024 : 512;
    const int SB = 32 * moe_scale_entry_bytes(QT);
    const int PPB = QT == MOE_Q8_0 ? 2 : 1;
    const size_t qoff = moe_piece_offset(QT, K, g, kb0 * PPB);
    const size_t soff = moe_quant_bytes(QT, R, K) + moe_scale_offset(QT, K, g, kb0);
    const int nq = nbr * QB / 16, ns = nbr * SB / 16;
    for (int i = threadIdx.x; i < nq + ns; i += GV_THREADS) {
        const bool q = i < nq;
        const size_t off = q ? qoff + (size_t)i * 16 : soff + (size_t)(i - nq) * 16;
        const uint4 v = __ldcs((const uint4 *)(src_mat + off));
        *(uint4 *)(smem + (q ? L.quant + (size_t)i * 16 : L.scale + (size_t)(i - nq) * 16)) = v;
        __stcs((uint4 *)(dst_mat + off), v);
    }
}

template <int XT>
__device__ __forceinline__ float load_x(const void *x, size_t i) {
    if (XT == MOE_BF16) return __bfloat162float(((const __nv_bfloat16 *)x)[i]);
    return ((const float *)x)[i];
}

// ------------------------------------------------------------------ G1: gate / up

template <int QT, int XT>
__global__ void __launch_bounds__(GV_THREADS) gateup_kernel(FfnParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int RTF = p.F / 32;
    int u = blockIdx.x;
    const int ks = u % p.KS; u /= p.KS;
    const int g = u % RTF;   u /= RTF;
    const int m = u & 1;
    const int a = u >> 1;
    const int *ints = p.ws_ints;
    if (a >= ints[0]) return;                       // uniform: fewer active experts than the grid
    const int e = ints[ws_active_off() + a];
    const int slot = p.slot_table ? p.slot_table[e] : e;
    if (slot < 0 || slot >= p.n_slots) {
        if (threadIdx.x == 0) moe_set_status(p.status, MOE_ERR_INVALID);
        return;
    }
    const int K = p.H, nbr = (K / 32) / p.KS, kb0 = ks * nbr, Kr = nbr * 32;
    const UnitSmem L = unit_smem(QT, nbr, p.ntok);
    const uint8_t *mat = p.pool + (size_t)slot * p.slot_bytes + moe_expert_matrix_offset(QT, p.H, p.F, m);
    const uint8_t *fill = p.fill_src ? (const uint8_t *)p.fill_src[e] : nullptr;
    bool ready = false, ok = true;
    if (fill) {
        // visible to every warp after the first __syncthreads of the token loop
        fill_unit<QT>(fill + moe_expert_matrix_offset(QT, p.H, p.F, m), (uint8_t *)mat, p.F, K, g, kb0, nbr, smem, L);
        ready = true;
    } else if (threadIdx.x == 0) {
        issue_unit_copies<QT>(mat, p.F, K, g, kb0, nbr, smem, L);
    }
    __syncthreads();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int b0, b1;
    warp_blocks(nbr, warp, b0, b1);
    float *act = (float *)(smem + L.act);
    float *asum = (float *)(smem + L.asum);
    float *red = (float *)(smem + L.red);
    const int pos0 = ints[ws_aoff_off(p.E) + a];
    const int n_e = ints[ws_aoff_off(p.E) + a + 1] - pos0;
    const int *routes = ints + ws_routes_off(p.E);

    for (int tg = 0; tg < n_e; tg += GV_TOK) {
        const int nt = min(GV_TOK, n_e - tg), ntp = pow2_tokens(nt);
        for (int i = threadIdx.x; i < ntp * Kr; i += GV_THREADS) {
            const int t = i / Kr, c = i % Kr;
            float v = 0.f;
            if (t < nt) {
                const int tok = routes[pos0 + tg + t] / p.k;
                v = load_x<XT>(p.x, (size_t)tok * p.H + (size_t)kb0 * 32 + c);
                if (QT == MOE_Q4_SM) v *= q4_act_scale(c);
            }
            act[i] = v;
        }
        __syncthreads();
        compute_asum<QT>(act, asum, ntp, nbr, Kr);
        __syncthreads();
        if (!ready) {
            if (b1 > b0) ok = mbar_wait_bounded((uint64_t *)(smem + L.bars) + warp, 0, p.status);
            ready = true;
        }
        float acc[GV_TOK];
#pragma unroll
        for (int t = 0; t < GV_TOK; ++t) acc[t] = 0.f;
        if (ok) tile_dot_dispatch<QT>(ntp, smem + L.quant, smem + L.scale, act, asum, Kr, nbr, b0, b1, lane, acc);
#pragma unroll
        for (int t = 0; t < GV_TOK; ++t)
            if (t < ntp) red[((size_t)warp * GV_TOK + t) * 32 + lane] = acc[t];
        __syncthreads();
        for (int t = warp; t < nt; t += GV_WARPS) {
            const float s = reduce_warps(red, t, lane);
            p.gu[(((size_t)ks * 2 + m) * p.RT + pos0 + tg + t) * p.F + 32 * g + lane] = s;
        }
        __syncthreads();
    }
    // never leave with this warp's copies in flight (a timed-out wait gets a second bounded wait)
    if ((!ready || !ok) && b1 > b0) mbar_wait_bounded((uint64_t *)(smem + L.bars) + warp, 0, p.status);
}

// ------------------------------------------------------------------ G2: down + weighted scatter

template <int QT>
__global__ void __launch_bounds__(GV_THREADS) down_kernel(FfnParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int RTH = p.H / 32;
    const int g = blockIdx.x % RTH;
    const int a = blockIdx.x / RTH;
    const int *ints = p.ws_ints;
    if (a >= ints[0]) return;
    const int e = ints[ws_active_off() + a];
    const int slot = p.slot_table ? p.slot_table[e] : e;
    if (slot < 0 || slot >= p.n_slots) {
        if (threadIdx.x == 0) moe_set_status(p.status, MOE_ERR_INVALID);
        return;
    }
    const int K = p.F, nbr = K / 32, Kr = K;
    const UnitSmem L = unit_smem(QT, nbr, p.ntok);
    const uint8_t *mat = p.pool + (size_t)slot * p.slot_bytes + moe_expert_matrix_offset(QT, p.H, p.F, 2);
    const uint8_t *fill = p.fill_src ? (const uint8_t *)p.fill_src[e] : nullptr;
    bool ready = false, ok = true;
    if (fill) {
        fill_unit<QT>(fill + moe_expert_matrix_offset(QT, p.H, p.F, 2), (uint8_t *)mat, p.H, K, g, 0, nbr, smem, L);
        ready = true;
    } else if (threadIdx.x == 0) {
        issue_unit_copies<QT>(mat, p.H, K, g, 0, nbr, smem, L);
    }
    __syncthreads();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int b0, b1;
    warp_blocks(nbr, warp, b0, b1);
    float *act = (float *)(smem + L.act);
    float *asum = (float *)(smem + L.asum);
    float *red = (float *)(smem + L.red);
    const int pos0 = ints[ws_aoff_off(p.E) + a];
    const int n_e = ints[ws_aoff_off(p.E) + a + 1] - pos0;
    const int *routes = ints + ws_routes_off(p.E);

    for (int tg = 0; tg < n_e; tg += GV_TOK) {
        const int nt = min(GV_TOK, n_e - tg), ntp = pow2_tokens(nt);
        // h = silu(gate) * up from the K-split partial dot products (fixed ks order)
        for (int i = threadIdx.x; i < ntp * Kr; i += GV_THREADS) {
            const int t = i / Kr, c = i % Kr;
            float v = 0.f;
            if (t < nt) {
                const size_t pos = (size_t)pos0 + tg + t;
                float gs = 0.f, us = 0.f;
                for (int ks = 0; ks < p.KS; ++ks) {
                    gs += p.gu[(((size_t)ks * 2 + 0) * p.RT + pos) * p.F + c];
                    us += p.gu[(((size_t)ks * 2 + 1) * p.RT + pos) * p.F + c];
                }
                v = gs / (1.0f + expf(-gs)) * us;
                if (QT == MOE_Q4_SM) v *= q4_act_scale(c);
            }
            act[i] = v;
        }
        __syncthreads();
        compute_asum<QT>(act, asum, ntp, nbr, Kr);
        __syncthreads();
        if (!ready) {
            if (b1 > b0) ok = mbar_wait_bounded((uint64_t *)(smem + L.bars) + warp, 0, p.status);
            ready = true;
        }
        float acc[GV_TOK];
#pragma unroll
        for (int t = 0; t < GV_TOK; ++t) acc[t] = 0.f;
        if (ok) tile_dot_dispatch<QT>(ntp, smem + L.quant, smem + L.scale, act, asum, Kr, nbr, b0, b1, lane, acc);
#pragma unroll
        for (int t = 0; t < GV_TOK; ++t)
            if (t < ntp) red[((size_t)warp * GV_TOK + t) * 32 + lane] = acc[t];
        __syncthreads();
        for (int t = warp; t < nt; t += GV_WARPS) {
            const float s = reduce_warps(red, t, lane);
            const int r = routes[pos0 + tg + t];
            p.partial[(size_t)r * p.H + 32 * g + lane] = p.weights[r] * s;
        }
        __syncthreads();
    }
    // never leave with this warp's copies in flight (a timed-out wait gets a second bounded wait)
    if ((!ready || !ok) && b1 > b0) mbar_wait_bounded((uint64_t *)(smem + L.bars) + warp, 0, p.status);
}

// ------------------------------------------------------------------ P1: permute

// Stable counting sort of the routes r = t*k + j by expert (restricted to a subset),
// plus the ascending list of active experts and their route ranges.
__global__ void __launch_bounds__(256) permute_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                      const int32_t *__restrict__ subset, int n_subset,
                                                      int32_t *__restrict__ ints, int *status) {
    __shared__ int cnt[MOE_MAX_E], off[MOE_MAX_E + 1], run[MOE_MAX_E];
    __shared__ unsigned char insub[MOE_MAX_E];
    __shared__ int chunk_e[256];
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
    if (tid == 0) {
        int s = 0, na = 0;
        int *active = ints + ws_active_off();
        int *aoff = ints + ws_aoff_off(E);
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
    }
    __syncthreads();
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

template <typename Kern>
int launch_unit_kernel(Kern kern, int grid, size_t smem, const FfnParams &p, cudaStream_t s) {
    if (grid <= 0) return MOE_OK;
    MOE_TRY_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    kern<<<grid, GV_THREADS, smem, s>>>(p);
    MOE_TRY_CUDA(cudaGetLastError());
    return MOE_OK;
}

}  // namespace

int moe_gateup_ksplit(int qtype, int H) {
    const int nb = H / 32;
    int ks = 1;
    while (moe_quant_bytes(qtype, 32, H / ks) > GV_UNIT_QUANT && nb % (2 * ks) == 0) ks *= 2;
    return ks;
}

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

    FfnParams p;
    p.x = x;
    p.T = T; p.H = H; p.F = F; p.k = k; p.E = E;
    p.KS = moe_gateup_ksplit(qtype, H);
    p.RT = T * k;
    p.ids = ids;
    p.weights = weights;
    p.ws_ints = (const int32_t *)((char *)workspace + W.ints_off);
    p.gu = (float *)((char *)workspace + W.gu_off);
    p.slot_table = d_slot_table;
    p.n_slots = n_slots;
    p.pool = (const uint8_t *)pool;
    p.slot_bytes = slot_bytes;
    p.partial = partial;
    p.status = moe_status_word_device_ptr();
    p.ntok = pow2_tokens(T < GV_TOK ? T : GV_TOK);
    p.fill_src = (const unsigned long long *)d_fill_src;

    const int n_act_max = expert_subset ? n_subset : (T * k < E ? T * k : E);
    const int nb1 = (H / 32) / p.KS;
    const size_t smem1 = unit_smem(qtype, nb1, p.ntok).total;
    const size_t smem2 = unit_smem(qtype, F / 32, p.ntok).total;
    if (smem1 > 220 * 1024 || smem2 > 220 * 1024) return MOE_ERR_UNSUPPORTED;

    if (timing && timing->permute0) MOE_TRY_CUDA(cudaEventRecord(timing->permute0, s));
    permute_kernel<<<1, 256, 0, s>>>(ids, T * k, E, expert_subset, n_subset,
                                     (int32_t *)((char *)workspace + W.ints_off), p.status);
    MOE_TRY_CUDA(cudaGetLastError());
    if (timing && timing->permute1) MOE_TRY_CUDA(cudaEventRecord(timing->permute1, s));
    if (timing && timing->gateup0) MOE_TRY_CUDA(cudaEventRecord(timing->gateup0, s));
    const int grid1 = n_act_max * 2 * (F / 32) * p.KS;
    int rc;
    if (qtype == MOE_Q8_0)
        rc = xtype == MOE_F32 ? launch_unit_kernel(gateup_kernel<MOE_Q8_0, MOE_F32>, grid1, smem1, p, s)
                              : launch_unit_kernel(gateup_kernel<MOE_Q8_0, MOE_BF16>, grid1, smem1, p, s);
    else
        rc = xtype == MOE_F32 ? launch_unit_kernel(gateup_kernel<MOE_Q4_SM, MOE_F32>, grid1, smem1, p, s)
                              : launch_unit_kernel(gateup_kernel<MOE_Q4_SM, MOE_BF16>, grid1, smem1, p, s);
    if (rc != MOE_OK) return rc;
    if (timing && timing->gateup1) MOE_TRY_CUDA(cudaEventRecord(timing->gateup1, s));
    if (timing && timing->down0) MOE_TRY_CUDA(cudaEventRecord(timing->down0, s));
    const int grid2 = n_act_max * (H / 32);
    rc = qtype == MOE_Q8_0 ? launch_unit_kernel(down_kernel<MOE_Q8_0>, grid2, smem2, p, s)
                           : launch_unit_kernel(down_kernel<MOE_Q4_SM>, grid2, smem2, p, s);
    if (rc != MOE_OK) return rc;
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
