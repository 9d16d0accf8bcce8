// Router GEMV + top-k + softmax over the selected experts (R1).
//
// Gating as on page 1 ("llama.cpp MoE 模型卸载", section 3.1): logits = x.W_r + b,
// then the k largest, then a softmax — here taken over the k selected logits, which
// equals a full softmax renormalised over the selected experts; equal logits are
// ordered by ascending expert id.  Page 1 also batches the gating of several tokens
// into one matrix product (section 5.2); one launch here handles every token.
//
// GB300 mapping: a cluster of MOE_ROUTER_CLUSTER CTAs per group of up to 32 tokens.
// CTA r of the cluster owns rows [r*H/C, (r+1)*H/C) of W_r [H][E]: one bulk copy
// (TMA engine) brings that contiguous slice into shared memory, the CTA computes
// partial logits for its rows, and cluster rank 0 sums the C partials over
// distributed shared memory in rank order, adds the bias and selects the top-k
// with one warp per token.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "moe_ptx.cuh"

#define MOE_ROUTER_CLUSTER 8
#define MOE_ROUTER_TOKENS 32   // tokens per cluster
#define MOE_ROUTER_CHUNK 8     // tokens accumulated at once in registers
#define MOE_ROUTER_THREADS 256

namespace {

struct RouterSmem {
    // offsets (bytes) into dynamic shared memory
    size_t w, x, red, part, bar, total;
};

__host__ __device__ inline RouterSmem router_smem_layout(int H, int E) {
    RouterSmem L;
    const int HS = H / MOE_ROUTER_CLUSTER;
    const int NP = (E + 1) / 2;
    const int HSUB = MOE_ROUTER_THREADS / NP;
    size_t off = 0;
    L.w = off;     off += ((size_t)HS * E * 2 + 15) / 16 * 16 + 16;   // + pad for the odd-E pair
    L.x = off;     off += (size_t)MOE_ROUTER_TOKENS * HS * 4;
    L.red = off;   off += (size_t)HSUB * MOE_ROUTER_CHUNK * NP * 2 * 4;
    L.part = off;  off += (size_t)MOE_ROUTER_TOKENS * E * 4;
    L.bar = off;   off += 16;
    L.total = off;
    return L;
}

template <int XT>
__device__ __forceinline__ float load_x(const void *x, size_t i) {
    if (XT == MOE_BF16) return __bfloat162float(((const __nv_bfloat16 *)x)[i]);
    return ((const float *)x)[i];
}

// (v, id) ordering of the selection: larger logit first, then lower id.
__device__ __forceinline__ bool better(float v1, int i1, float v2, int i2) {
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Top-k of one token's logits held by a warp (lane l holds experts l, l+32, ...; -inf
// beyond E), larger first and ties to the lower id, then the softmax over the k selected;
// lanes 0..k-1 write ids/weights of row `row`.
__device__ __forceinline__ void select_topk_softmax(const float (&v)[MOE_MAX_E / 32], int E, int k, int lane,
                                                    size_t row, int32_t *__restrict__ ids,
                                                    float *__restrict__ weights, float min_w) {
    constexpr int NPL = MOE_MAX_E / 32;
    unsigned taken = 0;
    float sel_v[MOE_MAX_K];
    int sel_i[MOE_MAX_K];
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !(taken >> i & 1u) && better(v[i], e, bv, bi)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        sel_v[j] = bv;
        sel_i[j] = bi;
    }
    float denom = 0.f;
    for (int j = 0; j < k; ++j) denom += expf(sel_v[j] - sel_v[0]);
    if (lane < k) {
        float myv = sel_v[0];
        int myi = sel_i[0];
        for (int j = 1; j < k; ++j)
            if (j == lane) {
                myv = sel_v[j];
                myi = sel_i[j];
            }
        // a route whose weight is below the load threshold is dropped: id -1, weight 0
        const float w = expf(myv - sel_v[0]) / denom;
        const bool drop = w < min_w;
        ids[row * k + lane] = drop ? -1 : myi;
        weights[row * k + lane] = drop ? 0.f : w;
    }
}

template <int XT>
__global__ void __launch_bounds__(MOE_ROUTER_THREADS)
router_topk_kernel(const void *__restrict__ x, int T, int H, const uint16_t *__restrict__ w_router,
                   const float *__restrict__ bias, int E, int k, int32_t *__restrict__ ids,
                   float *__restrict__ weights, float *__restrict__ logits_out, int use_bulk,
                   int *status, float min_w) {
    extern __shared__ __align__(128) unsigned char smem[];
    const RouterSmem L = router_smem_layout(H, E);
    const uint16_t *w_s = (const uint16_t *)(smem + L.w);
    float *x_s = (float *)(smem + L.x);
    float *red = (float *)(smem + L.red);
    float *part = (float *)(smem + L.part);
    uint64_t *bar = (uint64_t *)(smem + L.bar);

    const int rank = (int)cluster_ctarank();
    const int HS = H / MOE_ROUTER_CLUSTER;
    const int h0 = rank * HS;
    const int t0 = blockIdx.y * MOE_ROUTER_TOKENS;
    const int TT = min(MOE_ROUTER_TOKENS, T - t0);
    const int tid = threadIdx.x;
    const size_t wbytes = (size_t)HS * E * 2;

    // ---- W_r slice -> shared memory (bulk copy when aligned, else plain loads)
    bool w_ok = true;
    if (use_bulk) {
        if (tid == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(bar, (uint32_t)wbytes);
            bulk_g2s((void *)w_s, w_router + (size_t)h0 * E, (uint32_t)wbytes, bar);
        }
    } else {
        for (size_t i = tid; i < (size_t)HS * E; i += MOE_ROUTER_THREADS)
            ((uint16_t *)w_s)[i] = w_router[(size_t)h0 * E + i];
    }
    if (tid == 0) ((uint16_t *)w_s)[(size_t)HS * E] = 0;  // pad read by the odd-E pair
    __shared__ float bias_s[MOE_MAX_E];
    if (rank == 0)
        for (int e = tid; e < E; e += MOE_ROUTER_THREADS) bias_s[e] = bias ? bias[e] : 0.f;
    pdl_wait();  // x comes from the previous kernel (the weights and the bias do not)
    pdl_trigger();
    // ---- x slice of this cluster's tokens
    for (int i = tid; i < TT * HS; i += MOE_ROUTER_THREADS) {
        const int t = i / HS, h = i % HS;
        x_s[i] = load_x<XT>(x, (size_t)(t0 + t) * H + h0 + h);
    }
    __syncthreads();
    if (use_bulk) w_ok = mbar_wait_bounded(bar, 0, status);

    const int NP = (E + 1) / 2;
    const int HSUB = MOE_ROUTER_THREADS / NP;
    const int pair = tid % NP, hsub = tid / NP;
    const bool active = hsub < HSUB;

    for (int c0 = 0; c0 < TT; c0 += MOE_ROUTER_CHUNK) {
        float acc0[MOE_ROUTER_CHUNK], acc1[MOE_ROUTER_CHUNK];
#pragma unroll
        for (int t = 0; t < MOE_ROUTER_CHUNK; ++t) acc0[t] = acc1[t] = 0.f;
        const int nt = min(MOE_ROUTER_CHUNK, TT - c0);
        if (active && w_ok) {
            for (int h = hsub; h < HS; h += HSUB) {
                // column 2*pair+1 == E (odd E) reads the next row or the pad; it is never stored
                const float w0 = __half2float(__ushort_as_half(w_s[(size_t)h * E + 2 * pair]));
                const float w1 = __half2float(__ushort_as_half(w_s[(size_t)h * E + 2 * pair + 1]));
#pragma unroll
                for (int t = 0; t < MOE_ROUTER_CHUNK; ++t) {
                    if (t < nt) {
                        const float xv = x_s[(c0 + t) * HS + h];
                        acc0[t] = fmaf(xv, w0, acc0[t]);
                        acc1[t] = fmaf(xv, w1, acc1[t]);
                    }
                }
            }
        }
        if (active) {
#pragma unroll
            for (int t = 0; t < MOE_ROUTER_CHUNK; ++t) {
                red[((size_t)hsub * MOE_ROUTER_CHUNK + t) * NP * 2 + 2 * pair] = acc0[t];
                red[((size_t)hsub * MOE_ROUTER_CHUNK + t) * NP * 2 + 2 * pair + 1] = acc1[t];
            }
        }
        __syncthreads();
        for (int i = tid; i < nt * E; i += MOE_ROUTER_THREADS) {
            const int t = i / E, e = i % E;
            float s = 0.f;
            for (int hs = 0; hs < HSUB; ++hs) s += red[((size_t)hs * MOE_ROUTER_CHUNK + t) * NP * 2 + e];
            part[(size_t)(c0 + t) * E + e] = s;
        }
        __syncthreads();
    }

    cluster_sync_all();  // every CTA's partial logits are complete and visible

    if (rank == 0) {
        const int warp = tid / 32, lane = tid % 32;
        constexpr int NPL = MOE_MAX_E / 32;
        for (int t = warp; t < TT; t += MOE_ROUTER_THREADS / 32) {
            float v[NPL];
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const int e = lane + 32 * i;
                v[i] = -INFINITY;
                if (e < E) {
                    float s = 0.f;
                    for (int r = 0; r < MOE_ROUTER_CLUSTER; ++r)
                        s += ld_cluster_f32(cluster_map(&part[(size_t)t * E + e], r));
                    if (bias) s += bias_s[e];
                    if (logits_out) logits_out[(size_t)(t0 + t) * E + e] = s;
                    v[i] = (s != s) ? -INFINITY : s;  // NaN never wins
                }
            }
            select_topk_softmax(v, E, k, lane, (size_t)(t0 + t), ids, weights, min_w);
        }
    }
    cluster_sync_all();  // rank 0 has finished reading the other CTAs' shared memory
}

// ------------------------------------------------------------------ many tokens (prefill)
//
// Above the decode batch limit the router is a small fp32 GEMM [T x H] . [H x E]: a cluster
// of up to 8 CTAs owns 32 tokens and every expert, each CTA walking its share of H in
// chunks of 32 rows, double-buffered in shared memory (x duplicated into (v, v) pairs, W_r
// converted to fp32).  Thread (ty, tx) keeps 4 tokens x EPT experts in registers and
// accumulates expert pairs with packed fp32x2 FMAs, in ascending h per logit within each
// chunk; chunk sums are added in order, the CTAs' partial logits are summed in rank order
// over distributed shared memory, and each rank runs the warp selection of the cluster
// kernel for its share of the tokens.

#define RT_TT 32
#define RT_KC 32
#define RT_XS (RT_TT + 2)  // float2 row stride of the x chunk (16-byte aligned, fewer conflicts)

__host__ __device__ inline size_t router_tiled_smem(int EP) {
    const size_t xs = 2 * (size_t)RT_KC * RT_XS * 8;
    const size_t ws = 2 * (size_t)RT_KC * EP * 4;
    const size_t lg = (size_t)RT_TT * EP * 4;
    return xs + (ws > lg ? ws : lg);
}

template <int XT, int EPT>
__global__ void __launch_bounds__(MOE_ROUTER_THREADS)
router_tiled_kernel(const void *__restrict__ x, int T, int H, const uint16_t *__restrict__ w_router,
                    const float *__restrict__ bias, int E, int k, int32_t *__restrict__ ids,
                    float *__restrict__ weights, float *__restrict__ logits_out, float min_w) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int EP = 32 * EPT;
    float2 *xs = (float2 *)smem;                                       // [2][KC][RT_XS]
    float *ws = (float *)(smem + 2 * (size_t)RT_KC * RT_XS * 8);       // [2][KC][EP]
    float *lg = ws;                                                    // [TT][EP] after the loop
    const int tid = threadIdx.x, tx = tid % 32, ty = tid / 32;
    // a cluster of C CTAs shares a 32-token tile; rank r sums chunks [c_lo, c_hi) of W_r
    const int C = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
    const int t0 = (blockIdx.x / C) * RT_TT;
    const int NC = H / RT_KC;
    const int c_lo = rank * NC / C, c_hi = (rank + 1) * NC / C;
    const int wn = RT_KC * E;                   // halfs per W_r chunk (contiguous rows)
    const int wv = wn / 8;                      // 16-byte vectors per chunk

    // columns E..EP-1 stay zero in both buffers
    for (int i = tid; i < 2 * RT_KC * EP; i += MOE_ROUTER_THREADS)
        if (i % EP >= E) ws[i] = 0.f;

    constexpr int WPT = (RT_KC * EP / 8 + MOE_ROUTER_THREADS - 1) / MOE_ROUTER_THREADS;
    float4 xr;                                  // this thread's x piece of a chunk
    uint4 wr[WPT];                              // this thread's W_r vectors of a chunk
    const int xt = tid / 8, xc = (tid % 8) * 4;  // token and first column of the x piece

    auto load = [&](int c) {
        const int h0 = c * RT_KC;
        xr = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t0 + xt < T) {
            const size_t off = (size_t)(t0 + xt) * H + h0 + xc;
            if (XT == MOE_BF16) {
                const uint2 b = *(const uint2 *)((const __nv_bfloat16 *)x + off);
                const float2 lo = __bfloat1622float2(*(const __nv_bfloat162 *)&b.x);
                const float2 hi = __bfloat1622float2(*(const __nv_bfloat162 *)&b.y);
                xr = make_float4(lo.x, lo.y, hi.x, hi.y);
            } else {
                xr = *(const float4 *)((const float *)x + off);
            }
        }
        // rows h0.. of W_r are 32*E contiguous halfs, a multiple of 8 starting 64*E*c bytes in
        const uint4 *src = (const uint4 *)(w_router + (size_t)h0 * E);
#pragma unroll
        for (int q = 0; q < WPT; ++q) {
            const int v = tid + q * MOE_ROUTER_THREADS;
            if (v < wv) wr[q] = src[v];
        }
    };
    auto store = [&](int buf) {
        float2 *xb = xs + (size_t)buf * RT_KC * RT_XS;
        xb[(xc + 0) * RT_XS + xt] = make_float2(xr.x, xr.x);
        xb[(xc + 1) * RT_XS + xt] = make_float2(xr.y, xr.y);
        xb[(xc + 2) * RT_XS + xt] = make_float2(xr.z, xr.z);
        xb[(xc + 3) * RT_XS + xt] = make_float2(xr.w, xr.w);
        float *wb = ws + (size_t)buf * RT_KC * EP;
#pragma unroll
        for (int q = 0; q < WPT; ++q) {
            const int v = tid + q * MOE_ROUTER_THREADS;
            if (v < wv) {
                const uint16_t *h = (const uint16_t *)&wr[q];
                int row = (8 * v) / E, e = (8 * v) % E;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    wb[row * EP + e] = __half2float(__ushort_as_half(h[j]));
                    if (++e == E) {
                        e = 0;
                        ++row;
                    }
                }
            }
        }
    };

    unsigned long long acc[4][EPT / 2];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int p = 0; p < EPT / 2; ++p) acc[t][p] = 0ull;

    if (c_lo < c_hi) load(c_lo);
    __syncthreads();  // zero fill of the padding columns before the first store
    if (c_lo < c_hi) store(c_lo & 1);
    __syncthreads();
    for (int c = c_lo; c < c_hi; ++c) {
        if (c + 1 < c_hi) load(c + 1);
        // each chunk's 32 products are summed on their own, then added to the total (keeps
        // the rounding error of a 2048-term logit near 1e-6)
        unsigned long long part[4][EPT / 2];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int p = 0; p < EPT / 2; ++p) part[t][p] = 0ull;
        const float2 *xb = xs + (size_t)(c & 1) * RT_KC * RT_XS;
        const float *wb = ws + (size_t)(c & 1) * RT_KC * EP;
#pragma unroll 4
        for (int kk = 0; kk < RT_KC; ++kk) {
            const float4 xa = *(const float4 *)&xb[kk * RT_XS + 4 * ty];      // (x0,x0,x1,x1)
            const float4 xc4 = *(const float4 *)&xb[kk * RT_XS + 4 * ty + 2]; // (x2,x2,x3,x3)
            const unsigned long long xd[4] = {f2_pack(xa.x, xa.y), f2_pack(xa.z, xa.w), f2_pack(xc4.x, xc4.y),
                                              f2_pack(xc4.z, xc4.w)};
#pragma unroll
            for (int q = 0; q < EPT / 4; ++q) {
                const float4 w4 = *(const float4 *)&wb[kk * EP + 128 * q + 4 * tx];
                const unsigned long long w01 = f2_pack(w4.x, w4.y), w23 = f2_pack(w4.z, w4.w);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    part[t][2 * q] = f2_fma(w01, xd[t], part[t][2 * q]);
                    part[t][2 * q + 1] = f2_fma(w23, xd[t], part[t][2 * q + 1]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int p = 0; p < EPT / 2; ++p) acc[t][p] = f2_add(acc[t][p], part[t][p]);
        if (c + 1 < c_hi) store((c + 1) & 1);
        __syncthreads();
    }
    // this rank's partial logits -> shared memory (the W_r buffers are free after the last barrier)
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
        for (int q = 0; q < EPT / 4; ++q)
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                float a, b;
                f2_unpack(acc[t][2 * q + p], a, b);
                const int e = 128 * q + 4 * tx + 2 * p;
                lg[(size_t)(4 * ty + t) * EP + e] = a;
                lg[(size_t)(4 * ty + t) * EP + e + 1] = b;
            }
    cluster_sync_all();  // every rank's partial logits are complete and visible
    // rank r selects tokens r, r + C, ...: the partials summed in rank order, then the bias
    const int warp = ty, lane = tx;
    for (int t = rank + C * warp; t < RT_TT && t0 + t < T; t += C * (MOE_ROUTER_THREADS / 32)) {
        float v[MOE_MAX_E / 32];
#pragma unroll
        for (int i = 0; i < MOE_MAX_E / 32; ++i) {
            const int e = lane + 32 * i;
            v[i] = -INFINITY;
            if (e < E) {
                float s = 0.f;
                for (int r = 0; r < C; ++r) s += ld_cluster_f32(cluster_map(&lg[(size_t)t * EP + e], r));
                if (bias) s += bias[e];
                if (logits_out) logits_out[(size_t)(t0 + t) * E + e] = s;
                v[i] = (s != s) ? -INFINITY : s;  // NaN never wins
            }
        }
        select_topk_softmax(v, E, k, lane, (size_t)(t0 + t), ids, weights, min_w);
    }
    cluster_sync_all();  // the other ranks have finished reading this CTA's shared memory
}

}  // namespace

namespace {

// ------------------------------------------------------------------ bf16 prefill on tensor cores
//
// With bf16 activations (the prefill path) the product runs on the tensor cores: bf16 values
// in the normal fp16 range are exact in fp16 (8 significant bits of 11), W_r is fp16, so every
// product of an m16n8k16 MMA (fp16 operands, fp32 accumulation) is exact and only the sums
// round.  A cluster of C CTAs owns 32 tokens and every expert (E a multiple of 32, at most
// 128), each CTA a share of H (C is chosen so that the grid covers the SMs twice); in a CTA
// warp w takes tokens 16 (w % 2).. and experts E/4 (w / 2)..; H is walked in chunks of 64
// rows, x (converted to fp16) and W_r double-buffered in shared memory, operand fragments
// loaded with ldmatrix.  Each chunk's products are summed on their own (four K = 16 MMAs)
// and then added to the total, as in the fp32 kernel; the CTAs' partial logits are summed in
// rank order over distributed shared memory, and each rank adds the bias and runs the warp
// selection for its share of the tokens.

#define RM_TT 32
#define RM_KC 64
#define RM_XS (RM_KC + 8)  // fp16 row stride of the x chunk (ldmatrix rows on distinct banks)

__host__ __device__ inline size_t router_mma_smem(int E) {
    const size_t xs = 2 * (size_t)RM_TT * RM_XS * 2;
    const size_t ws = 2 * (size_t)RM_KC * (E + 8) * 2;
    const size_t lg = (size_t)RM_TT * (E + 1) * 4;
    return xs + (ws > lg ? ws : lg);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// NTW = n-tiles (8 experts) per warp = E / 32.
template <int NTW>
__global__ void __launch_bounds__(MOE_ROUTER_THREADS)
router_mma_kernel(const __nv_bfloat16 *__restrict__ x, int T, int H, const uint16_t *__restrict__ w_router,
                  const float *__restrict__ bias, int E, int k, int32_t *__restrict__ ids,
                  float *__restrict__ weights, float *__restrict__ logits_out, float min_w) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int WS = E + 8;  // fp16 row stride of the W_r chunk
    __half *xs = (__half *)smem;                                        // [2][RM_TT][RM_XS]
    __half *ws = (__half *)(smem + 2 * (size_t)RM_TT * RM_XS * 2);      // [2][RM_KC][WS]
    float *lg = (float *)ws;                                            // [RM_TT][E + 1] after the loop
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int C = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
    const int t0 = (blockIdx.x / C) * RM_TT;
    const int tg = warp & 1, n_base = (warp >> 1) * (E / 4);
    const int NC = H / RM_KC;
    const int c_lo = rank * NC / C, c_hi = (rank + 1) * NC / C;
    const int wv = RM_KC * E / 8;  // 16-byte vectors of a W_r chunk
    constexpr int WPT = (RM_KC * 128 / 8 + MOE_ROUTER_THREADS - 1) / MOE_ROUTER_THREADS;

    uint4 xr, wr[WPT];
    const int xt = tid / 8, xc = (tid % 8) * 8;  // token and first column of this thread's x piece
    auto load = [&](int c) {
        const int h0 = c * RM_KC;
        xr = make_uint4(0u, 0u, 0u, 0u);
        if (t0 + xt < T) xr = *(const uint4 *)(x + (size_t)(t0 + xt) * H + h0 + xc);
        const uint4 *src = (const uint4 *)(w_router + (size_t)h0 * E);
#pragma unroll
        for (int q = 0; q < WPT; ++q) {
            const int v = tid + q * MOE_ROUTER_THREADS;
            if (v < wv) wr[q] = src[v];
        }
    };
    auto store = [&](int buf) {
        // bf16 -> fp16 (exact in the normal fp16 range)
        const uint32_t in[4] = {xr.x, xr.y, xr.z, xr.w};
        uint32_t outv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(*(const __nv_bfloat162 *)&in[i]);
            const __half2 h = __floats2half2_rn(f.x, f.y);
            outv[i] = *(const uint32_t *)&h;
        }
        *(uint4 *)(xs + ((size_t)buf * RM_TT + xt) * RM_XS + xc) = make_uint4(outv[0], outv[1], outv[2], outv[3]);
        const int vpr = E / 8;  // vectors per W_r row
#pragma unroll
        for (int q = 0; q < WPT; ++q) {
            const int v = tid + q * MOE_ROUTER_THREADS;
            if (v < wv) *(uint4 *)(ws + ((size_t)buf * RM_KC + v / vpr) * WS + (v % vpr) * 8) = wr[q];
        }
    };

    float tot[NTW][4], part[NTW][4];
#pragma unroll
    for (int j = 0; j < NTW; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[j][i] = 0.f;

    // ldmatrix lane addresses: A (x, 16 x 16) as four 8 x 8 matrices rows 0-7 / 8-15 x
    // columns 0-7 / 8-15; B (W_r, 16 x 8 per n-tile) as two transposed 8 x 8 matrices
    const int am = lane >> 3, ar = lane & 7;
    const int a_row = 16 * tg + (am & 1) * 8 + ar, a_col = (am >> 1) * 8;
    const int b_row = ((lane >> 3) & 1) * 8 + ar;
    const uint32_t xs_base = smem_u32(xs), ws_base = smem_u32(ws);

    if (c_lo < c_hi) {
        load(c_lo);
        store(c_lo & 1);
    }
    __syncthreads();
    for (int c = c_lo; c < c_hi; ++c) {
        if (c + 1 < c_hi) load(c + 1);
        const int buf = c & 1;
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) part[j][i] = 0.f;
#pragma unroll
        for (int ks = 0; ks < RM_KC / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(xs_base + (uint32_t)((((size_t)buf * RM_TT + a_row) * RM_XS + 16 * ks + a_col) * 2), a0, a1, a2,
                    a3);
#pragma unroll
            for (int j = 0; j < NTW; ++j) {
                uint32_t b0, b1;
                ldsm_x2_trans(ws_base + (uint32_t)((((size_t)buf * RM_KC + 16 * ks + b_row) * WS + n_base + 8 * j) * 2),
                              b0, b1);
                mma_f16_16816(part[j], a0, a1, a2, a3, b0, b1);
            }
        }
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) tot[j][i] += part[j][i];
        if (c + 1 < c_hi) store((c + 1) & 1);
        __syncthreads();
    }
    // logits -> shared memory (the W_r buffers are free after the last barrier): accumulator
    // element (row g, columns 2t, 2t+1) and (row g + 8, ...) of each n-tile
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int j = 0; j < NTW; ++j) {
        const int e = n_base + 8 * j + 2 * t4;
        const int r = 16 * tg + g;
        lg[(size_t)r * (E + 1) + e] = tot[j][0];
        lg[(size_t)r * (E + 1) + e + 1] = tot[j][1];
        lg[(size_t)(r + 8) * (E + 1) + e] = tot[j][2];
        lg[(size_t)(r + 8) * (E + 1) + e + 1] = tot[j][3];
    }
    cluster_sync_all();  // every rank's partial logits are complete and visible
    for (int t = rank + C * warp; t < RM_TT && t0 + t < T; t += C * (MOE_ROUTER_THREADS / 32)) {
        float v[MOE_MAX_E / 32];
#pragma unroll
        for (int i = 0; i < MOE_MAX_E / 32; ++i) {
            const int e = lane + 32 * i;
            v[i] = -INFINITY;
            if (e < E) {
                float sv = 0.f;
                for (int r = 0; r < C; ++r) sv += ld_cluster_f32(cluster_map(&lg[(size_t)t * (E + 1) + e], r));
                if (bias) sv += bias[e];
                if (logits_out) logits_out[(size_t)(t0 + t) * E + e] = sv;
                v[i] = (sv != sv) ? -INFINITY : sv;  // NaN never wins
            }
        }
        select_topk_softmax(v, E, k, lane, (size_t)(t0 + t), ids, weights, min_w);
    }
    cluster_sync_all();  // the other ranks have finished reading this CTA's shared memory
}

// SMs of the current device (queried at every call: a process may drive several devices).
int router_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
        return 1;
    return n;
}

template <int NTW>
int router_mma_launch_t(const void *x, int T, int H, const uint16_t *w_router, const float *bias, int E, int k,
                        int32_t *ids, float *weights, float *logits, float min_w, cudaStream_t st) {
    const size_t smem = router_mma_smem(E);
    MOE_TRY_CUDA(cudaFuncSetAttribute(router_mma_kernel<NTW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    const int tiles = (T + RM_TT - 1) / RM_TT, NC = H / RM_KC;
    int C = 1;  // CTAs per cluster splitting H: until the grid covers the SMs twice
    while (2 * C <= MOE_ROUTER_CLUSTER && 2 * C <= NC && tiles * C < 2 * router_sm_count()) C *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C * tiles, 1, 1);
    cfg.blockDim = dim3(MOE_ROUTER_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, router_mma_kernel<NTW>, (const __nv_bfloat16 *)x, T, H, w_router, bias, E,
                                    k, ids, weights, logits, min_w));
    return MOE_OK;
}

// The tensor-core router takes bf16 tokens with E a multiple of 32 up to 128 and H a multiple
// of 64 (16-byte aligned rows); anything else keeps the fp32 kernel.
bool router_mma_eligible(int xtype, int H, int E) {
    return xtype == MOE_BF16 && E % 32 == 0 && E <= 128 && H % RM_KC == 0;
}

int router_mma_launch(const void *x, int T, int H, const uint16_t *w_router, const float *bias, int E, int k,
                      int32_t *ids, float *weights, float *logits, float min_w, cudaStream_t st) {
    switch (E / 32) {
        case 1: return router_mma_launch_t<1>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st);
        case 2: return router_mma_launch_t<2>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st);
        case 3: return router_mma_launch_t<3>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st);
        default: return router_mma_launch_t<4>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st);
    }
}

template <int XT, int EPT>
int router_tiled_launch_t(const void *x, int T, int H, const uint16_t *w_router, const float *bias, int E,
                          int k, int32_t *ids, float *weights, float *logits, float min_w, cudaStream_t st) {
    const size_t smem = router_tiled_smem(32 * EPT);
    MOE_TRY_CUDA(cudaFuncSetAttribute(router_tiled_kernel<XT, EPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
    const int NC = H / RT_KC;
    int C = 1;  // CTAs per cluster splitting H (each keeps at least one chunk)
    while (2 * C <= MOE_ROUTER_CLUSTER && 2 * C <= NC) C *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C * ((T + RT_TT - 1) / RT_TT), 1, 1);
    cfg.blockDim = dim3(MOE_ROUTER_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, router_tiled_kernel<XT, EPT>, x, T, H, w_router, bias, E, k, ids, weights,
                                    logits, min_w));
    return MOE_OK;
}

int router_tiled_launch(const void *x, int xtype, int T, int H, const uint16_t *w_router, const float *bias,
                        int E, int k, int32_t *ids, float *weights, float *logits, float min_w, cudaStream_t st) {
    if (E <= 128)
        return xtype == MOE_F32
                   ? router_tiled_launch_t<MOE_F32, 4>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st)
                   : router_tiled_launch_t<MOE_BF16, 4>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st);
    return xtype == MOE_F32
               ? router_tiled_launch_t<MOE_F32, 8>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st)
               : router_tiled_launch_t<MOE_BF16, 8>(x, T, H, w_router, bias, E, k, ids, weights, logits, min_w, st);
}

}  // namespace

extern "C" int moe_router_topk(const void *x, int xtype, int T, int H, const uint16_t *w_router,
                               const float *bias, int E, int k, int32_t *ids, float *weights,
                               float *logits, moe_stream_t s) {
    return moe_router_topk_threshold(x, xtype, T, H, w_router, bias, E, k, 0.0f, ids, weights, logits, s);
}

extern "C" int moe_router_topk_threshold(const void *x, int xtype, int T, int H, const uint16_t *w_router,
                                         const float *bias, int E, int k, float min_weight, int32_t *ids,
                                         float *weights, float *logits, moe_stream_t s) {
    MOE_CHECK(T >= 0);
    MOE_CHECK(min_weight >= 0.0f && min_weight <= 1.0f);
    MOE_CHECK(xtype == MOE_F32 || xtype == MOE_BF16);
    MOE_CHECK(H > 0 && H % 32 == 0);
    MOE_CHECK(E >= 1 && E <= MOE_MAX_E && k >= 1 && k <= MOE_MAX_K && k <= E);
    if (T == 0) return MOE_OK;
    MOE_CHECK(x && w_router && ids && weights);
    if (T > MOE_DECODE_MAX_T && ((uintptr_t)x & 15) == 0 && ((uintptr_t)w_router & 15) == 0) {
        if (router_mma_eligible(xtype, H, E))
            return router_mma_launch(x, T, H, w_router, bias, E, k, ids, weights, logits, min_weight,
                                     moe_cuda_stream(s));
        return router_tiled_launch(x, xtype, T, H, w_router, bias, E, k, ids, weights, logits, min_weight,
                                   moe_cuda_stream(s));
    }
    const RouterSmem L = router_smem_layout(H, E);
    if (L.total > 200 * 1024) return MOE_ERR_UNSUPPORTED;
    const int HS = H / MOE_ROUTER_CLUSTER;
    const size_t wbytes = (size_t)HS * E * 2;
    const int use_bulk = ((uintptr_t)w_router % 16 == 0) && (wbytes % 16 == 0) &&
                         (((size_t)HS * E * 2) % 16 == 0);
    int *status = moe_status_word_device_ptr();

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(MOE_ROUTER_CLUSTER, (T + MOE_ROUTER_TOKENS - 1) / MOE_ROUTER_TOKENS, 1);
    cfg.blockDim = dim3(MOE_ROUTER_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = moe_cuda_stream(s);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = MOE_ROUTER_CLUSTER;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (xtype == MOE_F32) {
        MOE_TRY_CUDA(cudaFuncSetAttribute(router_topk_kernel<MOE_F32>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total));
        MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, router_topk_kernel<MOE_F32>, x, T, H, w_router, bias, E,
                                        k, ids, weights, logits, use_bulk, status, min_weight));
    } else {
        MOE_TRY_CUDA(cudaFuncSetAttribute(router_topk_kernel<MOE_BF16>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total));
        MOE_TRY_CUDA(cudaLaunchKernelEx(&cfg, router_topk_kernel<MOE_BF16>, x, T, H, w_router, bias,
                                        E, k, ids, weights, logits, use_bulk, status, min_weight));
    }
    return MOE_OK;
}
